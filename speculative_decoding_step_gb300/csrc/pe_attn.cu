// Paged GQA attention of the drafter rows over the drafter KV cache.
//
// A row of sequence b at position p attends to the cache positions 0..p of
// its sequence (the prefix plus the rows this round wrote: causal inside the
// draft block).  Keys are stored post-RoPE.  Scale 1/sqrt(head_dim).
//
// bf16: one work item = (sequence b, kv head g, position chunk [c0, c1)).
// The query tile packs every valid row of the sequence times the n_q/n_kv
// query heads of g (<= 128 query vectors), so each KV page is read once per
// (sequence, kv head).  Warps 0 and 6 stream the chunk's K and V pages with
// 3-D TMA loads (one 16-position page per load, 128-byte swizzle, pages past
// the range zero-filled) into two mbarrier rings of 64-position blocks (5
// stages at head_dim 64, 2 at head_dim 128: two CTAs share an SM); a block's
// keys are released when its S product completes, its values after its PV.
// Warp 1 issues the 5th-generation tensor-core MMAs: S = Q K^T (M = 128 query
// vectors, N = 64 positions) into one of three TMEM buffers (two at head_dim
// 128), and O += P V with P read from TMEM and V as an MN-major operand straight
// from the ring; it issues each S as soon as its keys have landed and each PV as
// soon as its P is written, so S runs up to two blocks ahead of the softmax.
// Warps 2..5 own one query vector each (its TMEM lane): mask, exponentiate
// (log2 domain) and write P as bf16 over the first half of S's columns.  A
// row's reference maximum only moves when a block exceeds it by 2^8, and then
// O is rescaled in TMEM, so the common block is one read of S and one write
// of P per row.  A range in one chunk is written directly; otherwise every
// chunk leaves (reference max, sum, unnormalised output) partials that a
// second, GPU-wide kernel merges in chunk order (deterministic).
//
// fp32: one warp per (row, query head); lanes stride over positions with an
// online softmax each, then merge.
#include <algorithm>
#include <cfloat>
#include <climits>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

namespace {

PE_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x by the hardware approximation (MUFU; subnormal results flush to zero).
PE_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A wait's outcome, made the same for the whole warp (warp-collective
// instructions follow it).
PE_DEV bool warp_ok(bool ok) { return __all_sync(0xFFFFFFFFu, ok); }

}  // namespace

constexpr int kAttnBlk = 64;          // kv positions per pipeline stage (4 pages) = MMA N of S
// key and value stages in flight: 5 + 5 x 8 KB (head_dim 64) or 2 + 2 x 16 KB (head_dim 128), so
// two CTAs fit per SM
// (a deeper value ring and a shallower key ring, 6 + 4 or 7 + 3, measured no faster)
template <int HD>
__host__ __device__ constexpr int attn_kstages() { return HD == 64 ? 5 : 2; }
template <int HD>
__host__ __device__ constexpr int attn_vstages() { return HD == 64 ? 5 : 2; }
constexpr int kAttnMaxStages = 5;
constexpr int kAttnThreads = 224;     // warp 0: K loads, warp 1: MMA, warps 2..5: softmax (thread = query row), warp 6: V loads
constexpr int kAttnSoftmax = 128;     // softmax threads
constexpr uint32_t kAttnTmemCols = 256;  // S buffers (64 columns each) + O (head_dim columns)
// S/P buffers in TMEM: three at head_dim 64 (S runs up to two blocks ahead of the softmax),
// two at head_dim 128 (O takes 128 of the 256 columns)
template <int HD>
__host__ __device__ constexpr int attn_sbufs() { return HD == 64 ? 3 : 2; }
constexpr int kAttnMaxSbufs = 3;
template <int HD>
__host__ __device__ constexpr uint32_t attn_tmem_o() { return (uint32_t)(attn_sbufs<HD>() * kAttnBlk); }
constexpr int kAttnItemRing = 4;      // item indices the producer may publish ahead
// Lazy rescaling: a row keeps its reference maximum until a block's maximum
// exceeds it by more than this (log2 units), so P <= 2^8 and O is rescaled rarely.
constexpr float kAttnRescaleLog2 = 8.f;
// Longest sleep of the MMA warp on one input while another may arrive first (ns).
constexpr uint32_t kAttnPollNs = 100;

// Shared-memory tile [HD/64 halves][ROWS][64 bf16]: 128-byte rows with the
// 128-byte swizzle that TMA applies (16-byte unit c of row r sits at c ^ (r % 8)).
template <int ROWS>
PE_DEV uint32_t tile_addr(uint32_t base, int row, int chunk) {
  return base + (uint32_t)((chunk >> 3) * ROWS * 128 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int HD>
struct AttnLayout {
  static constexpr uint32_t Q = kAttnRows * HD * 2;      // query tile
  static constexpr uint32_t KV = kAttnBlk * HD * 2;      // K (or V) of one stage
  static constexpr uint32_t VRING = Q + attn_kstages<HD>() * KV;  // the value ring follows the key ring
  static constexpr uint32_t BARS = VRING + attn_vstages<HD>() * KV;
  static constexpr uint32_t TOTAL = 1024 + BARS + 512;   // + alignment slack
};

// Barriers and flags after the tiles.
// K and V of a stage are separate rings: a stage's keys are released once its S product
// has completed, its values once its PV product has.
struct AttnCtrl {
  uint64_t kfull[kAttnMaxStages], kempty[kAttnMaxStages];
  uint64_t vfull[kAttnMaxStages], vempty[kAttnMaxStages];
  uint64_t q_full;      // softmax threads staged the item's query tile
  uint64_t s_full[kAttnMaxSbufs];  // S of a block is in its TMEM buffer (block % sbufs)
  uint64_t p_full[kAttnMaxSbufs];  // P of a block is in TMEM (over its S), O rescaled where needed
  uint64_t pv_item;     // one phase per item: its last PV product has completed
  uint64_t o_free;      // softmax threads read O of the item
  uint64_t drain;       // every MMA issued has completed
  uint64_t item_full[kAttnItemRing];   // the producer published the next item index
  uint64_t item_empty[kAttnItemRing];  // the V loader, the MMA thread and every softmax thread read it
  int item[kAttnItemRing];  // item index, -1: no more work
  uint32_t tmem;
  int abort;
};

static_assert(sizeof(AttnCtrl) <= 512, "attention control block");

// Consumer side of the item ring: the index of this CTA's ii-th item (-1: done),
// or -2 when the wait gave up (the kernel is unwinding).
PE_DEV int attn_next_item(AttnCtrl* ctl, int ii, int32_t* err, volatile int* abort_flag, uint64_t wait_ns) {
  const int k = ii % kAttnItemRing;
  if (!mbar_wait(smem_u32(&ctl->item_full[k]), (uint32_t)(ii / kAttnItemRing) & 1u, err, abort_flag, wait_ns)) return -2;
  const int it = *reinterpret_cast<volatile int*>(&ctl->item[k]);
  mbar_arrive(smem_u32(&ctl->item_empty[k]));
  return it;
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const AttnArgs a) {
  using Lay = AttnLayout<HD>;
  constexpr int CH = HD / 8;  // 16-byte units per row
  constexpr int SK = attn_kstages<HD>(), SV = attn_vstages<HD>();
  constexpr int NB = attn_sbufs<HD>();
  constexpr uint32_t TO = attn_tmem_o<HD>();  // first TMEM column of O
  static_assert(TO + HD <= kAttnTmemCols, "S buffers and O fit the allocation");
  static_assert(SV >= NB - 1, "a value stage's release orders the PV product a rescale waits for");
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(sm);
  AttnCtrl* ctl = reinterpret_cast<AttnCtrl*>(sm + Lay::BARS);
  volatile int* abort_flag = &ctl->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv;

  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int s = 0; s < SK; ++s) {
      mbar_init(smem_u32(&ctl->kfull[s]), 1);
      mbar_init(smem_u32(&ctl->kempty[s]), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(smem_u32(&ctl->vfull[s]), 1);
      mbar_init(smem_u32(&ctl->vempty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->q_full), kAttnSoftmax);
    for (int b = 0; b < NB; ++b) {
      mbar_init(smem_u32(&ctl->s_full[b]), 1);
      mbar_init(smem_u32(&ctl->p_full[b]), kAttnSoftmax);
    }
    mbar_init(smem_u32(&ctl->pv_item), 1);
    mbar_init(smem_u32(&ctl->o_free), kAttnSoftmax);
    mbar_init(smem_u32(&ctl->drain), 1);
    for (int k = 0; k < kAttnItemRing; ++k) {
      mbar_init(smem_u32(&ctl->item_full[k]), 1);
      mbar_init(smem_u32(&ctl->item_empty[k]), 2 + kAttnSoftmax);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem), kAttnTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  // Until a role's dependency wait (pdl_wait) it reads only what kernels before the previous
  // one wrote, all complete once this kernel has started: the work list, the sequences'
  // metadata, and cache pages wholly below the sequence's smallest position of this round.
  // The queries, the new rows' k / v and the outputs come after the wait (L2 loads before it).
  pdl_trigger();
  const int n_items = __ldcg(a.n_items);

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------------ TMA loaders (whole warps)
    // Warp 0 streams the keys and warp 6 the values of the same blocks, each into its own
    // ring: a key stage is reused as soon as its S product has completed, without waiting
    // for the block's PV product.  Warp 0 also takes the items (dynamic: long and short
    // ranges even out across SMs) and publishes them through the item ring; warp 6 reads
    // them from it like the other roles.  A warp reads the page ids of 8 blocks (32 pages)
    // at once, one per lane; lane 0 then issues the TMA loads.
    const bool is_v = warp == 6;
    const CUtensorMap* tm = is_v ? &tmV : &tmK;
    uint64_t* fullb = is_v ? ctl->vfull : ctl->kfull;
    uint64_t* emptyb = is_v ? ctl->vempty : ctl->kempty;
    const uint32_t ring = sQ + (is_v ? Lay::VRING : Lay::Q);
    const int S = is_v ? SV : SK;
    const uint64_t pol = l2_policy_evict_first();  // the prefix is read once per round
    const int oob = a.num_pages * a.page_size;     // a row past the pool: TMA fills zeros
    constexpr int kPagesPerBlk = kAttnBlk / 16;
    constexpr int kBlkPerBatch = 32 / kPagesPerBlk;
    int gi = 0;
    bool stop = false, waited = false;
    for (int ii = 0; !stop; ++ii) {
      int it = 0;
      if (lane == 0) {
        if (is_v) {
          it = attn_next_item(ctl, ii, a.err, abort_flag, a.wait_ns);
        } else {
          // CTA x's first item is item x (no round trip before the first loads); the
          // counter hands out the rest
          it = ii == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(a.work_counter, 1);
          if (it >= n_items) it = -1;
          const int k = ii % kAttnItemRing;
          bool ok = true;
          if (ii >= kAttnItemRing)
            ok = mbar_wait(smem_u32(&ctl->item_empty[k]), ((uint32_t)(ii / kAttnItemRing) & 1u) ^ 1u, a.err,
                           abort_flag, a.wait_ns);
          if (!ok) it = -2;
          else {
            ctl->item[k] = it;
            mbar_arrive(smem_u32(&ctl->item_full[k]));  // release: the index is visible to the waiters
          }
        }
      }
      it = __shfl_sync(0xFFFFFFFFu, it, 0);
      if (it < 0) {
        stop = it == -2;
        break;
      }
      const int4 item = __ldcg(a.items + it);
      const int b = item.x, g = item.y, c0 = item.z, c1 = item.w;
      const int nblk = (c1 - c0 + kAttnBlk - 1) / kAttnBlk;
      const int first_new = __ldcg(a.seq_minpos + b);  // no k / v of this round lies below it
      for (int blk0 = 0; blk0 < nblk && !stop; blk0 += kBlkPerBatch) {
        const int pos0 = c0 + (blk0 * kPagesPerBlk + lane) * 16;
        int y = oob;
        if (pos0 < c1) {
          const int pi = pos0 / a.page_size;
          if (pi >= a.max_pages) {
            set_err(a.err, PE_DEV_BAD_POSITION);
          } else {
            const int page = __ldg(a.block_table + (size_t)b * a.max_pages + pi);
            if (page < 0 || page >= a.num_pages) set_err(a.err, PE_DEV_BAD_PAGE);
            else y = page * a.page_size;
          }
        }
        const int nb = min(kBlkPerBatch, nblk - blk0);
        for (int bb = 0; bb < nb; ++bb, ++gi) {
          if (!waited && c0 + (blk0 + bb + 1) * kAttnBlk > first_new) {  // the block's pages may hold new rows
            pdl_wait();
            waited = true;
          }
          const int s = gi % S;
          bool ok = true;
          if (lane == 0 && gi >= S)
            ok = mbar_wait(smem_u32(&emptyb[s]), ((uint32_t)(gi / S) & 1u) ^ 1u, a.err, abort_flag, a.wait_ns);
          if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
            stop = true;
            break;
          }
          const uint32_t fb = smem_u32(&fullb[s]);
          const uint32_t dst = ring + (uint32_t)s * Lay::KV;
          if (lane == 0) mbar_expect_tx(fb, Lay::KV);
#pragma unroll
          for (int p = 0; p < kPagesPerBlk; ++p) {
            const int yp = __shfl_sync(0xFFFFFFFFu, y, bb * kPagesPerBlk + p);
            if (lane == 0) {
#pragma unroll
              for (int h = 0; h < HD / 64; ++h)
                tma_load_3d(dst + (uint32_t)(h * kAttnBlk * 128 + p * 16 * 128), tm, fb, h * 64, g, yp, pol);
            }
          }
        }
      }
    }
    if (stop && lane == 0) {
      // leave no bulk copy in flight into this CTA's shared memory
      for (int i = (gi > S ? gi - S : 0); i < gi; ++i)
        mbar_wait(smem_u32(&fullb[i % S]), (uint32_t)(i / S) & 1u, a.err, nullptr, a.wait_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Converged warp: every lane waits on the barriers; the elected lane takes the
    // items and issues every MMA and commit (a lone lane looping is far slower).
    const uint32_t id_s = idesc_bf16(kAttnRows, kAttnBlk);                 // S = Q K^T: N = positions
    const uint32_t id_o = idesc_bf16(kAttnRows, HD) | kIdescTransposeB;   // O += P V: V is MN-major
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      const bool ok = mbar_wait(bar, parity, a.err, abort_flag, a.wait_ns);
      return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
    };
    int gi = 0, ii = 0;
    bool stop = false;
    for (;; ++ii) {
      int it = 0;
      if (elect_one()) it = attn_next_item(ctl, ii, a.err, abort_flag, a.wait_ns);
      it = __shfl_sync(0xFFFFFFFFu, it, 0);
      if (it < 0) break;
      const int4 item = __ldcg(a.items + it);
      const int nblk = (item.w - item.z + kAttnBlk - 1) / kAttnBlk;
      if (!wait_all(smem_u32(&ctl->q_full), (uint32_t)ii & 1u)) break;
      tc_fence_after();
      // Two streams, issued as their inputs arrive: S of block ns once its K has landed and
      // its TMEM buffer is free (the PV of block ns - NB is issued: ns <= np + NB - 1), and the PV
      // of block np once its P is written (and, for an item's first PV, which overwrites
      // O, once the softmax threads have read the previous item's O).  Neither waits for
      // the other's input: a PV is never held back by the next block's K still loading.
      int ns = 0, np = 0;
      bool o_ok = ii == 0;
      uint64_t t_idle = 0;
      uint32_t n_idle = 0;
      while (np < nblk) {
        bool prog = false;
        if (ns < nblk && ns <= np + NB - 1) {
          const int x = gi + ns, s = x % SK;
          if (__shfl_sync(0xFFFFFFFFu, mbar_test_wait(smem_u32(&ctl->kfull[s]), (uint32_t)(x / SK) & 1u) ? 1 : 0, 0)) {
            tc_fence_after();
            if (elect_one()) {
              const uint32_t kbase = sQ + Lay::Q + (uint32_t)s * Lay::KV;
              const uint32_t d = tmem + (uint32_t)((x % NB) * kAttnBlk);
#pragma unroll
              for (int kk = 0; kk < HD / 16; ++kk) {
                const uint64_t ad = sdesc_k_sw128(sQ + (uint32_t)((kk >> 2) * kAttnRows * 128)) + 2 * (kk & 3);
                const uint64_t bd = sdesc_k_sw128(kbase + (uint32_t)((kk >> 2) * kAttnBlk * 128)) + 2 * (kk & 3);
                tc_mma_bf16(d, ad, bd, id_s, kk > 0 ? 1u : 0u);
              }
              tc_commit(smem_u32(&ctl->s_full[x % NB]));
              tc_commit(smem_u32(&ctl->kempty[s]));  // the stage's keys are read
            }
            __syncwarp();
            ++ns;
            prog = true;
          }
        }
        if (np < ns) {
          const int x = gi + np, s = x % SV;
          if (!o_ok)
            o_ok = __shfl_sync(0xFFFFFFFFu, mbar_test_wait(smem_u32(&ctl->o_free), (uint32_t)(ii - 1) & 1u) ? 1 : 0, 0);
          if (o_ok &&
              __shfl_sync(0xFFFFFFFFu,
                          (mbar_test_wait(smem_u32(&ctl->p_full[x % NB]), (uint32_t)(x / NB) & 1u) &&
                           mbar_test_wait(smem_u32(&ctl->vfull[s]), (uint32_t)(x / SV) & 1u))
                              ? 1
                              : 0,
                          0)) {
            tc_fence_after();
            if (elect_one()) {
              const uint32_t vbase = sQ + Lay::VRING + (uint32_t)s * Lay::KV;
              const uint32_t pa = tmem + (uint32_t)((x % NB) * kAttnBlk);
#pragma unroll
              for (int kk = 0; kk < kAttnBlk / 16; ++kk)
                tc_mma_bf16_tmem_a(tmem + TO, pa + 8u * kk,
                                   sdesc_mn_sw128(vbase + (uint32_t)kk * 2048u, kAttnBlk * 128), id_o,
                                   (np > 0 || kk > 0) ? 1u : 0u);
              if (np == nblk - 1) tc_commit(smem_u32(&ctl->pv_item));
              tc_commit(smem_u32(&ctl->vempty[s]));
            }
            __syncwarp();
            ++np;
            prog = true;
          }
        }
        if (prog) {
          n_idle = 0;
          continue;
        }
        if ((n_idle++ & 7) == 0) {
          // the same bounded wait as mbar_wait (checked every 8th idle turn): give up when
          // another role did, or after the limit
          if (*abort_flag) {
            stop = true;
            break;
          }
          const uint64_t now = global_timer_ns();
          if (n_idle == 1) {
            t_idle = now;
          } else if (now - t_idle > a.wait_ns) {
            if (elect_one()) {
              set_err(a.err, PE_DEV_TIMEOUT);
              *abort_flag = 1;
            }
            __syncwarp();
            stop = true;
            break;
          }
        }
        // Sleep on the input most likely to come next, for a short while (a hot loop of
        // tests would take issue slots from the softmax warps): a pending P, else the
        // next block's K.
        if (np < ns) {
          const int x = gi + np;
          mbar_try_wait_for(smem_u32(&ctl->p_full[x % NB]), (uint32_t)(x / NB) & 1u, kAttnPollNs);
        } else if (ns < nblk) {
          const int x = gi + ns;
          mbar_try_wait_for(smem_u32(&ctl->kfull[x % SK]), (uint32_t)(x / SK) & 1u, kAttnPollNs);
        }
        __syncwarp();
      }
      if (stop) break;
      gi += nblk;
    }
    // TMEM is freed only after every MMA issued here has completed
    if (elect_one()) tc_commit(smem_u32(&ctl->drain));
    __syncwarp();
    mbar_wait(smem_u32(&ctl->drain), 0, a.err, nullptr, a.wait_ns);
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 2..5)
    const int et = tid - 64;                        // 0..127
    const int r = (warp & 3) * 32 + lane;           // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;
    const __nv_bfloat16* qbuf = static_cast<const __nv_bfloat16*>(a.q);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const int ldq = a.n_q * HD;

    // query tile: row m = (row m / G of the sequence, head g*G + m % G); zeros past the valid rows
    bool waited = false;
    auto stage_q = [&](int it) {
      const int4 item = __ldcg(a.items + it);
      const int b = item.x, g = item.y;
      const int start = __ldcg(a.seq_start + b);
      const int M = min(__ldcg(a.seq_len + b) * G, kAttnRows);
      if (!waited) {  // the queries come from the previous kernel
        pdl_wait();
        waited = true;
      }
      // every load of this thread first (one round trip), then the shared-memory stores
      constexpr int PER = kAttnRows * CH / kAttnSoftmax;
      uint4 val[PER];
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int idx = et + k * kAttnSoftmax;
        const int m = idx / CH, ch = idx - (idx / CH) * CH;
        val[k] = make_uint4(0, 0, 0, 0);
        if (m < M) {
          const int i = m / G, j = m - (m / G) * G;
          val[k] = __ldg(reinterpret_cast<const uint4*>(qbuf + (size_t)(start + i) * ldq + (size_t)(g * G + j) * HD +
                                                        ch * 8));
        }
      }
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int idx = et + k * kAttnSoftmax;
        const int m = idx / CH, ch = idx - (idx / CH) * CH;
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(tile_addr<kAttnRows>(sQ, m, ch)), "r"(val[k].x),
                     "r"(val[k].y), "r"(val[k].z), "r"(val[k].w)
                     : "memory");
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
      mbar_arrive(smem_u32(&ctl->q_full));
    };
    int gi = 0, ii = 0;
    bool stop = false;
    int it = attn_next_item(ctl, 0, a.err, abort_flag, a.wait_ns), it_next = -1;
    if (it >= 0) stage_q(it);
    for (; it >= 0 && !stop; it = it_next, ++ii) {
      it_next = -1;
      const int4 item = a.items[it];
      const int b = item.x, g = item.y, c0 = item.z, c1 = item.w;
      const int start = a.seq_start[b];
      const int M = min(a.seq_len[b] * G, kAttnRows);
      const int nblk = (c1 - c0 + kAttnBlk - 1) / kAttnBlk;
      const int nc = a.n_chunks[b];
      const bool valid = r < M;
      // causal bound: positions <= lim (row's own position, clipped to the chunk)
      const int lim = valid ? min(a.tok_pos[start + r / G], c1 - 1) : -1;
      const bool warp_any = __any_sync(0xFFFFFFFFu, valid);
      int wmin = valid ? lim : INT_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wmin = min(wmin, __shfl_xor_sync(0xFFFFFFFFu, wmin, o));

      float m_ref = -INFINITY, l = 0.f;  // reference maximum (log2 units, scaled) and row sum
      for (int j = 0; j < nblk; ++j) {
        const int x = gi + j;
        if (!warp_ok(mbar_wait(smem_u32(&ctl->s_full[x % NB]), (uint32_t)(x / NB) & 1u, a.err, abort_flag, a.wait_ns))) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t sbuf = tmem + lane_base + (uint32_t)((x % NB) * kAttnBlk);
        if (warp_any) {
          float sc[kAttnBlk];
          tmem_load64(sbuf, sc);
          const int kb0 = c0 + j * kAttnBlk;
          if (kb0 + kAttnBlk - 1 > wmin) {  // some position of the block is masked for some row of the warp
#pragma unroll
            for (int c = 0; c < kAttnBlk; ++c) sc[c] = (kb0 + c <= lim) ? sc[c] : -INFINITY;
          }
          float mx8[8];  // eight independent chains
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = sc[e];
#pragma unroll
          for (int c = 8; c < kAttnBlk; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], sc[c]);
          float bm = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                           fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          bm *= sl2;
          const bool fresh = (m_ref == -INFINITY);
          const bool need = !fresh && bm > m_ref + kAttnRescaleLog2;
          if (__any_sync(0xFFFFFFFFu, need)) {
            // O holds the PV products of blocks before j of this item (j >= 1 since m_ref is finite)
            // (the release of block x-1's values is committed after its PV product; that
            // barrier is at most one phase short of it: S(x) completing implies every PV up
            // to block x-NB has completed, and SV >= NB - 1)
            const int xp = x - 1;
            if (!warp_ok(mbar_wait(smem_u32(&ctl->vempty[xp % SV]), (uint32_t)(xp / SV) & 1u, a.err, abort_flag,
                                   a.wait_ns))) {
              stop = true;
            } else {
              tc_fence_after();
              const float f = need ? ex2_approx(m_ref - bm) : 1.f;
#pragma unroll 1
              for (int c = 0; c < HD; c += 16) {
                float ov[16];
                tmem_load16(tmem + lane_base + TO + (uint32_t)c, ov);
#pragma unroll
                for (int e = 0; e < 16; ++e) ov[e] *= f;
                tmem_store16(tmem + lane_base + TO + (uint32_t)c, ov);
              }
              if (need) {
                l *= f;
                m_ref = bm;
              }
            }
          }
          if (fresh) m_ref = bm;  // first block with an unmasked position (or still -inf)
          // P = 2^(s * scale * log2e - m_ref).  Masked scores are -inf (2^-inf = 0); a row
          // with nothing unmasked yet has m_ref = -inf and takes offset -inf, so P = 0 there too.
          const float nmr = m_ref == -INFINITY ? -INFINITY : -m_ref;
          uint32_t pk[kAttnBlk / 2];
          float rs8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) rs8[e] = 0.f;
#pragma unroll
          for (int c = 0; c < kAttnBlk / 2; ++c) {
            const float p0 = ex2_approx(fmaf(sc[2 * c], sl2, nmr));
            const float p1 = ex2_approx(fmaf(sc[2 * c + 1], sl2, nmr));
            rs8[c & 7] += p0 + p1;
            pk[c] = pack_bf16(p0, p1);
          }
          l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
          tmem_store32(sbuf, pk);  // P over the first half of S's columns
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&ctl->p_full[x % NB]));
        if (stop) break;
      }
      if (stop) break;
      // every S product of this item has completed: the next item's query tile may go in
      it_next = attn_next_item(ctl, ii + 1, a.err, abort_flag, a.wait_ns);
      if (it_next == -2) break;
      if (it_next >= 0) stage_q(it_next);

      gi += nblk;
      // The item's PV products are complete (a barrier of its own, committed after the
      // item's last PV: a parity wait cannot tell a barrier two phases behind from one
      // that is done, so no per-block barrier serves here).
      if (!warp_ok(mbar_wait(smem_u32(&ctl->pv_item), (uint32_t)ii & 1u, a.err, abort_flag, a.wait_ns))) break;
      tc_fence_after();
      if (nc == 1) {
        // the item covers the whole range: normalise and write the output row directly
        if (warp_any) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16* dst = out + (size_t)(start + r / G) * ldq + (size_t)(g * G + r % G) * HD;
#pragma unroll 1
          for (int c = 0; c < HD; c += 16) {
            float ov[16];
            tmem_load16(tmem + lane_base + TO + (uint32_t)c, ov);
            if (valid) {
              uint4 w0, w1;
              w0.x = pack_bf16(ov[0] * inv, ov[1] * inv);   w0.y = pack_bf16(ov[2] * inv, ov[3] * inv);
              w0.z = pack_bf16(ov[4] * inv, ov[5] * inv);   w0.w = pack_bf16(ov[6] * inv, ov[7] * inv);
              w1.x = pack_bf16(ov[8] * inv, ov[9] * inv);   w1.y = pack_bf16(ov[10] * inv, ov[11] * inv);
              w1.z = pack_bf16(ov[12] * inv, ov[13] * inv); w1.w = pack_bf16(ov[14] * inv, ov[15] * inv);
              *reinterpret_cast<uint4*>(dst + c) = w0;
              *reinterpret_cast<uint4*>(dst + c + 8) = w1;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&ctl->o_free));
        continue;
      }
      const size_t ib = (size_t)it * kAttnRows;
      if (warp_any) {
#pragma unroll 1
        for (int c = 0; c < HD; c += 16) {
          float ov[16];
          tmem_load16(tmem + lane_base + TO + (uint32_t)c, ov);
          if (valid) {  // two 32-byte stores (a partial row is 256-byte aligned)
            float* dst = a.part_o + (ib + r) * HD + c;
            st_global_v8(dst, ov);
            st_global_v8(dst + 8, ov + 8);
          }
        }
        if (valid) {
          a.part_m[ib + r] = m_ref;
          a.part_l[ib + r] = l;
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&ctl->o_free));
    }
  }
  pdl_wait();  // no CTA completes before the previous kernel has (later kernels rely on the chain)
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kAttnTmemCols);
  }
}

template <int HD>
static cudaError_t launch_attn_typed(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int grid,
                                     cudaStream_t s) {
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)AttnLayout<HD>::TOTAL);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_pdl(attn_bf16_kernel<HD>, dim3(grid), dim3(kAttnThreads), (size_t)AttnLayout<HD>::TOTAL, s, tk, tv,
                    a);
}

// Merge of the chunks of every (sequence, kv head) whose range took more than
// one chunk: one warp per (sequence, kv head, group of 32 / LPR query vectors),
// LPR lanes per query vector holding 8 of its head_dim values each.
// out = sum_c w_c O_c / sum_c w_c l_c with w_c = 2^(m_c - max_c m_c); every sum
// runs in a fixed order (deterministic): the statistics lane by lane and then a
// tree over the vector's lanes, the weighted outputs in chunk order.
constexpr int kMergeThreads = 256;

template <int HD>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_rows_kernel(const AttnArgs a) {
  // the sequences' metadata come from the prologue, complete once this kernel has started:
  // they are read before the dependency wait, the partials after it
  bool waited = false;
  constexpr int LPR = HD / 8;      // lanes per query vector (8 values each)
  constexpr int RPW = 32 / LPR;    // query vectors per warp
  constexpr int GROUPS = kAttnRows / RPW;
  constexpr int CB = 2;            // chunks whose outputs are loaded with the statistics (CB <= LPR)
  static_assert(CB <= LPR, "a prefetched chunk's weight is held by a lane of its vector");
  const int G = a.n_q / a.n_kv, lane = threadIdx.x & 31, sub = lane % LPR, rw = lane / LPR;
  const int ldq = a.n_q * HD;
  const long long n_tasks = (long long)a.B * a.n_kv * GROUPS;
  const long long warps = (long long)gridDim.x * (kMergeThreads / 32);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  for (long long task = ((long long)blockIdx.x * kMergeThreads + threadIdx.x) >> 5; task < n_tasks; task += warps) {
    const int grp = (int)(task % GROUPS);
    const int bg = (int)(task / GROUPS);
    const int b = bg / a.n_kv, g = bg - (bg / a.n_kv) * a.n_kv;
    // the sequence's metadata in one round trip
    const int nc = __ldcg(a.n_chunks + b), len = __ldcg(a.seq_len + b), ibase = __ldcg(a.item_base + b),
              start = __ldcg(a.seq_start + b);
    const int M = min(len * G, kAttnRows);
    if (nc <= 1 || grp * RPW >= M) continue;  // the same for the whole warp
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    const int m = grp * RPW + rw;
    const bool valid = m < M;
    const size_t base = (size_t)(ibase + g * nc) * kAttnRows + m;  // partial row of chunk 0
    // one round trip for the data: the statistics of chunk `sub` (and of every LPR-th one
    // after it) and the outputs of the first CB chunks are all in flight together
    float mc_l = -INFINITY, lc_l = 0.f;
    if (valid && sub < nc) {
      mc_l = __ldcg(a.part_m + base + (size_t)sub * kAttnRows);
      lc_l = __ldcg(a.part_l + base + (size_t)sub * kAttnRows);
    }
    float o[CB][8];
#pragma unroll
    for (int k = 0; k < CB; ++k)
      if (valid && k < nc) ldcg_v8(a.part_o + (base + (size_t)k * kAttnRows) * HD + sub * 8, o[k]);
    float mx = mc_l;
    if (valid)
      for (int c = sub + LPR; c < nc; c += LPR) mx = fmaxf(mx, __ldcg(a.part_m + base + (size_t)c * kAttnRows));
#pragma unroll
    for (int o2 = LPR / 2; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o2));
    const float w_l = mc_l == -INFINITY ? 0.f : exp2f(mc_l - mx);  // weight of chunk `sub`
    float L = w_l * lc_l;
    if (valid)
      for (int c = sub + LPR; c < nc; c += LPR) {
        const float mc = __ldcg(a.part_m + base + (size_t)c * kAttnRows);
        L += (mc == -INFINITY ? 0.f : exp2f(mc - mx)) * __ldcg(a.part_l + base + (size_t)c * kAttnRows);
      }
#pragma unroll
    for (int o2 = LPR / 2; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o2);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const int lane0 = lane - sub;  // the vector's first lane
#pragma unroll
    for (int k = 0; k < CB; ++k) {  // chunk order; chunk k's weight lives in lane lane0 + k
      const float wk = __shfl_sync(0xFFFFFFFFu, w_l, lane0 + k);
      if (k < nc) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += wk * o[k][e];
      }
    }
    if (!valid) continue;
#pragma unroll 4
    for (int c = CB; c < nc; ++c) {  // long ranges: the rest, in chunk order
      const size_t pr = base + (size_t)c * kAttnRows;
      const float mc = __ldcg(a.part_m + pr);
      const float wk = mc == -INFINITY ? 0.f : exp2f(mc - mx);
      float u[8];
      ldcg_v8(a.part_o + pr * HD + sub * 8, u);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += wk * u[e];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* dst = out + (size_t)(start + m / G) * ldq + (size_t)(g * G + m % G) * HD + (size_t)sub * 8;
    uint4 pk;
    pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    pk.z = pack_bf16(acc[4] * inv, acc[5] * inv);
    pk.w = pack_bf16(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(dst) = pk;
  }
  if (!waited) {  // no CTA completes before the previous kernel has
    pdl_wait();
    pdl_trigger();
  }
}

// The same merge for few (sequence, kv head) pairs with many chunks each: one warp
// per (sequence, kv head, query vector), lanes over head_dim, the chunk statistics
// one chunk per lane and eight chunks' outputs in flight at once.  out = sum_c w_c O_c / sum_c w_c l_c with w_c = 2^(m_c - max_c m_c);
// the weighted sum runs in chunk order (deterministic).

template <int HD>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnArgs a) {
  bool waited = false;  // metadata before the dependency wait, partials after it (as above)
  constexpr int VPL = HD / 32;  // output values per lane
  constexpr int CB = 8;         // chunks whose outputs are in flight together
  const int G = a.n_q / a.n_kv, lane = threadIdx.x & 31;
  const int ldq = a.n_q * HD;
  const long long n_tasks = (long long)a.B * a.n_kv * kAttnRows;
  const long long warps = (long long)gridDim.x * (kMergeThreads / 32);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  for (long long task = ((long long)blockIdx.x * kMergeThreads + threadIdx.x) >> 5; task < n_tasks; task += warps) {
    const int m = (int)(task % kAttnRows);
    const int bg = (int)(task / kAttnRows);
    const int b = bg / a.n_kv, g = bg - (bg / a.n_kv) * a.n_kv;
    // the sequence's metadata in one round trip
    const int nc = __ldcg(a.n_chunks + b), len = __ldcg(a.seq_len + b), ibase = __ldcg(a.item_base + b),
              start = __ldcg(a.seq_start + b);
    if (nc <= 1 || m >= min(len * G, kAttnRows)) continue;
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    const size_t base = (size_t)(ibase + g * nc) * kAttnRows + m;  // partial row of chunk 0
    // chunk statistics (one chunk per lane) and the first CB chunks' outputs, all in flight together
    float mc_l = -INFINITY, lc_l = 0.f;
    if (lane < nc) {
      mc_l = __ldcg(a.part_m + base + (size_t)lane * kAttnRows);
      lc_l = __ldcg(a.part_l + base + (size_t)lane * kAttnRows);
    }
    float v[CB][VPL];
#pragma unroll
    for (int k = 0; k < CB; ++k)
      if (k < nc) {
        const float* src = a.part_o + (base + (size_t)k * kAttnRows) * HD + lane * VPL;
        if constexpr (VPL == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
          v[k][0] = t.x; v[k][1] = t.y; v[k][2] = t.z; v[k][3] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
          v[k][0] = t.x; v[k][1] = t.y;
        }
      }
    float mx = mc_l;
    for (int c = 32 + lane; c < nc; c += 32) mx = fmaxf(mx, __ldcg(a.part_m + base + (size_t)c * kAttnRows));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    const float w_l = mc_l == -INFINITY ? 0.f : exp2f(mc_l - mx);  // weight of chunk `lane`
    float L = w_l * lc_l;
    for (int c = 32 + lane; c < nc; c += 32) {
      const float mc = __ldcg(a.part_m + base + (size_t)c * kAttnRows);
      L += (mc == -INFINITY ? 0.f : exp2f(mc - mx)) * __ldcg(a.part_l + base + (size_t)c * kAttnRows);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
    float acc[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
#pragma unroll
    for (int k = 0; k < CB; ++k) {  // chunk order
      const float wk = __shfl_sync(0xFFFFFFFFu, w_l, k);
      if (k < nc) {
#pragma unroll
        for (int e = 0; e < VPL; ++e) acc[e] += wk * v[k][e];
      }
    }
    for (int c0 = CB; c0 < nc; c0 += CB) {  // long ranges: the rest, CB chunks' loads at a time
#pragma unroll
      for (int k = 0; k < CB; ++k) {
        const int c = c0 + k;
        if (c < nc) {
          const float* src = a.part_o + (base + (size_t)c * kAttnRows) * HD + lane * VPL;
#pragma unroll
          for (int e = 0; e < VPL; ++e) v[k][e] = __ldcg(src + e);
        }
      }
#pragma unroll
      for (int k = 0; k < CB; ++k) {  // chunk order
        const int c = c0 + k;
        const float wk = __shfl_sync(0xFFFFFFFFu, w_l, c & 31);  // lane c holds chunk c's weight for c < 32
        const float mc = (c >= 32 && c < nc) ? __ldcg(a.part_m + base + (size_t)c * kAttnRows) : 0.f;
        const float w = c < 32 ? wk : (mc == -INFINITY ? 0.f : exp2f(mc - mx));
        if (c < nc) {
#pragma unroll
          for (int e = 0; e < VPL; ++e) acc[e] += w * v[k][e];
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* dst = out + (size_t)(start + m / G) * ldq + (size_t)(g * G + m % G) * HD + (size_t)lane * VPL;
    if constexpr (VPL == 4) {
      uint2 pk;
      pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
      pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(dst) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
    }
  }
  if (!waited) {  // no CTA completes before the previous kernel has
    pdl_wait();
    pdl_trigger();
  }
}

// Many (sequence, kv head) pairs (large batches, few chunks each): several query vectors
// per warp, so that most warps do work; few pairs (small batches, many chunks each): a warp
// per query vector with its chunks spread over the lanes.
constexpr int kMergeRowsMinPairs = 128;

template <int HD>
static cudaError_t launch_merge_typed(const AttnArgs& a, int sms, cudaStream_t s) {
  const bool rows = (long long)a.B * a.n_kv >= kMergeRowsMinPairs;
  const int per_warp = rows ? 32 / (HD / 8) : 1;
  const long long warps = (long long)a.B * a.n_kv * (kAttnRows / per_warp);
  const long long need = (warps + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
  const int grid = (int)std::min<long long>(need, 64LL * sms);
  if (grid <= 0) return cudaSuccess;
  if (rows) return launch_pdl(attn_merge_rows_kernel<HD>, dim3(grid), dim3(kMergeThreads), 0, s, a);
  return launch_pdl(attn_merge_kernel<HD>, dim3(grid), dim3(kMergeThreads), 0, s, a);
}

cudaError_t launch_attention_bf16(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a, int grid,
                                  int sms, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidValue;
  if (a.head_dim == 64) e = launch_attn_typed<64>(tmK, tmV, a, grid, s);
  if (a.head_dim == 128) e = launch_attn_typed<128>(tmK, tmV, a, grid, s);
  if (e != cudaSuccess) return e;
  if (a.head_dim == 64) return launch_merge_typed<64>(a, sms, s);
  return launch_merge_typed<128>(a, sms, s);
}

// ============================================================================= fp32

template <int HD>
__global__ void __launch_bounds__(256) attn_f32_kernel(const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int n = min(*a.n_valid, a.n_rows);
  const int t = gw / a.n_q, h = gw - (gw / a.n_q) * a.n_q;
  if (t >= n) return;
  const int G = a.n_q / a.n_kv, g = h / G;
  const int b = a.tok_seq[t], p = a.tok_pos[t];
  const float* q = static_cast<const float*>(a.q) + (size_t)t * a.n_q * HD + (size_t)h * HD;
  const float* kc = static_cast<const float*>(a.k_cache);
  const float* vc = static_cast<const float*>(a.v_cache);
  float qr[HD];
#pragma unroll
  for (int e = 0; e < HD; ++e) qr[e] = q[e];
  float m = -INFINITY, l = 0.f, o[HD];
#pragma unroll
  for (int e = 0; e < HD; ++e) o[e] = 0.f;
  for (int pos = lane; pos <= p; pos += 32) {
    const int pi = pos / a.page_size;
    if (pi >= a.max_pages) { set_err(a.err, PE_DEV_BAD_POSITION); break; }
    const int page = a.block_table[(size_t)b * a.max_pages + pi];
    if (page < 0 || page >= a.num_pages) { set_err(a.err, PE_DEV_BAD_PAGE); continue; }
    const size_t off = (((size_t)page * a.page_size + pos % a.page_size) * a.n_kv + g) * HD;
    float sdot = 0.f;
#pragma unroll
    for (int e = 0; e < HD; ++e) sdot += qr[e] * kc[off + e];
    sdot *= a.scale;
    const float m_new = fmaxf(m, sdot);
    const float c = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float w = expf(sdot - m_new);
    l = l * c + w;
#pragma unroll
    for (int e = 0; e < HD; ++e) o[e] = o[e] * c + w * vc[off + e];
    m = m_new;
  }
  float M = m;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, s));
  const float f = (m == -INFINITY) ? 0.f : expf(m - M);
  float L = l * f;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, s);
  float* out = static_cast<float*>(a.out) + (size_t)t * a.n_q * HD + (size_t)h * HD;
#pragma unroll
  for (int e = 0; e < HD; ++e) {
    float v = o[e] * f;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, s);
    if (lane == (e & 31)) out[e] = v / L;
  }
}

cudaError_t launch_attention_f32(const AttnArgs& a, cudaStream_t s) {
  const long long warps = (long long)a.n_rows * a.n_q;
  const int grid = (int)((warps * 32 + 255) / 256);
  if (grid == 0) return cudaSuccess;
  if (a.head_dim == 64) return launch_pdl(attn_f32_kernel<64>, dim3(grid), dim3(256), 0, s, a);
  if (a.head_dim == 128) return launch_pdl(attn_f32_kernel<128>, dim3(grid), dim3(256), 0, s, a);
  return cudaErrorInvalidValue;
}

}  // namespace pe
