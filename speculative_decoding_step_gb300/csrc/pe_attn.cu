// Paged GQA attention of the drafter rows over the drafter KV cache.
//
// A row of sequence b at position p attends to the cache positions 0..p of
// its sequence (the prefix plus the rows this round wrote: causal inside the
// draft block).  Keys are stored post-RoPE.  Scale 1/sqrt(head_dim).
//
// bf16: one work item = (sequence b, kv head g, position chunk [c0, c1)).
// The query tile packs every valid row of the sequence times the n_q/n_kv
// query heads of g (<= 128 query vectors), so each KV page is read once per
// (sequence, kv head).  One producer warp streams the chunk's K and V pages
// with 3-D TMA loads (one 16-position page per load, 128-byte swizzle,
// pages past the range zero-filled) into a 4-stage mbarrier ring; eight
// compute warps run QK^T and PV on warp-level tensor-core MMAs (m16n8k16
// bf16, fp32 accumulate) with an online softmax, without any block-wide
// barrier in the loop.  A range in one chunk is written directly; otherwise
// every chunk leaves (max, sum, unnormalised output) partials and the last
// chunk to finish merges them in chunk order (deterministic).
//
// fp32: one warp per (row, query head); lanes stride over positions with an
// online softmax each, then merge.
#include <cfloat>
#include <climits>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

namespace {

PE_DEV void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
PE_DEV void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
PE_DEV void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
PE_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace

constexpr int kAttnBlk = 64;            // kv positions per pipeline stage (4 pages)
constexpr int kAttnStages = 4;          // stages in flight
constexpr int kAttnComputeWarps = 8;    // 16 query rows each
constexpr int kAttnThreads = 32 * (kAttnComputeWarps + 1);  // + one TMA producer warp

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
  static constexpr uint32_t STAGE = 2 * KV;
  static constexpr uint32_t BARS = Q + kAttnStages * STAGE;
  static constexpr uint32_t TOTAL = 1024 + BARS + 128;   // + alignment slack
};

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, HD == 64 ? 2 : 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const AttnArgs a) {
  using Lay = AttnLayout<HD>;
  constexpr int CH = HD / 8;  // 16-byte units per row
  constexpr int S = kAttnStages;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(sm);
  const uint32_t sRing = sQ + Lay::Q;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lay::BARS);
  uint64_t* empty = full + S;
  volatile int* last_s = reinterpret_cast<volatile int*>(empty + S);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv;

  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kAttnComputeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int n_items = *a.n_items;

  if (warp == kAttnComputeWarps) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();  // the prefix is read once per round
      const int oob = a.num_pages * a.page_size;     // a row past the pool: TMA fills zeros
      int gi = 0;
      bool stop = false;
      for (int it = blockIdx.x; it < n_items && !stop; it += gridDim.x) {
        const int4 item = a.items[it];
        const int b = item.x, g = item.y, c0 = item.z, c1 = item.w;
        const int nblk = (c1 - c0 + kAttnBlk - 1) / kAttnBlk;
        for (int blk = 0; blk < nblk; ++blk, ++gi) {
          const int s = gi % S;
          const uint32_t use = (uint32_t)(gi / S);
          if (gi >= S && !mbar_wait(smem_u32(empty + s), (use & 1u) ^ 1u, a.err, nullptr)) {
            stop = true;
            break;
          }
          const uint32_t fb = smem_u32(full + s);
          mbar_expect_tx(fb, Lay::STAGE);
          const uint32_t kdst = sRing + (uint32_t)s * Lay::STAGE;
#pragma unroll
          for (int p = 0; p < kAttnBlk / 16; ++p) {
            const int pos0 = c0 + blk * kAttnBlk + p * 16;
            int y = oob;
            if (pos0 < c1) {
              const int pi = pos0 / a.page_size;
              if (pi >= a.max_pages) {
                set_err(a.err, PE_DEV_BAD_POSITION);
              } else {
                const int page = a.block_table[(size_t)b * a.max_pages + pi];
                if (page < 0 || page >= a.num_pages) set_err(a.err, PE_DEV_BAD_PAGE);
                else y = page * a.page_size;
              }
            }
#pragma unroll
            for (int h = 0; h < HD / 64; ++h) {
              const uint32_t off = (uint32_t)(h * kAttnBlk * 128 + p * 16 * 128);
              tma_load_3d(kdst + off, &tmK, fb, h * 64, g, y, pol);
              tma_load_3d(kdst + Lay::KV + off, &tmV, fb, h * 64, g, y, pol);
            }
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ compute warps
    const float scale_log2 = a.scale * 1.4426950408889634f;
    const __nv_bfloat16* qbuf = static_cast<const __nv_bfloat16*>(a.q);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const int ldq = a.n_q * HD;
    int gi = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const int4 item = a.items[it];
      const int b = item.x, g = item.y, c0 = item.z, c1 = item.w;
      const int start = a.seq_start[b], nb = a.seq_len[b];
      const int M = min(nb * G, kAttnRows);
      const int nblk = (c1 - c0 + kAttnBlk - 1) / kAttnBlk;
      const int nc = a.n_chunks[b];

      // query tile: row m = (row m / G of the sequence, head g*G + m % G); zeros past the valid rows
      named_bar_sync(1, 32 * kAttnComputeWarps);  // every warp holds its fragments of the previous tile
      for (int idx = tid; idx < kAttnRows * CH; idx += 32 * kAttnComputeWarps) {
        const int m = idx / CH, ch = idx - (idx / CH) * CH;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (m < M) {
          const int i = m / G, j = m - (m / G) * G;
          val = *reinterpret_cast<const uint4*>(qbuf + (size_t)(start + i) * ldq + (size_t)(g * G + j) * HD + ch * 8);
        }
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(tile_addr<kAttnRows>(sQ, m, ch)), "r"(val.x),
                     "r"(val.y), "r"(val.z), "r"(val.w)
                     : "memory");
      }
      named_bar_sync(1, 32 * kAttnComputeWarps);

      const bool active = warp * 16 < M;
      const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
      const int p0 = r0 < M ? a.tok_pos[start + r0 / G] : -1;
      const int p1 = r1 < M ? a.tok_pos[start + r1 / G] : -1;
      // smallest causal bound of the warp's rows; rows past M bound nothing (they are discarded)
      int pmin = min(r0 < M ? p0 : INT_MAX, r1 < M ? p1 : INT_MAX);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pmin = min(pmin, __shfl_xor_sync(0xFFFFFFFFu, pmin, o));
      uint32_t qf[HD / 16][4];
      if (active) {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          ldmatrix_x4(tile_addr<kAttnRows>(sQ, warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), qf[kk][0], qf[kk][1],
                      qf[kk][2], qf[kk][3]);
      }
      float o[HD / 8][4];
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

      for (int blk = 0; blk < nblk; ++blk, ++gi) {
        const int s = gi % S;
        mbar_wait(smem_u32(full + s), (uint32_t)(gi / S) & 1u, a.err, nullptr);
        if (active) {
          const uint32_t kbase = sRing + (uint32_t)s * Lay::STAGE;
          const uint32_t vbase = kbase + Lay::KV;
#pragma unroll 1
          for (int hb = 0; hb < kAttnBlk / 32; ++hb) {  // 32 positions at a time (bounds the score registers)
            float sc[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
              for (int np = 0; np < 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(tile_addr<kAttnBlk>(kbase, hb * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3),
                                                kk * 2 + ((lane >> 3) & 1)),
                            b0, b1, b2, b3);
                mma_bf16_16816(sc[2 * np], qf[kk], b0, b1);
                mma_bf16_16816(sc[2 * np + 1], qf[kk], b2, b3);
              }
            }
            // scale, causal mask (only where this half reaches the end of the range or a row's
            // position), online softmax (log2 domain)
            const int kb0 = c0 + blk * kAttnBlk + hb * 32;
            float mx[2] = {-INFINITY, -INFINITY};
            if (kb0 + 32 <= c1 && kb0 + 31 <= pmin) {
#pragma unroll
              for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  sc[n][e] *= scale_log2;
                  mx[e >> 1] = fmaxf(mx[e >> 1], sc[n][e]);
                }
            } else {
#pragma unroll
              for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int pos = kb0 + n * 8 + 2 * (lane & 3) + (e & 1);
                  const int rp = e < 2 ? p0 : p1;
                  sc[n][e] = (pos < c1 && pos <= rp) ? sc[n][e] * scale_log2 : -INFINITY;
                  mx[e >> 1] = fmaxf(mx[e >> 1], sc[n][e]);
                }
            }
            float corr[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xFFFFFFFFu, mx[h], 1));
              mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xFFFFFFFFu, mx[h], 2));
              const float m_new = fmaxf(m_run[h], mx[h]);
              corr[h] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[h] - m_new);
              m_run[h] = m_new;
            }
            float rs[2] = {0.f, 0.f};
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float mr = m_run[e >> 1];
                const float pv = (mr == -INFINITY) ? 0.f : exp2f(sc[n][e] - mr);
                sc[n][e] = pv;
                rs[e >> 1] += pv;
              }
            l_run[0] = l_run[0] * corr[0] + rs[0];
            l_run[1] = l_run[1] * corr[1] + rs[1];
#pragma unroll
            for (int n = 0; n < HD / 8; ++n) {
              o[n][0] *= corr[0];
              o[n][1] *= corr[0];
              o[n][2] *= corr[1];
              o[n][3] *= corr[1];
            }
            // O += P V over these 32 positions
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              uint32_t pa[4];
              pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
              pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
              pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
              pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
              for (int np = 0; np < HD / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(tile_addr<kAttnBlk>(vbase, hb * 32 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                                      np * 2 + (lane >> 4)),
                                  b0, b1, b2, b3);
                mma_bf16_16816(o[2 * np], pa, b0, b1);
                mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
      }

      // ---- results of this item
      if (active) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 1);
          l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 2);
        }
      }
      if (nc == 1) {
        // the item covers the whole range: normalise and write the output rows directly
        if (active) {
          const float i0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f, i1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
#pragma unroll
          for (int n = 0; n < HD / 8; ++n) {
            const int col = n * 8 + 2 * (lane & 3);
            if (r0 < M)
              *reinterpret_cast<uint32_t*>(out + (size_t)(start + r0 / G) * ldq + (size_t)(g * G + r0 % G) * HD + col) =
                  pack_bf16(o[n][0] * i0, o[n][1] * i0);
            if (r1 < M)
              *reinterpret_cast<uint32_t*>(out + (size_t)(start + r1 / G) * ldq + (size_t)(g * G + r1 % G) * HD + col) =
                  pack_bf16(o[n][2] * i1, o[n][3] * i1);
          }
        }
        continue;
      }
      const size_t ib = (size_t)it * kAttnRows;
      if (active) {
        if ((lane & 3) == 0) {
          if (r0 < M) { a.part_m[ib + r0] = m_run[0]; a.part_l[ib + r0] = l_run[0]; }
          if (r1 < M) { a.part_m[ib + r1] = m_run[1]; a.part_l[ib + r1] = l_run[1]; }
        }
#pragma unroll
        for (int n = 0; n < HD / 8; ++n) {
          const int col = n * 8 + 2 * (lane & 3);
          if (r0 < M) *reinterpret_cast<float2*>(a.part_o + (ib + r0) * HD + col) = make_float2(o[n][0], o[n][1]);
          if (r1 < M) *reinterpret_cast<float2*>(a.part_o + (ib + r1) * HD + col) = make_float2(o[n][2], o[n][3]);
        }
      }
      // the last chunk of (sequence, kv head) to finish merges all chunks, in chunk order
      __threadfence();
      named_bar_sync(1, 32 * kAttnComputeWarps);
      if (tid == 0) {
        const int old = atomicAdd(a.counters + b * a.n_kv + g, 1);
        *last_s = (old == nc - 1) ? 1 : 0;
      }
      named_bar_sync(1, 32 * kAttnComputeWarps);
      if (*last_s) {
        __threadfence();
        const int base = a.item_base[b] + g * nc;
        for (int idx = tid; idx < M * (HD / 4); idx += 32 * kAttnComputeWarps) {
          const int m = idx / (HD / 4), e4 = idx - (idx / (HD / 4)) * (HD / 4);
          // chunk statistics first (independent loads), then the weighted sum, in chunk order
          float Mx = -INFINITY;
#pragma unroll 4
          for (int c = 0; c < nc; ++c) Mx = fmaxf(Mx, __ldcg(a.part_m + (size_t)(base + c) * kAttnRows + m));
          float L = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
          for (int c = 0; c < nc; ++c) {
            const size_t pr = (size_t)(base + c) * kAttnRows + m;
            const float mc = __ldcg(a.part_m + pr);
            const float lc = __ldcg(a.part_l + pr);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part_o + pr * HD) + e4);
            const float wgt = mc == -INFINITY ? 0.f : exp2f(mc - Mx);
            L += wgt * lc;
            acc.x += wgt * v.x; acc.y += wgt * v.y; acc.z += wgt * v.z; acc.w += wgt * v.w;
          }
          const float inv = L > 0.f ? 1.f / L : 0.f;
          __nv_bfloat16* dst = out + (size_t)(start + m / G) * ldq + (size_t)(g * G + m % G) * HD + 4 * e4;
          uint2 pk;
          pk.x = pack_bf16(acc.x * inv, acc.y * inv);
          pk.y = pack_bf16(acc.z * inv, acc.w * inv);
          *reinterpret_cast<uint2*>(dst) = pk;
        }
        if (tid == 0) a.counters[b * a.n_kv + g] = 0;  // ready for the next layer
      }
    }
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

cudaError_t launch_attention_bf16(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a, int grid,
                                  cudaStream_t s) {
  if (a.head_dim == 64) return launch_attn_typed<64>(tmK, tmV, a, grid, s);
  if (a.head_dim == 128) return launch_attn_typed<128>(tmK, tmV, a, grid, s);
  return cudaErrorInvalidValue;
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
