// Paged GQA attention of the drafter rows over the drafter KV cache.
//
// A row of sequence b at position p attends to the cache positions 0..p of
// its sequence (the prefix plus the rows this round wrote: causal inside the
// draft block).  Keys are stored post-RoPE.  Scale 1/sqrt(head_dim).
//
// bf16: one work item = (sequence b, kv head g, position chunk [c0, c1)).
// The query tile packs every valid row of the sequence times the n_q/n_kv
// query heads of g (<= 128 query vectors), so each KV page is read once per
// (sequence, kv head).  QK^T and PV run on warp-level tensor-core MMAs
// (m16n8k16 bf16, fp32 accumulate) with an online softmax; KV blocks of 64
// positions are double-buffered with cp.async through a page-table gather.
// Items write (max, sum, unnormalised output) partials; a combine kernel
// merges the chunks of each row in chunk order (deterministic).
//
// fp32: one warp per (row, query head); lanes stride over positions with an
// online softmax each, then merge.
#include <cfloat>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

namespace {

PE_DEV void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
PE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
PE_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

// [rows][HD] bf16 tile with 16-byte chunks XOR-swizzled by (row % 8): conflict-free ldmatrix.
template <int HD>
PE_DEV uint32_t swz(uint32_t base, int row, int chunk) {
  return base + (uint32_t)(row * HD * 2) + (uint32_t)(((chunk ^ (row & 7))) * 16);
}

}  // namespace

constexpr int kAttnBlk = 64;      // kv positions per pipeline block
constexpr int kAttnThreads = 256; // 8 warps x 16 query rows
constexpr int kAttnStages = 3;    // cp.async ring depth (blocks in flight)

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, HD == 64 ? 2 : 1) attn_bf16_kernel(const AttnArgs a) {
  constexpr int CH = HD / 8;  // 16-byte chunks per row
  constexpr int S = kAttnStages;
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sQ = smem_u32(sm);
  const uint32_t sK = sQ + kAttnRows * HD * 2;
  const uint32_t sV = sK + S * kAttnBlk * HD * 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  const __nv_bfloat16* qbuf = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  const int ldq = a.n_q * HD;
  pdl_wait();
  pdl_trigger();
  const int n_items = *a.n_items;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int4 item = a.items[it];
    const int b = item.x, g = item.y, c0 = item.z, c1 = item.w;
    const int start = a.seq_start[b], nb = a.seq_len[b];
    const int M = min(nb * G, kAttnRows);

    // ---- query tile (zeros past the valid rows)
    for (int idx = tid; idx < kAttnRows * CH; idx += kAttnThreads) {
      const int m = idx / CH, ch = idx - (idx / CH) * CH;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (m < M) {
        const int i = m / G, j = m - (m / G) * G;
        val = *reinterpret_cast<const uint4*>(qbuf + (size_t)(start + i) * ldq + (size_t)(g * G + j) * HD + ch * 8);
      }
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(swz<HD>(sQ, m, ch)), "r"(val.x), "r"(val.y),
                   "r"(val.z), "r"(val.w)
                   : "memory");
    }

    auto load_block = [&](int blk, int buf) {
      const int kb0 = c0 + blk * kAttnBlk;
      for (int idx = tid; idx < 2 * kAttnBlk * CH; idx += kAttnThreads) {
        const int which = idx / (kAttnBlk * CH);
        const int rem = idx - which * (kAttnBlk * CH);
        const int r = rem / CH, ch = rem - (rem / CH) * CH;
        const int pos = kb0 + r;
        bool valid = pos < c1;
        const __nv_bfloat16* src = kc;
        if (valid && pos / a.page_size >= a.max_pages) {
          set_err(a.err, PE_DEV_BAD_POSITION);
          valid = false;
        }
        if (valid) {
          const int page = a.block_table[(size_t)b * a.max_pages + pos / a.page_size];
          if (page < 0 || page >= a.num_pages) {
            set_err(a.err, PE_DEV_BAD_PAGE);
            valid = false;
          } else {
            const size_t off = (((size_t)page * a.page_size + pos % a.page_size) * a.n_kv + g) * HD + ch * 8;
            src = (which == 0 ? kc : vc) + off;
          }
        }
        const uint32_t base = (which == 0 ? sK : sV) + (uint32_t)(buf * kAttnBlk * HD * 2);
        cp_async16(swz<HD>(base, r, ch), src, valid);
      }
    };

    const int nblk = (c1 - c0 + kAttnBlk - 1) / kAttnBlk;
    for (int st = 0; st < S - 1; ++st) {  // prologue: S-1 blocks in flight (empty groups keep the count)
      if (st < nblk) load_block(st, st);
      cp_async_commit();
    }
    __syncthreads();  // query tile visible

    // ---- per-warp state: rows 16*warp + lane/4 and +8
    const bool active = warp * 16 < M;
    const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
    const int p0 = r0 < M ? a.tok_pos[start + r0 / G] : -1;
    const int p1 = r1 < M ? a.tok_pos[start + r1 / G] : -1;
    uint32_t qf[HD / 16][4];
    if (active) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int row = warp * 16 + (lane & 15);
        const int ch = kk * 2 + (lane >> 4);
        ldmatrix_x4(swz<HD>(sQ, row, ch), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    float o[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int blk = 0; blk < nblk; ++blk) {
      const int buf = blk % S;
      cp_async_wait<S - 2>();  // block blk has landed
      __syncthreads();         // ... for every thread; and block blk-1's stage is free again
      if (blk + S - 1 < nblk) load_block(blk + S - 1, (blk + S - 1) % S);
      cp_async_commit();
      if (active) {
        const uint32_t kbase = sK + (uint32_t)(buf * kAttnBlk * HD * 2);
        const uint32_t vbase = sV + (uint32_t)(buf * kAttnBlk * HD * 2);
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            uint32_t b0, b1, b2, b3;
            const int row = np * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int ch = kk * 2 + ((lane >> 3) & 1);
            ldmatrix_x4(swz<HD>(kbase, row, ch), b0, b1, b2, b3);
            mma_bf16_16816(s[2 * np], qf[kk], b0, b1);
            mma_bf16_16816(s[2 * np + 1], qf[kk], b2, b3);
          }
        }
        // scale, causal mask, online softmax (log2 domain)
        const int kb0 = c0 + blk * kAttnBlk;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = kb0 + n * 8 + 2 * (lane & 3) + (e & 1);
            const int rp = e < 2 ? p0 : p1;
            const bool ok = pos < c1 && pos <= rp;
            s[n][e] = ok ? s[n][e] * scale_log2 : -INFINITY;
            mx[e >> 1] = fmaxf(mx[e >> 1], s[n][e]);
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
        for (int n = 0; n < 8; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mr = m_run[e >> 1];
            const float p = (mr == -INFINITY) ? 0.f : exp2f(s[n][e] - mr);
            s[n][e] = p;
            rs[e >> 1] += p;
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
        // O += P V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t pa[4];
          pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
          pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
          pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
          pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
          for (int np = 0; np < HD / 16; ++np) {
            uint32_t b0, b1, b2, b3;
            const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int ch = np * 2 + (lane >> 4);
            ldmatrix_x4_trans(swz<HD>(vbase, row, ch), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * np], pa, b0, b1);
            mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
          }
        }
      }
    }
    cp_async_wait<0>();

    // ---- partials: row max (log2 domain), row sum, unnormalised output
    if (active) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(0xFFFFFFFFu, l_run[h], 2);
      }
      const size_t ib = (size_t)it * kAttnRows;
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
    __syncthreads();  // query tile reused by the next item
  }
}

// Merge the chunks of every (row, query head), in chunk order.
template <int HD>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int n = min(*a.n_valid, a.n_rows);
  const int t = gw / a.n_q, h = gw - (gw / a.n_q) * a.n_q;
  if (t >= n) return;
  const int G = a.n_q / a.n_kv;
  const int b = a.tok_seq[t];
  const int i = t - a.seq_start[b];
  const int g = h / G, j = h - g * G;
  const int m = i * G + j;
  const int nc = a.n_chunks[b];
  const int base = a.item_base[b] + g * nc;
  float M = -INFINITY;
  for (int c = 0; c < nc; ++c) M = fmaxf(M, a.part_m[(size_t)(base + c) * kAttnRows + m]);
  float L = 0.f;
  constexpr int PER = HD / 32;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int c = 0; c < nc; ++c) {
    const size_t ib = (size_t)(base + c) * kAttnRows + m;
    const float mc = a.part_m[ib];
    if (mc == -INFINITY) continue;
    const float w = exp2f(mc - M);
    L += w * a.part_l[ib];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += w * a.part_o[ib * HD + lane + 32 * e];
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (size_t)t * a.n_q * HD + (size_t)h * HD;
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) out[lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
}

template <int HD>
static size_t attn_smem() {
  return (size_t)kAttnRows * HD * 2 + 2 * (size_t)kAttnStages * kAttnBlk * HD * 2;
}

cudaError_t launch_attention_bf16(const AttnArgs& a, int grid, cudaStream_t s) {
  if (a.head_dim == 64) {
    static bool cfg = false;
    if (!cfg) {
      cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)attn_smem<64>());
      if (e != cudaSuccess) return e;
      cfg = true;
    }
    return launch_pdl(attn_bf16_kernel<64>, dim3(grid), dim3(kAttnThreads), attn_smem<64>(), s, a);
  } else if (a.head_dim == 128) {
    static bool cfg = false;
    if (!cfg) {
      cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)attn_smem<128>());
      if (e != cudaSuccess) return e;
      cfg = true;
    }
    return launch_pdl(attn_bf16_kernel<128>, dim3(grid), dim3(kAttnThreads), attn_smem<128>(), s, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention_combine_bf16(const AttnArgs& a, cudaStream_t s) {
  const long long warps = (long long)a.n_rows * a.n_q;
  const int grid = (int)((warps * 32 + 255) / 256);
  if (grid == 0) return cudaSuccess;
  if (a.head_dim == 64) return launch_pdl(attn_combine_kernel<64>, dim3(grid), dim3(256), 0, s, a);
  if (a.head_dim == 128) return launch_pdl(attn_combine_kernel<128>, dim3(grid), dim3(256), 0, s, a);
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
