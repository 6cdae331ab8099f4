// Indexing and bandwidth stages of the P-EAGLE drafting round:
//   prepare_batch  -- stage (a): one pass over the B*2K padded rows
//   verify         -- stage (e): greedy verification (+ next round's verify batch)
//   forward_init   -- per compacted row metadata and the attention work list
//   scatter        -- stage (b): drafter input rows moved with bulk async copies
//   rmsnorm        -- row RMSNorm of the fp32 residual stream
#include <climits>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

// ============================================================================= stage (a)
// P-EAGLE: Parallel Speculative Decoding in vLLM, "vLLM implementation details":
// one fused pass copies the previous token ids and positions, inserts the bonus
// token, fills the parallel-draft slots with the MASK id and emits the rejected
// mask, the MASK mask and the hidden-state map; "KV cache and CUDA Graphs":
// rejected tokens map to PADDING_SLOT_ID (-1).  Valid rows are compacted with a
// warp-ballot + block prefix sum so the drafter pass never touches them.

constexpr int kPrepThreads = 1024;

PE_DEV void prepare_body(const PrepArgs& a) {
  __shared__ int warp_off[32];
  __shared__ int carry_s;
  __shared__ int chunk_total_s;
  const int S = 2 * a.K, R = a.B * S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  if (tid == 0) carry_s = 0;
  __syncthreads();

  for (int base = 0; base < R; base += blockDim.x) {
    const int row = base + tid;
    int valid = 0, draft_k = -1, b = 0;
    if (row < R) {
      b = row / S;
      const int r = row % S;
      int acc = a.num_accepted[b];
      if (acc < 0 || acc > a.K) {
        set_err(a.err, PE_DEV_BAD_ACCEPTED);
        acc = acc < 0 ? 0 : a.K;
      }
      const int32_t* pt = a.prev_tokens + (size_t)b * (a.K + 1);
      const int32_t* pp = a.prev_pos + (size_t)b * (a.K + 1);
      int tok, pos, hmap, rej = 0, msk = 0;
      if (r < acc) {                 // accepted context row: token at p+1, hidden state of p
        tok = pt[r + 1];
        pos = pp[r];
        hmap = b * (a.K + 1) + r;
      } else if (r == acc) {         // NTP row: bonus token with h_context
        tok = a.bonus[b];
        pos = pp[acc];
        hmap = b * (a.K + 1) + acc;
        draft_k = 0;
      } else if (r <= a.K) {         // rejected draft position
        tok = 0;
        pos = pp[r];
        hmap = b * (a.K + 1) + r;
        rej = 1;
      } else {                       // MASK slot m = r - K
        const int m = r - a.K;
        tok = a.vocab;
        pos = pp[acc] + m;
        hmap = -1;
        msk = 1;
        draft_k = m;
      }
      if (!msk && (tok < 0 || tok >= a.vocab)) set_err(a.err, PE_DEV_BAD_TOKEN);
      long long slot = -1;
      if (!rej) {
        const int pi = pos / a.page_size;
        if (pos < 0 || pi >= a.max_pages) {
          set_err(a.err, PE_DEV_BAD_POSITION);
        } else {
          const int page = a.block_table[(size_t)b * a.max_pages + pi];
          if (page < 0 || page >= a.num_pages) set_err(a.err, PE_DEV_BAD_PAGE);
          else slot = (long long)page * a.page_size + pos % a.page_size;
        }
      }
      a.input_ids[row] = tok;
      a.positions[row] = pos;
      a.slot_mapping[row] = slot;
      a.is_rejected[row] = (uint8_t)rej;
      a.is_mask[row] = (uint8_t)msk;
      a.hidden_map[row] = hmap;
      valid = !rej;
    }
    // block-wide exclusive prefix sum of `valid` (warp ballots, then a scan of warp totals)
    const unsigned ballot = __ballot_sync(0xFFFFFFFFu, valid);
    const int lane_prefix = __popc(ballot & ((1u << lane) - 1u));
    if (lane == 0) warp_off[warp] = __popc(ballot);
    __syncthreads();
    if (warp == 0) {
      const int v = lane < nwarps ? warp_off[lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
      }
      if (lane < nwarps) warp_off[lane] = incl - v;
      if (lane == 31) chunk_total_s = incl;
    }
    __syncthreads();
    if (valid) {
      const int idx = carry_s + warp_off[warp] + lane_prefix;
      a.row_list[idx] = row;
      if (draft_k >= 0) a.draft_rows[b * a.K + draft_k] = idx;
    }
    __syncthreads();
    if (tid == 0) carry_s += chunk_total_s;
    __syncthreads();
  }
  for (int i = carry_s + tid; i < R; i += blockDim.x) a.row_list[i] = -1;
  if (tid == 0) *a.n_valid = carry_s;
}

__global__ void __launch_bounds__(kPrepThreads) prepare_kernel(const PrepArgs a) {
  pdl_wait();
  pdl_trigger();
  prepare_body(a);
}

cudaError_t launch_prepare(const PrepArgs& a, cudaStream_t s) {
  const int R = a.B * 2 * a.K;
  const int threads = R >= kPrepThreads ? kPrepThreads : ((R + 31) / 32) * 32;
  return launch_pdl(prepare_kernel, dim3(1), dim3(threads), 0, s, a);
}

// ============================================================================= stage (e)
// vLLM Speculators: parallel drafting for speculative decoding, "Production
// integration in vLLM": verification preserves the target's output; greedy
// form: accept the longest prefix of drafts equal to the target's tokens,
// then take the target's token at the first mismatch as the bonus token.

__global__ void verify_kernel(const VerifyArgs a) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < a.B) verify_seq(a, b);
}
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s) {
  const int threads = 128;
  return launch_pdl(verify_kernel, dim3((a.B + threads - 1) / threads), dim3(threads), 0, s, a);
}

// ============================================================================= DFlash-style KV injection
// vLLM Speculators: parallel drafting for speculative decoding, "DFlash": the verifier's
// hidden states are projected into the drafter's KV cache.  Each element j of sequence b's
// previous verify batch (hidden row b*(K+1) + j) is written at its position's slot when
// j <= num_accepted[b] (the accepted drafts and the bonus token's position); a rejected
// element gets slot -1 (no write).

__global__ void inject_init_kernel(const InjectArgs a) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int S = a.K + 1;
  if (i >= a.B * S) return;
  const int b = i / S, j = i - b * S;
  int acc = a.num_accepted[b];
  if (acc < 0 || acc > a.K) {
    set_err(a.err, PE_DEV_BAD_ACCEPTED);
    acc = -1;  // nothing of this sequence is written
  }
  const int p = a.prev_pos[i];
  long long slot = -1;
  if (j <= acc) {
    const int pi = p / a.page_size;
    if (p < 0 || pi >= a.max_pages) {
      set_err(a.err, PE_DEV_BAD_POSITION);
    } else {
      const int page = a.block_table[(size_t)b * a.max_pages + pi];
      if (page < 0 || page >= a.num_pages) set_err(a.err, PE_DEV_BAD_PAGE);
      else slot = (long long)page * a.page_size + p % a.page_size;
    }
  }
  a.tok_pos[i] = p < 0 ? 0 : p;
  a.tok_slot[i] = slot;
}

cudaError_t launch_inject_init(const InjectArgs& a, cudaStream_t s) {
  const int n = a.B * (a.K + 1), threads = 256;
  return launch_pdl(inject_init_kernel, dim3((n + threads - 1) / threads), dim3(threads), 0, s, a);
}

// ============================================================================= forward prologue

constexpr int kInitThreads = 1024;

PE_DEV void init_body(const InitArgs& a) {
  const int tid = threadIdx.x;
  int n = *a.n_valid;
  if (n < 0 || n > a.R) {
    if (tid == 0) set_err(a.err, PE_DEV_BAD_ROW);
    n = n < 0 ? 0 : a.R;
  }
  const int S = 2 * a.K;
  for (int i = tid; i < a.n_counters; i += blockDim.x) a.counters[i] = 0;
  for (int i = tid; i < a.T; i += blockDim.x) a.keys[i] = 0ull;
  for (int b = tid; b < a.B; b += blockDim.x) {
    a.seq_start[b] = INT_MAX;
    a.seq_len[b] = 0;
    a.seq_maxpos[b] = -1;
    a.seq_minpos[b] = INT_MAX;
  }
  __syncthreads();
  for (int t = tid; t < a.R; t += blockDim.x) {
    if (t < n) {
      const int row = a.row_list[t];
      if (row < 0 || row >= a.R) {
        set_err(a.err, PE_DEV_BAD_ROW);
        a.tok_pos[t] = 0;
        a.tok_slot[t] = -1;
        a.tok_seq[t] = 0;
        continue;
      }
      const int b = row / S;
      const int pos = a.positions[row];
      a.tok_pos[t] = pos;
      a.tok_slot[t] = a.slot_mapping[row];
      a.tok_seq[t] = b;
      atomicMin(&a.seq_start[b], t);
      atomicAdd(&a.seq_len[b], 1);
      atomicMax(&a.seq_maxpos[b], pos);
      atomicMin(&a.seq_minpos[b], pos);
    } else {
      a.tok_pos[t] = 0;
      a.tok_slot[t] = -1;
      a.tok_seq[t] = 0;
    }
  }
  __syncthreads();
  // Attention work list: every (sequence, kv head) splits its causal range
  // 0..maxpos into equal chunks; the chunk length is set so that the whole
  // batch yields about target_items items.  Total length by a block reduction,
  // per-sequence item offsets by a warp scan (both in fixed order).
  __shared__ long long red_s[kInitThreads / 32];
  __shared__ int chunk_s;
  long long part = 0;
  for (int b = tid; b < a.B; b += blockDim.x) part += a.seq_len[b] > 0 ? a.seq_maxpos[b] + 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
  if ((tid & 31) == 0) red_s[tid >> 5] = part;
  __syncthreads();
  if (tid < 32) {
    long long total = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += red_s[w];
    long long per = (total * a.n_kv + a.target_items - 1) / a.target_items;
    per = ((per + 63) / 64) * 64;
    const int chunk = (int)(per < a.min_chunk ? a.min_chunk : per);
    int carry = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + tid;
      const int L = (b < a.B && a.seq_len[b] > 0) ? a.seq_maxpos[b] + 1 : 0;
      const int nc = (L + chunk - 1) / chunk;
      const int v = nc * a.n_kv;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (tid >= o) incl += n;
      }
      if (b < a.B) {
        a.n_chunks[b] = nc;
        a.item_base[b] = carry + incl - v;
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (tid == 0) {
      if (carry > a.max_items) {  // cannot happen with the host's sizing; keep the list in bounds
        set_err(a.err, PE_DEV_BAD_ROW);
        carry = 0;
      }
      *a.n_items = carry;
      chunk_s = chunk;
    }
  }
  __syncthreads();
  const int chunk = chunk_s;
  if (*a.n_items == 0) return;
  for (int b = tid; b < a.B; b += blockDim.x) {
    const int L = a.seq_len[b] > 0 ? a.seq_maxpos[b] + 1 : 0;
    const int nc = a.n_chunks[b];
    int it = a.item_base[b];
    for (int g = 0; g < a.n_kv; ++g)
      for (int c = 0; c < nc; ++c) {
        const int c0 = c * chunk;
        const int c1 = c0 + chunk < L ? c0 + chunk : L;
        a.items[it++] = make_int4(b, g, c0, c1);
      }
  }
}

// One L2 prefetch per 2 MB (a translation page of large allocations) of every warmed weight
// range, spread over the threads of CTAs 0 .. n_cta - 1; nothing waits for them.  The
// weights do not depend on earlier kernels.  (One per 64 KB gave the same B = 8 round and a
// 1.4 us slower B = 1 round.)
PE_DEV void warm_weight_translations(const InitArgs& a, int n_cta) {
  constexpr long long kPiece = 2 << 20;
  const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x, stride = (long long)n_cta * blockDim.x;
  for (int r = 0; r < a.warm_n; ++r) {
    const long long n = a.warm_bytes[r] / kPiece;
    for (long long i = i0; i < n; i += stride) prefetch_l2(a.warm_base[r] + i * kPiece);
  }
}

__global__ void __launch_bounds__(kInitThreads) forward_init_kernel(const InitArgs a) {
  warm_weight_translations(a, gridDim.x);
  pdl_wait();
  pdl_trigger();
  init_body(a);
}

cudaError_t launch_forward_init(const InitArgs& a, cudaStream_t s) {
  return launch_pdl(forward_init_kernel, dim3(1), dim3(kInitThreads), 0, s, a);
}

// ============================================================================= stage (b)
// P-EAGLE: Parallel Speculative Decoding in vLLM, step 2 "Parallel Drafting"
// and "Hidden-state management": each valid row is concat(emb(token), hidden),
// hidden = target hidden state (context / NTP rows) or the learned h_shared
// (MASK rows).  Rows are moved HBM -> shared -> HBM with bulk async copies;
// the MASK row (emb(mask), h_shared) is staged in shared memory once per CTA
// and stored to every MASK row the CTA owns.

constexpr int kScatterRowsPerCta = 4;

// Copies of up to RPC input rows by one thread (it issues every copy): row k goes to x0
// row dst[k]; kind 1: concat(emb[tok], hidden[hmp]), kind 2: the MASK row
// concat(emb(mask), h_shared), staged in shared memory once; kind 0: nothing.
PE_DEV void copy_rows(const ScatterArgs& a, const int (&kind)[kScatterRowsPerCta], const int (&tok)[kScatterRowsPerCta],
                      const int (&hmp)[kScatterRowsPerCta], const int (&dst)[kScatterRowsPerCta]) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar;
  constexpr int RPC = kScatterRowsPerCta;
  const uint32_t rb = (uint32_t)a.d * a.elem_bytes;  // bytes of one half row
  const uint8_t* emb = static_cast<const uint8_t*>(a.emb);
  const uint8_t* hid = static_cast<const uint8_t*>(a.hidden);
  uint8_t* x0 = static_cast<uint8_t*>(a.x0);
  const uint32_t base = smem_u32(sm);
  const uint32_t mask_slot = base + (uint32_t)(2 * RPC) * rb;  // [emb(mask) | h_shared]
  uint32_t bytes = 0;
  bool any_mask = false;
#pragma unroll
  for (int k = 0; k < RPC; ++k) {
    if (kind[k] == 1) bytes += 2 * rb;
    if (kind[k] == 2) any_mask = true;
  }
  if (any_mask) bytes += 2 * rb;
  if (bytes == 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  mbar_expect_tx(b, bytes);
#pragma unroll
  for (int k = 0; k < RPC; ++k) {
    if (kind[k] != 1) continue;
    bulk_g2s(base + (uint32_t)(2 * k) * rb, emb + (size_t)tok[k] * rb, rb, b);
    bulk_g2s(base + (uint32_t)(2 * k + 1) * rb, hid + (size_t)hmp[k] * rb, rb, b);
  }
  if (any_mask) {
    bulk_g2s(mask_slot, emb + (size_t)a.vocab * rb, rb, b);
    bulk_g2s(mask_slot + rb, a.h_shared, rb, b);
  }
  if (!mbar_wait(b, 0, a.err, nullptr)) return;
  fence_proxy_async_smem();
#pragma unroll
  for (int k = 0; k < RPC; ++k) {
    uint8_t* d = x0 + (size_t)dst[k] * 2 * rb;
    if (kind[k] == 1) {
      bulk_s2g(d, base + (uint32_t)(2 * k) * rb, rb);
      bulk_s2g(d + rb, base + (uint32_t)(2 * k + 1) * rb, rb);
    } else if (kind[k] == 2) {
      bulk_s2g(d, mask_slot, 2 * rb);
    }
  }
  bulk_commit();
  bulk_wait_all();
}

// One CTA's rows of the compacted list (pe_scatter_hidden): rows i0 .. i0 + RPC - 1.
PE_DEV void scatter_body(const ScatterArgs& a, int cta) {
  constexpr int RPC = kScatterRowsPerCta;
  const int i0 = cta * RPC;
  // the row count and this CTA's rows in one round trip (rows past the count are -1
  // padding), then every row's metadata in a second one
  int n = *a.n_valid;
  int rows[RPC];
#pragma unroll
  for (int k = 0; k < RPC; ++k) rows[k] = i0 + k < a.R ? a.row_list[i0 + k] : -1;
  n = n < 0 ? 0 : (n > a.R ? a.R : n);
  if (i0 >= n) return;
  const int i1 = i0 + RPC < n ? i0 + RPC : n;
  int msk[RPC], tok[RPC], hmp[RPC], kind[RPC], dst[RPC];
#pragma unroll
  for (int k = 0; k < RPC; ++k) {
    const int row = rows[k];
    const bool ok = i0 + k < i1 && row >= 0 && row < a.R;
    msk[k] = ok ? a.is_mask[row] : 0;
    tok[k] = ok ? a.input_ids[row] : 0;
    hmp[k] = ok ? a.hidden_map[row] : 0;
  }
#pragma unroll
  for (int k = 0; k < RPC; ++k) {
    kind[k] = 0;
    dst[k] = i0 + k;
    if (i0 + k >= i1) continue;
    const int row = rows[k];
    if (row < 0 || row >= a.R) { set_err(a.err, PE_DEV_BAD_ROW); continue; }
    if (msk[k]) { kind[k] = 2; continue; }
    if (tok[k] < 0 || tok[k] > a.vocab) { set_err(a.err, PE_DEV_BAD_TOKEN); continue; }
    if (hmp[k] < 0 || hmp[k] >= a.n_hidden) { set_err(a.err, PE_DEV_BAD_ROW); continue; }
    kind[k] = 1;
  }
  copy_rows(a, kind, tok, hmp, dst);
}

// The input rows of sequence b straight from the previous verify batch (pe_step): the
// sequence's valid rows are, in the rebuild's order, its copy slots 0..a (accepted
// context rows, then the NTP row) and its K-1 MASK rows; they land at compacted rows
// base + 0 .. base + a + K - 1, base = the valid rows of the sequences before b.  CTA
// group `grp` copies the sequence's valid rows grp*RPC .. grp*RPC + RPC - 1.
PE_DEV void scatter_seq_body(const PrepArgs& p, const ScatterArgs& a, int b, int grp, int base) {
  constexpr int RPC = kScatterRowsPerCta;
  const int K = p.K;
  int acc = p.num_accepted[b];
  acc = acc < 0 ? 0 : (acc > K ? K : acc);  // the rebuild reports a bad count and clamps it the same way
  const int v0 = grp * RPC, nv = acc + K;
  if (v0 >= nv) return;
  int kind[RPC], tok[RPC], hmp[RPC], dst[RPC];
#pragma unroll
  for (int k = 0; k < RPC; ++k) {
    const int v = v0 + k;
    kind[k] = 0;
    tok[k] = hmp[k] = 0;
    dst[k] = base + v;
    if (v >= nv) continue;
    if (v > acc) { kind[k] = 2; continue; }  // MASK row m = v - acc
    tok[k] = v < acc ? p.prev_tokens[(size_t)b * (K + 1) + v + 1] : p.bonus[b];
    hmp[k] = b * (K + 1) + v;
    if (tok[k] < 0 || tok[k] >= a.vocab) { set_err(a.err, PE_DEV_BAD_TOKEN); continue; }
    kind[k] = 1;
  }
  copy_rows(a, kind, tok, hmp, dst);
}

__global__ void __launch_bounds__(32) scatter_kernel(const ScatterArgs a) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) scatter_body(a, blockIdx.x);
}

size_t scatter_smem_bytes(int d, int elem_bytes) {
  return (size_t)(2 * kScatterRowsPerCta + 2) * (size_t)d * (size_t)elem_bytes;
}

cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t s) {
  const size_t smem = scatter_smem_bytes(a.d, a.elem_bytes);
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kScatterSmemMax);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int grid = (a.R + kScatterRowsPerCta - 1) / kScatterRowsPerCta;
  return launch_pdl(scatter_kernel, dim3(grid), dim3(32), smem, s, a);
}

// Block-wide exclusive prefix sum of v in thread order (every thread of the CTA calls it);
// `total` receives the sum over the CTA.  warp_s: 33 ints of shared memory.
PE_DEV int block_exclusive_scan(int v, int* warp_s, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_s[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? warp_s[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) warp_s[lane] = wi - w;
    if (lane == 31) warp_s[32] = wi;
  }
  __syncthreads();
  const int r = warp_s[warp] + incl - v;
  total = warp_s[32];
  __syncthreads();  // warp_s may be reused
  return r;
}

// pe_step's batch rebuild and forward prologue in one CTA, with the same results as the
// rebuild followed by the prologue (prepare_body, init_body), in fewer memory round trips:
// a sequence's valid rows are contiguous in the compacted list (its copy slots 0..a, then
// its K-1 MASK rows), so the accepted counts alone give each sequence's offset (a prefix sum
// of a + K over the sequences before it), its row count and, with its positions, its largest
// position; every padded row then finds its compacted index directly and writes the
// prologue's per-row metadata in the same pass.  Sequences are taken kStepSeqChunk at a time,
// one thread each.
constexpr int kStepPrologueThreads = 512;
constexpr int kStepSeqChunk = kStepPrologueThreads;

// Inputs of one padded row that do not depend on the accepted counts (loaded before the
// counts are known, so that they share a round trip with them).
struct StepRowIn {
  int tok_ctx, pos_own, bonus;
};

PE_DEV StepRowIn step_row_inputs(const PrepArgs& a, int row, int r1, int K, int S) {
  StepRowIn in{0, 0, 0};
  if (row >= r1) return in;
  const int bb = row / S, r = row - bb * S;
  if (r < K) in.tok_ctx = a.prev_tokens[(size_t)bb * (K + 1) + r + 1];
  if (r <= K) {
    in.pos_own = a.prev_pos[(size_t)bb * (K + 1) + r];
    in.bonus = a.bonus[bb];
  }
  return in;
}

// One padded row of the rebuilt batch and, for a valid row, its compacted entry and the
// prologue's per-row metadata.  acc_s / base_s / ppac_s: the row's sequence's accepted
// count, first compacted row and NTP position (index bb - c0).
PE_DEV void step_write_row(const PrepArgs& a, const InitArgs& ia, int row, const StepRowIn& in, int c0,
                           const int* acc_s, const int* base_s, const int* ppac_s) {
  const int K = a.K, S = 2 * K;
  const int bb = row / S, r = row - bb * S, li = bb - c0;
  const int ac = acc_s[li];
  int tok, pos, hmap, rej = 0, msk = 0, draft_k = -1;
  if (r < ac) {          // accepted context row: token at p+1, hidden state of p
    tok = in.tok_ctx;
    pos = in.pos_own;
    hmap = bb * (K + 1) + r;
  } else if (r == ac) {  // NTP row: bonus token with h_context
    tok = in.bonus;
    pos = in.pos_own;
    hmap = bb * (K + 1) + ac;
    draft_k = 0;
  } else if (r <= K) {   // rejected draft position
    tok = 0;
    pos = in.pos_own;
    hmap = bb * (K + 1) + r;
    rej = 1;
  } else {               // MASK slot m = r - K
    const int m = r - K;
    tok = a.vocab;
    pos = ppac_s[li] + m;
    hmap = -1;
    msk = 1;
    draft_k = m;
  }
  if (!msk && (tok < 0 || tok >= a.vocab)) set_err(a.err, PE_DEV_BAD_TOKEN);
  long long slot = -1;
  if (!rej) {
    const int pi = pos / a.page_size;
    if (pos < 0 || pi >= a.max_pages) {
      set_err(a.err, PE_DEV_BAD_POSITION);
    } else {
      const int page = a.block_table[(size_t)bb * a.max_pages + pi];
      if (page < 0 || page >= a.num_pages) set_err(a.err, PE_DEV_BAD_PAGE);
      else slot = (long long)page * a.page_size + pos % a.page_size;
    }
  }
  a.input_ids[row] = tok;
  a.positions[row] = pos;
  a.slot_mapping[row] = slot;
  a.is_rejected[row] = (uint8_t)rej;
  a.is_mask[row] = (uint8_t)msk;
  a.hidden_map[row] = hmap;
  if (!rej) {
    const int idx = base_s[li] + (r <= ac ? r : r - (K - ac));
    a.row_list[idx] = row;
    if (draft_k >= 0) a.draft_rows[bb * K + draft_k] = idx;
    ia.tok_pos[idx] = pos;
    ia.tok_slot[idx] = slot;
    ia.tok_seq[idx] = bb;
  }
}

constexpr int kStepRowsPf = 2;  // rows per thread whose inputs are loaded with the accepted counts

PE_DEV void step_meta_body(const PrepArgs& a, const InitArgs& ia) {
  __shared__ int warp_s[33];
  __shared__ int acc_s[kStepSeqChunk], base_s[kStepSeqChunk], ppac_s[kStepSeqChunk];
  __shared__ int ib_s[kStepSeqChunk], nc_s[kStepSeqChunk], rng_s[kStepSeqChunk];
  __shared__ long long len_s[kStepPrologueThreads / 32];
  __shared__ int chunk_s;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int K = a.K, S = 2 * K, R = a.B * S;
  const bool one_chunk = a.B <= kStepSeqChunk;  // every sequence has a thread of its own
  for (int i = tid; i < ia.n_counters; i += NT) ia.counters[i] = 0;
  for (int i = tid; i < ia.T; i += NT) ia.keys[i] = 0ull;
  int carry = 0;           // compacted rows of the sequences before the chunk (the same in every thread)
  long long len_part = 0;  // this thread's share of the summed causal ranges
  int my_range = 0;        // (one chunk) the causal range of this thread's sequence: largest position + 1
  for (int c0 = 0; c0 < a.B; c0 += kStepSeqChunk) {
    const int b = c0 + tid;
    const bool own = tid < kStepSeqChunk && b < a.B;
    const int r0 = c0 * S, r1 = min(a.B, c0 + kStepSeqChunk) * S;
    // one round trip for everything that does not depend on the accepted counts: the
    // sequence's count and first eight positions, and the inputs of this thread's first rows
    const int32_t* pp = a.prev_pos + (size_t)b * (K + 1);
    int acc = own ? a.num_accepted[b] : 0;
    int pv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pv[k] = (own && k <= K) ? pp[k] : 0;
    StepRowIn rin[kStepRowsPf];
#pragma unroll
    for (int j = 0; j < kStepRowsPf; ++j) rin[j] = step_row_inputs(a, r0 + tid + j * NT, r1, K, S);
    if (own && (acc < 0 || acc > K)) {
      set_err(a.err, PE_DEV_BAD_ACCEPTED);
      acc = acc < 0 ? 0 : K;
    }
    int total = 0;
    const int excl = block_exclusive_scan(own ? acc + K : 0, warp_s, total);
    if (own) {
      // the largest and smallest positions of the sequence's valid rows: its context rows
      // (0..a-1), its NTP row (a) and the MASK rows after it (the last at NTP + K - 1)
      int ppa = pv[0], mx = INT_MIN, mn = INT_MAX;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k == acc) ppa = pv[k];
        if (k < acc) {
          mx = max(mx, pv[k]);
          mn = min(mn, pv[k]);
        }
      }
      if (acc >= 8) ppa = pp[acc];
      for (int r8 = 8; r8 < acc; r8 += 8) {  // more than eight context rows (K > 8)
        int v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = r8 + k < acc ? pp[r8 + k] : ppa;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mx = max(mx, v[k]);
          mn = min(mn, v[k]);
        }
      }
      mx = max(mx, ppa + K - 1);
      mn = min(mn, ppa);
      acc_s[tid] = acc;
      base_s[tid] = carry + excl;
      ppac_s[tid] = ppa;
      ia.seq_start[b] = carry + excl;
      ia.seq_len[b] = acc + K;
      ia.seq_maxpos[b] = mx;
      ia.seq_minpos[b] = mn;
      len_part += (long long)mx + 1;
      my_range = mx + 1;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kStepRowsPf; ++j) {
      const int row = r0 + tid + j * NT;
      if (row < r1) step_write_row(a, ia, row, rin[j], c0, acc_s, base_s, ppac_s);
    }
    for (int row = r0 + tid + kStepRowsPf * NT; row < r1; row += NT)
      step_write_row(a, ia, row, step_row_inputs(a, row, r1, K, S), c0, acc_s, base_s, ppac_s);
    carry += total;
    __syncthreads();  // acc_s / base_s / ppac_s are refilled by the next chunk
  }
  if (tid == 0) *a.n_valid = carry;
  for (int i = carry + tid; i < R; i += NT) {
    a.row_list[i] = -1;
    ia.tok_pos[i] = 0;
    ia.tok_slot[i] = -1;
    ia.tok_seq[i] = 0;
  }
  // attention work list, as the prologue builds it: the chunk length from the summed causal
  // ranges, then per sequence its chunk count and item offset (a prefix sum in sequence order)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) len_part += __shfl_xor_sync(0xFFFFFFFFu, len_part, o);
  if ((tid & 31) == 0) len_s[tid >> 5] = len_part;
  __syncthreads();
  if (tid == 0) {
    long long tot = 0;
    for (int w = 0; w < NT / 32; ++w) tot += len_s[w];
    long long per = (tot * ia.n_kv + ia.target_items - 1) / ia.target_items;
    per = ((per + 63) / 64) * 64;
    chunk_s = (int)(per < ia.min_chunk ? ia.min_chunk : per);
  }
  __syncthreads();
  const int chunk = chunk_s;
  int items = 0;
  for (int c0 = 0; c0 < a.B; c0 += kStepSeqChunk) {
    const int b = c0 + tid;
    const bool own = tid < kStepSeqChunk && b < a.B;
    const int range = own ? (one_chunk ? my_range : ia.seq_maxpos[b] + 1) : 0;
    const int nc = (range + chunk - 1) / chunk;
    int total = 0;
    const int excl = block_exclusive_scan(nc * ia.n_kv, warp_s, total);
    if (own) {
      ia.n_chunks[b] = nc;
      ia.item_base[b] = items + excl;
      ib_s[tid] = excl;  // read only with one chunk (items is then 0 here)
      nc_s[tid] = nc;
      rng_s[tid] = range;
    }
    items += total;
  }
  if (items > ia.max_items) {  // cannot happen with the host's sizing; keep the list in bounds
    if (tid == 0) set_err(ia.err, PE_DEV_BAD_ROW);
    items = 0;
  }
  if (tid == 0) *ia.n_items = items;
  if (items == 0) return;
  if (one_chunk) {
    // every thread writes items: item i belongs to the last sequence whose first item is at
    // most i (every sequence has at least n_kv items, so the first items increase)
    __syncthreads();
    for (int i = tid; i < items; i += NT) {
      int lo = 0, hi = a.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ib_s[mid] <= i) lo = mid;
        else hi = mid - 1;
      }
      const int k = i - ib_s[lo], nc = nc_s[lo];
      const int g = k / nc, c = k - g * nc;
      const int c0 = c * chunk;
      ia.items[i] = make_int4(lo, g, c0, min(c0 + chunk, rng_s[lo]));
    }
    return;
  }
  for (int b = tid; b < a.B; b += NT) {
    const int L = ia.seq_maxpos[b] + 1;
    const int nc = ia.n_chunks[b];
    int it = ia.item_base[b];
    for (int g = 0; g < ia.n_kv; ++g)
      for (int c = 0; c < nc; ++c) {
        const int c0 = c * chunk;
        const int c1 = c0 + chunk < L ? c0 + chunk : L;
        ia.items[it++] = make_int4(b, g, c0, c1);
      }
  }
}

// pe_step's first launch: the batch rebuild, the input rows and the forward prologue.  The
// last CTA rebuilds the batch (metadata, compaction) and then builds the prologue from it;
// every other CTA copies up to RPC input rows of one sequence, finding where they land from
// the accepted counts alone (the rows of the sequences before it), so no CTA waits for the
// rebuild.
__global__ void __launch_bounds__(kStepPrologueThreads)
    step_prologue_kernel(const PrepArgs pa, const ScatterArgs sa, const InitArgs ia, int groups) {
  __shared__ int part_s[kStepPrologueThreads / 32];
  // the input-row CTAs warm the weights' translations; the metadata CTA (the last) is the
  // longest and leaves them out
  if (blockIdx.x != gridDim.x - 1) warm_weight_translations(ia, gridDim.x - 1);
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == gridDim.x - 1) {
    step_meta_body(pa, ia);
    return;
  }
  const int b = blockIdx.x / groups, grp = blockIdx.x - b * groups;
  int part = 0;  // valid rows of sequences 0 .. b-1, each a + K (a clamped to [0, K])
  for (int bb = threadIdx.x; bb < b; bb += blockDim.x) {
    const int x = pa.num_accepted[bb];
    part += (x < 0 ? 0 : (x > pa.K ? pa.K : x)) + pa.K;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
  if ((threadIdx.x & 31) == 0) part_s[threadIdx.x >> 5] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    int base = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) base += part_s[w];
    scatter_seq_body(pa, sa, b, grp, base);
  }
}

cudaError_t launch_step_prologue(const PrepArgs& pa, const ScatterArgs& sa, const InitArgs& ia, cudaStream_t s) {
  const size_t smem = scatter_smem_bytes(sa.d, sa.elem_bytes);
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(step_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kScatterSmemMax);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int groups = (2 * pa.K + kScatterRowsPerCta - 1) / kScatterRowsPerCta;  // a + K <= 2K rows per sequence
  const int grid = pa.B * groups + 1;
  return launch_pdl(step_prologue_kernel, dim3(grid), dim3(kStepPrologueThreads), smem, s, pa, sa, ia, groups);
}

// ============================================================================= RMSNorm
// y = x / sqrt(mean(x^2) + eps) * g.  One CTA per row; the row stays in
// registers between the sum of squares and the scaling; the sum runs in a
// fixed order (per-thread partials, warp butterflies, then warp totals in
// warp order), so the result does not depend on scheduling.

constexpr int kNormThreads = 256;

template <typename OutT>
PE_DEV void store4(OutT* y, float a, float b, float c, float d);
template <>
PE_DEV void store4<float>(float* y, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(y) = make_float4(a, b, c, d);
}
template <>
PE_DEV void store4<__nv_bfloat16>(__nv_bfloat16* y, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 v;
  v.x = *reinterpret_cast<uint32_t*>(&lo);
  v.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(y) = v;
}

constexpr int kNormMaxSplits = 16;  // split-K ways a GEMM may leave to the norm

// MS: the most split-K partials the producing GEMM may have left to sum (8 or 16; 0: none).
// The partial loads in flight take KC * MS float4 registers (128 registers): with at most 8
// splits a thread's four float4 groups load in one round trip instead of two.  The
// instantiation without partials keeps the register count low (several CTAs fit on an SM,
// and a many-row norm runs in one wave).
template <typename OutT, typename GT, int VPT, int MS>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const NormArgs a) {
  constexpr bool SPLIT = MS > 0;
  __shared__ float warp_ss[kNormThreads / 32];
  const int row = blockIdx.x, tid = threadIdx.x;
  const int nv = a.d / 4;
  // the gains are weights: load them before waiting for the previous kernel
  float gn[VPT][4];
  const GT* g = static_cast<const GT*>(a.g);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int j = tid + k * kNormThreads;
#pragma unroll
    for (int e = 0; e < 4; ++e) gn[k][e] = j < nv ? to_float<GT>(g[4 * j + e]) : 0.f;
  }
  // every count / index this row needs, in one round trip (before the dependency wait when
  // the kernel that wrote them has completed by the time this one starts)
  if (!a.meta_ready) pdl_wait();
  const int dev_n = a.n_rows_dev != nullptr ? __ldcg(a.n_rows_dev) : a.n_rows;
  const int dev_g = !SPLIT ? 0
                    : (a.g_ntok_dev == nullptr ? a.g_ntok
                       : (a.g_ntok_dev == a.n_rows_dev ? dev_n : __ldcg(a.g_ntok_dev)));
  const int mapped = a.row_map != nullptr ? __ldcg(a.row_map + row) : row;
  if (a.meta_ready) pdl_wait();
  pdl_trigger();
  const int n = min(a.n_rows, dev_n);
  if (row >= n) return;
  const int src = mapped;
  if (a.row_map != nullptr && (src < 0 || src >= a.src_rows)) {
    if (tid == 0) set_err(a.err, PE_DEV_BAD_ROW);
    return;
  }
  float4 v[VPT];
  float ss = 0.f;
  if constexpr (SPLIT) {
    // x_new = x + the producing GEMM's split-K partials (split order).  Units are numbered
    // as the GEMM numbers them over its live token tiles: ((tile_f * ntl + tile_t) * splits + split).
    const int n_eff = min(a.g_ntok, max(dev_g, a.g_ntok_min));
    const int ntl = min(a.n_t, (n_eff + a.bn - 1) / a.bn);
    const int tile_t = src / a.bn, tt = src - tile_t * a.bn;
    const size_t tile_floats = (size_t)a.bn * 128;
    constexpr int KC0 = MS <= 8 ? 4 : 2;
    constexpr int KC = VPT < KC0 ? VPT : KC0;  // groups of four features whose loads are in flight together
#pragma unroll
    for (int k0 = 0; k0 < VPT; k0 += KC) {
      float4 q[KC][MS > 0 ? MS : 1];
#pragma unroll
      for (int kc = 0; kc < KC; ++kc) {
        const int k = k0 + kc, j = tid + k * kNormThreads;
        v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < nv) {
          if (a.x != nullptr) v[k] = reinterpret_cast<const float4*>(a.x + (size_t)src * a.d)[j];
          const int f = 4 * j, tile_f = f >> 7;
          const float* p = a.part + ((size_t)(tile_f * ntl + tile_t) * a.n_splits) * tile_floats +
                           (size_t)tt * 128 + (f & 127);
#pragma unroll
          for (int sp = 0; sp < MS; ++sp)
            if (sp < a.n_splits) q[kc][sp] = __ldcg(reinterpret_cast<const float4*>(p + (size_t)sp * tile_floats));
        }
      }
#pragma unroll
      for (int kc = 0; kc < KC; ++kc) {
        const int k = k0 + kc, j = tid + k * kNormThreads;
        if (j < nv) {
#pragma unroll
          for (int sp = 0; sp < MS; ++sp)  // split order
            if (sp < a.n_splits) {
              v[k].x += q[kc][sp].x; v[k].y += q[kc][sp].y; v[k].z += q[kc][sp].z; v[k].w += q[kc][sp].w;
            }
          if (a.x_out != nullptr) reinterpret_cast<float4*>(a.x_out + (size_t)src * a.d)[j] = v[k];
        }
      }
    }
  } else {
    const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)src * a.d);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * kNormThreads;
      v[k] = j < nv ? xr[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    ss += v[k].x * v[k].x;
    ss += v[k].y * v[k].y;
    ss += v[k].z * v[k].z;
    ss += v[k].w * v[k].w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if ((tid & 31) == 0) warp_ss[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += warp_ss[w];
  const float inv = 1.0f / sqrtf(tot / (float)a.d + a.eps);
  OutT* y = static_cast<OutT*>(a.y) + (size_t)row * a.d;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int j = tid + k * kNormThreads;
    if (j < nv)
      store4<OutT>(y + 4 * j, v[k].x * inv * gn[k][0], v[k].y * inv * gn[k][1], v[k].z * inv * gn[k][2],
                   v[k].w * inv * gn[k][3]);
  }
}

template <typename OutT, typename GT, int SPLIT>
static cudaError_t launch_norm_typed(const NormArgs& a, cudaStream_t s) {
  const int per = (a.d / 4 + kNormThreads - 1) / kNormThreads;  // float4 per thread
  const dim3 grid(a.n_rows), block(kNormThreads);
  if (per <= 1) return launch_pdl(rmsnorm_kernel<OutT, GT, 1, SPLIT>, grid, block, 0, s, a);
  if (per <= 2) return launch_pdl(rmsnorm_kernel<OutT, GT, 2, SPLIT>, grid, block, 0, s, a);
  if (per <= 4) return launch_pdl(rmsnorm_kernel<OutT, GT, 4, SPLIT>, grid, block, 0, s, a);
  if (per <= 8) return launch_pdl(rmsnorm_kernel<OutT, GT, 8, SPLIT>, grid, block, 0, s, a);
  if (per <= 16) return launch_pdl(rmsnorm_kernel<OutT, GT, 16, SPLIT>, grid, block, 0, s, a);
  return cudaErrorInvalidValue;  // d > 16384 is rejected by the config check
}

cudaError_t launch_rmsnorm(const NormArgs& a, pe_dtype dt, cudaStream_t s) {
  if (a.n_rows == 0) return cudaSuccess;
  if (a.n_splits > kNormMaxSplits) return cudaErrorInvalidValue;
  if (a.n_splits > 8) {
    if (dt == PE_BF16) return launch_norm_typed<__nv_bfloat16, __nv_bfloat16, kNormMaxSplits>(a, s);
    return launch_norm_typed<float, float, kNormMaxSplits>(a, s);
  }
  if (a.n_splits > 0) {
    if (dt == PE_BF16) return launch_norm_typed<__nv_bfloat16, __nv_bfloat16, 8>(a, s);
    return launch_norm_typed<float, float, 8>(a, s);
  }
  if (dt == PE_BF16) return launch_norm_typed<__nv_bfloat16, __nv_bfloat16, 0>(a, s);
  return launch_norm_typed<float, float, 0>(a, s);
}

}  // namespace pe
