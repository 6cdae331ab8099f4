// Internal interface between the C-ABI layer (pe_api.cu) and the kernels.
// Every struct is passed to a kernel by value; every pointer is a device pointer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pe.h"

namespace pe {

// Counts every kernel launch of the library (reported by pe_kernel_launches).
void count_launch(int n = 1);

// Programmatic dependent launch on (default on; PE_PDL=0 in the environment turns it off).
bool pdl_enabled();

// Limit of every bounded pipeline wait in the kernels launched from now on (pe_set_wait_limit_ns).
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
uint64_t wait_limit_ns();
// The pipeline stage the next tensor-core GEMM launch leaves unarmed in CTA 0, then -1 again
// (pe_test_skip_pipeline_stage); -1: none.
int take_drop_stage();

// Launch with the programmatic-stream-serialization attribute so the kernel's
// prologue may overlap the previous kernel's tail (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ----------------------------------------------------------------------------- batch metadata

struct PrepArgs {
  int B, K, vocab, max_pages, num_pages, page_size;
  const int32_t *prev_tokens, *prev_pos, *num_accepted, *bonus, *block_table;
  int32_t *input_ids, *positions;
  int64_t* slot_mapping;
  uint8_t *is_rejected, *is_mask;
  int32_t *hidden_map, *row_list, *n_valid, *draft_rows, *err;
};
cudaError_t launch_prepare(const PrepArgs& a, cudaStream_t s);

struct ScatterArgs {
  int R, d, elem_bytes, vocab, n_hidden;
  const void *emb, *h_shared, *hidden;
  const int32_t* input_ids;
  const uint8_t* is_mask;
  const int32_t *hidden_map, *row_list, *n_valid;
  void* x0;
  int32_t* err;
};
cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t s);
// Shared memory of one input-row CTA (its rows' embedding and hidden halves plus the
// MASK row); a config whose rows need more than kScatterSmemMax is rejected up front.
constexpr size_t kScatterSmemMax = 200 * 1024;
size_t scatter_smem_bytes(int d, int elem_bytes);

struct VerifyArgs {
  int B, K;
  const int32_t *draft, *target;
  int32_t *acc_out, *bonus_out;
  // optional: next round's verify batch (pe_step), built from the rebuilt batch of this
  // round (compacted row list, draft-row list, row positions and token ids) so that the
  // outputs may overwrite the caller's state arrays that the rebuild read
  const int32_t *row_list, *draft_rows, *positions, *input_ids;
  int32_t *next_tokens, *next_pos;
};
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s);

// Greedy verification of sequence b (vLLM Speculators: parallel drafting for
// speculative decoding, "Production integration in vLLM": the target's output is
// preserved): the longest prefix of drafts equal to the target's tokens, then the
// target's token at the first mismatch as the bonus; optionally the next round's
// verify batch [bonus, drafts] at the positions after the NTP position.  The NTP
// row (the first draft row: the bonus token at the last accepted position) is read
// from the rebuilt batch, never from the previous round's state arrays.
__device__ __forceinline__ void verify_seq(const VerifyArgs& a, int b) {
  const int32_t* d = a.draft + (size_t)b * a.K;
  const int32_t* t = a.target + (size_t)b * (a.K + 1);
  int acc = 0;
  while (acc < a.K && d[acc] == t[acc]) ++acc;
  if (a.next_tokens != nullptr) {
    const int ntp = a.row_list[a.draft_rows[(size_t)b * a.K]];  // padded NTP row of sequence b
    const int p0 = a.positions[ntp] + 1;
    int32_t* nt = a.next_tokens + (size_t)b * (a.K + 1);
    int32_t* np = a.next_pos + (size_t)b * (a.K + 1);
    nt[0] = a.input_ids[ntp];
    for (int k = 0; k < a.K; ++k) nt[k + 1] = d[k];
    for (int j = 0; j <= a.K; ++j) np[j] = p0 + j;
  }
  a.acc_out[b] = acc;
  a.bonus_out[b] = t[acc];
}

// Non-greedy drafting and rejection-sampling verification; see pe_sample.cu.  Each
// draw over a vocabulary row keeps one statistic pair per 512 entries in the
// workspace (sample_stats_bytes).
struct SampleArgs {
  int B, K, V;
  const float* logits;  // [B*K][V]
  const float* u;       // [B*K] uniforms in [0, 1)
  float inv_t2;         // log2(e) / temperature
  float2* stats;        // workspace: [B*K][steps], one per 512 vocabulary entries
  int32_t* drafts;      // [B*K]
  float* lse;           // [B*K]
  int32_t* err;
};
cudaError_t launch_sample_drafts(const SampleArgs& a, int sms, cudaStream_t s);

struct VerifySampledArgs {
  int B, K, V;
  const int32_t* drafts;      // [B*K]
  const float *logits, *lse;  // [B*K][V], [B*K] (natural log)
  float inv_t2;               // log2(e) / temperature
  const float* target_probs;  // [B][K+1][V]
  const float *u_accept, *u_resample;  // [B*K], [B]
  float2* stats;              // workspace: [B][steps]
  int32_t* acc_ws;            // workspace: [B] accepted counts (statistics launch -> draw launch)
  int32_t *acc_out, *bonus_out;
  int32_t* err;
};
cudaError_t launch_verify_sampled(const VerifySampledArgs& a, int sms, cudaStream_t s);
size_t sample_stats_bytes(int rows, int vocab);

// Forward prologue: per compacted row metadata, per sequence ranges, the
// attention work list, and zeroing of the pass's counters and argmax keys.
constexpr int kWarmRanges = 17;  // fc and the four matrices of each of the first four layers
struct InitArgs {
  int B, K, R, T, n_kv;
  const int32_t *row_list, *n_valid, *positions;
  const int64_t* slot_mapping;
  int32_t *tok_pos, *tok_seq;
  int64_t* tok_slot;
  int32_t *seq_start, *seq_len, *seq_maxpos;
  int32_t* seq_minpos;       // smallest position of the sequence's valid rows (INT_MAX: none)
  int target_items, max_items, min_chunk;
  int4* items;
  int32_t *n_items, *item_base, *n_chunks;
  int32_t* counters;
  int n_counters;
  unsigned long long* keys;
  int32_t* err;
  // The round's layer weight matrices (fc, the first layers' four): the prologue touches
  // one line per 2 MB of each, so that their address translations are in place before the
  // GEMMs stream them (the first touch of each page otherwise stalls every GEMM's first loads).
  const uint8_t* warm_base[kWarmRanges];
  long long warm_bytes[kWarmRanges];
  int warm_n;
};
cudaError_t launch_forward_init(const InitArgs& a, cudaStream_t s);
// DFlash-style KV injection: position and cache slot of every element of the previous verify
// batch (hidden row i = b*(K+1) + j): slot -1 for j > num_accepted[b].
struct InjectArgs {
  int B, K, max_pages, num_pages, page_size;
  const int32_t *prev_pos, *num_accepted, *block_table;
  int32_t* tok_pos;
  int64_t* tok_slot;
  int32_t* err;
};
cudaError_t launch_inject_init(const InjectArgs& a, cudaStream_t s);
// pe_step's first launch: the batch rebuild (PrepArgs), the input rows (ScatterArgs, every
// CTA placing one sequence's rows itself) and the forward prologue (InitArgs).
cudaError_t launch_step_prologue(const PrepArgs& pa, const ScatterArgs& sa, const InitArgs& ia, cudaStream_t s);

// ----------------------------------------------------------------------------- RMSNorm

struct NormArgs {
  const float* x;            // residual stream [rows][d] fp32 (nullable when partials carry the whole value)
  int d;
  const int32_t* row_map;    // output row i reads x[row_map[i]] (nullable: identity)
  int n_rows;                // host upper bound of output rows
  const int32_t* n_rows_dev; // actual count (nullable)
  int src_rows;              // bound on source rows (device check)
  const void* g;             // gains [d], storage dtype
  float eps;
  void* y;                   // [rows][d], bf16 (bf16 configs) or fp32
  // Split-K partials of the GEMM that produced (or adds to) x, reduced here instead of in the
  // GEMM: x_new = x + sum of n_splits partials, in split order.  n_splits = 0: x as it is.
  const float* part;         // [units][bn][128] fp32, units numbered as the GEMM's (tile_f, tile_t, split)
  int n_splits, bn, n_t;     // the GEMM's splits, token tile and token tiles
  int g_ntok, g_ntok_min;    // the GEMM's token rows: host bound, rows that certainly exist
  const int32_t* g_ntok_dev; // the GEMM's device row count (nullable)
  float* x_out;              // nullable: where x_new is written ([rows][d], may alias x)
  int32_t* err;
  int meta_ready;            // the row counts and row map were written by a kernel that has completed
                             //   when this one starts: read them before the dependency wait
};
cudaError_t launch_rmsnorm(const NormArgs& a, pe_dtype dt, cudaStream_t s);

// ----------------------------------------------------------------------------- GEMM + fused epilogues

enum Epi : int {
  EPI_STORE_F32 = 0,  // x[t][f] = acc                 (fc)
  EPI_ADD_F32 = 1,    // x[t][f] += acc                (o-proj, down: residual add)
  EPI_SWIGLU = 2,     // u[t][f] = silu(gate) * up     (gate/up, paired rows)
  EPI_QKV_ROPE = 3,   // RoPE(q,k); q -> q buffer; k,v -> paged cache at the row's slot
  EPI_ARGMAX = 4,     // LM head: per-token max / argmax over the vocabulary
  EPI_ARGMAX_BAL = 5, // the same with equal k-block ranges per CTA (tensor-core kernel only)
};

struct GemmArgs {
  int n_out;             // output units: features; SwiGLU: F; QKV: (head, pair) units = heads*hd/2
  int k_dim;             // reduction length
  int n_tok;             // token rows (host upper bound)
  const int32_t* n_tok_dev;  // actual token rows (nullable)
  // tensor-core tiling (ignored by the fp32 kernel)
  int bn;                // token columns per tile (MMA N)
  int n_t, n_f;          // token tiles, weight tiles; work units = n_t * n_f * k_splits
  int n_tok_min;         // token rows that certainly exist (every tile below it is computed)
  int tok_major;         // units numbered token tile after token tile (weight tile fastest): a CTA's
                         // first weight tile is then known before the row count, and prefetched
  int kb_total, k_splits, stages;  // k stages over the whole K (each ka 64-wide atoms)
  int ka;                          // 64-wide k atoms per pipeline stage (1 or 2)
  uint32_t stage_bytes;
  int nbuf;              // TMEM accumulator buffers (2: epilogue overlaps the next unit's MMAs)
  int acc_stride;        // TMEM columns per accumulator buffer
  uint32_t tmem_cols;    // TMEM columns allocated (power of two >= 32)
  // fp32 kernel operands
  const void* W;         // [rows][k_dim]
  const void* X;         // [tokens][ldx]
  int ldx;
  // epilogue
  float* out_f32;        // residual stream [tokens][ld_out]
  void* out_act;         // SwiGLU output / q buffer (bf16 or fp32 by config)
  int ld_out;
  int n_q, n_kv, head_dim;
  int head0;             // QKV: heads of this GEMM start at head0 of the q | k | v concatenation (0; KV
                         //   injection: n_q, the GEMM covering the k and v heads only)
  // RoPE: turns per position of pair index i, theta^(-2i/head_dim) / (2 pi), split into
  // a float and the float nearest its remainder (i < head_dim / 2 <= 64)
  float rope_tf_hi[64], rope_tf_lo[64];
  const int32_t* tok_pos;
  const int64_t* tok_slot;
  void *k_cache, *v_cache;
  unsigned long long* keys;  // LM head: one key per token (zero before the launch)
  float* logits_dbg;         // nullable [tokens][n_out]
  int32_t* done_counter;     // LM head: CTAs finished (zero before the launch)
  float* partial;            // split K: [grid][planes][bn][128] fp32 partial tiles (column-major per plane)
  int32_t* tile_cnt;         // EPI_ARGMAX_BAL: [grid][8] arrivals per cut tile and epilogue warp (zero
                             //   before the launch); the pieces' partials go to `partial` as [grid][2][bn][128]
  int32_t* draft_out;        // LM head: argmax per token
  VerifyArgs verify;         // LM head: greedy verification of the drafts by the finishing CTA
  int has_verify;            //   (pe_step); 0: none
  uint64_t wait_ns;          // limit of every pipeline wait (wait_limit_ns())
  int drop_stage;            // test of the wait-expiry path: CTA 0 leaves this pipeline stage unarmed (-1: none)
  int32_t* err;
  int meta_ready;            // the row count was written by a kernel that has completed when this one
                             //   starts (every kernel from the first QKV GEMM on): read it before the
                             //   dependency wait
};

// Tensor-core GEMM (tcgen05 + TMA): D[f][t] = W[f][:] . X[t][:], weights on the MMA M side.
// Persistent: `grid` CTAs (at most one per SM) stride over the work units.  With
// k_splits > 1 every CTA (pair) owns exactly one unit and writes its fp32 partial tile to
// `partial`; the consumer sums the splits (RMSNorm, or launch_splitk_finish).
// cg = 2: clusters of two CTAs, each unit one MMA of M = 256 over the pair (grid even;
// the token operand's tensor map has boxes of bn / 2 rows); not for EPI_ARGMAX_BAL.
cudaError_t launch_gemm_tc(int epi, int cg, const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                           int grid, size_t smem_bytes, cudaStream_t s);
// Clusters of two CTAs of this GEMM epilogue with this much shared memory that fit on the
// GPU at once (0 if the query fails).
int gemm_tc_max_pairs(int epi, size_t smem_bytes);
// Sum of a split-K QKV or gate/up GEMM's partials and its epilogue (the same GemmArgs).
cudaError_t launch_splitk_finish(int epi, const GemmArgs& a, int sms, cudaStream_t s);
// fp32 CUDA-core GEMM for fp32 configurations (same epilogues).
cudaError_t launch_gemm_f32(int epi, const GemmArgs& a, cudaStream_t s);

constexpr int kTcEpiWarps = 8;         // at most: two per TMEM lane quarter, each taking half of the token columns
constexpr int kTcThreads = 64 + 32 * kTcEpiWarps;  // warp 0: TMA, warp 1: MMA, warps 2-9: epilogue
// Threads of a tensor-core GEMM launch: eight epilogue warps for token tiles of at least 64
// columns, four (one per lane quarter) for narrower ones, whose epilogue is a chunk or two.
constexpr int gemm_tc_threads(int bn) { return bn >= 64 ? kTcThreads : 64 + 32 * 4; }
constexpr int kTcBM = 128;             // weight rows per tile
constexpr int kTcBK = 64;              // k per atom (one 128-byte swizzle row); a stage holds 1 or 2 atoms
constexpr int kTcCtrlBytes = 1024;     // barriers + TMEM slot + flags
constexpr int kTcSmemOptIn = 232448;   // largest dynamic shared memory per block (227 KB)
// dynamic shared memory: alignment slack + stage ring + control block + argmax keys (4 warps * n_t * bn)
size_t gemm_tc_smem_bytes(int stages, uint32_t stage_bytes, int red_entries);

// ----------------------------------------------------------------------------- attention

struct AttnArgs {
  int B, n_q, n_kv, head_dim, max_pages, page_size, num_pages;
  float scale;               // 1/sqrt(head_dim)
  const void* q;             // [rows][n_q*hd], post-RoPE
  const void *k_cache, *v_cache;
  const int32_t* block_table;
  const int32_t *tok_pos, *tok_seq, *seq_start, *seq_len, *n_valid;
  // smallest position of each sequence's rows: every k / v this round writes for the
  // sequence lies at or after it, so cache pages wholly below it may be read before the
  // kernel that writes the new rows has finished
  const int32_t* seq_minpos;
  const int4* items;         // (b, g, c0, c1)
  const int32_t *n_items, *item_base, *n_chunks;
  float *part_m, *part_l, *part_o;  // [items][128], [items][128], [items][128][hd]
  int32_t* work_counter;     // items handed out so far (zero before the launch)
  void* out;                 // [rows][n_q*hd]
  int n_rows;                // host upper bound on rows
  uint64_t wait_ns;          // limit of every pipeline wait (wait_limit_ns())
  int32_t* err;
};
constexpr int kAttnRows = 128;    // query rows (row x GQA head) per work item
// tmK / tmV: the layer's K and V pools as bf16 [num_pages*16][n_kv][hd], 128-byte swizzle, box 64 x 1 x 16.
// Launches the attention kernel (`grid` CTAs) and then the chunk merge.
cudaError_t launch_attention_bf16(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a, int grid,
                                  int sms, cudaStream_t s);
cudaError_t launch_attention_f32(const AttnArgs& a, cudaStream_t s);

}  // namespace pe
