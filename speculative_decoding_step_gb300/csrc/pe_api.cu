// C ABI of the P-EAGLE drafting round: argument validation, the workspace
// plan, TMA descriptors and the launch sequence of every stage.  Nothing here
// allocates device memory or synchronises the stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "pe_internal.h"

namespace pe {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("PE_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return on;
}

static std::atomic<uint64_t> g_wait_ns{0};    // 0: the kernels' default limit
static std::atomic<int> g_drop_stage{-1};
uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_ns.load(std::memory_order_relaxed);
  return v == 0 ? kDefaultWaitNs : v;
}
int take_drop_stage() { return g_drop_stage.exchange(-1, std::memory_order_relaxed); }

namespace {

// Caller-created events recorded at stage boundaries (tracing).
std::mutex g_trace_mu;
std::vector<cudaEvent_t> g_trace;

void trace(int point, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (point >= 0 && point < (int)g_trace.size()) cudaEventRecord(g_trace[point], s);
}

constexpr int kMaxRows = 1 << 16;        // B*2K
constexpr int kAttnItemsPerSlot = 4;     // attention work items aimed for, per resident CTA (load balance)
constexpr int kAttnMinChunk = 256;       // shortest position chunk of a work item (bounds the chunks to merge)
constexpr int kTcMaxStages = 12;
constexpr int kMinStagesKa2 = 3;        // ring depth below which a stage keeps one k atom
constexpr int kMaxSplits = 16;           // split-K ways per tile (the RMSNorm that sums deferred partials takes up to 16)

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Clusters of two GEMM CTAs (about 200 KB of shared memory each, one per SM) that fit on
// the GPU at once: fewer than half the SMs when a GPU processing cluster has an odd number
// of SMs.  Without a device (host-only use of the plan): half the SMs.
int max_pairs(int sms) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return sms / 2;
  if (cached[dev] == 0) {
    const int n = gemm_tc_max_pairs(EPI_ADD_F32, (size_t)kTcSmemOptIn);
    cached[dev] = n > 0 ? std::min(n, sms / 2) : sms / 2;
  }
  return cached[dev];
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int round_up(int x, int m) { return (x + m - 1) / m * m; }
size_t elem_bytes(pe_dtype dt) { return dt == PE_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ----------------------------------------------------------------------------- GEMM plan

struct GemmPlan {
  int epi = 0, bn = 16, n_t = 1, n_f = 1, k_splits = 1, kb_total = 1, stages = 2, grid = 1;
  int cg = 1;  // CTAs per MMA: 2 = CTA pairs (M = 256), each taking in half the token operand
  int nbuf = 1, acc_stride = 16;
  int balanced = 0;
  int ka = 1;  // 64-wide k atoms per stage
  uint32_t tmem_cols = 32;
  uint32_t stage_bytes = 0;
  size_t smem = 0;
  int tiles = 0;
};

// Work decomposition of one GEMM: 128 weight rows x bn token rows per tile.
// With fewer tiles than SMs, split K so that nearly every SM streams weights:
// every CTA owns exactly one unit and leaves an fp32 partial tile for the
// consumer to sum; each split keeps at least four 64-wide k blocks.
//
// Many token rows (more than one 256-row tile), or an LM head whose token tile is at
// least 128 rows: CTA pairs (cg = 2).  The GEMM is then bound by how fast each SM takes
// in its operands (measured: about 95 GB/s per SM from L2 with 32 KB boxes), not by the
// tensor pipe: a pair's MMA of 256 weight rows has each CTA take in 128 weight rows and
// half of the token tile, a quarter less per flop at 128 tokens than one CTA's 128 x 128
// tile.  Layer GEMMs then use 128-token tiles (64 rows per CTA), which keeps enough units
// to fill the GPU at B = 64.  `max_pairs`: clusters of two that fit on the GPU at once.
GemmPlan plan_gemm(int epi, int n_f_tiles, int n_tok, int k_dim, int sms, int max_pairs) {
  GemmPlan g;
  g.epi = epi;
  const bool paired = (epi == EPI_SWIGLU || epi == EPI_QKV_ROPE);
  if (n_tok <= 256 || epi == EPI_ARGMAX) {  // one token tile, or the LM head (vocabulary tiles are plenty)
    g.n_t = (n_tok + 255) / 256;
    g.bn = round_up((n_tok + g.n_t - 1) / g.n_t, 16);
    g.cg = (epi == EPI_ARGMAX && g.bn >= 128) ? 2 : 1;
  } else {  // many rows: 128-row token tiles give enough units to fill the GPU without split K
    g.bn = 128;
    g.n_t = (n_tok + g.bn - 1) / g.bn;
    g.cg = 2;
  }
  const int slots = g.cg == 2 ? std::max(1, max_pairs) : sms;  // units that run at once
  g.n_f = n_f_tiles;
  g.tiles = g.n_f * g.n_t;
  const int unit_tiles = ((g.n_f + g.cg - 1) / g.cg) * g.n_t;  // work units per k split
  // epilogue scratch after the ring, in 8-byte words: the LM head's per-warp keys, or the
  // QKV epilogue's token positions and slots (two buffers of bn x 12 bytes)
  const int red = epi == EPI_ARGMAX ? 4 * g.n_t * g.bn : (epi == EPI_QKV_ROPE ? 3 * g.bn : 0);
  const long long avail = kTcSmemOptIn - 1024 - kTcCtrlBytes - (long long)red * 8;
  // Two k atoms per stage (one TMA box of both per operand: half the boxes per byte, half
  // the barrier round trips per MMA) while the ring still holds kMinStagesKa2 stages.
  const int bnl = g.bn / g.cg;  // token rows a CTA loads
  auto stage_bytes = [&](int ka) {
    return (uint32_t)ka * ((paired ? 2u : 1u) * kTcBM * kTcBK * 2 + (uint32_t)bnl * kTcBK * 2);
  };
  g.ka = avail / stage_bytes(2) >= kMinStagesKa2 ? 2 : 1;
  const int atoms = (k_dim + kTcBK - 1) / kTcBK;
  g.kb_total = (atoms + g.ka - 1) / g.ka;  // the last stage's second atom may lie past K: zeros
  g.stage_bytes = stage_bytes(g.ka);
  g.stages = (int)std::min<long long>(kTcMaxStages, avail / g.stage_bytes);
  g.smem = gemm_tc_smem_bytes(g.stages, g.stage_bytes, red);
  if (epi != EPI_ARGMAX && unit_tiles < slots)
    g.k_splits = std::max(1, std::min(kMaxSplits, std::min(slots / unit_tiles, g.kb_total * g.ka / 4)));
  const int acc_cols = (paired ? 2 : 1) * g.bn;
  g.nbuf = 2 * acc_cols <= 512 ? 2 : 1;
  g.acc_stride = acc_cols;
  const int need = g.nbuf * acc_cols;
  g.tmem_cols = need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
  const int units = unit_tiles * g.k_splits;
  g.grid = g.cg * (g.k_splits > 1 ? units : std::min(units, slots));
  // LM head with one token tile: equal k-block ranges per CTA when the last wave of
  // vocabulary tiles is at most three quarters full (a range then spans more than a
  // tile).  One SM streams at most about 53 GB/s (measured), little above its
  // 1/152 share of HBM bandwidth, so a last wave of n CTAs runs at about n/152 of
  // the HBM rate; a nearly full last wave costs less than exchanging the partial
  // sums of the cut tiles.
  const int last_wave = g.tiles % sms;
  if (epi == EPI_ARGMAX && g.cg == 1 && g.n_t == 1 && g.tiles > sms && last_wave != 0 && 4 * last_wave <= 3 * sms)
    g.balanced = 1;
  return g;
}

struct Plan {
  int R = 0, T = 0, S = 0, sms = 0, max_items = 0, attn_grid = 0, attn_target = 0, n_counters = 0;
  GemmPlan fc, qkv, o, gu, down, lm;
  GemmPlan inj, injkv;  // KV injection: W_inj over the verify batch's hidden rows, then the k | v heads
  // workspace offsets
  size_t tok_pos, tok_seq, tok_slot, seq_start, seq_len, seq_maxpos, seq_minpos, item_base, n_chunks, n_items, items;
  size_t done, keys, x, y, q, ao, u, yl, part_m, part_l, part_o, split_part;
  size_t st_ids, st_pos, st_slot, st_rej, st_mask, st_hmap, st_rows, st_nvalid, st_draft, st_x0;
  size_t samp, samp_acc;
  size_t total = 0;
};

Plan make_plan(const pe_config& c) {
  Plan p;
  p.S = 2 * c.K;
  p.R = c.B * p.S;
  p.T = c.B * c.K;
  p.sms = num_sms();
  const int half = c.head_dim / 2;
  const int heads = c.n_q + 2 * c.n_kv;
  const int hpt = kTcBM / half;
  const int mp = c.dtype == PE_BF16 ? max_pairs(p.sms) : 0;
  p.fc = plan_gemm(EPI_STORE_F32, (c.d + kTcBM - 1) / kTcBM, p.R, 2 * c.d, p.sms, mp);
  p.qkv = plan_gemm(EPI_QKV_ROPE, (heads + hpt - 1) / hpt, p.R, c.d, p.sms, mp);
  p.o = plan_gemm(EPI_ADD_F32, (c.d + kTcBM - 1) / kTcBM, p.R, c.n_q * c.head_dim, p.sms, mp);
  p.gu = plan_gemm(EPI_SWIGLU, (c.ffn + kTcBM - 1) / kTcBM, p.R, c.d, p.sms, mp);
  p.down = plan_gemm(EPI_ADD_F32, (c.d + kTcBM - 1) / kTcBM, p.R, c.ffn, p.sms, mp);
  p.lm = plan_gemm(EPI_ARGMAX, (c.vocab + kTcBM - 1) / kTcBM, p.T, c.d, p.sms, mp);
  const int n_inj = c.B * (c.K + 1);
  p.inj = plan_gemm(EPI_STORE_F32, (c.d + kTcBM - 1) / kTcBM, n_inj, c.d, p.sms, mp);
  p.injkv = plan_gemm(EPI_QKV_ROPE, (2 * c.n_kv + hpt - 1) / hpt, n_inj, c.d, p.sms, mp);
  // attention items: the work list aims at attn_target items; rounding adds at
  // most one per (sequence, kv head), and no (sequence, kv head) can have more
  // chunks than its longest possible range holds minimum chunks
  const int attn_slots = 2 * p.sms;  // resident attention CTAs (two per SM)
  p.attn_target = kAttnItemsPerSlot * attn_slots;
  const long long per_pair = ((long long)c.max_pages_per_seq * c.page_size + kAttnMinChunk - 1) / kAttnMinChunk;
  p.max_items = (int)std::min<long long>(p.attn_target + (long long)c.B * c.n_kv, per_pair * c.B * c.n_kv);
  p.attn_grid = std::min(p.max_items, attn_slots);

  const size_t eb = elem_bytes(c.dtype);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  p.tok_pos = take(4 * (size_t)p.R);
  p.tok_seq = take(4 * (size_t)p.R);
  p.tok_slot = take(8 * (size_t)p.R);
  p.seq_start = take(4 * (size_t)c.B);
  p.seq_len = take(4 * (size_t)c.B);
  p.seq_maxpos = take(4 * (size_t)c.B);
  p.seq_minpos = take(4 * (size_t)c.B);
  p.item_base = take(4 * (size_t)c.B);
  p.n_chunks = take(4 * (size_t)c.B);
  p.n_items = take(4);
  p.items = take(16 * (size_t)p.max_items);
  // LM-head completion counter, one attention work counter per layer, then the
  // balanced LM head's arrival counters (4 per CTA)
  p.n_counters = 1 + c.n_layers + kTcEpiWarps * p.sms;
  p.done = take(4 * (size_t)p.n_counters);
  p.keys = take(8 * (size_t)p.T);
  p.x = take(4 * (size_t)p.R * c.d);
  p.y = take(eb * (size_t)p.R * c.d);
  p.q = take(eb * (size_t)p.R * c.n_q * c.head_dim);
  p.ao = take(eb * (size_t)p.R * c.n_q * c.head_dim);
  p.u = take(eb * (size_t)p.R * c.ffn);
  p.yl = take(eb * (size_t)p.T * c.d);
  size_t split_bytes = 0;  // fp32 partial tiles of the largest split-K launch (one per unit)
  for (const GemmPlan* g : {&p.fc, &p.qkv, &p.o, &p.gu, &p.down, &p.inj, &p.injkv})
    if (g->k_splits > 1) {
      const bool paired = g->epi == EPI_SWIGLU || g->epi == EPI_QKV_ROPE;
      split_bytes = std::max(split_bytes, (size_t)g->n_f * g->n_t * g->k_splits * (paired ? 2 : 1) * g->bn * kTcBM * 4);
    }
  if (p.lm.balanced) split_bytes = std::max(split_bytes, (size_t)p.lm.grid * 2 * p.lm.bn * kTcBM * 4);
  p.split_part = c.dtype == PE_BF16 && split_bytes > 0 ? take(split_bytes) : 0;
  if (c.dtype == PE_BF16) {
    p.part_m = take(4 * (size_t)p.max_items * kAttnRows);
    p.part_l = take(4 * (size_t)p.max_items * kAttnRows);
    p.part_o = take(4 * (size_t)p.max_items * kAttnRows * c.head_dim);
  } else {
    p.part_m = p.part_l = p.part_o = 0;
  }
  // pe_step: batch metadata and input rows
  p.st_ids = take(4 * (size_t)p.R);
  p.st_pos = take(4 * (size_t)p.R);
  p.st_slot = take(8 * (size_t)p.R);
  p.st_rej = take((size_t)p.R);
  p.st_mask = take((size_t)p.R);
  p.st_hmap = take(4 * (size_t)p.R);
  p.st_rows = take(4 * (size_t)p.R);
  p.st_nvalid = take(4);
  p.st_draft = take(4 * (size_t)p.T);
  p.st_x0 = take(eb * (size_t)p.R * 2 * c.d);
  p.samp = take(sample_stats_bytes(p.T, c.vocab));  // pe_sample_drafts / pe_verify_sampled
  p.samp_acc = take(4 * (size_t)c.B);
  p.total = off;
  return p;
}

// ----------------------------------------------------------------------------- TMA descriptors

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor of `rank` dims (dims[0] innermost), 128-byte swizzle, zero fill out of bounds.
bool make_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
               const uint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                        reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides_bytes),
                        reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows][cols] row-major, box of box_rows x 64 columns
// GEMM operands view K as [K/64][64] (K a multiple of 64): a box of `ka` atoms lands as
// ka consecutive [box rows][64] tiles, each 128-byte swizzled.

// [rows][cols] as [cols/64][rows][64]: box of box_rows rows x ka atoms
bool tmap_matrix(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, int ka) {
  const uint64_t dims[3] = {(uint64_t)kTcBK, rows, cols / kTcBK};
  const uint64_t strides[2] = {cols * 2, (uint64_t)kTcBK * 2};
  const uint32_t box[3] = {(uint32_t)kTcBK, box_rows, (uint32_t)ka};
  return make_tmap(m, base, 3, dims, strides, box);
}

// w_gate_up [2F][d] as [d/64][2][F][64]: one box = 128 rows of both halves x ka atoms,
// landing per atom as the gate tile then the up tile
bool tmap_gate_up(CUtensorMap* m, const void* base, uint64_t F, uint64_t d, int ka) {
  const uint64_t dims[4] = {(uint64_t)kTcBK, F, 2, d / kTcBK};
  const uint64_t strides[3] = {d * 2, F * d * 2, (uint64_t)kTcBK * 2};
  const uint32_t box[4] = {(uint32_t)kTcBK, (uint32_t)kTcBM, 2, (uint32_t)ka};
  return make_tmap(m, base, 4, dims, strides, box);
}

// wqkv [heads*hd][d] as [d/64][2][heads][hd/2][64] (the half index outside the heads):
// one box = both halves of 128/(hd/2) heads x ka atoms, landing per atom as the tile of
// the heads' first halves then the tile of their second halves
bool tmap_qkv(CUtensorMap* m, const void* base, uint64_t heads, uint64_t hd, uint64_t d, int ka) {
  const uint64_t half = hd / 2;
  const uint64_t dims[5] = {(uint64_t)kTcBK, half, heads, 2, d / kTcBK};
  const uint64_t strides[4] = {d * 2, hd * d * 2, half * d * 2, (uint64_t)kTcBK * 2};
  const uint32_t box[5] = {(uint32_t)kTcBK, (uint32_t)half, (uint32_t)(kTcBM / half), 2, (uint32_t)ka};
  return make_tmap(m, base, 5, dims, strides, box);
}

// paged K or V pool [num_pages*16][n_kv][hd] as a 3-D tensor (hd innermost); box = 64 dims x 1 head x 16 positions
bool tmap_kv(CUtensorMap* m, const void* base, const pe_config& c, int num_pages) {
  const uint64_t dims[3] = {(uint64_t)c.head_dim, (uint64_t)c.n_kv, (uint64_t)num_pages * c.page_size};
  const uint64_t strides[2] = {(uint64_t)c.head_dim * 2, (uint64_t)c.n_kv * c.head_dim * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)c.page_size};
  return make_tmap(m, base, 3, dims, strides, box);
}

// ----------------------------------------------------------------------------- validation

pe_status check_cfg(const pe_config* c) {
  if (c == nullptr) return PE_ERR_INVALID_ARG;
  if (c->dtype != PE_F32 && c->dtype != PE_BF16) return PE_ERR_INVALID_ARG;
  if (c->B < 1 || c->K < 1 || c->d < 8 || c->n_q < 1 || c->n_kv < 1 || c->ffn < 1 || c->vocab < 2 ||
      c->n_layers < 1 || c->max_pages_per_seq < 1)
    return PE_ERR_SHAPE;
  if (c->n_q % c->n_kv != 0) return PE_ERR_SHAPE;
  if (c->page_size != 16) return PE_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return PE_ERR_UNSUPPORTED;
  if ((long long)c->B * 2 * c->K > kMaxRows) return PE_ERR_SHAPE;
  if (c->d > 16384) return PE_ERR_UNSUPPORTED;  // RMSNorm keeps a row in registers
  if (scatter_smem_bytes(c->d, (int)elem_bytes(c->dtype)) > kScatterSmemMax) return PE_ERR_UNSUPPORTED;  // staged rows
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return PE_ERR_INVALID_ARG;
  const size_t eb = elem_bytes(c->dtype);
  if ((c->d * eb) % 16 != 0 || c->d % 4 != 0) return PE_ERR_UNSUPPORTED;  // bulk row copies, float4 norm
  if (c->dtype == PE_BF16) {
    // tensor-core GEMM operands are tiled in 64-wide k atoms along every contraction
    // (d, 2d, ffn, n_q * head_dim; head_dim is 64 or 128)
    if (c->d % 64 != 0 || c->ffn % 64 != 0) return PE_ERR_UNSUPPORTED;
    if (2 * c->K * (c->n_q / c->n_kv) > kAttnRows) return PE_ERR_UNSUPPORTED;  // one query tile per item
  }
  return PE_OK;
}

#define PE_TRY_CUDA(expr)                         \
  do {                                            \
    if ((expr) != cudaSuccess) return PE_ERR_CUDA; \
  } while (0)

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// RoPE turn frequencies in double, stored as hi + lo floats.
void set_rope_table(GemmArgs& g, float theta, int hd) {
  for (int i = 0; i < 64; ++i) {
    const double tf = i < hd / 2 ? std::pow((double)theta, -2.0 * i / hd) / (2.0 * 3.14159265358979323846) : 0.0;
    g.rope_tf_hi[i] = (float)tf;
    g.rope_tf_lo[i] = (float)(tf - (double)g.rope_tf_hi[i]);
  }
}

// ----------------------------------------------------------------------------- one GEMM launch

struct GemmCall {
  int epi;
  const GemmPlan* plan;
  const void* W;
  const void* X;  // [tokens][k_dim]
  int k_dim, n_out, n_tok;
  const int32_t* n_tok_dev;
  // tensor-map shapes of W
  int w_kind;  // 0: matrix [w_rows][k_dim], 1: gate/up, 2: qkv
  uint64_t w_rows;
};

pe_status run_gemm(const pe_config& c, const Plan& p, void* ws, const GemmCall& call, GemmArgs a, cudaStream_t s) {
  a.n_out = call.n_out;
  a.k_dim = call.k_dim;
  a.n_tok = call.n_tok;
  a.n_tok_dev = call.n_tok_dev;
  a.W = call.W;
  a.X = call.X;
  a.ldx = call.k_dim;
  if (c.dtype == PE_F32) {
    PE_TRY_CUDA(launch_gemm_f32(call.epi, a, s));
    return PE_OK;
  }
  const GemmPlan& g = *call.plan;
  a.bn = g.bn;
  a.kb_total = g.kb_total;
  a.ka = g.ka;
  a.k_splits = g.k_splits;
  a.stages = g.stages;
  a.stage_bytes = g.stage_bytes;
  a.n_t = g.n_t;
  a.n_f = g.n_f;
  a.nbuf = g.nbuf;
  a.acc_stride = g.acc_stride;
  a.tmem_cols = g.tmem_cols;
  a.n_tok_min = call.n_tok_dev != nullptr ? std::min(call.n_tok, c.B * c.K) : call.n_tok;
  // many-row GEMMs on pairs that (at the usual row counts) run one wave: weight tile fastest,
  // so that every CTA prefetches its first weight stages before the dependency wait; the
  // multi-wave gate/up and the LM head keep a weight tile's token tiles side by side (L2 reuse)
  a.tok_major = (g.cg == 2 && g.n_t > 1 && call.epi != EPI_SWIGLU && call.epi != EPI_ARGMAX) ? 1 : 0;
  a.wait_ns = wait_limit_ns();
  a.drop_stage = take_drop_stage();
  if (g.k_splits > 1 || g.balanced) a.partial = at<float>(ws, p.split_part);
  if (g.balanced) a.tile_cnt = at<int32_t>(ws, p.done) + 1 + c.n_layers;
  CUtensorMap tw, tx;
  bool ok;
  if (call.w_kind == 1) ok = tmap_gate_up(&tw, call.W, (uint64_t)c.ffn, (uint64_t)c.d, g.ka);
  else if (call.w_kind == 2)  // w_rows: heads of W (0: all of q | k | v)
    ok = tmap_qkv(&tw, call.W, call.w_rows ? call.w_rows : (uint64_t)(c.n_q + 2 * c.n_kv), (uint64_t)c.head_dim,
                  (uint64_t)c.d, g.ka);
  else ok = tmap_matrix(&tw, call.W, call.w_rows, (uint64_t)call.k_dim, (uint32_t)kTcBM, g.ka);
  ok = ok && tmap_matrix(&tx, call.X, (uint64_t)call.n_tok, (uint64_t)call.k_dim, (uint32_t)(g.bn / g.cg), g.ka);
  if (!ok) return PE_ERR_CUDA;
  PE_TRY_CUDA(launch_gemm_tc(g.balanced ? EPI_ARGMAX_BAL : call.epi, g.cg, tw, tx, a, g.grid, g.smem, s));
  if (g.k_splits > 1 && (call.epi == EPI_QKV_ROPE || call.epi == EPI_SWIGLU))
    PE_TRY_CUDA(launch_splitk_finish(call.epi, a, p.sms, s));
  return PE_OK;
}

pe_status check_weights(const pe_config& c, const pe_weights* w) {
  if (w == nullptr || w->emb == nullptr || w->h_shared == nullptr || w->fc == nullptr || w->norm_final == nullptr ||
      w->lm_head == nullptr || w->norm_attn == nullptr || w->wqkv == nullptr || w->wo == nullptr ||
      w->norm_mlp == nullptr || w->w_gate_up == nullptr || w->w_down == nullptr)
    return PE_ERR_INVALID_ARG;
  const void* ptrs[5] = {w->emb, w->h_shared, w->fc, w->norm_final, w->lm_head};
  for (const void* q : ptrs)
    if (!aligned16(q)) return PE_ERR_INVALID_ARG;
  for (int l = 0; l < c.n_layers; ++l) {
    const void* lp[6] = {w->norm_attn[l], w->wqkv[l], w->wo[l], w->norm_mlp[l], w->w_gate_up[l], w->w_down[l]};
    for (const void* q : lp)
      if (q == nullptr || !aligned16(q)) return PE_ERR_INVALID_ARG;
  }
  return PE_OK;
}

pe_status check_kv(const pe_config& c, const pe_kv* kv) {
  if (kv == nullptr || kv->k_cache == nullptr || kv->v_cache == nullptr || kv->num_pages < 1) return PE_ERR_INVALID_ARG;
  for (int l = 0; l < c.n_layers; ++l)
    if (kv->k_cache[l] == nullptr || kv->v_cache[l] == nullptr || !aligned16(kv->k_cache[l]) ||
        !aligned16(kv->v_cache[l]))
      return PE_ERR_INVALID_ARG;
  return PE_OK;
}

// pe_step's outputs against its inputs: an output may be exactly its paired state input
// (next_prev_tokens / prev_tokens, next_prev_pos / prev_pos, num_accepted_out /
// num_accepted, bonus_out / bonus); otherwise no output may overlap an input or another
// output.  The error word and the part of the workspace the round uses count as outputs.
// Byte ranges from the config's shapes.
struct Span {
  uintptr_t lo, hi;
};
bool overlaps(const Span& a, const Span& b) { return a.lo < b.hi && b.lo < a.hi; }
Span span_of(const void* p, size_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + bytes};
}
bool step_aliasing_ok(const pe_config& c, const int32_t* block_table, const int32_t* prev_tokens,
                      const int32_t* prev_pos, const int32_t* num_accepted, const int32_t* bonus,
                      const void* target_hidden, const int32_t* target_tokens, const int32_t* draft_tokens,
                      const int32_t* num_accepted_out, const int32_t* bonus_out, const int32_t* next_prev_tokens,
                      const int32_t* next_prev_pos, const float* logits_dbg, const int32_t* err_word,
                      const void* workspace, size_t workspace_used) {
  const size_t B = (size_t)c.B, K = (size_t)c.K;
  const Span in[7] = {span_of(block_table, 4 * B * (size_t)c.max_pages_per_seq), span_of(prev_tokens, 4 * B * (K + 1)),
                      span_of(prev_pos, 4 * B * (K + 1)), span_of(num_accepted, 4 * B), span_of(bonus, 4 * B),
                      span_of(target_hidden, elem_bytes(c.dtype) * B * (K + 1) * (size_t)c.d),
                      span_of(target_tokens, 4 * B * (K + 1))};
  // outputs, each with the index of the input it may replace exactly (-1: none)
  const Span out[8] = {span_of(draft_tokens, 4 * B * K), span_of(num_accepted_out, 4 * B),
                       span_of(bonus_out, 4 * B), span_of(next_prev_tokens, 4 * B * (K + 1)),
                       span_of(next_prev_pos, 4 * B * (K + 1)),
                       span_of(logits_dbg, logits_dbg ? 4 * B * K * (size_t)c.vocab : 0), span_of(err_word, 4),
                       span_of(workspace, workspace_used)};
  const int pair[8] = {-1, 3, 4, 1, 2, -1, -1, -1};
  for (int o = 0; o < 8; ++o) {
    for (int i = 0; i < 7; ++i) {
      if (!overlaps(out[o], in[i])) continue;
      if (i == pair[o] && out[o].lo == in[i].lo && out[o].hi == in[i].hi) continue;
      return false;
    }
    for (int o2 = 0; o2 < o; ++o2)
      if (overlaps(out[o], out[o2])) return false;
  }
  return true;
}

PrepArgs make_prep_args(const pe_config& c, const int32_t* prev_tokens, const int32_t* prev_pos,
                        const int32_t* num_accepted, const int32_t* bonus, const int32_t* block_table, int32_t num_pages,
                        int32_t* input_ids, int32_t* positions, int64_t* slot_mapping, uint8_t* is_rejected,
                        uint8_t* is_mask, int32_t* hidden_map, int32_t* row_list, int32_t* n_valid, int32_t* draft_rows,
                        int32_t* err) {
  PrepArgs a{};
  a.B = c.B; a.K = c.K; a.vocab = c.vocab; a.max_pages = c.max_pages_per_seq; a.num_pages = num_pages;
  a.page_size = c.page_size; a.prev_tokens = prev_tokens; a.prev_pos = prev_pos; a.num_accepted = num_accepted;
  a.bonus = bonus; a.block_table = block_table; a.input_ids = input_ids; a.positions = positions;
  a.slot_mapping = slot_mapping; a.is_rejected = is_rejected; a.is_mask = is_mask; a.hidden_map = hidden_map;
  a.row_list = row_list; a.n_valid = n_valid; a.draft_rows = draft_rows; a.err = err;
  return a;
}

ScatterArgs make_scatter_args(const pe_config& c, const pe_weights* w, const void* target_hidden,
                              const int32_t* input_ids, const uint8_t* is_mask, const int32_t* hidden_map,
                              const int32_t* row_list, const int32_t* n_valid, void* x0, int32_t* err) {
  ScatterArgs a{};
  a.R = c.B * 2 * c.K; a.d = c.d; a.elem_bytes = (int)elem_bytes(c.dtype); a.vocab = c.vocab;
  a.n_hidden = c.B * (c.K + 1); a.emb = w->emb; a.h_shared = w->h_shared; a.hidden = target_hidden;
  a.input_ids = input_ids; a.is_mask = is_mask; a.hidden_map = hidden_map; a.row_list = row_list;
  a.n_valid = n_valid; a.x0 = x0; a.err = err;
  return a;
}

InitArgs make_init_args(const pe_config& c, const Plan& p, void* ws, const int32_t* row_list, const int32_t* n_valid,
                        const int32_t* positions, const int64_t* slot_mapping, int32_t* err) {
  InitArgs ia{};
  ia.B = c.B; ia.K = c.K; ia.R = p.R; ia.T = p.T; ia.n_kv = c.n_kv;
  ia.row_list = row_list; ia.n_valid = n_valid; ia.positions = positions; ia.slot_mapping = slot_mapping;
  ia.tok_pos = at<int32_t>(ws, p.tok_pos); ia.tok_seq = at<int32_t>(ws, p.tok_seq);
  ia.tok_slot = at<int64_t>(ws, p.tok_slot);
  ia.seq_start = at<int32_t>(ws, p.seq_start); ia.seq_len = at<int32_t>(ws, p.seq_len);
  ia.seq_maxpos = at<int32_t>(ws, p.seq_maxpos);
  ia.seq_minpos = at<int32_t>(ws, p.seq_minpos);
  ia.target_items = p.attn_target; ia.max_items = p.max_items; ia.min_chunk = kAttnMinChunk;
  ia.items = at<int4>(ws, p.items); ia.n_items = at<int32_t>(ws, p.n_items);
  ia.item_base = at<int32_t>(ws, p.item_base); ia.n_chunks = at<int32_t>(ws, p.n_chunks);
  ia.counters = at<int32_t>(ws, p.done); ia.n_counters = p.n_counters;
  ia.keys = at<unsigned long long>(ws, p.keys); ia.err = err;
  return ia;
}

// The weight matrices the prologue warms (bf16 storage; fp32 configurations run the CUDA-core
// path, which is not limited by the first loads).
void set_warm_ranges(InitArgs& ia, const pe_config& c, const pe_weights* w) {
  ia.warm_n = 0;
  if (c.dtype != PE_BF16) return;
  const long long d = c.d, hd = c.head_dim, F = c.ffn;
  auto add = [&](const void* base, long long elems) {
    if (ia.warm_n < kWarmRanges && base != nullptr) {
      ia.warm_base[ia.warm_n] = static_cast<const uint8_t*>(base);
      ia.warm_bytes[ia.warm_n++] = 2 * elems;
    }
  };
  add(w->fc, 2 * d * d);
  for (int l = 0; l < c.n_layers && l < (kWarmRanges - 1) / 4; ++l) {
    add(w->wqkv[l], (long long)(c.n_q + 2 * c.n_kv) * hd * d);
    add(w->wo[l], d * c.n_q * hd);
    add(w->w_gate_up[l], 2 * F * d);
    add(w->w_down[l], d * F);
  }
  // not the LM head: it streams long enough for its own first touches to overlap, and its
  // ~600 pages would make a prologue that finds every translation missing 10-20 us longer
}

pe_status forward_impl(const pe_config& c, const pe_weights* w, const pe_kv* kv, const int32_t* block_table,
                       const void* x0, const int32_t* positions, const int64_t* slot_mapping,
                       const int32_t* row_list, const int32_t* n_valid, const int32_t* draft_rows, void* ws,
                       const Plan& p, int32_t* draft_tokens, float* logits_dbg, int32_t* err, cudaStream_t s,
                       bool init_done = false, const VerifyArgs* verify = nullptr) {
  const bool bf16 = c.dtype == PE_BF16;
  const int hd = c.head_dim;
  // prologue (already run by pe_step's fused batch-rebuild kernel when init_done)
  InitArgs ia = make_init_args(c, p, ws, row_list, n_valid, positions, slot_mapping, err);
  set_warm_ranges(ia, c, w);
  if (!init_done) PE_TRY_CUDA(launch_forward_init(ia, s));
  trace(3, s);


  GemmArgs base{};
  base.n_q = c.n_q; base.n_kv = c.n_kv; base.head_dim = hd; set_rope_table(base, c.rope_theta, hd);
  base.tok_pos = ia.tok_pos; base.tok_slot = ia.tok_slot; base.err = err;
  // Every kernel from the first QKV GEMM on starts only after the prologue has completed (its
  // predecessor triggers dependents after its own dependency wait, or the one before does), so
  // it may read the prologue's row count and maps before its own wait; fc and the norm after it
  // may start while the prologue still runs.
  base.meta_ready = 1;

  float* x = at<float>(ws, p.x);
  void* y = at<uint8_t>(ws, p.y);
  void* qb = at<uint8_t>(ws, p.q);
  void* ao = at<uint8_t>(ws, p.ao);
  void* u = at<uint8_t>(ws, p.u);
  void* yl = at<uint8_t>(ws, p.yl);
  const int heads = c.n_q + 2 * c.n_kv;

  // fc, o-proj and down leave their split-K partials to the RMSNorm that follows them, which
  // sums them (plus the residual) while it normalises (QKV and gate/up: splitk_finish_kernel)
  auto deferred = [&](const GemmPlan& g) { return bf16 && g.k_splits > 1; };
  auto norm_after = [&](NormArgs& n, const GemmPlan& g, bool residual, bool keep_x) {
    if (deferred(g)) {
      n.part = at<float>(ws, p.split_part); n.n_splits = g.k_splits; n.bn = g.bn; n.n_t = g.n_t;
      n.g_ntok = p.R; n.g_ntok_dev = n_valid; n.g_ntok_min = std::min(p.R, c.B * c.K);
      n.x = residual ? x : nullptr; n.x_out = keep_x ? x : nullptr;
    } else {
      n.part = nullptr; n.n_splits = 0; n.x = x; n.x_out = nullptr;
    }
  };

  // fc: x = X0 . W_fc^T
  {
    GemmArgs a = base;
    a.out_f32 = x; a.ld_out = c.d;
    a.meta_ready = 0;
    GemmCall call{EPI_STORE_F32, &p.fc, w->fc, x0, 2 * c.d, c.d, p.R, n_valid, 0, (uint64_t)c.d};
    pe_status st = run_gemm(c, p, ws, call, a, s);
    if (st != PE_OK) return st;
  }
  trace(4, s);
  NormArgs na{};
  na.x = x; na.d = c.d; na.row_map = nullptr; na.n_rows = p.R; na.n_rows_dev = n_valid; na.src_rows = p.R;
  na.eps = c.rms_eps; na.y = y; na.err = err;

  AttnArgs at_{};
  at_.B = c.B; at_.n_q = c.n_q; at_.n_kv = c.n_kv; at_.head_dim = hd; at_.max_pages = c.max_pages_per_seq;
  at_.page_size = c.page_size; at_.num_pages = kv->num_pages; at_.scale = 1.0f / sqrtf((float)hd);
  at_.q = qb; at_.block_table = block_table; at_.tok_pos = ia.tok_pos; at_.tok_seq = ia.tok_seq;
  at_.seq_start = ia.seq_start; at_.seq_len = ia.seq_len; at_.n_valid = n_valid; at_.items = ia.items;
  at_.seq_minpos = ia.seq_minpos;
  at_.n_items = ia.n_items; at_.item_base = ia.item_base; at_.n_chunks = ia.n_chunks;
  at_.part_m = bf16 ? at<float>(ws, p.part_m) : nullptr;
  at_.part_l = bf16 ? at<float>(ws, p.part_l) : nullptr;
  at_.part_o = bf16 ? at<float>(ws, p.part_o) : nullptr;
  at_.out = ao; at_.n_rows = p.R; at_.err = err; at_.wait_ns = wait_limit_ns();

  for (int l = 0; l < c.n_layers; ++l) {
    const int tp = 5 + 7 * l;
    na.g = w->norm_attn[l];
    na.meta_ready = l == 0 ? 0 : 1;
    if (l == 0) norm_after(na, p.fc, false, true);
    else norm_after(na, p.down, true, true);
    PE_TRY_CUDA(launch_rmsnorm(na, c.dtype, s));
    trace(tp + 0, s);
    {
      GemmArgs a = base;
      a.out_act = qb; a.ld_out = c.n_q * hd; a.k_cache = kv->k_cache[l]; a.v_cache = kv->v_cache[l];
      GemmCall call{EPI_QKV_ROPE, &p.qkv, w->wqkv[l], y, c.d, heads * hd / 2, p.R, n_valid, 2, 0};
      pe_status st = run_gemm(c, p, ws, call, a, s);
      if (st != PE_OK) return st;
    }
    trace(tp + 1, s);
    at_.k_cache = kv->k_cache[l];
    at_.v_cache = kv->v_cache[l];
    at_.work_counter = at<int32_t>(ws, p.done) + 1 + l;
    if (bf16) {
      CUtensorMap tk, tv;
      if (!tmap_kv(&tk, kv->k_cache[l], c, kv->num_pages) || !tmap_kv(&tv, kv->v_cache[l], c, kv->num_pages))
        return PE_ERR_CUDA;
      PE_TRY_CUDA(launch_attention_bf16(tk, tv, at_, p.attn_grid, p.sms, s));
    } else {
      PE_TRY_CUDA(launch_attention_f32(at_, s));
    }
    trace(tp + 2, s);
    {
      GemmArgs a = base;
      a.out_f32 = x; a.ld_out = c.d;
      GemmCall call{EPI_ADD_F32, &p.o, w->wo[l], ao, c.n_q * hd, c.d, p.R, n_valid, 0, (uint64_t)c.d};
      pe_status st = run_gemm(c, p, ws, call, a, s);
      if (st != PE_OK) return st;
    }
    trace(tp + 3, s);
    na.g = w->norm_mlp[l];
    na.meta_ready = 1;
    norm_after(na, p.o, true, true);
    PE_TRY_CUDA(launch_rmsnorm(na, c.dtype, s));
    trace(tp + 4, s);
    {
      GemmArgs a = base;
      a.out_act = u; a.ld_out = c.ffn;
      GemmCall call{EPI_SWIGLU, &p.gu, w->w_gate_up[l], y, c.d, c.ffn, p.R, n_valid, 1, 0};
      pe_status st = run_gemm(c, p, ws, call, a, s);
      if (st != PE_OK) return st;
    }
    trace(tp + 5, s);
    {
      GemmArgs a = base;
      a.out_f32 = x; a.ld_out = c.d;
      GemmCall call{EPI_ADD_F32, &p.down, w->w_down[l], u, c.ffn, c.d, p.R, n_valid, 0, (uint64_t)c.d};
      pe_status st = run_gemm(c, p, ws, call, a, s);
      if (st != PE_OK) return st;
    }
    trace(tp + 6, s);
  }
  const int tf = 5 + 7 * c.n_layers;
  // final norm of the draft rows (in draft order), then LM head + argmax
  NormArgs nf = na;
  nf.row_map = draft_rows; nf.n_rows = p.T; nf.n_rows_dev = nullptr; nf.src_rows = p.R; nf.g = w->norm_final;
  nf.meta_ready = 1;
  nf.y = yl;
  norm_after(nf, p.down, true, false);  // the residual after the last layer is needed only here
  PE_TRY_CUDA(launch_rmsnorm(nf, c.dtype, s));
  trace(tf, s);
  {
    GemmArgs a = base;
    a.keys = ia.keys; a.logits_dbg = logits_dbg; a.done_counter = at<int32_t>(ws, p.done);
    a.draft_out = draft_tokens;
    if (verify != nullptr) {
      a.verify = *verify;
      a.has_verify = 1;
    }
    GemmCall call{EPI_ARGMAX, &p.lm, w->lm_head, yl, c.d, c.vocab, p.T, nullptr, 0, (uint64_t)c.vocab};
    pe_status st = run_gemm(c, p, ws, call, a, s);
    if (st != PE_OK) return st;
  }
  trace(tf + 1, s);
  return PE_OK;
}

}  // namespace
}  // namespace pe

using namespace pe;

extern "C" {

const char* pe_status_str(pe_status st) {
  switch (st) {
    case PE_OK: return "ok";
    case PE_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer or bad value)";
    case PE_ERR_SHAPE: return "inconsistent or out-of-range sizes";
    case PE_ERR_UNSUPPORTED: return "configuration not supported by this build";
    case PE_ERR_CUDA: return "CUDA launch or runtime call failed";
    case PE_ERR_DEVICE_CHECK: return "a device-side check fired";
    case PE_ERR_TIMEOUT: return "a bounded device wait timed out";
  }
  return "unknown status";
}

pe_status pe_check_config(const pe_config* cfg) { return check_cfg(cfg); }

size_t pe_workspace_bytes(const pe_config* cfg) {
  if (check_cfg(cfg) != PE_OK) return 0;
  return make_plan(*cfg).total;
}

pe_status pe_prepare_batch(const pe_config* cfg, const int32_t* prev_tokens, const int32_t* prev_pos,
                           const int32_t* num_accepted, const int32_t* bonus, const int32_t* block_table,
                           int32_t num_pages, int32_t* input_ids, int32_t* positions, int64_t* slot_mapping,
                           uint8_t* is_rejected, uint8_t* is_mask, int32_t* hidden_map, int32_t* row_list,
                           int32_t* n_valid, int32_t* draft_rows, int32_t* err_word, pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  if (!prev_tokens || !prev_pos || !num_accepted || !bonus || !block_table || !input_ids || !positions ||
      !slot_mapping || !is_rejected || !is_mask || !hidden_map || !row_list || !n_valid || !draft_rows || !err_word)
    return PE_ERR_INVALID_ARG;
  if (num_pages < 1) return PE_ERR_SHAPE;
  const PrepArgs a = make_prep_args(*cfg, prev_tokens, prev_pos, num_accepted, bonus, block_table, num_pages, input_ids,
                                    positions, slot_mapping, is_rejected, is_mask, hidden_map, row_list, n_valid,
                                    draft_rows, err_word);
  if (launch_prepare(a, (cudaStream_t)stream) != cudaSuccess) return PE_ERR_CUDA;
  return PE_OK;
}

pe_status pe_scatter_hidden(const pe_config* cfg, const pe_weights* w, const void* target_hidden,
                            const int32_t* input_ids, const uint8_t* is_mask, const int32_t* hidden_map,
                            const int32_t* row_list, const int32_t* n_valid, void* x0, int32_t* err_word,
                            pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  if (w == nullptr || !w->emb || !w->h_shared || !target_hidden || !input_ids || !is_mask || !hidden_map ||
      !row_list || !n_valid || !x0 || !err_word)
    return PE_ERR_INVALID_ARG;
  if (!aligned16(w->emb) || !aligned16(w->h_shared) || !aligned16(target_hidden) || !aligned16(x0))
    return PE_ERR_INVALID_ARG;
  const ScatterArgs a =
      make_scatter_args(*cfg, w, target_hidden, input_ids, is_mask, hidden_map, row_list, n_valid, x0, err_word);
  if (launch_scatter(a, (cudaStream_t)stream) != cudaSuccess) return PE_ERR_CUDA;
  return PE_OK;
}

pe_status pe_draft_forward(const pe_config* cfg, const pe_weights* w, const pe_kv* kv, const int32_t* block_table,
                           const void* x0, const int32_t* positions, const int64_t* slot_mapping,
                           const int32_t* row_list, const int32_t* n_valid, const int32_t* draft_rows,
                           void* workspace, size_t workspace_bytes, int32_t* draft_tokens, float* logits_dbg,
                           int32_t* err_word, pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  if ((st = check_weights(*cfg, w)) != PE_OK) return st;
  if ((st = check_kv(*cfg, kv)) != PE_OK) return st;
  if (!block_table || !x0 || !positions || !slot_mapping || !row_list || !n_valid || !draft_rows || !workspace ||
      !draft_tokens || !err_word)
    return PE_ERR_INVALID_ARG;
  if (!aligned16(x0) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PE_ERR_INVALID_ARG;
  const Plan p = make_plan(*cfg);
  if (workspace_bytes < p.total) return PE_ERR_SHAPE;
  for (int i = 0; i < 3; ++i) trace(i, (cudaStream_t)stream);
  return forward_impl(*cfg, w, kv, block_table, x0, positions, slot_mapping, row_list, n_valid, draft_rows,
                      workspace, p, draft_tokens, logits_dbg, err_word, (cudaStream_t)stream);
}

pe_status pe_verify(const pe_config* cfg, const int32_t* draft_tokens, const int32_t* target_tokens,
                    int32_t* num_accepted_out, int32_t* bonus_out, pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  if (!draft_tokens || !target_tokens || !num_accepted_out || !bonus_out) return PE_ERR_INVALID_ARG;
  VerifyArgs a{};
  a.B = cfg->B; a.K = cfg->K; a.draft = draft_tokens; a.target = target_tokens; a.acc_out = num_accepted_out;
  a.bonus_out = bonus_out;
  if (launch_verify(a, (cudaStream_t)stream) != cudaSuccess) return PE_ERR_CUDA;
  return PE_OK;
}

pe_status pe_step(const pe_config* cfg, const pe_weights* w, const pe_kv* kv, const int32_t* block_table,
                  const int32_t* prev_tokens, const int32_t* prev_pos, const int32_t* num_accepted,
                  const int32_t* bonus, const void* target_hidden, const int32_t* target_tokens, void* workspace,
                  size_t workspace_bytes, int32_t* draft_tokens, int32_t* num_accepted_out, int32_t* bonus_out,
                  int32_t* next_prev_tokens, int32_t* next_prev_pos, float* logits_dbg, int32_t* err_word,
                  pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  if ((st = check_weights(*cfg, w)) != PE_OK) return st;
  if ((st = check_kv(*cfg, kv)) != PE_OK) return st;
  if (!block_table || !prev_tokens || !prev_pos || !num_accepted || !bonus || !target_hidden || !target_tokens ||
      !workspace || !draft_tokens || !num_accepted_out || !bonus_out || !next_prev_tokens || !next_prev_pos ||
      !err_word)
    return PE_ERR_INVALID_ARG;
  if (!aligned16(target_hidden) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PE_ERR_INVALID_ARG;
  const Plan p = make_plan(*cfg);
  // the workspace bytes this round would use (a workspace that is too short fails below)
  if (!step_aliasing_ok(*cfg, block_table, prev_tokens, prev_pos, num_accepted, bonus, target_hidden, target_tokens,
                        draft_tokens, num_accepted_out, bonus_out, next_prev_tokens, next_prev_pos, logits_dbg,
                        err_word, workspace, std::min(workspace_bytes, p.total)))
    return PE_ERR_INVALID_ARG;
  if (workspace_bytes < p.total) return PE_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  int32_t* ids = at<int32_t>(ws, p.st_ids);
  int32_t* pos = at<int32_t>(ws, p.st_pos);
  int64_t* slot = at<int64_t>(ws, p.st_slot);
  uint8_t* rej = at<uint8_t>(ws, p.st_rej);
  uint8_t* msk = at<uint8_t>(ws, p.st_mask);
  int32_t* hmap = at<int32_t>(ws, p.st_hmap);
  int32_t* rows = at<int32_t>(ws, p.st_rows);
  int32_t* nval = at<int32_t>(ws, p.st_nvalid);
  int32_t* drows = at<int32_t>(ws, p.st_draft);
  void* x0 = at<uint8_t>(ws, p.st_x0);
  // the batch rebuild, the input rows and the forward prologue in one launch
  if (!w->emb || !w->h_shared || !aligned16(w->emb) || !aligned16(w->h_shared)) return PE_ERR_INVALID_ARG;
  const PrepArgs pa = make_prep_args(*cfg, prev_tokens, prev_pos, num_accepted, bonus, block_table, kv->num_pages, ids,
                                     pos, slot, rej, msk, hmap, rows, nval, drows, err_word);
  const ScatterArgs sa = make_scatter_args(*cfg, w, target_hidden, ids, msk, hmap, rows, nval, x0, err_word);
  InitArgs ia = make_init_args(*cfg, p, ws, rows, nval, pos, slot, err_word);
  set_warm_ranges(ia, *cfg, w);
  trace(0, s);
  PE_TRY_CUDA(launch_step_prologue(pa, sa, ia, s));
  trace(1, s);
  trace(2, s);
  VerifyArgs va{};
  va.B = cfg->B; va.K = cfg->K; va.draft = draft_tokens; va.target = target_tokens; va.acc_out = num_accepted_out;
  va.bonus_out = bonus_out; va.row_list = rows; va.draft_rows = drows; va.positions = pos; va.input_ids = ids;
  va.next_tokens = next_prev_tokens; va.next_pos = next_prev_pos;
  const bool bf16 = cfg->dtype == PE_BF16;  // the tensor-core LM head verifies in its finishing CTA
  st = forward_impl(*cfg, w, kv, block_table, x0, pos, slot, rows, nval, drows, ws, p, draft_tokens, logits_dbg,
                    err_word, s, true, bf16 ? &va : nullptr);
  if (st != PE_OK) return st;
  if (!bf16 && launch_verify(va, s) != cudaSuccess) return PE_ERR_CUDA;
  trace(7 + 7 * cfg->n_layers, s);
  return PE_OK;
}

pe_status pe_sample_drafts(const pe_config* cfg, const float* logits, const float* u_draft, float temperature,
                           void* workspace, size_t workspace_bytes, int32_t* draft_tokens, float* lse,
                           int32_t* err_word, pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  if (!logits || !u_draft || !workspace || !draft_tokens || !lse || !err_word) return PE_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return PE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PE_ERR_INVALID_ARG;
  const Plan p = make_plan(*cfg);
  if (workspace_bytes < p.total) return PE_ERR_SHAPE;
  SampleArgs a{};
  a.B = cfg->B; a.K = cfg->K; a.V = cfg->vocab;
  a.logits = logits; a.u = u_draft; a.inv_t2 = (float)(1.4426950408889634 / (double)temperature);
  a.stats = at<float2>(workspace, p.samp);
  a.drafts = draft_tokens; a.lse = lse; a.err = err_word;
  PE_TRY_CUDA(launch_sample_drafts(a, p.sms, (cudaStream_t)stream));
  return PE_OK;
}

pe_status pe_verify_sampled(const pe_config* cfg, const int32_t* draft_tokens, const float* logits, const float* lse,
                            float temperature, const float* target_probs, const float* u_accept,
                            const float* u_resample, void* workspace, size_t workspace_bytes,
                            int32_t* num_accepted_out, int32_t* bonus_out, int32_t* err_word, pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  if (!draft_tokens || !logits || !lse || !target_probs || !u_accept || !u_resample || !workspace ||
      !num_accepted_out || !bonus_out || !err_word)
    return PE_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return PE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PE_ERR_INVALID_ARG;
  const Plan p = make_plan(*cfg);
  if (workspace_bytes < p.total) return PE_ERR_SHAPE;
  VerifySampledArgs a{};
  a.B = cfg->B; a.K = cfg->K; a.V = cfg->vocab;
  a.drafts = draft_tokens; a.logits = logits; a.lse = lse; a.inv_t2 = (float)(1.4426950408889634 / (double)temperature);
  a.target_probs = target_probs; a.u_accept = u_accept; a.u_resample = u_resample;
  a.stats = at<float2>(workspace, p.samp);
  a.acc_ws = at<int32_t>(workspace, p.samp_acc);
  a.acc_out = num_accepted_out; a.bonus_out = bonus_out; a.err = err_word;
  PE_TRY_CUDA(launch_verify_sampled(a, p.sms, (cudaStream_t)stream));
  return PE_OK;
}

pe_status pe_inject_kv(const pe_config* cfg, const pe_weights* w, const void* w_inj, const pe_kv* kv,
                       const int32_t* block_table, const int32_t* prev_pos, const int32_t* num_accepted,
                       const void* target_hidden, void* workspace, size_t workspace_bytes, int32_t* err_word,
                       pe_stream_t stream) {
  pe_status st = check_cfg(cfg);
  if (st != PE_OK) return st;
  const pe_config& c = *cfg;
  if (w == nullptr || w->norm_attn == nullptr || w->wqkv == nullptr) return PE_ERR_INVALID_ARG;
  for (int l = 0; l < c.n_layers; ++l)
    if (!w->norm_attn[l] || !w->wqkv[l] || !aligned16(w->norm_attn[l]) || !aligned16(w->wqkv[l]))
      return PE_ERR_INVALID_ARG;
  if ((st = check_kv(c, kv)) != PE_OK) return st;
  if (!w_inj || !block_table || !prev_pos || !num_accepted || !target_hidden || !workspace || !err_word)
    return PE_ERR_INVALID_ARG;
  if (!aligned16(w_inj) || !aligned16(target_hidden) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PE_ERR_INVALID_ARG;
  const Plan p = make_plan(c);
  if (workspace_bytes < p.total) return PE_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  const bool bf16 = c.dtype == PE_BF16;
  const int NI = c.B * (c.K + 1);
  const int hd = c.head_dim;
  InjectArgs ia{};
  ia.B = c.B; ia.K = c.K; ia.max_pages = c.max_pages_per_seq; ia.num_pages = kv->num_pages;
  ia.page_size = c.page_size; ia.prev_pos = prev_pos; ia.num_accepted = num_accepted; ia.block_table = block_table;
  ia.tok_pos = at<int32_t>(ws, p.tok_pos); ia.tok_slot = at<int64_t>(ws, p.tok_slot); ia.err = err_word;
  PE_TRY_CUDA(launch_inject_init(ia, s));

  GemmArgs base{};
  base.n_q = c.n_q; base.n_kv = c.n_kv; base.head_dim = hd; set_rope_table(base, c.rope_theta, hd);
  base.tok_pos = ia.tok_pos; base.tok_slot = ia.tok_slot; base.err = err_word;
  float* x = at<float>(ws, p.x);
  void* y = at<uint8_t>(ws, p.y);
  // x = H . W_inj^T over every element of the verify batch (the rejected ones are computed but
  // never written: their slot is -1)
  {
    GemmArgs a = base;
    a.out_f32 = x; a.ld_out = c.d;
    GemmCall call{EPI_STORE_F32, &p.inj, w_inj, target_hidden, c.d, c.d, NI, nullptr, 0, (uint64_t)c.d};
    if ((st = run_gemm(c, p, ws, call, a, s)) != PE_OK) return st;
  }
  for (int l = 0; l < c.n_layers; ++l) {
    NormArgs n{};
    n.x = x; n.d = c.d; n.row_map = nullptr; n.n_rows = NI; n.n_rows_dev = nullptr; n.src_rows = NI;
    n.g = w->norm_attn[l]; n.eps = c.rms_eps; n.y = y; n.err = err_word;
    if (bf16 && p.inj.k_splits > 1 && l == 0) {  // the first norm also sums W_inj's split-K partials
      n.part = at<float>(ws, p.split_part); n.n_splits = p.inj.k_splits; n.bn = p.inj.bn; n.n_t = p.inj.n_t;
      n.g_ntok = NI; n.g_ntok_dev = nullptr; n.g_ntok_min = NI; n.x = nullptr; n.x_out = x;
    }
    PE_TRY_CUDA(launch_rmsnorm(n, c.dtype, s));
    GemmArgs a = base;
    a.out_act = at<uint8_t>(ws, p.q); a.ld_out = c.n_q * hd;  // no q heads here: never written
    a.k_cache = kv->k_cache[l]; a.v_cache = kv->v_cache[l];
    a.head0 = c.n_q;
    const void* wkv = static_cast<const uint8_t*>(w->wqkv[l]) + (size_t)c.n_q * hd * c.d * elem_bytes(c.dtype);
    GemmCall call{EPI_QKV_ROPE, &p.injkv, wkv, y, c.d, c.n_kv * hd, NI, nullptr, 2, (uint64_t)(2 * c.n_kv)};
    if ((st = run_gemm(c, p, ws, call, a, s)) != PE_OK) return st;
  }
  return PE_OK;
}

pe_status pe_set_trace_events(void* const* events, int32_t n_events) {
  if (n_events < 0 || (n_events > 0 && events == nullptr)) return PE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace.assign(n_events, nullptr);
  for (int i = 0; i < n_events; ++i) g_trace[i] = static_cast<cudaEvent_t>(events[i]);
  return PE_OK;
}

int32_t pe_trace_points(const pe_config* cfg) {
  if (check_cfg(cfg) != PE_OK) return 0;
  return 8 + 7 * cfg->n_layers;
}

uint64_t pe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

pe_status pe_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns, std::memory_order_relaxed);
  return PE_OK;
}

pe_status pe_test_skip_pipeline_stage(int32_t stage) {
  if (stage < -1) return PE_ERR_INVALID_ARG;
  g_drop_stage.store(stage, std::memory_order_relaxed);
  return PE_OK;
}

}  // extern "C"
