// Dense contractions of the drafter pass with fused epilogues:
//   fc (2d -> d), QKV + RoPE + paged KV write, o-proj + residual,
//   gate/up + SwiGLU, down + residual, LM head + argmax.
//
// bf16 configurations run on the 5th-generation tensor cores: weights stream
// through a TMA -> shared-memory ring (128-byte swizzle) and one elected thread
// issues tcgen05.mma with fp32 accumulators in tensor memory.  The weight
// matrix sits on the MMA's M side (128 weight rows per tile) and the few
// token rows on its N side, so a batch of 16..256 rows reads every weight
// byte once.  Split-K spreads small matrices over all SMs; the splits leave
// fp32 partials in L2 and the consuming kernel sums them in a fixed order, so
// the result does not depend on scheduling.
// The LM head never writes logits: each
// CTA reduces its 128 vocabulary rows to a (max, argmax) key per token and
// folds it into a global 64-bit atomicMax; the last CTA decodes the keys.
//
// fp32 configurations run a CUDA-core kernel with the same epilogues.
#include <mutex>
#include <vector>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

// ============================================================================= epilogues

// Rotate-half RoPE of the pair (x1, x2) = (v[i], v[i + hd/2]) at position pos.
// tf = theta^(-2i/hd) / (2 pi) as hi + lo floats: the angle in turns, pos * tf,
// is reduced to [-1/2, 1/2] without loss (the rounding error of pos * tf.hi is
// recovered by an fma; subtracting the nearest integer is exact), so the
// hardware sine / cosine only ever sees |angle| <= pi.
PE_DEV void rope_pair(float x1, float x2, int pos, float2 tf, float& o1, float& o2) {
  const float p = (float)pos;  // exact below 2^24
  const float h = p * tf.x;
  const float e = fmaf(p, tf.x, -h);
  const float r = (h - rintf(h)) + fmaf(p, tf.y, e);
  float s, c;
  __sincosf(r * 6.283185307179586f, &s, &c);
  o1 = x1 * c - x2 * s;
  o2 = x2 * c + x1 * s;
}

// unit = head * (hd/2) + i for the pair (i, i + hd/2) of `head` in the
// q | k | v concatenation.  q and k are rotated; q goes to the q buffer, k and
// v to the paged cache at the token's slot (no write for slot -1).
// As epi_qkv, with the token's position and KV slot already loaded.
template <typename T>
PE_DEV void qkv_store(const GemmArgs& a, int unit, int t, float x1, float x2, float2 tf, int pos, long long slot) {
  const int half = a.head_dim >> 1;
  const int head = unit / half + a.head0, i = unit - (unit / half) * half;
  if (head < a.n_q + a.n_kv) rope_pair(x1, x2, pos, tf, x1, x2);
  if (head < a.n_q) {
    T* q = static_cast<T*>(a.out_act) + (size_t)t * a.ld_out + (size_t)head * a.head_dim + i;
    q[0] = from_float<T>(x1);
    q[half] = from_float<T>(x2);
    return;
  }
  if (slot < 0) return;
  const bool is_k = head < a.n_q + a.n_kv;
  const int g = is_k ? head - a.n_q : head - a.n_q - a.n_kv;
  T* c = static_cast<T*>(is_k ? a.k_cache : a.v_cache) + ((size_t)slot * a.n_kv + g) * a.head_dim + i;
  c[0] = from_float<T>(x1);
  c[half] = from_float<T>(x2);
}

template <typename T>
PE_DEV void epi_qkv(const GemmArgs& a, int unit, int t, float x1, float x2, float2 tf) {
  const int half = a.head_dim >> 1;
  const int head = unit / half + a.head0, i = unit - (unit / half) * half;
  if (head < a.n_q + a.n_kv) rope_pair(x1, x2, a.tok_pos[t], tf, x1, x2);
  if (head < a.n_q) {
    T* q = static_cast<T*>(a.out_act) + (size_t)t * a.ld_out + (size_t)head * a.head_dim + i;
    q[0] = from_float<T>(x1);
    q[half] = from_float<T>(x2);
    return;
  }
  const long long slot = a.tok_slot[t];
  if (slot < 0) return;
  const bool is_k = head < a.n_q + a.n_kv;
  const int g = is_k ? head - a.n_q : head - a.n_q - a.n_kv;
  T* c = static_cast<T*>(is_k ? a.k_cache : a.v_cache) + ((size_t)slot * a.n_kv + g) * a.head_dim + i;
  c[0] = from_float<T>(x1);
  c[half] = from_float<T>(x2);
}

template <int EPI, typename T>
PE_DEV void epi_elem(const GemmArgs& a, int unit, int t, float v, float v2, float2 tf) {
  if (EPI == EPI_STORE_F32) {
    a.out_f32[(size_t)t * a.ld_out + unit] = v;
  } else if (EPI == EPI_ADD_F32) {
    float* o = a.out_f32 + (size_t)t * a.ld_out + unit;
    *o = *o + v;
  } else if (EPI == EPI_SWIGLU) {
    static_cast<T*>(a.out_act)[(size_t)t * a.ld_out + unit] = from_float<T>(silu(v) * v2);
  } else if (EPI == EPI_QKV_ROPE) {
    epi_qkv<T>(a, unit, t, v, v2, tf);
  }
}

// Epilogue of one output unit over up to 16 consecutive tokens t0..t0+nv-1 (the
// persistent GEMM's own epilogue; the split-K finish uses epi_elem).  Every load the
// epilogue needs (residual values, token positions and slots) is issued before the
// first store: interleaving them would make each token a separate memory round trip,
// because the compiler cannot prove the stores and the later loads disjoint.  The
// token loops are unrolled so that the 16-value arrays stay in registers (a rolled
// loop indexes them dynamically, which puts them in local memory: measured 14 us per
// 128 x 128 SwiGLU unit).
template <int EPI, typename T>
PE_DEV void epi_chunk(const GemmArgs& a, int unit, int t0, int nv, const float (&v)[16], const float (&v2)[16],
                      float2 tf, const int* pos_s, const long long* slot_s) {
  if (EPI == EPI_STORE_F32) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < nv) a.out_f32[(size_t)(t0 + j) * a.ld_out + unit] = v[j];
  } else if (EPI == EPI_ADD_F32) {
    float old[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) old[j] = j < nv ? a.out_f32[(size_t)(t0 + j) * a.ld_out + unit] : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < nv) a.out_f32[(size_t)(t0 + j) * a.ld_out + unit] = old[j] + v[j];
  } else if (EPI == EPI_SWIGLU) {
    T* o = static_cast<T*>(a.out_act) + (size_t)t0 * a.ld_out + unit;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < nv) o[(size_t)j * a.ld_out] = from_float<T>(silu(v[j]) * v2[j]);
  } else if (EPI == EPI_QKV_ROPE) {
    const int half = a.head_dim >> 1;
    const int head = unit / half + a.head0, i = unit - (unit / half) * half;
    const bool is_q = head < a.n_q, rotated = head < a.n_q + a.n_kv;
    int pos[16];
    long long slot[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {  // this chunk's tokens, staged in shared memory per unit
      pos[j] = (j < nv && rotated) ? pos_s[j] : 0;
      slot[j] = (j < nv && !is_q) ? slot_s[j] : -1;
    }
    T* qdst = static_cast<T*>(a.out_act) + (size_t)t0 * a.ld_out + (size_t)head * a.head_dim + i;
    const int g = rotated ? head - a.n_q : head - a.n_q - a.n_kv;
    T* cache = static_cast<T*>(rotated ? a.k_cache : a.v_cache) + (size_t)g * a.head_dim + i;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= nv) break;
      float x1 = v[j], x2 = v2[j];
      if (rotated) rope_pair(v[j], v2[j], pos[j], tf, x1, x2);
      if (is_q) {
        qdst[(size_t)j * a.ld_out] = from_float<T>(x1);
        qdst[(size_t)j * a.ld_out + half] = from_float<T>(x2);
      } else if (slot[j] >= 0) {
        T* c = cache + (size_t)slot[j] * a.n_kv * a.head_dim;
        c[0] = from_float<T>(x1);
        c[half] = from_float<T>(x2);
      }
    }
  }
}

// RoPE turn frequency of the pair index of `unit` (hi + lo).
PE_DEV float2 rope_tf(const GemmArgs& a, int unit) {
  const int i = unit % (a.head_dim >> 1);
  return make_float2(a.rope_tf_hi[i], a.rope_tf_lo[i]);
}

// Last CTA of the LM head: turn the per-token keys into token ids.
PE_DEV void argmax_finish(const GemmArgs& a, int n_tok, int thread, int nthreads) {
  for (int t = thread; t < n_tok; t += nthreads) {
    const unsigned long long k = __ldcg(a.keys + t);
    a.draft_out[t] = argmax_key_index(k);
  }
}


// ============================================================================= tensor-core kernel
//
// Persistent: CTA b processes work units b, b + grid, b + 2*grid, ...; a unit is
// (k split, token tile, weight tile).  Roles: warp 0 lane 0 issues TMA loads
// into a ring of `stages` shared-memory stages (continuously across units),
// warp 1 lane 0 issues tcgen05.mma into one of `nbuf` TMEM accumulators, warps
// 2..5 run the epilogue of unit i while the MMAs of unit i+1 fill the other
// accumulator.  Before waiting on the previous kernel (pdl_wait) the producer
// already streams the weights of its first unit (balanced LM head: its first
// stages, across pieces): they never depend on it.
//
// Split K: one unit per CTA.  Each split writes its fp32 partial tile
// column-major to the workspace and exits; the kernel that consumes the output
// sums the splits in split order: the RMSNorm that follows fc, o-proj and down
// (adding the residual), or splitk_finish_kernel for QKV (RoPE, q, KV cache)
// and gate/up (SwiGLU).  No CTA waits for another, and the weight stream of a
// small GEMM is spread over nearly all SMs.

size_t gemm_tc_smem_bytes(int stages, uint32_t stage_bytes, int red_entries) {
  return 1024 /*alignment slack*/ + (size_t)stages * stage_bytes + kTcCtrlBytes + (size_t)red_entries * 8;
}

// Token rows of this launch: the device count, never below the rows every
// valid batch has (B*K), so that units whose weights were prefetched before
// pdl_wait() are always processed.  Rows between the two hold stale data;
// their outputs land in scratch rows and their KV slot is -1.
PE_DEV int effective_ntok(const GemmArgs& a) {
  int n = a.n_tok;
  if (a.n_tok_dev != nullptr) {
    const int d = __ldcg(a.n_tok_dev);
    if (d < a.n_tok_min) set_err(a.err, PE_DEV_BAD_ROW);
    n = min(n, max(d, a.n_tok_min));
  }
  return n;
}

struct Unit {
  int tile_t, tile_f, split, kb0, kb1;
  int bnd, side;  // balanced LM head: schedule boundary cutting this tile (-1: none), piece 0 / 1
};

// Token tiles holding at least one of this launch's rows.  Units are numbered
// over these only, so the rows' padding never lands on a CTA's schedule.
PE_DEV int live_token_tiles(const GemmArgs& a, int n_tok) {
  return min(a.n_t, (n_tok + a.bn - 1) / a.bn);
}

// nfp: weight tiles of a unit's kind (pair tiles on CTA pairs).
PE_DEV Unit decode_unit(const GemmArgs& a, int u, int n_t_live, int nfp) {
  Unit w;
  w.split = u % a.k_splits;  // splits of a tile are consecutive (one arrival counter per tile)
  const int r = u / a.k_splits;
  if (a.tok_major) {         // weight tile fastest: unit r's weight tile does not depend on the rows
    w.tile_f = r % nfp;
    w.tile_t = r / nfp;
  } else {
    w.tile_t = r % n_t_live;   // token tiles of a weight tile run side by side (L2 reuse)
    w.tile_f = r / n_t_live;
  }
  w.kb0 = (int)((long long)w.split * a.kb_total / a.k_splits);
  w.kb1 = (int)((long long)(w.split + 1) * a.kb_total / a.k_splits);
  w.bnd = -1;
  w.side = 0;
  return w;
}

// A CTA's work.  Default: units blockIdx.x, blockIdx.x + gridDim.x, ...; a CTA pair
// (CG = 2) takes units p, p + pairs, ... with p = blockIdx.x / 2, a unit's weight tile
// then being 256 rows (1-CTA tiles 2 * tile_f and 2 * tile_f + 1, one per CTA).
// Balanced LM head (EPI_ARGMAX_BAL: one token tile, more vocabulary tiles than
// CTAs): the n_f * kb_total k blocks, tile after tile, are cut into gridDim.x
// contiguous ranges of equal length, so every CTA streams the same number of
// weight bytes instead of some CTAs taking one whole tile more than the rest.  A
// range is at least a tile long, so a tile is cut by at most one range boundary,
// into two pieces (side 0: its first k blocks, side 1: the rest).
struct Sched {
  int cur, end;
};

template <int EPI, int CG>
PE_DEV Sched sched_begin(const GemmArgs& a, int n_t_live) {
  Sched sc;
  if (EPI == EPI_ARGMAX_BAL) {
    const long long W = (long long)a.n_f * a.kb_total;
    sc.cur = (int)(W * blockIdx.x / gridDim.x);
    sc.end = (int)(W * (blockIdx.x + 1) / gridDim.x);
  } else {
    sc.cur = blockIdx.x / CG;
    sc.end = n_t_live * ((a.n_f + CG - 1) / CG) * a.k_splits;
  }
  return sc;
}

template <int EPI, int CG>
PE_DEV bool sched_next(const GemmArgs& a, Sched& sc, int n_t_live, Unit& w) {
  if (sc.cur >= sc.end) return false;
  if (EPI == EPI_ARGMAX_BAL) {
    const int KB = a.kb_total;
    w.tile_t = 0;
    w.split = 0;
    w.tile_f = sc.cur / KB;
    w.kb0 = sc.cur - w.tile_f * KB;
    w.kb1 = min(KB, w.kb0 + (sc.end - sc.cur));
    // boundary b lies between the ranges of CTAs b - 1 and b
    w.bnd = w.kb0 > 0 ? (int)blockIdx.x : (w.kb1 < KB ? (int)blockIdx.x + 1 : -1);
    w.side = w.kb0 > 0 ? 1 : 0;
    sc.cur += w.kb1 - w.kb0;
  } else {
    w = decode_unit(a, sc.cur, n_t_live, (a.n_f + CG - 1) / CG);
    sc.cur += gridDim.x / CG;
  }
  return true;
}

// One stage of weights: a.ka 64-wide k atoms from atom `ka0` on, in one TMA box per
// operand (the tensor maps view K as [K/64][64], so a box of ka atoms lands as ka
// consecutive 128-byte-swizzled [128 rows][64] tiles).  One large box instead of ka
// small ones: a single SM's TMA throughput is set by the number of boxes (measured:
// 46 GB/s with 16 KB boxes, 95 GB/s with 32 KB boxes).
// Paired operands (gate/up, the heads' first/second halves) come in the same box and
// land per atom as two consecutive 128-row tiles: [ka][2][128][64].
// CG = 2: the copy completes on the leader CTA's barrier (fb is a cluster address).
template <int EPI, int CG>
PE_DEV void issue_w(const CUtensorMap* tmW, const GemmArgs& a, uint32_t sa, uint32_t fb, int ka0, int tile_f,
                    uint64_t pol) {
  if (EPI == EPI_SWIGLU) {  // W viewed as [K/64][2][F][64]
    if (CG == 2) tma_load_4d_pair(sa, tmW, fb, 0, tile_f * kTcBM, 0, ka0, pol);
    else tma_load_4d(sa, tmW, fb, 0, tile_f * kTcBM, 0, ka0, pol);
  } else if (EPI == EPI_QKV_ROPE) {  // W viewed as [K/64][2][heads][hd/2][64]
    const int hpt = kTcBM / (a.head_dim >> 1);
    if (CG == 2) tma_load_5d_pair(sa, tmW, fb, 0, 0, tile_f * hpt, 0, ka0, pol);
    else tma_load_5d(sa, tmW, fb, 0, 0, tile_f * hpt, 0, ka0, pol);
  } else {
    if (CG == 2) tma_load_3d_pair(sa, tmW, fb, 0, tile_f * kTcBM, ka0, pol);
    else tma_load_3d(sa, tmW, fb, 0, tile_f * kTcBM, ka0, pol);
  }
}

template <int EPI>
PE_DEV void apply16(const GemmArgs& a, int unit, int t0, int n_tok, const float (&v)[16], const float (&v2)[16],
                    float2 tf, const int* pos_s, const long long* slot_s) {
  if (unit >= a.n_out) return;
  epi_chunk<EPI, __nv_bfloat16>(a, unit, t0, max(0, min(16, n_tok - t0)), v, v2, tf, pos_s, slot_s);
}

PE_DEV unsigned long long umax64(unsigned long long x, unsigned long long y) { return x > y ? x : y; }

// (max, argmax) keys of 16 token columns over the warp's 32 rows by a
// transpose-reduce: each exchange round halves the columns a lane keeps, so
// after 4 rounds lane l owns one column (bits 4..1 of l) and a final round
// joins the lane pair holding it -- 16 exchanges instead of 5 per column.
// The even lane folds its column into this warp's running keys (no atomics:
// every address has one writer).
PE_DEV void argmax16(const GemmArgs& a, int unit, int t0, int n_tok, const float (&v)[16],
                     unsigned long long* red_w, int lane) {
  // keys without branches (a branch per value held this loop at ~0.8 us per 16 columns);
  // a non-finite logit is reported once per call, the debug logits written in a loop of
  // their own
  unsigned long long k[16];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const bool live = unit < a.n_out && t0 + j < n_tok;
    bad |= live && !isfinite(v[j]);
    k[j] = live ? argmax_key(v[j], (uint32_t)unit) : 0ull;
  }
  if (bad) set_err(a.err, PE_DEV_NONFINITE);
  if (a.logits_dbg != nullptr) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (unit < a.n_out && t0 + j < n_tok) a.logits_dbg[(size_t)(t0 + j) * a.n_out + unit] = v[j];
  }
  const bool h1 = (lane >> 4) & 1, h2 = (lane >> 3) & 1, h3 = (lane >> 2) & 1, h4 = (lane >> 1) & 1;
  unsigned long long k8[8], k4[4], k2[2];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const unsigned long long mine = h1 ? k[8 + i] : k[i], other = h1 ? k[i] : k[8 + i];
    k8[i] = umax64(mine, __shfl_xor_sync(0xFFFFFFFFu, other, 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const unsigned long long mine = h2 ? k8[4 + i] : k8[i], other = h2 ? k8[i] : k8[4 + i];
    k4[i] = umax64(mine, __shfl_xor_sync(0xFFFFFFFFu, other, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const unsigned long long mine = h3 ? k4[2 + i] : k4[i], other = h3 ? k4[i] : k4[2 + i];
    k2[i] = umax64(mine, __shfl_xor_sync(0xFFFFFFFFu, other, 4));
  }
  unsigned long long k1 = umax64(h4 ? k2[1] : k2[0], __shfl_xor_sync(0xFFFFFFFFu, h4 ? k2[0] : k2[1], 2));
  k1 = umax64(k1, __shfl_xor_sync(0xFFFFFFFFu, k1, 1));
  const int col = (h1 ? 8 : 0) + (h2 ? 4 : 0) + (h3 ? 2 : 0) + (h4 ? 1 : 0);
  if ((lane & 1) == 0 && k1 > red_w[col]) red_w[col] = k1;
}

// Epilogue of one piece of a vocabulary tile cut by a schedule boundary (balanced
// LM head).  Each epilogue warp stores its 32 rows of the piece's fp32
// accumulator over its half of the column chunks ([boundary][side][token column][128
// rows]); of the two warps (one per piece) that hold the same rows and columns, the one
// that arrives second adds the other piece and takes the argmax of the full sums.
// fp32 addition is commutative, so the sum is the same whichever piece is first.
PE_DEV void argmax_piece(const GemmArgs& a, const Unit& w, uint32_t tl, int unit, int n_tok,
                         unsigned long long* red_w, int r, int lane, int h, int hs) {
  const int BN = a.bn;
  const size_t plane = (size_t)BN * kTcBM;
  float* mine = a.partial + (size_t)(2 * w.bnd + w.side) * plane + r;
  const float* other = a.partial + (size_t)(2 * w.bnd + 1 - w.side) * plane + r;
  for (int c = h; c < BN / 16; c += hs) {
    float v[16];
    tmem_load16(tl + (uint32_t)(c * 16), v);
#pragma unroll
    for (int j = 0; j < 16; ++j) mine[(size_t)(c * 16 + j) * kTcBM] = v[j];
  }
  __threadfence();
  __syncwarp();
  int* cnt = a.tile_cnt + kTcEpiWarps * w.bnd + 2 * (r >> 5) + h;
  int old = 0;
  if (lane == 0) old = atomicAdd(cnt, 1);
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  if (old == 0) return;  // the other piece finishes this tile
  __threadfence();
  for (int c = h; c < BN / 16; c += hs) {
    float v[16], o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = __ldcg(other + (size_t)(c * 16 + j) * kTcBM);
    tmem_load16(tl + (uint32_t)(c * 16), v);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] += o[j];
    argmax16(a, unit, c * 16, n_tok, v, red_w + c * 16, lane);
  }
  if (lane == 0) *cnt = 0;
}

// CG = 2 (a CTA pair per unit, M = 256): the weight tile of a unit is 256 rows, 128 per
// CTA, and its BN token columns are split in halves, BN / 2 rows loaded by each CTA; the
// leader (rank 0) issues every MMA, whose D rows land in the tensor memory of the CTA that
// holds them, so each CTA's epilogue handles its own 128 weight rows over all BN tokens.
// Each CTA takes in half the token operand per unit that a single CTA does.  Both CTAs'
// copies of a stage complete on the leader's barrier (armed for both); the leader's commits
// free the stage and publish the accumulator in both CTAs; the epilogue warps of both
// return an accumulator to the leader.
template <int EPI, int CG>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmArgs a) {
  constexpr bool PAIRED = (EPI == EPI_SWIGLU || EPI == EPI_QKV_ROPE);
  constexpr bool ARGMAX = (EPI == EPI_ARGMAX || EPI == EPI_ARGMAX_BAL);
  constexpr bool BAL = (EPI == EPI_ARGMAX_BAL);
  static_assert(CG == 1 || (CG == 2 && !BAL), "CTA pairs: every epilogue but the balanced LM head");
  constexpr uint32_t A_ATOM = kTcBM * kTcBK * 2;  // one 64-wide k atom of 128 weight rows
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int EW = (int)(blockDim.x >> 5) - 2;  // epilogue warps: 4 or 8 (gemm_tc_threads)
  const int BN = a.bn;         // MMA N: token columns of a unit
  const int BNL = BN / CG;     // token rows this CTA loads per unit
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int U = a.n_t * ((a.n_f + CG - 1) / CG) * a.k_splits;  // units of the largest row count
  const int S = a.stages;
  const int NT = a.n_t * BN;  // argmax keys per warp
  uint8_t* ctrl = smem + (size_t)S * a.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;
  unsigned long long* red = reinterpret_cast<unsigned long long*>(ctrl + kTcCtrlBytes);  // [4 warps][NT]
  const uint32_t b_off = (PAIRED ? 2u : 1u) * (uint32_t)a.ka * A_ATOM;  // weights: [ka][PAIRED ? 2 : 1][128][64]

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(tfull + b), 1);
      mbar_init(smem_u32(tempty + b), EW * CG);  // one arrival per epilogue warp (of both CTAs)
    }

    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (ARGMAX)
    for (int j = threadIdx.x; j < 4 * NT; j += blockDim.x) red[j] = 0ull;
  if (warp == 1) {
    if (CG == 2) {
      tmem_alloc_cg2(smem_u32(tmem_slot), a.tmem_cols);
      tmem_relinquish_cg2();
    } else {
      tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
      tmem_relinquish();
    }
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (CG == 2) cluster_sync();  // both CTAs' barriers are initialised before any arrival crosses over
  pdl_trigger();
  int issued = 0;  // k-block stages the producer issued (its drain after an abort)

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (converged) and waits on the barriers; one
    // elected lane arms the barriers and issues the copies.  Stage index and
    // phase advance incrementally: no division per k block.
    const uint64_t pol_w = l2_policy_evict_first();  // weights: read once
    const uint64_t pol_x = l2_policy_evict_last();   // activations: re-read by every weight tile
    // wait-expiry test: CTA 0 never arms this stage, so the MMA warp's wait on it runs out
    const int drop = blockIdx.x == 0 ? a.drop_stage : -1;
    const uint32_t tx = (uint32_t)CG * a.stage_bytes;  // the leader's barrier counts both CTAs' copies
    auto fbar = [&](int st) { return CG == 2 ? mapa_shared(smem_u32(full + st), 0) : smem_u32(full + st); };
    // the weights do not depend on earlier kernels: start the first stages now
    int npre = 0;
    if (BAL) {  // the first S k blocks of the range, across pieces
      Sched s0 = sched_begin<EPI, CG>(a, 1);
      Unit w;
      while (npre < S && sched_next<EPI, CG>(a, s0, 1, w))
        for (int kb = w.kb0; kb < w.kb1 && npre < S; ++kb, ++npre)
          if (npre != drop && elect_one()) {
            const uint32_t sa = smem_u32(smem + (size_t)npre * a.stage_bytes);
            mbar_expect_tx(smem_u32(full + npre), a.stage_bytes);
            issue_w<EPI, CG>(&tmW, a, sa, smem_u32(full + npre), kb * a.ka, w.tile_f, pol_w);
          }
    } else if ((a.n_t == 1 || a.tok_major) &&
               (int)blockIdx.x / CG < U / a.n_t * min(a.n_t, (a.n_tok_min + BN - 1) / BN)) {
      // the CTA's first unit exists whatever the row count (it lies within the token tiles of
      // the rows that certainly exist), and its weight tile does not depend on the count
      const Unit w = decode_unit(a, (int)blockIdx.x / CG, 1, (a.n_f + CG - 1) / CG);
      npre = min(S, w.kb1 - w.kb0);
      if (elect_one())
        for (int i = 0; i < npre; ++i) {
          if (i == drop) continue;
          const uint32_t sa = smem_u32(smem + (size_t)i * a.stage_bytes);
          if (leader) mbar_expect_tx(smem_u32(full + i), tx);
          issue_w<EPI, CG>(&tmW, a, sa, fbar(i), (w.kb0 + i) * a.ka, CG * w.tile_f + (int)rank, pol_w);
        }
    }
    __syncwarp();
    const int n_tok_early = a.meta_ready ? effective_ntok(a) : 0;
    pdl_wait();
    const int n_tok = a.meta_ready ? n_tok_early : effective_ntok(a);
    const int ntl = live_token_tiles(a, n_tok);
    int it = 0, s = 0;
    uint32_t ph = 0;  // (it / S) & 1
    bool stop = false;
    Sched sc = sched_begin<EPI, CG>(a, ntl);
    Unit w;
    while (!stop && sched_next<EPI, CG>(a, sc, ntl, w)) {
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
        const uint32_t sa = smem_u32(smem + (size_t)s * a.stage_bytes);
        if (it >= npre && it >= S) {
          const bool ok = mbar_wait(smem_u32(empty + s), ph ^ 1u, a.err, abort_flag, a.wait_ns);
          if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
            stop = true;
            break;
          }
        }
        if (it != drop && elect_one()) {
          const uint32_t fb = fbar(s);
          if (it >= npre) {
            if (leader) mbar_expect_tx(smem_u32(full + s), tx);
            issue_w<EPI, CG>(&tmW, a, sa, fb, kb * a.ka, CG * w.tile_f + (int)rank, pol_w);
          }
          if (CG == 2)
            tma_load_3d_pair(sa + b_off, &tmX, fb, 0, w.tile_t * BN + (int)rank * BNL, kb * a.ka, pol_x);
          else
            tma_load_3d(sa + b_off, &tmX, fb, 0, w.tile_t * BN, kb * a.ka, pol_x);
        }
        __syncwarp();
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    issued = it;
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (the leader of a pair)
    // Converged warp; the elected lane issues every MMA and commit.
    if (CG == 1 || leader) {
      const int n_tok_early = a.meta_ready ? effective_ntok(a) : 0;
      pdl_wait();
      const int n_tok = a.meta_ready ? n_tok_early : effective_ntok(a);
      const int ntl = live_token_tiles(a, n_tok);
      const uint32_t idesc = idesc_bf16(kTcBM * CG, BN);
      int i = 0, s = 0;
      uint32_t ph = 0;  // (it / S) & 1 over this CTA's k blocks
      bool stop = false;
      Sched sc = sched_begin<EPI, CG>(a, ntl);
      Unit w;
      while (!stop && sched_next<EPI, CG>(a, sc, ntl, w)) {
        const int buf = i % a.nbuf;
        if (i >= a.nbuf) {
          const bool ok =
              mbar_wait(smem_u32(tempty + buf), (uint32_t)((i / a.nbuf) - 1) & 1u, a.err, abort_flag, a.wait_ns);
          if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
            stop = true;
            break;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * a.acc_stride);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const bool ok = mbar_wait(smem_u32(full + s), ph, a.err, abort_flag, a.wait_ns);
          if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
            stop = true;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sa = smem_u32(smem + (size_t)s * a.stage_bytes);
#pragma unroll
            for (int at = 0; at < 2; ++at) {  // the stage's k atoms (a.ka of them)
              if (at < a.ka) {
                const uint64_t da = sdesc_k_sw128(sa + (uint32_t)(PAIRED ? 2 * at : at) * A_ATOM);
                const uint64_t da2 = sdesc_k_sw128(sa + (uint32_t)(2 * at + 1) * A_ATOM);
                const uint64_t db = sdesc_k_sw128(sa + b_off + (uint32_t)(at * BNL * kTcBK * 2));
#pragma unroll
                for (int kk = 0; kk < kTcBK / 16; ++kk) {
                  const uint32_t accum = (kb > w.kb0 || at > 0 || kk > 0) ? 1u : 0u;
                  if (CG == 2) {
                    tc_mma_bf16_pair(d, da + 2 * kk, db + 2 * kk, idesc, accum);
                    if (PAIRED) tc_mma_bf16_pair(d + (uint32_t)BN, da2 + 2 * kk, db + 2 * kk, idesc, accum);
                  } else {
                    tc_mma_bf16(d, da + 2 * kk, db + 2 * kk, idesc, accum);
                    if (PAIRED) tc_mma_bf16(d + (uint32_t)BN, da2 + 2 * kk, db + 2 * kk, idesc, accum);
                  }
                }
              }
            }
            if (CG == 2) tc_commit_pair(smem_u32(empty + s));
            else tc_commit(smem_u32(empty + s));
          }
          __syncwarp();
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (elect_one()) {
          if (CG == 2) tc_commit_pair(smem_u32(tfull + buf));
          else tc_commit(smem_u32(tfull + buf));
        }
        __syncwarp();
        ++i;
      }
      // After a wait gave up: every MMA issued so far completes before the tensor memory is
      // freed (the last commit tracks all of them).
      if (stop && i > 0) {
        const int lb = (i - 1) % a.nbuf;
        mbar_wait(smem_u32(tfull + lb), (uint32_t)((i - 1) / a.nbuf) & 1u, a.err, nullptr, a.wait_ns);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..9)
    // Two warps per TMEM lane quarter: each takes every other 16-column chunk of the
    // accumulator, so that an epilogue (argmax over a 224-token tile: ~10 us with one warp
    // per quarter, as long as the next unit's MMAs) stays hidden behind the next unit.
    const int n_tok_early = a.meta_ready ? effective_ntok(a) : 0;
    pdl_wait();
    const int n_tok = a.meta_ready ? n_tok_early : effective_ntok(a);
    const int q = warp & 3;                // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;         // which half of the column chunks (0 with four warps)
    const int hs = EW >> 2;                // chunk stride: the number of halves
    const int r = q * 32 + lane;           // row of the tile = TMEM lane
    unsigned long long* red_w = red + (size_t)q * NT;  // per quarter; the halves' columns are disjoint
    const int ntl = live_token_tiles(a, n_tok);
    int i = 0;
    Sched sc = sched_begin<EPI, CG>(a, ntl);
    Unit w;
    while (sched_next<EPI, CG>(a, sc, ntl, w)) {
      const int buf = i % a.nbuf;
      const int tbase = w.tile_t * BN;
      // QKV: the tile's token positions and KV slots, loaded once per unit by the epilogue
      // warps into shared memory (two buffers by unit parity, so the next unit's loads never
      // overwrite a buffer still being read) instead of a round trip per chunk, while the
      // unit's MMAs run.  Every epilogue warp passes the barrier once per unit.
      int* pos_s = nullptr;
      long long* slot_s = nullptr;
      if (EPI == EPI_QKV_ROPE && a.k_splits == 1) {
        slot_s = reinterpret_cast<long long*>(red) + (size_t)(i & 1) * BN;
        pos_s = reinterpret_cast<int*>(reinterpret_cast<long long*>(red) + 2 * (size_t)BN) + (size_t)(i & 1) * BN;
        for (int t = threadIdx.x - 64; t < BN; t += 32 * EW) {
          const int tok = tbase + t;
          pos_s[t] = tok < n_tok ? a.tok_pos[tok] : 0;
          slot_s[t] = tok < n_tok ? a.tok_slot[tok] : -1;
        }
        named_bar_sync(1, 32 * EW);
      }
      // after an abort the accumulator may be incomplete: skip its epilogue
      const bool ok =
          mbar_wait(smem_u32(tfull + buf), (uint32_t)(i / a.nbuf) & 1u, a.err, abort_flag, a.wait_ns) && !*abort_flag;
      tc_fence_after();
      const int tf = CG * w.tile_f + (int)rank;  // this CTA's 128-row weight tile
      const int unit = tf * kTcBM + r;
      const uint32_t tl = tmem + (uint32_t)(buf * a.acc_stride) + ((uint32_t)(q * 32) << 16);
      if (BAL && ok && w.bnd >= 0) {
        argmax_piece(a, w, tl, unit, n_tok, red_w, r, lane, h, hs);
      } else if (ok && a.k_splits == 1) {
        const float2 tf2 = (EPI == EPI_QKV_ROPE) ? rope_tf(a, unit) : make_float2(0.f, 0.f);
        for (int c = h; c < BN / 16; c += hs) {
          float v[16], v2[16];
          tmem_load16(tl + (uint32_t)(c * 16), v);
          if (PAIRED) tmem_load16(tl + (uint32_t)(BN + c * 16), v2);
          if (ARGMAX)
            argmax16(a, unit, tbase + c * 16, n_tok, v, red_w + tbase + c * 16, lane);
          else
            apply16<EPI>(a, unit, tbase + c * 16, n_tok, v, v2, tf2, pos_s + c * 16, slot_s + c * 16);
        }
      } else if (ok && tf < a.n_f) {
        // split K (one unit per CTA): this split's fp32 partial tile straight from TMEM to
        // the workspace, column-major ([plane][token column][128 rows]: a warp's stores of
        // one column are 128 contiguous bytes), at the unit's index over the live token
        // tiles.  The next kernel sums the splits.
        const size_t pu = ((size_t)tf * ntl + w.tile_t) * a.k_splits + w.split;
        float* P = a.partial + pu * (PAIRED ? 2 : 1) * BN * kTcBM + r;
        const int cend = (PAIRED ? 2 : 1) * BN;
        // 64-column TMEM loads at 64-aligned columns; the halves take alternate loads
        for (int c = 0; c < cend;) {
          if ((c & 63) == 0 && c + 64 <= cend) {
            if (((c >> 6) & (hs - 1)) == h) {
              float v[64];
              tmem_load64(tl + (uint32_t)c, v);
#pragma unroll
              for (int j = 0; j < 64; ++j) P[(size_t)(c + j) * kTcBM] = v[j];
            }
            c += 64;
          } else {
            if (((c >> 4) & (hs - 1)) == h) {
              float v[16];
              tmem_load16(tl + (uint32_t)c, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) P[(size_t)(c + j) * kTcBM] = v[j];
            }
            c += 16;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // accumulator free for a later unit
        if (CG == 2) mbar_arrive_cluster(mapa_shared(smem_u32(tempty + buf), 0));
        else mbar_arrive(smem_u32(tempty + buf));
      }
      ++i;
    }
    if (ARGMAX) {
      const int ET = 32 * EW;  // epilogue threads
      named_bar_sync(1, ET);
      const int ethread = threadIdx.x - 64;
      for (int j = ethread; j < NT; j += ET) {  // key index = token = tile_t * BN + column
        const unsigned long long k =
            umax64(umax64(red[j], red[NT + j]), umax64(red[2 * NT + j], red[3 * NT + j]));
        if (j < n_tok && k != 0ull) atomicMax(a.keys + j, k);
      }
      __threadfence();
      named_bar_sync(1, ET);
      if (ethread == 0) {
        const int old = atomicAdd(a.done_counter, 1);
        *last_flag = (old == (int)gridDim.x - 1) ? 1 : 0;
      }
      named_bar_sync(1, ET);
      if (*last_flag) {
        __threadfence();
        argmax_finish(a, n_tok, ethread, ET);
        if (ethread == 0) *a.done_counter = 0;
        if (a.has_verify) {  // every draft token is known: verify them here
          named_bar_sync(1, ET);
          for (int b = ethread; b < a.verify.B; b += ET) verify_seq(a.verify, b);
        }
      }
    }
  }

  __syncthreads();
  // After a wait gave up (every role has left its loop, so the flag is final): leave no bulk
  // copy in flight into this CTA's shared memory.  The stages still in the ring are the last
  // S issued; each wait is bounded.  In a pair the leader's barriers count both CTAs' copies,
  // so the leader drains for both (the peer stops issuing when a wait of its own gives up,
  // at least one wait limit after its last copy was issued).
  if (warp == 0 && *abort_flag && leader) {
    const int drop = blockIdx.x == 0 ? a.drop_stage : -1;
    for (int i = issued > S ? issued - S : 0; i < issued; ++i)
      if (i != drop) mbar_wait(smem_u32(full + (i % S)), (uint32_t)(i / S) & 1u, a.err, nullptr, a.wait_ns);
    __syncwarp();
  }
  __syncthreads();
  if (CG == 2) cluster_sync();  // neither CTA frees its tensor memory or exits while the pair works
  if (warp == 1) {
    tc_fence_after();
    if (CG == 2) tmem_dealloc_cg2(tmem, a.tmem_cols);
    else tmem_dealloc(tmem, a.tmem_cols);
  }
}

// Opt every GEMM variant into the largest dynamic shared memory once per
// device (an upper bound only; each launch passes its own size).
template <int EPI, int CG>
static cudaError_t ensure_smem_attr() {
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<EPI, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemOptIn);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

template <int EPI, int CG>
static cudaError_t launch_tc_typed(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a, int grid,
                                   size_t smem, cudaStream_t s) {
  const cudaError_t e = ensure_smem_attr<EPI, CG>();
  if (e != cudaSuccess) return e;
  if constexpr (CG == 1) {
    return launch_pdl(gemm_tc_kernel<EPI, 1>, dim3(grid), dim3(gemm_tc_threads(a.bn)), smem, s, tmW, tmX, a);
  } else {
  // a pair per cluster, with programmatic dependent launch
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gemm_tc_threads(a.bn));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<EPI, 2>, tmW, tmX, a);
  }
}

cudaError_t launch_gemm_tc(int epi, int cg, const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                           int grid, size_t smem, cudaStream_t s) {
  if (cg == 2) {
    if (grid % 2 != 0) return cudaErrorInvalidValue;
    switch (epi) {
      case EPI_STORE_F32: return launch_tc_typed<EPI_STORE_F32, 2>(tmW, tmX, a, grid, smem, s);
      case EPI_ADD_F32: return launch_tc_typed<EPI_ADD_F32, 2>(tmW, tmX, a, grid, smem, s);
      case EPI_SWIGLU: return launch_tc_typed<EPI_SWIGLU, 2>(tmW, tmX, a, grid, smem, s);
      case EPI_QKV_ROPE: return launch_tc_typed<EPI_QKV_ROPE, 2>(tmW, tmX, a, grid, smem, s);
      case EPI_ARGMAX: return launch_tc_typed<EPI_ARGMAX, 2>(tmW, tmX, a, grid, smem, s);
    }
    return cudaErrorInvalidValue;
  }
  switch (epi) {
    case EPI_STORE_F32: return launch_tc_typed<EPI_STORE_F32, 1>(tmW, tmX, a, grid, smem, s);
    case EPI_ADD_F32: return launch_tc_typed<EPI_ADD_F32, 1>(tmW, tmX, a, grid, smem, s);
    case EPI_SWIGLU: return launch_tc_typed<EPI_SWIGLU, 1>(tmW, tmX, a, grid, smem, s);
    case EPI_QKV_ROPE: return launch_tc_typed<EPI_QKV_ROPE, 1>(tmW, tmX, a, grid, smem, s);
    case EPI_ARGMAX: return launch_tc_typed<EPI_ARGMAX, 1>(tmW, tmX, a, grid, smem, s);
    case EPI_ARGMAX_BAL: return launch_tc_typed<EPI_ARGMAX_BAL, 1>(tmW, tmX, a, grid, smem, s);
  }
  return cudaErrorInvalidValue;
}

// Clusters of two CTAs of this GEMM that fit on the GPU at once (0 if the query fails).
int gemm_tc_max_pairs(int epi, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (epi) {
    case EPI_STORE_F32:
      if (ensure_smem_attr<EPI_STORE_F32, 2>() == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<EPI_STORE_F32, 2>, &cfg);
      break;
    case EPI_ADD_F32:
      if (ensure_smem_attr<EPI_ADD_F32, 2>() == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<EPI_ADD_F32, 2>, &cfg);
      break;
    case EPI_SWIGLU:
      if (ensure_smem_attr<EPI_SWIGLU, 2>() == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<EPI_SWIGLU, 2>, &cfg);
      break;
    case EPI_QKV_ROPE:
      if (ensure_smem_attr<EPI_QKV_ROPE, 2>() == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<EPI_QKV_ROPE, 2>, &cfg);
      break;
    case EPI_ARGMAX:
      if (ensure_smem_attr<EPI_ARGMAX, 2>() == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<EPI_ARGMAX, 2>, &cfg);
      break;
  }
  return e == cudaSuccess ? n : 0;
}

// ============================================================================= split-K finish
//
// Sum of the split-K partials of a QKV or gate/up GEMM and its epilogue, one
// thread per output unit and kFinishTok consecutive tokens: RoPE + q + KV-cache
// write, or SwiGLU.  A block of 128 threads covers one weight tile's 128 units;
// every load of a thread (all splits of both planes, the tokens' positions and
// slots) is in flight before the sums, which run in split order.
constexpr int kFinishThreads = 128;
constexpr int kFinishMaxSplits = 16;
constexpr int kFinishTok = 2;

template <int EPI, int MAXS>  // MAXS >= k_splits: bounds the registers holding the loads
__global__ void __launch_bounds__(kFinishThreads) splitk_finish_kernel(const GemmArgs a) {
  const int n_tok_early = a.meta_ready ? effective_ntok(a) : 0;
  pdl_wait();
  pdl_trigger();
  const int n_tok = a.meta_ready ? n_tok_early : effective_ntok(a);
  const int ntl = live_token_tiles(a, n_tok);
  const int ns = a.k_splits, BN = a.bn;
  const size_t tile_floats = (size_t)2 * BN * kTcBM;  // both planes
  const int r = threadIdx.x;
  const int groups = (n_tok + kFinishTok - 1) / kFinishTok;
  const long long items = (long long)a.n_f * groups;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int tile_f = (int)(it / groups), t0 = (int)(it - (long long)tile_f * groups) * kFinishTok;
    const int unit = tile_f * kTcBM + r;
    if (unit >= a.n_out) continue;
    float x1[kFinishTok][MAXS], x2[kFinishTok][MAXS];
    int pos[kFinishTok];
    long long slot[kFinishTok];
#pragma unroll
    for (int k = 0; k < kFinishTok; ++k) {
      const int t = t0 + k;
      if (t < n_tok) {
        const int tile_t = t / BN, tt = t - tile_t * BN;
        const float* p = a.partial + (size_t)(tile_f * ntl + tile_t) * ns * tile_floats + (size_t)tt * kTcBM + r;
#pragma unroll
        for (int sp = 0; sp < MAXS; ++sp)
          if (sp < ns) {
            x1[k][sp] = __ldcg(p + (size_t)sp * tile_floats);
            x2[k][sp] = __ldcg(p + (size_t)sp * tile_floats + (size_t)BN * kTcBM);
          }
        if (EPI == EPI_QKV_ROPE) {
          pos[k] = a.tok_pos[t];
          slot[k] = a.tok_slot[t];
        }
      }
    }
    const float2 tf = (EPI == EPI_QKV_ROPE) ? rope_tf(a, unit) : make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kFinishTok; ++k) {
      const int t = t0 + k;
      if (t >= n_tok) break;
      float v = 0.f, v2 = 0.f;
#pragma unroll
      for (int sp = 0; sp < MAXS; ++sp)
        if (sp < ns) {
          v += x1[k][sp];
          v2 += x2[k][sp];
        }
      if (EPI == EPI_SWIGLU) {
        static_cast<__nv_bfloat16*>(a.out_act)[(size_t)t * a.ld_out + unit] = __float2bfloat16_rn(silu(v) * v2);
      } else {
        qkv_store<__nv_bfloat16>(a, unit, t, v, v2, tf, pos[k], slot[k]);
      }
    }
  }
}

template <int EPI>
static cudaError_t launch_finish_typed(const GemmArgs& a, int grid, cudaStream_t s) {
  if (a.k_splits <= 4) return launch_pdl(splitk_finish_kernel<EPI, 4>, dim3(grid), dim3(kFinishThreads), 0, s, a);
  if (a.k_splits <= 8) return launch_pdl(splitk_finish_kernel<EPI, 8>, dim3(grid), dim3(kFinishThreads), 0, s, a);
  return launch_pdl(splitk_finish_kernel<EPI, kFinishMaxSplits>, dim3(grid), dim3(kFinishThreads), 0, s, a);
}

cudaError_t launch_splitk_finish(int epi, const GemmArgs& a, int sms, cudaStream_t s) {
  if (a.k_splits > kFinishMaxSplits) return cudaErrorInvalidValue;
  const long long items = (long long)a.n_f * ((a.n_tok + kFinishTok - 1) / kFinishTok);
  const int grid = (int)std::min<long long>(items, 16LL * sms);
  if (grid <= 0) return cudaSuccess;
  if (epi == EPI_QKV_ROPE) return launch_finish_typed<EPI_QKV_ROPE>(a, grid, s);
  if (epi == EPI_SWIGLU) return launch_finish_typed<EPI_SWIGLU>(a, grid, s);
  return cudaErrorInvalidValue;
}

// ============================================================================= fp32 CUDA-core kernel
// One warp per output unit (a feature, a gate/up pair or a RoPE pair): lanes
// split the reduction, each lane keeps partial sums for 8 tokens at a time,
// then a butterfly reduction gives every lane the full sums.

constexpr int kF32Warps = 8;
constexpr int kF32Tok = 8;

template <int EPI>
__global__ void __launch_bounds__(kF32Warps * 32) gemm_f32_kernel(const GemmArgs a) {
  constexpr bool PAIRED = (EPI == EPI_SWIGLU || EPI == EPI_QKV_ROPE);
  __shared__ int last_s;
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kF32Warps + warp;
  int n_tok = a.n_tok;
  if (a.n_tok_dev != nullptr) n_tok = min(n_tok, *a.n_tok_dev);
  const float* W = static_cast<const float*>(a.W);
  const float* X = static_cast<const float*>(a.X);
  if (unit < a.n_out) {
    int row1 = unit, row2 = unit;
    if (EPI == EPI_SWIGLU) row2 = a.n_out + unit;
    if (EPI == EPI_QKV_ROPE) {
      const int half = a.head_dim >> 1;
      const int head = unit / half, i = unit - head * half;
      row1 = head * a.head_dim + i;
      row2 = row1 + half;
    }
    const float2 tf = (EPI == EPI_QKV_ROPE) ? rope_tf(a, unit) : make_float2(0.f, 0.f);
    const float* w1 = W + (size_t)row1 * a.k_dim;
    const float* w2 = W + (size_t)row2 * a.k_dim;
    for (int t0 = 0; t0 < n_tok; t0 += kF32Tok) {
      float acc1[kF32Tok], acc2[kF32Tok];
#pragma unroll
      for (int j = 0; j < kF32Tok; ++j) acc1[j] = acc2[j] = 0.f;
      for (int k = lane; k < a.k_dim; k += 32) {
        const float wa = w1[k];
        const float wb = PAIRED ? w2[k] : 0.f;
#pragma unroll
        for (int j = 0; j < kF32Tok; ++j)
          if (t0 + j < n_tok) {
            const float x = X[(size_t)(t0 + j) * a.ldx + k];
            acc1[j] += wa * x;
            if (PAIRED) acc2[j] += wb * x;
          }
      }
#pragma unroll
      for (int j = 0; j < kF32Tok; ++j)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          acc1[j] += __shfl_xor_sync(0xFFFFFFFFu, acc1[j], o);
          if (PAIRED) acc2[j] += __shfl_xor_sync(0xFFFFFFFFu, acc2[j], o);
        }
#pragma unroll
      for (int j = 0; j < kF32Tok; ++j) {
        const int t = t0 + j;
        if (t >= n_tok || lane != j) continue;
        if (EPI == EPI_ARGMAX) {
          if (!isfinite(acc1[j])) set_err(a.err, PE_DEV_NONFINITE);
          if (a.logits_dbg != nullptr) a.logits_dbg[(size_t)t * a.n_out + unit] = acc1[j];
          atomicMax(a.keys + t, argmax_key(acc1[j], (uint32_t)unit));
        } else {
          epi_elem<EPI, float>(a, unit, t, acc1[j], acc2[j], tf);
        }
      }
    }
  }
  if (EPI == EPI_ARGMAX) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_s = (atomicAdd(a.done_counter, 1) == (int)gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (last_s) {
      __threadfence();
      argmax_finish(a, n_tok, threadIdx.x, blockDim.x);
      if (threadIdx.x == 0) *a.done_counter = 0;
    }
  }
}

cudaError_t launch_gemm_f32(int epi, const GemmArgs& a, cudaStream_t s) {
  const int grid = (a.n_out + kF32Warps - 1) / kF32Warps;
  const int threads = kF32Warps * 32;
  switch (epi) {
    case EPI_STORE_F32: return launch_pdl(gemm_f32_kernel<EPI_STORE_F32>, dim3(grid), dim3(threads), 0, s, a);
    case EPI_ADD_F32: return launch_pdl(gemm_f32_kernel<EPI_ADD_F32>, dim3(grid), dim3(threads), 0, s, a);
    case EPI_SWIGLU: return launch_pdl(gemm_f32_kernel<EPI_SWIGLU>, dim3(grid), dim3(threads), 0, s, a);
    case EPI_QKV_ROPE: return launch_pdl(gemm_f32_kernel<EPI_QKV_ROPE>, dim3(grid), dim3(threads), 0, s, a);
    case EPI_ARGMAX: return launch_pdl(gemm_f32_kernel<EPI_ARGMAX>, dim3(grid), dim3(threads), 0, s, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pe
