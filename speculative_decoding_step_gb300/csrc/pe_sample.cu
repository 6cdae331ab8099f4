// Non-greedy drafting and verification by rejection sampling (speculative sampling).
//
// vLLM Speculators: parallel drafting for speculative decoding, closing paragraph of
// "Production integration in vLLM": verification by rejection sampling keeps the
// target model's output distribution.  The steps are the standard scheme that does
// so: draft tokens drawn from the drafter's temperature softmax q, draft k accepted
// with probability min(1, p_k / q_k), the first rejected one replaced by a draw from
// the normalised residual max(0, p_k - q_k), and a bonus token drawn from the target
// when every draft is accepted.  Every random number is a caller-supplied uniform.
//
// A draw over a vocabulary row runs in two launches:
//   phase A  many CTAs per row, each over a contiguous range of 512-entry steps: one
//            statistic pair per step into the workspace (drafting: the step's
//            maximum of z = logit / T and its sum of exp(z - that maximum), in base
//            2; verification: the step's sums of residual weights and of target
//            probabilities)
//   phase B  one warp per row: the row total from the step statistics in a fixed
//            order, the step where the running sum passes u times the total, and the
//            entry within that step (one reload of 512 entries)
// Draws are deterministic: every sum runs in a fixed order (a step: each lane's 16
// consecutive entries in order, then a butterfly over the lanes; the steps: each lane
// of the phase B warp adds a contiguous range of steps in order, then the lane totals
// are added in lane order).  The draw is the first entry at which that running sum
// exceeds u times the total; an entry of weight zero is never drawn, and where
// rounding leaves no such entry the last entry of positive weight is taken.
#include <math.h>

#include <algorithm>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

constexpr int kSampPerLane = 16;   // consecutive vocabulary entries of a lane in a step
constexpr int kSampStep = 32 * kSampPerLane;  // entries per step
constexpr int kSampBatch = 2;      // steps whose loads a warp keeps in flight together
constexpr int kSampAThreads = 256;
constexpr int kSampCtasPerSm = 4;  // phase A CTAs resident per SM (256 threads, <= 64 registers)
constexpr int kSampBWarps = 4;     // phase B rows per CTA (one warp each)

PE_DEV float samp_warp_sum(float v) {  // every lane gets the same value
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
PE_DEV float samp_warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
PE_DEV float samp_warp_scan(float v) {  // inclusive, lane order
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// A lane's 16 consecutive values of a row from v0 (a multiple of 16); zeros past n.
// `vec`: the row is 16-byte aligned and n a multiple of 4, so vector loads serve.
struct Lane16 {
  float v[kSampPerLane];
};
PE_DEV Lane16 ld16(const float* row, int v0, int n, bool vec) {
  Lane16 r;
#pragma unroll
  for (int q = 0; q < kSampPerLane; q += 4) {
    if (vec && v0 + q < n) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(row + v0 + q));
      r.v[q] = x.x; r.v[q + 1] = x.y; r.v[q + 2] = x.z; r.v[q + 3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) r.v[q + e] = v0 + q + e < n ? __ldg(row + v0 + q + e) : 0.f;
    }
  }
  return r;
}
PE_DEV Lane16 zero16() {
  Lane16 r;
#pragma unroll
  for (int q = 0; q < kSampPerLane; ++q) r.v[q] = 0.f;
  return r;
}
PE_DEV bool vec_ok(const float* p, int n) { return (n & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
PE_DEV float sum16(const Lane16& w) {  // in index order
  float t = 0.f;
#pragma unroll
  for (int q = 0; q < kSampPerLane; ++q) t += w.v[q];
  return t;
}

// Exponentials run in base 2: z2 = logit * (log2(e) / T), weights 2^(z2 - m2) with the
// hardware approximation (relative error a few units in the last place, far below the
// rounding of the running sums).
PE_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 2^(z2 - m2) of a lane's logits (zero past n).  m2 is the maximum of a range that holds
// these entries; when it is -inf every entry is -inf (a masked range) and every weight 0
// (not 2^(-inf + inf), which is NaN).
PE_DEV Lane16 exp16(const Lane16& x, int v0, int n, float inv_t2, float m2) {
  Lane16 r;
  const bool empty = m2 == -INFINITY;
#pragma unroll
  for (int q = 0; q < kSampPerLane; ++q) r.v[q] = v0 + q < n && !empty ? ex2(x.v[q] * inv_t2 - m2) : 0.f;
  return r;
}
// max(0, p - q) of a lane's entries (zero past n), q = 2^(z2 - lse2)
PE_DEV Lane16 resid16(const Lane16& p, const Lane16& x, int v0, int n, float inv_t2, float lse2) {
  Lane16 r;
#pragma unroll
  for (int q = 0; q < kSampPerLane; ++q)
    r.v[q] = v0 + q < n ? fmaxf(0.f, p.v[q] - ex2(x.v[q] * inv_t2 - lse2)) : 0.f;
  return r;
}
constexpr float kLog2e = 1.4426950408889634f;

// Accepted count of sequence b, by one whole warp (lane j tests draft k0 + j, 32 at a
// time; the first failing test ends the count); -1 - k when draft k is outside the
// vocabulary (counted as rejected).  Every lane returns the same value.
PE_DEV int accept_count(const VerifySampledArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  for (int k0 = 0; k0 < a.K; k0 += 32) {
    const int k = k0 + lane;
    bool fail = false, bad = false;
    if (k < a.K) {
      const int row = b * a.K + k;
      const int x = a.drafts[row];
      if (x < 0 || x >= a.V) {
        bad = fail = true;
      } else {
        const float qx = ex2(a.logits[(size_t)row * a.V + x] * a.inv_t2 - a.lse[row] * kLog2e);
        const float px = a.target_probs[((size_t)b * (a.K + 1) + k) * a.V + x];
        fail = !(a.u_accept[row] * qx < px);  // accepted with probability min(1, px / qx)
      }
    }
    const unsigned f = __ballot_sync(0xFFFFFFFFu, fail);
    if (f) {
      const int j = __ffs(f) - 1;
      const bool jb = __shfl_sync(0xFFFFFFFFu, bad, j);
      return jb ? -1 - (k0 + j) : k0 + j;
    }
  }
  return a.K;
}

// Phase A: this warp's contiguous range of steps within the CTA's range of the row.
PE_DEV void step_range(int steps, int g, int G, int& s_lo, int& s_hi) {
  const int per_cta = (steps + G - 1) / G;
  const int c_lo = min(steps, g * per_cta), c_hi = min(steps, c_lo + per_cta);
  const int warps = kSampAThreads / 32, warp = threadIdx.x >> 5;
  const int per_w = (c_hi - c_lo + warps - 1) / warps;
  s_lo = min(c_hi, c_lo + warp * per_w);
  s_hi = min(c_hi, s_lo + per_w);
}

__global__ void __launch_bounds__(kSampAThreads, kSampCtasPerSm) sample_stats_kernel(const SampleArgs a) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, lane = threadIdx.x & 31;
  const int V = a.V, steps = (V + kSampStep - 1) / kSampStep;
  const float* l = a.logits + (size_t)row * V;
  const bool vec = vec_ok(l, V);
  float2* st = a.stats + (size_t)row * steps;
  int s_lo, s_hi;
  step_range(steps, blockIdx.x, gridDim.x, s_lo, s_hi);
  bool bad = false;
  for (int s0 = s_lo; s0 < s_hi; s0 += kSampBatch) {
    Lane16 x[kSampBatch];
#pragma unroll
    for (int j = 0; j < kSampBatch; ++j)
      x[j] = s0 + j < s_hi ? ld16(l, (s0 + j) * kSampStep + kSampPerLane * lane, V, vec) : zero16();
#pragma unroll
    for (int j = 0; j < kSampBatch; ++j) {
      if (s0 + j < s_hi) {
        const int v0 = (s0 + j) * kSampStep + kSampPerLane * lane;
        if ((s0 + j + 1) * kSampStep <= V) {
          // a step inside the row: no bounds per entry, and the non-finite check once on
          // the sum (a NaN logit makes its weight NaN, a +inf one makes the maximum +inf
          // and its weight 2^(inf - inf) = NaN), with the same values as the general path
          float lm = -INFINITY;
#pragma unroll
          for (int q = 0; q < kSampPerLane; ++q) lm = fmaxf(lm, x[j].v[q] * a.inv_t2);
          const float m = samp_warp_max(lm);
          float t = 0.f;
          if (m != -INFINITY) {
#pragma unroll
            for (int q = 0; q < kSampPerLane; ++q) t += ex2(x[j].v[q] * a.inv_t2 - m);
          }
          const float sm = samp_warp_sum(t);
          bad |= sm != sm;
          if (lane == 0) st[s0 + j] = make_float2(m, sm);
        } else {
          float lm = -INFINITY;
#pragma unroll
          for (int q = 0; q < kSampPerLane; ++q) {
            if (v0 + q < V) {
              const float z = x[j].v[q] * a.inv_t2;
              bad |= z != z || z == INFINITY;  // NaN or +inf; a -inf logit is a masked entry
              lm = fmaxf(lm, z);
            }
          }
          const float m = samp_warp_max(lm);  // -inf: the whole step is masked, its sum 0
          const float sm = samp_warp_sum(sum16(exp16(x[j], v0, V, a.inv_t2, m)));
          if (lane == 0) st[s0 + j] = make_float2(m, sm);
        }
      }
    }
  }
  if (bad) set_err(a.err, PE_DEV_NONFINITE);
}

__global__ void __launch_bounds__(kSampAThreads, kSampCtasPerSm) verify_stats_kernel(const VerifySampledArgs a) {
  __shared__ int s_acc;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y, lane = threadIdx.x & 31;
  const int V = a.V, K = a.K, steps = (V + kSampStep - 1) / kSampStep;
  if (threadIdx.x < 32) {
    const int c = accept_count(a, b);
    if (threadIdx.x == 0) {
      s_acc = c < 0 ? -1 - c : c;
      if (blockIdx.x == 0) {  // the draw launch takes the count from here, not a recomputation
        a.acc_ws[b] = s_acc;
        if (c < 0) set_err(a.err, PE_DEV_BAD_TOKEN);
      }
    }
  }
  __syncthreads();
  const int acc = s_acc;
  const float* p = a.target_probs + ((size_t)b * (K + 1) + acc) * V;
  const bool pvec = vec_ok(p, V);
  const bool res = acc < K;
  const float* l = res ? a.logits + (size_t)(b * K + acc) * V : p;
  const bool lvec = vec_ok(l, V);
  const float ls2 = res ? a.lse[b * K + acc] * kLog2e : 0.f;
  float2* st = a.stats + (size_t)b * steps;
  int s_lo, s_hi;
  step_range(steps, blockIdx.x, gridDim.x, s_lo, s_hi);
  // one step of both rows in flight (as many bytes as two steps of one row)
  constexpr int kVB = kSampBatch / 2;
  for (int s0 = s_lo; s0 < s_hi; s0 += kVB) {
    Lane16 pp[kVB], x[kVB];
#pragma unroll
    for (int j = 0; j < kVB; ++j) {
      const int v0 = (s0 + j) * kSampStep + kSampPerLane * lane;
      const bool live = s0 + j < s_hi;
      pp[j] = live ? ld16(p, v0, V, pvec) : zero16();
      x[j] = live && res ? ld16(l, v0, V, lvec) : zero16();
    }
#pragma unroll
    for (int j = 0; j < kVB; ++j) {
      if (s0 + j < s_hi) {
        const int v0 = (s0 + j) * kSampStep + kSampPerLane * lane;
        const float sp = samp_warp_sum(sum16(pp[j]));
        const float sr = res ? samp_warp_sum(sum16(resid16(pp[j], x[j], v0, V, a.inv_t2, ls2))) : sp;
        if (lane == 0) st[s0 + j] = make_float2(sr, sp);
      }
    }
  }
}

// Phase B body shared by both draws: the warp of one row finds the step where the running
// sum of step weights sw(s) passes u times their total, then the entry within that step
// from its entry weights ew(v0) (a lane's 16 weights from v0).  Returns the entry (-1 when the
// total is not positive and finite); *total gets the total.
template <typename SW, typename EW>
PE_DEV int warp_draw(int steps, float u, const SW& sw, const EW& ew, float* total) {
  const int lane = threadIdx.x & 31;
  const int per = (steps + 31) / 32;
  const int lo = min(steps, lane * per), hi = min(steps, lo + per);
  float mine = 0.f;
#pragma unroll 8
  for (int s = lo; s < hi; ++s) mine += sw(s);
  // lane totals in lane order: every lane computes the same total and its own prefix
  float tot = 0.f, pre = 0.f;
  for (int i = 0; i < 32; ++i) {
    const float x = __shfl_sync(0xFFFFFFFFu, mine, i);
    if (i == lane) pre = tot;
    tot += x;
  }
  *total = tot;
  if (!(tot > 0.f) || !isfinite(tot)) return -1;
  const float t = u * tot;
  // the lane whose range the running sum passes t in (else the last with weight)
  const unsigned hit_l = __ballot_sync(0xFFFFFFFFu, mine > 0.f && pre + mine > t);
  const unsigned pos_l = __ballot_sync(0xFFFFFFFFu, mine > 0.f);
  const bool cross = hit_l != 0;
  const int L = cross ? __ffs(hit_l) - 1 : 31 - __clz(pos_l);  // pos_l != 0: tot > 0
  float r = __shfl_sync(0xFFFFFFFFu, pre, L);
  const int a_lo = min(steps, L * per), a_hi = min(steps, a_lo + per);
  // the step within lane L's range, 32 steps at a time
  int sc = -1, last_s = -1;
  for (int c0 = a_lo; c0 < a_hi && sc < 0; c0 += 32) {
    const float x = c0 + lane < a_hi ? sw(c0 + lane) : 0.f;
    const float inc = samp_warp_scan(x);
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, x > 0.f);
    if (pos) last_s = c0 + 31 - __clz(pos);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, cross && x > 0.f && r + inc > t);
    if (hit) {
      const int k = __ffs(hit) - 1;
      sc = c0 + k;
      r += __shfl_sync(0xFFFFFFFFu, inc - x, k);
    } else {
      r += __shfl_sync(0xFFFFFFFFu, inc, 31);
    }
  }
  const bool in_step = sc >= 0;
  if (!in_step) sc = last_s;  // lane L's range has weight, so last_s >= 0
  const Lane16 x = ew(sc * kSampStep + kSampPerLane * lane);
  const float lt = sum16(x);
  const float inc = samp_warp_scan(lt);
  float c = r + (inc - lt);
  int first = -1, last = -1;
#pragma unroll
  for (int q = 0; q < kSampPerLane; ++q) {
    c += x.v[q];
    if (x.v[q] > 0.f) {
      last = kSampPerLane * lane + q;
      if (first < 0 && in_step && c > t) first = kSampPerLane * lane + q;
    }
  }
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, first >= 0);
  const unsigned pos = __ballot_sync(0xFFFFFFFFu, last >= 0);
  if (hit) return sc * kSampStep + __shfl_sync(0xFFFFFFFFu, first, __ffs(hit) - 1);
  if (pos) return sc * kSampStep + __shfl_sync(0xFFFFFFFFu, last, 31 - __clz(pos));
  return -1;  // a step of positive total whose entries all rounded to zero
}

__global__ void __launch_bounds__(32 * kSampBWarps) sample_draw_kernel(const SampleArgs a) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * kSampBWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= a.B * a.K) return;
  const int V = a.V, steps = (V + kSampStep - 1) / kSampStep;
  const float2* st = a.stats + (size_t)row * steps;
  const float* l = a.logits + (size_t)row * V;
  const bool vec = vec_ok(l, V);
  float m = -INFINITY;
  for (int s = lane; s < steps; s += 32) m = fmaxf(m, st[s].x);
  m = samp_warp_max(m);
  float tot = 0.f;
  int x = -1;
  if (isfinite(m))
    x = warp_draw(
        steps, a.u[row], [&](int s) { const float2 v = st[s]; return v.x == -INFINITY ? 0.f : v.y * ex2(v.x - m); },
        [&](int v0) { return exp16(ld16(l, v0, V, vec), v0, V, a.inv_t2, m); }, &tot);
  if (lane == 0) {
    if (x < 0) {
      set_err(a.err, PE_DEV_NONFINITE);
      a.drafts[row] = 0;
      a.lse[row] = NAN;
    } else {
      a.drafts[row] = x;
      a.lse[row] = (m + log2f(tot)) * 0.6931471805599453f;  // natural log
    }
  }
}

__global__ void __launch_bounds__(32 * kSampBWarps) verify_draw_kernel(const VerifySampledArgs a) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * kSampBWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const int V = a.V, K = a.K, steps = (V + kSampStep - 1) / kSampStep;
  const int acc = a.acc_ws[b];  // decided once, by the statistics launch
  const float2* st = a.stats + (size_t)b * steps;
  const float* p = a.target_probs + ((size_t)b * (K + 1) + acc) * V;
  const bool pvec = vec_ok(p, V);
  float tot = 0.f;
  int x = -1;
  if (acc < K) {  // the residual of the first rejected draft
    const float* l = a.logits + (size_t)(b * K + acc) * V;
    const bool lvec = vec_ok(l, V);
    const float ls2 = a.lse[b * K + acc] * kLog2e;
    x = warp_draw(
        steps, a.u_resample[b], [&](int s) { return st[s].x; },
        [&](int v0) { return resid16(ld16(p, v0, V, pvec), ld16(l, v0, V, lvec), v0, V, a.inv_t2, ls2); }, &tot);
  }
  if (x < 0)  // every draft accepted, or an empty residual: the target's distribution itself
    x = warp_draw(
        steps, a.u_resample[b], [&](int s) { return st[s].y; }, [&](int v0) { return ld16(p, v0, V, pvec); },
        &tot);
  if (lane == 0) {
    if (x < 0) {
      set_err(a.err, PE_DEV_NONFINITE);  // a target distribution with no positive finite mass
      x = 0;
    }
    a.acc_out[b] = acc;
    a.bonus_out[b] = x;
  }
}

// CTAs per row in phase A: as many as fit on the GPU at once over all rows (one wave),
// at least a batch of steps per warp.
static int phase_a_ctas(int rows, int steps, int sms) {
  const int by_sm = kSampCtasPerSm * sms / rows;
  const int by_steps = std::max(1, steps / (kSampBatch * (kSampAThreads / 32)));
  return std::max(1, std::min(by_sm, by_steps));
}

cudaError_t launch_sample_drafts(const SampleArgs& a, int sms, cudaStream_t s) {
  const int rows = a.B * a.K, steps = (a.V + kSampStep - 1) / kSampStep;
  cudaError_t e =
      launch_pdl(sample_stats_kernel, dim3(phase_a_ctas(rows, steps, sms), rows), dim3(kSampAThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(sample_draw_kernel, dim3((rows + kSampBWarps - 1) / kSampBWarps), dim3(32 * kSampBWarps), 0, s,
                    a);
}

cudaError_t launch_verify_sampled(const VerifySampledArgs& a, int sms, cudaStream_t s) {
  const int steps = (a.V + kSampStep - 1) / kSampStep;
  cudaError_t e =
      launch_pdl(verify_stats_kernel, dim3(phase_a_ctas(a.B, steps, sms), a.B), dim3(kSampAThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(verify_draw_kernel, dim3((a.B + kSampBWarps - 1) / kSampBWarps), dim3(32 * kSampBWarps), 0, s,
                    a);
}

size_t sample_stats_bytes(int rows, int vocab) {
  return (size_t)rows * ((vocab + kSampStep - 1) / kSampStep) * sizeof(float2);
}

}  // namespace pe
