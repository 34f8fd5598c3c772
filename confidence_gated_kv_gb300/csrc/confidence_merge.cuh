// Merge of the per-chunk confidence partials of one sequence (one warp).
//
// CONF-KV (gist.science/de/paper/2605.24786, Konfidenzschätzung;
// paper.rainbus.top/paper/2605.24786, 核心方法 and Algorithm 1 steps 3-4):
// c = w_H (1 - H / log V) + w_m sigmoid(log p(1) - log p(2)) + w_p p(1),
// N = N_high if c >= tau else N_low.  From chunk partials (M_j, S_j, T_j)
// with S_j = sum exp(z - M_j), T_j = sum (z - M_j) exp(z - M_j):
// S = sum_j S_j e^(M_j - M), T = sum_j e^(M_j - M) (T_j + (M_j - M) S_j),
// H = log S - T / S, p(1) = e^(z1 - M) / S, log p(1) - log p(2) = z1 - z2.
//
// Arithmetic.  Float64 runs at a small fraction of the fp32 rate on this
// GPU, so the sums are compensated fp32: each running sum is an unevaluated
// pair (hi, lo) updated with Knuth's TwoSum, which keeps the rounding error
// of the additions near 2^-44 relative.  Every term of S and of T has one
// sign (z - M <= 0), so the error of c is set by the fp32 exp and log of
// single terms, a few 1e-8 absolute.
#pragma once
#include <cfloat>
#include "confkv_internal.cuh"

namespace confkv {

struct Top2 {
  float z1, z2;
  int i1;
};

__device__ __forceinline__ Top2 top2_merge(Top2 a, Top2 b) {
  Top2 r;
  if (a.z1 > b.z1 || (a.z1 == b.z1 && a.i1 < b.i1)) {
    r.z1 = a.z1; r.i1 = a.i1; r.z2 = fmaxf(a.z2, b.z1);
  } else {
    r.z1 = b.z1; r.i1 = b.i1; r.z2 = fmaxf(b.z2, a.z1);
  }
  return r;
}

// Compensated fp32 sum: value hi + lo.
struct FSum {
  float hi, lo;
};

// TwoSum: s = a + b exactly as s + e (no multiplications, so no FMA contraction)
__device__ __forceinline__ FSum fsum_add(FSum a, float b) {
  const float s = a.hi + b;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b - bb);
  return FSum{s, a.lo + e};
}

__device__ __forceinline__ FSum fsum_add(FSum a, FSum b) {
  FSum r = fsum_add(a, b.hi);
  r.lo += b.lo;
  return r;
}

__device__ __forceinline__ FSum fsum_shfl_xor(FSum a, int o) {
  return FSum{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}

// Called by all 32 lanes of one warp; publishes c (d.cval, conf_out) and the
// budget of every layer of sequence b.
__device__ __forceinline__ void conf_merge_warp(const Shape& s, const Dev& d, int b,
                                                int32_t* budget, float* conf_out) {
  const int lane = threadIdx.x & 31;
  const ConfPartial* cp = d.conf + (size_t)b * s.SV;
  float M = -FLT_MAX;
  for (int i = lane; i < s.SV; i += 32) M = fmaxf(M, cp[i].M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  FSum S{0.f, 0.f}, T{0.f, 0.f};
  Top2 tp{-FLT_MAX, -FLT_MAX, 0x7fffffff};
  for (int i = lane; i < s.SV; i += 32) {
    const ConfPartial p = cp[i];
    if (p.M > -FLT_MAX) {
      const float dm = p.M - M;
      const float f = expf(dm);
      S = fsum_add(S, p.S * f);
      S = fsum_add(S, p.Se * f);
      T = fsum_add(T, (p.T + dm * p.S) * f);
      T = fsum_add(T, (p.Te + dm * p.Se) * f);
    }
    tp = top2_merge(tp, Top2{p.z1, p.z2, p.i1});
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S = fsum_add(S, fsum_shfl_xor(S, o));
    T = fsum_add(T, fsum_shfl_xor(T, o));
    Top2 other{__shfl_xor_sync(0xffffffffu, tp.z1, o), __shfl_xor_sync(0xffffffffu, tp.z2, o),
               __shfl_xor_sync(0xffffffffu, tp.i1, o)};
    tp = top2_merge(tp, other);
  }
  const float Sv = S.hi + S.lo, Tv = T.hi + T.lo;
  const float H = logf(Sv) - Tv / Sv;
  const float Hhat = H / logf((float)s.V);
  const float m = tp.z1 - tp.z2;
  const float p1 = expf(tp.z1 - M) / Sv;
  const float c = (float)s.wH * (1.0f - Hhat) + (float)s.wm * (1.0f / (1.0f + expf(-m))) +
                  (float)s.wp * p1;
  const bool high = c >= (float)s.tau;   // compared in fp32, the precision of c
  for (int l = lane; l < s.L; l += 32) budget[(size_t)b * s.L + l] = high ? d.n_high[l] : d.n_low[l];
  if (lane == 0) {
    d.cval[b] = (double)c;
    if (conf_out) conf_out[b] = c;
  }
}

}  // namespace confkv
