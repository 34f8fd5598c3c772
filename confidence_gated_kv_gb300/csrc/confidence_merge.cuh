// Merge of the per-chunk confidence partials of one sequence (one warp).
//
// CONF-KV (gist.science/de/paper/2605.24786, Konfidenzschätzung;
// paper.rainbus.top/paper/2605.24786, 核心方法 and Algorithm 1 steps 3-4):
// c = w_H (1 - H / log V) + w_m sigmoid(log p(1) - log p(2)) + w_p p(1),
// N = N_high if c >= tau else N_low.  From chunk partials (M_j, S_j, T_j)
// with S_j = sum exp(z - M_j), T_j = sum (z - M_j) exp(z - M_j):
// S = sum_j S_j e^(M_j - M), T = sum_j e^(M_j - M) (T_j + (M_j - M) S_j),
// H = log S - T / S, p(1) = e^(z1 - M) / S, log p(1) - log p(2) = z1 - z2.
// Sums and the final formula run in float64.
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
  double S = 0.0, T = 0.0;
  Top2 tp{-FLT_MAX, -FLT_MAX, 0x7fffffff};
  for (int i = lane; i < s.SV; i += 32) {
    const ConfPartial p = cp[i];
    if (p.M > -FLT_MAX) {
      const double dm = (double)p.M - (double)M;
      const double f = exp(dm);
      S += p.S * f;
      T += f * (p.T + dm * p.S);
    }
    tp = top2_merge(tp, Top2{p.z1, p.z2, p.i1});
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S += __shfl_xor_sync(0xffffffffu, S, o);
    T += __shfl_xor_sync(0xffffffffu, T, o);
    Top2 other{__shfl_xor_sync(0xffffffffu, tp.z1, o), __shfl_xor_sync(0xffffffffu, tp.z2, o),
               __shfl_xor_sync(0xffffffffu, tp.i1, o)};
    tp = top2_merge(tp, other);
  }
  const double H = log(S) - T / S;
  const double Hhat = H / log((double)s.V);
  const double m = (double)tp.z1 - (double)tp.z2;
  const double p1 = exp((double)tp.z1 - (double)M) / S;
  const double c = s.wH * (1.0 - Hhat) + s.wm * (1.0 / (1.0 + exp(-m))) + s.wp * p1;
  const bool high = c >= s.tau;
  for (int l = lane; l < s.L; l += 32) budget[(size_t)b * s.L + l] = high ? d.n_high[l] : d.n_low[l];
  if (lane == 0) {
    d.cval[b] = c;
    if (conf_out) conf_out[b] = (float)c;
  }
}

}  // namespace confkv
