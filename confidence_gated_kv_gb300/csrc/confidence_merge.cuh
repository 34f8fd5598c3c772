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

// (S, T) of a running maximum m_old carried over to a larger one m_new:
// S <- S e^(m_old - m_new), T <- e^(m_old - m_new) (T + (m_old - m_new) S).
__device__ __forceinline__ void conf_rescale(FSum& S, FSum& T, float m_old, float m_new) {
  if (m_old == -FLT_MAX) return;   // nothing summed yet (S = T = 0)
  const float dm = m_old - m_new;
  const float f = expf(dm);
  T = fsum_add(T, dm * S.hi);
  T = fsum_add(T, dm * S.lo);
  T = FSum{T.hi * f, T.lo * f};
  S = FSum{S.hi * f, S.lo * f};
}

// Partial (M, S, T, top 2) of vocabulary chunk `part` of sequence b, computed
// by one warp in a single pass over the logits: each lane keeps its own
// running maximum and carries its sums over when it moves, then the lanes are
// brought to the chunk maximum and summed.  Called by all 32 lanes.  kIn:
// loads in flight per lane (each lane takes its elements in increasing order
// whatever kIn is, so the result does not depend on it).
template <int kIn = 8>
__device__ __forceinline__ void conf_partial_warp(const Shape& s, const Dev& d,
                                                  const float* __restrict__ logits, int b, int part) {
  const int lane = threadIdx.x & 31;
  const int V = s.V;
  const int chunk = (V + s.SV - 1) / s.SV;
  const int v0 = part * chunk, v1 = min(V, v0 + chunk);
  const float* z = logits + (size_t)b * V;
  float m = -FLT_MAX;
  FSum S{0.f, 0.f}, T{0.f, 0.f};
  Top2 tp{-FLT_MAX, -FLT_MAX, 0x7fffffff};
  for (int base = v0; base < v1; base += 32 * kIn) {
    float x[kIn];
#pragma unroll
    for (int j = 0; j < kIn; ++j) {
      const int idx = base + 32 * j + lane;
      x[j] = idx < v1 ? __ldg(z + idx) : -FLT_MAX;
    }
#pragma unroll
    for (int j = 0; j < kIn; ++j) {
      const int idx = base + 32 * j + lane;
      if (idx < v1) {
        if (x[j] > m) {
          conf_rescale(S, T, m, x[j]);
          m = x[j];
        }
        const float dz = x[j] - m;
        const float e = expf(dz);
        S = fsum_add(S, e);
        T = fsum_add(T, dz * e);
        tp = top2_merge(tp, Top2{x[j], -FLT_MAX, idx});
      }
    }
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  conf_rescale(S, T, m, M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S = fsum_add(S, fsum_shfl_xor(S, o));
    T = fsum_add(T, fsum_shfl_xor(T, o));
    Top2 other{__shfl_xor_sync(0xffffffffu, tp.z1, o), __shfl_xor_sync(0xffffffffu, tp.z2, o),
               __shfl_xor_sync(0xffffffffu, tp.i1, o)};
    tp = top2_merge(tp, other);
  }
  if (lane == 0) {
    ConfPartial cp;
    cp.M = (v1 > v0) ? M : -FLT_MAX;
    cp.z1 = tp.z1;
    cp.z2 = tp.z2;
    cp.i1 = tp.i1;
    cp.S = S.hi;
    cp.Se = S.lo;
    cp.T = T.hi;
    cp.Te = T.lo;
    d.conf[(size_t)b * s.SV + part] = cp;
  }
}

static_assert(sizeof(ConfPartial) == 32, "ConfPartial is read as two 16-byte words");

// One chunk partial read from L2 (written by other CTAs of the same kernel
// in the attention-side reduction).
__device__ __forceinline__ ConfPartial load_partial(const ConfPartial* p) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
  const float4 c = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  ConfPartial r;
  r.M = a.x;
  r.z1 = a.y;
  r.z2 = a.z;
  r.i1 = __float_as_int(a.w);
  r.S = c.x;
  r.Se = c.y;
  r.T = c.z;
  r.Te = c.w;
  return r;
}

// c of one sequence from its SV chunk partials cp[0 .. SV) over a vocabulary
// of V, with the weights (wH, wm, wp).  Called by all 32 lanes of one warp;
// every lane returns c.  One pass: each lane folds its partials into a
// running (M, S, T) with the same rescaling as the single-chunk pass, four
// partials loaded at a time; then the lanes are brought to the common
// maximum and summed.
__device__ __forceinline__ float conf_merge_c(const ConfPartial* __restrict__ cp, int SV, int V,
                                              float wH, float wm, float wp) {
  const int lane = threadIdx.x & 31;
  float m = -FLT_MAX;
  FSum S{0.f, 0.f}, T{0.f, 0.f};
  Top2 tp{-FLT_MAX, -FLT_MAX, 0x7fffffff};
  for (int i0 = lane; i0 < SV; i0 += 32 * 4) {
    ConfPartial p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + 32 * j;
      if (i < SV) {
        p[j] = load_partial(cp + i);
      } else {
        p[j].M = -FLT_MAX;
        p[j].z1 = p[j].z2 = -FLT_MAX;
        p[j].i1 = 0x7fffffff;
        p[j].S = p[j].Se = p[j].T = p[j].Te = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (p[j].M > -FLT_MAX) {
        if (p[j].M > m) {
          conf_rescale(S, T, m, p[j].M);
          m = p[j].M;
        }
        const float dm = p[j].M - m;
        const float f = expf(dm);
        S = fsum_add(S, p[j].S * f);
        S = fsum_add(S, p[j].Se * f);
        T = fsum_add(T, (p[j].T + dm * p[j].S) * f);
        T = fsum_add(T, (p[j].Te + dm * p[j].Se) * f);
      }
      tp = top2_merge(tp, Top2{p[j].z1, p[j].z2, p[j].i1});
    }
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  conf_rescale(S, T, m, M);
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
  const float Hhat = H / logf((float)V);
  const float mg = tp.z1 - tp.z2;
  const float p1 = expf(tp.z1 - M) / Sv;
  return wH * (1.0f - Hhat) + wm * (1.0f / (1.0f + expf(-mg))) + wp * p1;
}

// Merges the partials of sequence b and publishes c (d.cval, conf_out) and
// the budget of every layer of the sequence.  Called by all 32 lanes of one
// warp.
__device__ __forceinline__ void conf_merge_warp(const Shape& s, const Dev& d, int b, int32_t* budget,
                                                float* conf_out) {
  const int lane = threadIdx.x & 31;
  const float c = conf_merge_c(d.conf + (size_t)b * s.SV, s.SV, s.V, (float)s.wH, (float)s.wm, (float)s.wp);
  const bool high = c >= (float)s.tau;   // compared in fp32, the precision of c
  for (int l = lane; l < s.L; l += 32) budget[(size_t)b * s.L + l] = high ? d.n_high[l] : d.n_low[l];
  if (lane == 0) {
    d.cval[b] = (double)c;
    if (conf_out) conf_out[b] = c;
  }
}

}  // namespace confkv
