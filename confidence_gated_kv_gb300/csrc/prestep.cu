// First kernel of a decode step: (a) the vocabulary-wide reduction of the
// logits that feeds the confidence score, split into per-chunk partials, and
// (b) the append of the new token's K/V to the FP16 ring.
//
// (a) CONF-KV (paper.rainbus.top/paper/2605.24786, 方法步骤详情, Algorithm 1
// steps 2-3; gist.science/de/paper/2605.24786, Konfidenzschätzung): c needs
// the entropy of p = softmax(z), the top-two log-probabilities and p(1).  One
// pass gives everything: with M = max z, S = sum exp(z - M) and
// T = sum (z - M) exp(z - M), the entropy is H = log S - T / S, p(1) = 1 / S
// and log p(1) - log p(2) = z(1) - z(2).  Each block reduces one chunk of the
// vocabulary of one sequence to (M, S, T, z(1), z(2)); the chunks of a
// sequence are merged in float64 by one warp of the attention kernel, off its
// critical path (confidence_merge.cuh).
//
// (b) Algorithm 1 step 13 appends the new K/V in FP16.  The ring has W + 16
// slots, so slot t mod (W + 16) is always free when token t arrives (its
// previous occupant, position t - W - 16, left the window 16 steps ago), and
// the attention kernel reads the new token as an ordinary ring entry.
#include <cuda_runtime.h>
#include <cfloat>
#include "confidence_merge.cuh"

namespace confkv {

constexpr int kConfThreads = 256;
constexpr int kConfPerThread = 16;   // chunk <= 4096 logits

__device__ void conf_block(const Shape& s, const Dev& d, const float* __restrict__ logits, int b,
                           int part) {
  __shared__ float red_f[kConfThreads / 32];
  __shared__ double red_s[kConfThreads / 32], red_t[kConfThreads / 32];
  __shared__ Top2 red_top[kConfThreads / 32];
  const int V = s.V;
  const int chunk = (V + s.SV - 1) / s.SV;
  const int v0 = part * chunk, v1 = min(V, v0 + chunk);
  const float* z = logits + (size_t)b * V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  float x[kConfPerThread];
  Top2 tp{-FLT_MAX, -FLT_MAX, 0x7fffffff};
  float mx = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < kConfPerThread; ++i) {
    const int idx = v0 + i * kConfThreads + threadIdx.x;
    x[i] = idx < v1 ? __ldg(z + idx) : -FLT_MAX;
    if (idx < v1) {
      mx = fmaxf(mx, x[i]);
      Top2 one{x[i], -FLT_MAX, idx};
      tp = top2_merge(tp, one);
    }
  }
  // block maximum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_f[warp] = mx;
  __syncthreads();
  float M = red_f[0];
  for (int w = 1; w < kConfThreads / 32; ++w) M = fmaxf(M, red_f[w]);

  float sf = 0.f, tf = 0.f;
#pragma unroll
  for (int i = 0; i < kConfPerThread; ++i) {
    const int idx = v0 + i * kConfThreads + threadIdx.x;
    if (idx < v1) {
      const float dz = x[i] - M;
      const float e = expf(dz);
      sf += e;
      tf += dz * e;
    }
  }
  double S = sf, T = tf;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S += __shfl_xor_sync(0xffffffffu, S, o);
    T += __shfl_xor_sync(0xffffffffu, T, o);
    Top2 other{__shfl_xor_sync(0xffffffffu, tp.z1, o), __shfl_xor_sync(0xffffffffu, tp.z2, o),
               __shfl_xor_sync(0xffffffffu, tp.i1, o)};
    tp = top2_merge(tp, other);
  }
  if (lane == 0) {
    red_s[warp] = S;
    red_t[warp] = T;
    red_top[warp] = tp;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double S0 = 0.0, T0 = 0.0;
    Top2 t0 = red_top[0];
    for (int w = 0; w < kConfThreads / 32; ++w) {
      S0 += red_s[w];
      T0 += red_t[w];
      if (w) t0 = top2_merge(t0, red_top[w]);
    }
    ConfPartial cp;
    cp.M = (v1 > v0) ? M : -FLT_MAX;
    cp.z1 = t0.z1;
    cp.z2 = t0.z2;
    cp.i1 = t0.i1;
    cp.S = S0;
    cp.T = T0;
    d.conf[(size_t)b * s.SV + part] = cp;
  }
}

// Append token t of sequence b, layer l to ring slot t mod WR (all KV heads).
__device__ void append_block(const Shape& s, const Dev& d, long long step, int l, int b,
                             const __half* __restrict__ k_new, const __half* __restrict__ v_new) {
  const int t = d.T0[b] + (int)step;
  const int rs = t % s.WR;
  const int D = s.D;
  char* k16b = reinterpret_cast<char*>(d.k16);
  char* v16b = reinterpret_cast<char*>(d.v16);
  for (int i = threadIdx.x; i < s.Hkv * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    const size_t u = unit_index(s, l, b, h);
    const size_t blk_base = (u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;
    const size_t src = u * D + c;   // [l][b][kvh][D]
    *reinterpret_cast<__half*>(k16b + blk_base + k16_offset(D, rs & 15, c)) = k_new[src];
    *reinterpret_cast<__half*>(v16b + blk_base + v16_offset(D, rs & 15, c)) = v_new[src];
  }
  if (threadIdx.x == 0) {
    const size_t lb = lb_index(s, l, b);
    d.pos[lb * s.S + s.cap + rs] = t;
    d.ema[lb * s.S + s.cap + rs] = 0.f;
  }
}

__global__ void __launch_bounds__(kConfThreads) prestep_kernel(Shape s, Dev d, long long step,
                                                               const float* __restrict__ logits,
                                                               const __half* __restrict__ k_new,
                                                               const __half* __restrict__ v_new) {
  const int nconf = s.B * s.SV;
  if ((int)blockIdx.x < nconf) {
    conf_block(s, d, logits, blockIdx.x / s.SV, blockIdx.x % s.SV);
  } else {
    const int i = blockIdx.x - nconf;
    append_block(s, d, step, i / s.B, i % s.B, k_new, v_new);
  }
}

int launch_prestep(const Shape& s, const Dev& d, long long step, const float* logits,
                   const void* k_new, const void* v_new, cudaStream_t stream) {
  const unsigned grid = (unsigned)(s.B * s.SV + s.L * s.B);
  prestep_kernel<<<grid, kConfThreads, 0, stream>>>(s, d, step, logits,
                                                    static_cast<const __half*>(k_new),
                                                    static_cast<const __half*>(v_new));
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace confkv
