// Prefill ingestion: per-(sequence, layer, KV head, channel) absmax scales and
// the initial cache layout.
//
// The pages do not describe prefill; the scales follow the rule that INT8 is
// kept per head and per channel (CONF-KV, gist.science/de/paper/2605.24786,
// Technischer Zusammenfassung, Systemintegration) with the scale fixed from
// the absmax of the prefill: s = absmax / 127 (float32), s = 1 when the
// channel is all zero.  Positions >= T0 - W start in the FP16 window; older
// positions are quantised: code = clamp(rint(x / s), -127, 127).
#include <cuda_runtime.h>
#include "confkv_internal.cuh"

namespace confkv {

__device__ __forceinline__ float scale_from_absmax(uint32_t bits) {
  float a = __uint_as_float(bits);
  return a > 0.f ? __fdiv_rn(a, 127.0f) : 1.0f;
}

// Stored byte of code = clamp(rint(x / s), -127, 127): the code + 128.
__device__ __forceinline__ uint8_t quant_code(float x, float s) {
  float r = rintf(__fdiv_rn(x, s));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return (uint8_t)((int)r + kCodeBias);
}

// grid: (units, token splits); block: D threads (one channel each).
__global__ void prefill_absmax_kernel(Shape s, Dev d, const __half* __restrict__ k,
                                      const __half* __restrict__ v, long long t_max) {
  const int u = blockIdx.x;
  const int b = (u / s.Hkv) % s.B;
  const int T0 = d.T0[b];
  const int per = (T0 + gridDim.y - 1) / gridDim.y;
  const int t0 = blockIdx.y * per, t1 = min(T0, t0 + per);
  const int c = threadIdx.x;
  const size_t base = (size_t)u * t_max * s.D + c;
  float mk = 0.f, mv = 0.f;
  for (int tau = t0; tau < t1; ++tau) {
    mk = fmaxf(mk, fabsf(__half2float(k[base + (size_t)tau * s.D])));
    mv = fmaxf(mv, fabsf(__half2float(v[base + (size_t)tau * s.D])));
  }
  const size_t nu = (size_t)s.L * s.B * s.Hkv * s.D;
  if (t1 > t0) {
    atomicMax(&d.absmax[(size_t)u * s.D + c], __float_as_uint(mk));
    atomicMax(&d.absmax[nu + (size_t)u * s.D + c], __float_as_uint(mv));
  }
}

// grid: (units, token blocks of 16); block: 256 threads over (tau, channel).
__global__ void prefill_place_kernel(Shape s, Dev d, const __half* __restrict__ k,
                                     const __half* __restrict__ v, long long t_max) {
  const int u = blockIdx.x;
  const int h = u % s.Hkv;
  const int b = (u / s.Hkv) % s.B;
  const int l = u / (s.Hkv * s.B);
  const int T0 = d.T0[b];
  const int blk = blockIdx.y;
  const int D = s.D;
  const size_t nu = (size_t)s.L * s.B * s.Hkv * D;
  const int n8 = max(0, T0 - s.W);
  const size_t lb = lb_index(s, l, b);

  if (blk == 0) {
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
      d.sK[(size_t)u * D + c] = scale_from_absmax(d.absmax[(size_t)u * D + c]);
      d.sV[(size_t)u * D + c] = scale_from_absmax(d.absmax[nu + (size_t)u * D + c]);
    }
    if (h == 0 && threadIdx.x == 0) d.n8[lb] = n8;
  }
  for (int i = threadIdx.x; i < 16 * D; i += blockDim.x) {
    const int tau = i / D, c = i % D;
    const int p = blk * 16 + tau;
    if (p >= T0) continue;
    const size_t src = ((size_t)u * t_max + p) * D + c;
    const float xk = __half2float(k[src]);
    const float xv = __half2float(v[src]);
    if (p < n8) {
      const float sk = scale_from_absmax(d.absmax[(size_t)u * D + c]);
      const float sv = scale_from_absmax(d.absmax[nu + (size_t)u * D + c]);
      const size_t blk_base = ((size_t)u * (s.cstride / 16) + (p >> 4)) * 16 * D;
      d.k8[blk_base + k8_offset(D, p & 15, c)] = quant_code(xk, sk);
      d.v8[blk_base + v8_offset(D, p & 15, c)] = quant_code(xv, sv);
      if (h == 0 && c == 0) {
        d.pos[lb * s.S + p] = p;
        d.ema[lb * s.S + p] = 0.f;
      }
    } else {
      const int rs = p % s.WR;
      const size_t blk_base = ((size_t)u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;  // bytes
      char* k16b = reinterpret_cast<char*>(d.k16);
      char* v16b = reinterpret_cast<char*>(d.v16);
      *reinterpret_cast<__half*>(k16b + blk_base + k16_offset(D, rs & 15, c)) = k[src];
      *reinterpret_cast<__half*>(v16b + blk_base + v16_offset(D, rs & 15, c)) = v[src];
      if (h == 0 && c == 0) {
        d.pos[lb * s.S + s.cap + rs] = p;
        d.ema[lb * s.S + s.cap + rs] = 0.f;
      }
    }
  }
}

int launch_prefill(const Shape& s, const Dev& d, const void* k, const void* v, long long t_max,
                   const int32_t* T0_host, cudaStream_t stream) {
  int tmax0 = 0;
  for (int b = 0; b < s.B; ++b) tmax0 = T0_host[b] > tmax0 ? T0_host[b] : tmax0;
  const size_t units = (size_t)s.L * s.B * s.Hkv;
  const size_t nu = units * s.D;
  cudaMemsetAsync(d.absmax, 0, 2 * nu * sizeof(uint32_t), stream);
  cudaMemsetAsync(d.pos, 0xFF, (size_t)s.L * s.B * s.S * sizeof(int32_t), stream);
  cudaMemsetAsync(d.ema, 0, (size_t)s.L * s.B * s.S * sizeof(float), stream);
  cudaMemsetAsync(d.k16, 0, units * s.WR * s.D * sizeof(__half), stream);
  cudaMemsetAsync(d.v16, 0, units * s.WR * s.D * sizeof(__half), stream);
  cudaMemsetAsync(d.k8, kCodeBias, units * (size_t)s.cstride * s.D, stream);
  cudaMemsetAsync(d.v8, kCodeBias, units * (size_t)s.cstride * s.D, stream);
  // Sequences with T0 = 0 still need their scales (1.0) and n8 = 0.
  int tsplit = tmax0 > 0 ? (tmax0 + 1023) / 1024 : 1;
  if (tsplit > 64) tsplit = 64;
  prefill_absmax_kernel<<<dim3((unsigned)units, tsplit), s.D, 0, stream>>>(
      s, d, static_cast<const __half*>(k), static_cast<const __half*>(v), t_max);
  const int nblk = tmax0 > 0 ? (tmax0 + 15) / 16 : 1;
  prefill_place_kernel<<<dim3((unsigned)units, nblk), 256, 0, stream>>>(
      s, d, static_cast<const __half*>(k), static_cast<const __half*>(v), t_max);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace confkv
