// Confidence of B next-token distributions without any device allocation.
//
// Who needs this: code that may not call cudaMalloc (or any allocating
// routine) at the point where it wants the confidence score -- for example an
// inference server plug-in whose host process owns every device buffer
// through its own pool, a real-time loop that forbids allocation after
// start-up, or a caller that must not risk the implicit synchronisation an
// allocation can cause.  Such a caller passes only its input logits and its
// output array; the per-chunk partial results of the reduction live in the
// fixed scratch array below, which this library reserves once on every GPU
// that loads it and keeps until the process exits.
//
// The arithmetic is the same one-pass reduction as the decode step's
// confidence kernel: per vocabulary chunk M = max z, S = sum exp(z - M),
// T = sum (z - M) exp(z - M) and the two largest logits; the chunks are merged
// in float64 and c = w_H (1 - H / log V) + w_m sigmoid(z1 - z2) + w_p / S,
// with H = log S - T / S.
#include <cuda_runtime.h>
#include <cfloat>
#include <climits>
#include <cmath>
#include <mutex>

#include "../../include/confkv.h"

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 16;                    // chunk of at most 4096 logits
constexpr int kChunk = kThreads * kPerThread;
constexpr int kMaxPartials = CONFKV_NOALLOC_MAX_PARTIALS;
constexpr int kMaxDevices = 64;

struct Partial {
  float M, z1, z2;
  int i1;
  double S, T;
};

// Scratch shared by every call on a device: B * ceil(V / 4096) partials at
// most.  Every call overwrites the entries it uses before reading them.
static __device__ __align__(256) Partial g_noalloc_partials[kMaxPartials];

struct Top {
  float z1, z2;
  int i1;
};

__device__ __forceinline__ Top top_merge(Top a, Top b) {
  Top r;
  if (a.z1 > b.z1 || (a.z1 == b.z1 && a.i1 < b.i1)) {
    r.z1 = a.z1; r.i1 = a.i1; r.z2 = fmaxf(a.z2, b.z1);
  } else {
    r.z1 = b.z1; r.i1 = b.i1; r.z2 = fmaxf(b.z2, a.z1);
  }
  return r;
}

// grid: B * parts blocks; block (b, part) reduces one chunk of row b.
__global__ void __launch_bounds__(kThreads) noalloc_partial_kernel(const float* __restrict__ logits,
                                                                   int V, int parts,
                                                                   Partial* __restrict__ scratch) {
  __shared__ float red_f[kThreads / 32];
  __shared__ double red_s[kThreads / 32], red_t[kThreads / 32];
  __shared__ Top red_top[kThreads / 32];
  const int b = blockIdx.x / parts, part = blockIdx.x % parts;
  const int chunk = (V + parts - 1) / parts;
  const int v0 = part * chunk, v1 = min(V, v0 + chunk);
  const float* z = logits + (size_t)b * V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float x[kPerThread];
  Top tp{-FLT_MAX, -FLT_MAX, INT_MAX};
  float mx = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int idx = v0 + i * kThreads + threadIdx.x;
    x[i] = idx < v1 ? z[idx] : -FLT_MAX;
    if (idx < v1) {
      mx = fmaxf(mx, x[i]);
      tp = top_merge(tp, Top{x[i], -FLT_MAX, idx});
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_f[warp] = mx;
  __syncthreads();
  float M = red_f[0];
  for (int w = 1; w < kThreads / 32; ++w) M = fmaxf(M, red_f[w]);
  float sf = 0.f, tf = 0.f;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int idx = v0 + i * kThreads + threadIdx.x;
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
    Top other{__shfl_xor_sync(0xffffffffu, tp.z1, o), __shfl_xor_sync(0xffffffffu, tp.z2, o),
              __shfl_xor_sync(0xffffffffu, tp.i1, o)};
    tp = top_merge(tp, other);
  }
  if (lane == 0) {
    red_s[warp] = S;
    red_t[warp] = T;
    red_top[warp] = tp;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Partial p;
    double s0 = 0.0, t0 = 0.0;
    Top t = red_top[0];
    for (int w = 0; w < kThreads / 32; ++w) {
      s0 += red_s[w];
      t0 += red_t[w];
      if (w) t = top_merge(t, red_top[w]);
    }
    p.M = v1 > v0 ? M : -FLT_MAX;
    p.z1 = t.z1;
    p.z2 = t.z2;
    p.i1 = t.i1;
    p.S = s0;
    p.T = t0;
    scratch[(size_t)b * parts + part] = p;
  }
}

// grid: B blocks of one warp; merges the partials of row b into c.
__global__ void noalloc_merge_kernel(const Partial* __restrict__ scratch, int parts, int V,
                                     double wH, double wm, double wp, float* __restrict__ conf) {
  const int b = blockIdx.x, lane = threadIdx.x;
  const Partial* cp = scratch + (size_t)b * parts;
  float M = -FLT_MAX;
  for (int i = lane; i < parts; i += 32) M = fmaxf(M, cp[i].M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  double S = 0.0, T = 0.0;
  Top tp{-FLT_MAX, -FLT_MAX, INT_MAX};
  for (int i = lane; i < parts; i += 32) {
    const Partial p = cp[i];
    if (p.M > -FLT_MAX) {
      const double dm = (double)p.M - (double)M;
      const double f = exp(dm);
      S += p.S * f;
      T += f * (p.T + dm * p.S);
    }
    tp = top_merge(tp, Top{p.z1, p.z2, p.i1});
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S += __shfl_xor_sync(0xffffffffu, S, o);
    T += __shfl_xor_sync(0xffffffffu, T, o);
    Top other{__shfl_xor_sync(0xffffffffu, tp.z1, o), __shfl_xor_sync(0xffffffffu, tp.z2, o),
              __shfl_xor_sync(0xffffffffu, tp.i1, o)};
    tp = top_merge(tp, other);
  }
  if (lane == 0) {
    const double H = log(S) - T / S;
    const double Hhat = H / log((double)V);
    const double m = (double)tp.z1 - (double)tp.z2;
    const double p1 = exp((double)tp.z1 - (double)M) / S;
    const double c = wH * (1.0 - Hhat) + wm * (1.0 / (1.0 + exp(-m))) + wp * p1;
    conf[b] = (float)c;
  }
}

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code cannot use the array's name as a device pointer).
int scratch_on_current_device(Partial** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CONFKV_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return CONFKV_EINVAL;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p) return CONFKV_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<Partial*>(g_scratch_addr[dev]);
  return CONFKV_OK;
}

}  // namespace

extern "C" int confkv_confidence_noalloc(const float* logits, int32_t B, int32_t V, double w_H,
                                         double w_m, double w_p, float* confidence, void* stream) {
  if (!logits || !confidence || B < 1 || V < 2) return CONFKV_EINVAL;
  if (reinterpret_cast<uintptr_t>(logits) % 4 || reinterpret_cast<uintptr_t>(confidence) % 4)
    return CONFKV_EINVAL;
  if (!std::isfinite(w_H) || !std::isfinite(w_m) || !std::isfinite(w_p)) return CONFKV_EINVAL;
  const long long parts = (V + (long long)kChunk - 1) / kChunk;
  if ((long long)B * parts > kMaxPartials) return CONFKV_ECAPACITY;
  Partial* scratch = nullptr;
  const int r = scratch_on_current_device(&scratch);
  if (r != CONFKV_OK) return r;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  noalloc_partial_kernel<<<(unsigned)(B * parts), kThreads, 0, st>>>(logits, V, (int)parts, scratch);
  noalloc_merge_kernel<<<(unsigned)B, 32, 0, st>>>(scratch, (int)parts, V, w_H, w_m, w_p, confidence);
  return cudaGetLastError() == cudaSuccess ? CONFKV_OK : CONFKV_ECUDA;
}
