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
// vocabulary of one sequence to (M, S, T, z(1), z(2)), the sums in
// compensated fp32; the chunks of a sequence are merged by one warp of the
// attention kernel, off its critical path (confidence_merge.cuh).
//
// (b) Algorithm 1 step 13 appends the new K/V in FP16.  The ring has W + 16
// slots, so slot t mod (W + 16) is always free when token t arrives (its
// previous occupant, position t - W - 16, left the window 16 steps ago), and
// the attention kernel reads the new token as an ordinary ring entry.
//
// One launch holds both parts: the first B * SV blocks reduce vocabulary
// chunks of at most 4096 logits, the rest append 32 units each, so the grid
// fits on the GPU in one wave.
#include <cuda_runtime.h>
#include <cfloat>
#include "confidence_merge.cuh"

namespace confkv {

constexpr int kConfThreads = 256;
constexpr int kConfPerThread = 16;   // chunk <= 4096 logits

__device__ void conf_block(const Shape& s, const Dev& d, const float* __restrict__ logits, int b,
                           int part) {
  __shared__ float red_f[kConfThreads / 32];
  __shared__ FSum red_s[kConfThreads / 32], red_t[kConfThreads / 32];
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
  }
#pragma unroll
  for (int i = 0; i < kConfPerThread; ++i) {
    const int idx = v0 + i * kConfThreads + threadIdx.x;
    if (idx < v1) {
      mx = fmaxf(mx, x[i]);
      tp = top2_merge(tp, Top2{x[i], -FLT_MAX, idx});
    }
  }
  // block maximum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_f[warp] = mx;
  __syncthreads();
  float M = red_f[0];
  for (int w = 1; w < kConfThreads / 32; ++w) M = fmaxf(M, red_f[w]);

  FSum S{0.f, 0.f}, T{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kConfPerThread; ++i) {
    const int idx = v0 + i * kConfThreads + threadIdx.x;
    if (idx < v1) {
      const float dz = x[i] - M;
      const float e = expf(dz);
      S = fsum_add(S, e);
      T = fsum_add(T, dz * e);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S = fsum_add(S, fsum_shfl_xor(S, o));
    T = fsum_add(T, fsum_shfl_xor(T, o));
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
    FSum S0 = red_s[0], T0 = red_t[0];
    Top2 t0 = red_top[0];
    for (int w = 1; w < kConfThreads / 32; ++w) {
      S0 = fsum_add(S0, red_s[w]);
      T0 = fsum_add(T0, red_t[w]);
      t0 = top2_merge(t0, red_top[w]);
    }
    ConfPartial cp;
    cp.M = (v1 > v0) ? M : -FLT_MAX;
    cp.z1 = t0.z1;
    cp.z2 = t0.z2;
    cp.i1 = t0.i1;
    cp.S = S0.hi;
    cp.Se = S0.lo;
    cp.T = T0.hi;
    cp.Te = T0.lo;
    d.conf[(size_t)b * s.SV + part] = cp;
  }
}

// Append the new token of every unit u = (l, b, kvh) in [u0, u1) to ring slot
// t mod WR.  One warp per unit, four units in flight per warp: lane i writes
// the 8 bytes of K that hold channels 16(i/4) + 2(i%4) + {0, 1, 8, 9} of the
// interleaved FP16 block (one aligned store) and V channels i, i + 32, ...
template <int D, bool kDevStep>
__device__ void append_units(const Shape& s, const Dev& d, long long step_arg, int u0, int u1,
                             const __half* __restrict__ k_new, const __half* __restrict__ v_new) {
  constexpr int kU = 4;
  constexpr int kV = D / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int kc0 = 16 * (lane >> 2) + 2 * (lane & 3);
  char* k16b = reinterpret_cast<char*>(d.k16);
  char* v16b = reinterpret_cast<char*>(d.v16);
  const int nwarps = blockDim.x >> 5;
  uint2 kx[kU];
  unsigned short vx[kU][kV];
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    const int u = u0 + warp + j * nwarps;
    if (u >= u1) break;
    const unsigned short* kn = reinterpret_cast<const unsigned short*>(k_new) + (size_t)u * D;
    const unsigned short* vn = reinterpret_cast<const unsigned short*>(v_new) + (size_t)u * D;
    if (lane < D / 4) {
      kx[j].x = *reinterpret_cast<const uint32_t*>(kn + kc0);
      kx[j].y = *reinterpret_cast<const uint32_t*>(kn + kc0 + 8);
    }
#pragma unroll
    for (int i = 0; i < kV; ++i) vx[j][i] = vn[lane + 32 * i];
  }
  // a step inside a graph reservation reads the step index from the device
  // (after the payload loads are in flight); other steps take the argument
  const long long step = kDevStep ? __ldcg(d.step_dev) : step_arg;
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    const int u = u0 + warp + j * nwarps;
    if (u >= u1) break;
    const int lbi = u / s.Hkv, h = u - lbi * s.Hkv;
    const int b = lbi % s.B;
    const int t = d.T0[b] + (int)step;
    const int rs = t % s.WR;
    const size_t blk = ((size_t)u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;
    if (lane < D / 4) *reinterpret_cast<uint2*>(k16b + blk + k16_offset(D, rs & 15, kc0)) = kx[j];
#pragma unroll
    for (int i = 0; i < kV; ++i)
      *reinterpret_cast<unsigned short*>(v16b + blk + v16_offset(D, rs & 15, lane + 32 * i)) = vx[j][i];
    if (h == 0 && lane == 0) {
      d.pos[(size_t)lbi * s.S + s.cap + rs] = t;
      d.ema[(size_t)lbi * s.S + s.cap + rs] = 0.f;
    }
  }
}

// The (layer, sequence) groups sorted by their INT8 length, longest first,
// ties by index: d.order[rank] = group.  The attention kernel deals its units
// to CTAs in snake order over this list, which balances the CTAs' streams
// (a unit's time follows its bytes, and the INT8 region is the part of a
// unit's length that varies).  The rank of a group is the number of groups
// that sort before it; kSortPerBlock groups per block, four threads per
// group each counting over a quarter of the keys.
constexpr int kSortPerBlock = kConfThreads / 4;

__device__ void order_block(const Shape& s, const Dev& d, int part) {
  __shared__ int key[kSortMaxGroups];
  const int n = s.L * s.B;
  for (int i = threadIdx.x; i < n; i += kConfThreads) key[i] = d.n8[i];
  __syncthreads();
  const int i = part * kSortPerBlock + (threadIdx.x >> 2), q = threadIdx.x & 3;
  int r = 0;
  if (i < n) {
    const int ki = key[i];
    for (int j = q; j < n; j += 4) {
      const int kj = key[j];
      r += (kj > ki) | ((kj == ki) & (j < i));
    }
  }
  r += __shfl_xor_sync(0xffffffffu, r, 1);
  r += __shfl_xor_sync(0xffffffffu, r, 2);
  if (i < n && q == 0) d.order[r] = i;
  if (part == 0 && threadIdx.x == 0) *d.queue = 0u;
}

__host__ __device__ inline int sort_blocks(const Shape& s, const Dev& d) {
  return d.sorted ? (s.L * s.B + kSortPerBlock - 1) / kSortPerBlock : 0;
}

constexpr int kAppendUnitsPerBlock = 4 * (kConfThreads / 32);

template <int D, bool kDevStep>
__global__ void __launch_bounds__(kConfThreads) prestep_kernel(Shape s, Dev d, long long step,
                                                               const float* __restrict__ logits,
                                                               const __half* __restrict__ k_new,
                                                               const __half* __restrict__ v_new,
                                                               int nconf) {
  pdl_wait();
  if ((int)blockIdx.x < nconf) {
    conf_block(s, d, logits, blockIdx.x / s.SV, blockIdx.x % s.SV);
  } else if ((int)blockIdx.x >= (int)gridDim.x - sort_blocks(s, d)) {
    order_block(s, d, (int)blockIdx.x - ((int)gridDim.x - sort_blocks(s, d)));
  } else {
    const int units = s.L * s.B * s.Hkv;
    const int u0 = ((int)blockIdx.x - nconf) * kAppendUnitsPerBlock;
    append_units<D, kDevStep>(s, d, step, u0, min(units, u0 + kAppendUnitsPerBlock), k_new, v_new);
  }
}

int launch_prestep(const Shape& s, const Dev& d, long long step, const float* logits,
                   const void* k_new, const void* v_new, bool conf, cudaStream_t stream) {
  const int units = s.L * s.B * s.Hkv;
  const int nconf = conf ? s.B * s.SV : 0;
  const unsigned grid =
      (unsigned)(nconf + (units + kAppendUnitsPerBlock - 1) / kAppendUnitsPerBlock + sort_blocks(s, d));
  const __half* kn = static_cast<const __half*>(k_new);
  const __half* vn = static_cast<const __half*>(v_new);
  const dim3 g(grid), blk(kConfThreads);
  cudaError_t e;
  if (step >= 0)
    e = s.D == 128 ? launch_pdl(prestep_kernel<128, false>, g, blk, 0, stream, s, d, step, logits, kn, vn, nconf)
                   : launch_pdl(prestep_kernel<64, false>, g, blk, 0, stream, s, d, step, logits, kn, vn, nconf);
  else
    e = s.D == 128 ? launch_pdl(prestep_kernel<128, true>, g, blk, 0, stream, s, d, step, logits, kn, vn, nconf)
                   : launch_pdl(prestep_kernel<64, true>, g, blk, 0, stream, s, d, step, logits, kn, vn, nconf);
  return e == cudaSuccess ? 0 : -1;
}

}  // namespace confkv
