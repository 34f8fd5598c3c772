// Last kernel of a decode step, one CTA per (layer, sequence): confidence and
// budget, EMA update, ranking, bottom-k selection, evicted-position output,
// compaction of the INT8 region and requantisation of the token that leaves
// the FP16 window.
//
// CONF-KV (paper.rainbus.top/paper/2605.24786, 方法步骤详情, Algorithm 1):
//   step 3   c = w_H (1 - H/log V) + w_m sigmoid(log p(1) - log p(2)) + w_p p(1)
//   step 4   N = N_high if c >= tau else N_low       (tau = 0.7, 核心方法)
//   step 5   a_i <- lam a_i + (1 - lam) A_i          (lam = 0.9, 前置知识)
//   steps 6-9  if |C| > N: rank the non-protected entries by
//            s_i = alpha a_hat_i + (1 - alpha) r_hat_i (alpha = 0.65) and evict
//            the |C| - N lowest, then compact the survivors
//   step 10  quantise to INT8 the retained entries older than the newest W
// Readings taken where the pages are open: the new token is attended but not
// a candidate; a_hat, r_hat are min-max normalised over the candidates (r by
// absolute position); candidates are the positions < t - P; ties go to the
// older position; the new token's EMA starts from 0.
//
// Compaction fills every evicted INT8 slot below the new length from the
// survivors above it (at most k moves), so the region stays dense without
// an indirection table (gist.science/de/paper/2605.24786, Systemintegration:
// contiguous compaction).  Evicted FP16 ring slots are just marked empty.
#include <cuda_runtime.h>
#include <cfloat>
#include <climits>
#include "confkv_internal.cuh"

namespace confkv {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

// Stored byte of code = clamp(rint(x / s), -127, 127): the code + 128.
__device__ __forceinline__ uint8_t quant_code_sel(float x, float s) {
  float r = rintf(__fdiv_rn(x, s));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return (uint8_t)((int)r + kCodeBias);
}

template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, Op op, T* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  T r = red[0];
  for (int w = 1; w < kSelWarps; ++w) r = op(r, red[w]);
  return r;
}

struct MinOp { template <typename T> __device__ T operator()(T a, T b) const { return a < b ? a : b; } };
struct MaxOp { template <typename T> __device__ T operator()(T a, T b) const { return a > b ? a : b; } };
struct AddOp { template <typename T> __device__ T operator()(T a, T b) const { return a + b; } };

__global__ void __launch_bounds__(kSelThreads) select_kernel(Shape s, Dev d, long long step,
                                                             int32_t* __restrict__ budget_out,
                                                             float* __restrict__ conf_out,
                                                             int32_t* __restrict__ evicted_out,
                                                             int32_t* __restrict__ nevict_out,
                                                             int sort_cap) {
  extern __shared__ __align__(16) uint32_t dsm[];
  uint32_t* bitmap = dsm;                                  // [cap/32] evicted INT8 slots
  int32_t* list = reinterpret_cast<int32_t*>(dsm + s.cap / 32);   // [sort_cap]
  __shared__ unsigned long long red64[kSelWarps];
  __shared__ float redf[kSelWarps];
  __shared__ int redi[kSelWarps];
  __shared__ int hist[256];
  __shared__ int sN, s_cnt, s_k8, s_digit, s_remaining;
  __shared__ unsigned long long s_prefix, s_mask;

  const int l = blockIdx.x / s.B, b = blockIdx.x % s.B;
  const size_t lb = lb_index(s, l, b);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t* pos = d.pos + lb * s.S;
  float* ema = d.ema + lb * s.S;
  uint32_t* keys = d.scratch + lb * s.S;
  const int t = d.T0[b] + (int)step;
  const int n8 = d.n8[lb];

  // ------------------------------------------------ 1. confidence and budget
  if (warp == 0) {
    const ConfPartial* cp = d.conf + (size_t)b * s.SV;
    float M = -FLT_MAX;
    for (int i = lane; i < s.SV; i += 32) M = fmaxf(M, cp[i].M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    double S = 0.0, T = 0.0;
    float z1 = -FLT_MAX, z2 = -FLT_MAX;
    int i1 = INT_MAX;
    for (int i = lane; i < s.SV; i += 32) {
      const ConfPartial p = cp[i];
      if (p.M > -FLT_MAX) {
        const double dm = (double)p.M - (double)M;
        const double f = exp(dm);
        S += p.S * f;
        T += f * (p.T + dm * p.S);
      }
      // merge top-2
      if (p.z1 > z1 || (p.z1 == z1 && p.i1 < i1)) {
        z2 = fmaxf(z1, p.z2);
        z1 = p.z1;
        i1 = p.i1;
      } else {
        z2 = fmaxf(z2, p.z1);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      S += __shfl_xor_sync(0xffffffffu, S, o);
      T += __shfl_xor_sync(0xffffffffu, T, o);
      const float oz1 = __shfl_xor_sync(0xffffffffu, z1, o);
      const float oz2 = __shfl_xor_sync(0xffffffffu, z2, o);
      const int oi1 = __shfl_xor_sync(0xffffffffu, i1, o);
      if (oz1 > z1 || (oz1 == z1 && oi1 < i1)) {
        z2 = fmaxf(z1, oz2);
        z1 = oz1;
        i1 = oi1;
      } else {
        z2 = fmaxf(z2, oz1);
      }
    }
    if (lane == 0) {
      const double H = log(S) - T / S;
      const double Hhat = H / log((double)s.V);
      const double m = (double)z1 - (double)z2;
      const double p1 = exp((double)z1 - (double)M) / S;
      const double sig = 1.0 / (1.0 + exp(-m));
      const double c = s.wH * (1.0 - Hhat) + s.wm * sig + s.wp * p1;
      const int N = (c >= s.tau) ? d.n_high[l] : d.n_low[l];
      sN = N;
      budget_out[(size_t)b * s.L + l] = N;
      if (l == 0 && conf_out) conf_out[b] = (float)c;
    }
  }
  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_k8 = 0;
  }
  for (int w = threadIdx.x; w < s.cap / 32; w += kSelThreads) bitmap[w] = 0u;
  __syncthreads();
  const int N = sN;

  // ------------------------------------------------ 2. EMA update
  // Virtual index i < n8: INT8 slot i; otherwise ring slot cap + (i - n8).
  const int nvirt = n8 + s.WR;
  const float lam = s.lam, inv_hq = 1.0f / (float)s.Hq;
  int nring = 0;
  for (int i = threadIdx.x; i < nvirt; i += kSelThreads) {
    const int slot = i < n8 ? i : s.cap + (i - n8);
    if (i >= n8 && pos[slot] < 0) continue;
    nring += (i >= n8);
    float A = 0.f;
    for (int h = 0; h < s.Hkv; ++h) A += d.mass[(lb * s.Hkv + h) * s.S + slot];
    A *= inv_hq;
    ema[slot] = fmaf(lam, ema[slot], (1.0f - lam) * A);
  }
  nring = block_reduce(nring, AddOp(), redi);
  const int n = n8 + nring - 1;          // resident entries, new token excluded
  const int k = max(0, n - N);
  const int thr = t - s.P;               // candidates: pos < t - P

  // ------------------------------------------------ 3. rank and select
  unsigned long long threshold = 0ull;
  if (k > 0) {
    float amin = FLT_MAX, amax = -FLT_MAX;
    int pmin = INT_MAX, pmax = INT_MIN;
    for (int i = threadIdx.x; i < nvirt; i += kSelThreads) {
      const int slot = i < n8 ? i : s.cap + (i - n8);
      const int p = pos[slot];
      if (p < 0 || p >= thr) continue;
      const float a = ema[slot];
      amin = fminf(amin, a); amax = fmaxf(amax, a);
      pmin = min(pmin, p); pmax = max(pmax, p);
    }
    amin = block_reduce(amin, MinOp(), redf);
    amax = block_reduce(amax, MaxOp(), redf);
    pmin = block_reduce(pmin, MinOp(), redi);
    pmax = block_reduce(pmax, MaxOp(), redi);
    const float arng = amax - amin;
    const float prng = (float)(pmax - pmin);
    const float alpha = s.alpha;
    unsigned long long best = ~0ull;
    for (int i = threadIdx.x; i < nvirt; i += kSelThreads) {
      const int slot = i < n8 ? i : s.cap + (i - n8);
      const int p = pos[slot];
      if (p < 0 || p >= thr) continue;
      const float ah = arng > 0.f ? (ema[slot] - amin) / arng : 0.f;
      const float rh = prng > 0.f ? (float)(p - pmin) / prng : 0.f;
      const float sc = alpha * ah + (1.0f - alpha) * rh;
      const uint32_t key = __float_as_uint(sc);
      keys[slot] = key;
      const unsigned long long comp = ((unsigned long long)key << 32) | (uint32_t)p;
      best = comp < best ? comp : best;
    }
    if (k == 1) {
      threshold = block_reduce(best, MinOp(), red64);
    } else {
      __syncthreads();
      if (threadIdx.x == 0) {
        s_prefix = 0ull;
        s_mask = 0ull;
        s_remaining = k;
      }
      for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        const unsigned long long prefix = s_prefix, mask = s_mask;
        for (int i = threadIdx.x; i < nvirt; i += kSelThreads) {
          const int slot = i < n8 ? i : s.cap + (i - n8);
          const int p = pos[slot];
          if (p < 0 || p >= thr) continue;
          const unsigned long long comp = ((unsigned long long)keys[slot] << 32) | (uint32_t)p;
          if ((comp & mask) == prefix) atomicAdd(&hist[(comp >> shift) & 255], 1);
        }
        __syncthreads();
        if (warp == 0) {
          // find the digit at which the running count reaches `remaining`
          const int rem = s_remaining;
          int cnt[8], run = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            cnt[j] = hist[lane * 8 + j];
            run += cnt[j];
          }
          int incl = run;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
          }
          int before = incl - run;
          if (before < rem && rem <= incl) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (before < rem && rem <= before + cnt[j]) {
                s_digit = lane * 8 + j;
                s_remaining = rem - before;
                // all elements with this digit are taken: stop refining
                if (cnt[j] == rem - before) s_remaining = -(rem - before);
              }
              before += cnt[j];
            }
          }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
          s_prefix |= (unsigned long long)s_digit << shift;
          s_mask |= 255ull << shift;
        }
        __syncthreads();
        if (s_remaining < 0) break;
      }
      threshold = s_prefix | ~s_mask;
    }
    // ---------------------------------------------- 4. mark the evicted
    for (int i = threadIdx.x; i < nvirt; i += kSelThreads) {
      const int slot = i < n8 ? i : s.cap + (i - n8);
      const int p = pos[slot];
      if (p < 0 || p >= thr) continue;
      const unsigned long long comp = ((unsigned long long)keys[slot] << 32) | (uint32_t)p;
      if (comp > threshold) continue;
      const int idx = atomicAdd(&s_cnt, 1);
      if (idx < sort_cap) list[idx] = p;
      if (i < n8) {
        atomicOr(&bitmap[slot >> 5], 1u << (slot & 31));
        atomicAdd(&s_k8, 1);
      } else {
        pos[slot] = -1;   // evicted ring entry: the slot becomes empty
      }
    }
  }
  __syncthreads();
  const int cnt = s_cnt;
  if (threadIdx.x == 0 && cnt != k) atomicOr(d.status, kStatusBadCount);
  if (threadIdx.x == 0 && cnt > s.max_evict) atomicOr(d.status, kStatusEvictBound);

  // ------------------------------------------------ 5. sorted evicted positions
  const int nlist = min(cnt, min(sort_cap, s.max_evict));
  if (nlist > 1) {
    int np2 = 1;
    while (np2 < nlist) np2 <<= 1;
    for (int i = nlist + threadIdx.x; i < np2; i += kSelThreads) list[i] = INT_MAX;
    __syncthreads();
    for (int size = 2; size <= np2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < np2; i += kSelThreads) {
          const int j = i ^ stride;
          if (j > i) {
            const bool up = (i & size) == 0;
            const int a = list[i], c = list[j];
            if ((a > c) == up) {
              list[i] = c;
              list[j] = a;
            }
          }
        }
        __syncthreads();
      }
    }
  }
  int32_t* ev = evicted_out + lb * s.max_evict;
  for (int i = threadIdx.x; i < nlist; i += kSelThreads) ev[i] = list[i];
  if (threadIdx.x == 0) nevict_out[lb] = cnt;

  // ------------------------------------------------ 6. compaction (tail fill)
  const int k8 = s_k8;
  const int n8p = n8 - k8;
  int moves = 0;
  if (k8 > 0) {
    // holes: evicted slots < n8p; movers: surviving slots in [n8p, n8).
    uint32_t* hole = keys;                       // [moves]
    uint32_t* mover = keys + (s.S >> 1);         // [moves]
    const int nw = (n8 + 31) >> 5;
    int base_h = 0, base_m = 0;
    for (int w0 = 0; w0 < nw; w0 += kSelThreads) {
      const int w = w0 + threadIdx.x;
      uint32_t hb = 0u, mb = 0u;
      if (w < nw) {
        const uint32_t bits = bitmap[w];
        for (int j = 0; j < 32; ++j) {
          const int slot = w * 32 + j;
          if (slot < n8p) hb |= ((bits >> j) & 1u) << j;
          else if (slot < n8) mb |= ((~bits >> j) & 1u) << j;
        }
      }
      // exclusive scans of the per-word counts across the block
      int ch = __popc(hb), cm = __popc(mb);
      int ih = ch, im = cm;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int vh = __shfl_up_sync(0xffffffffu, ih, o);
        const int vm = __shfl_up_sync(0xffffffffu, im, o);
        if (lane >= o) { ih += vh; im += vm; }
      }
      __syncthreads();
      if (lane == 31) { redi[warp] = ih; red64[warp] = (unsigned long long)im; }
      __syncthreads();
      int offh = base_h, offm = base_m;
      for (int ww = 0; ww < warp; ++ww) { offh += redi[ww]; offm += (int)red64[ww]; }
      int rh = offh + ih - ch, rm = offm + im - cm;
      while (hb) { const int j = __ffs(hb) - 1; hb &= hb - 1; hole[rh++] = w * 32 + j; }
      while (mb) { const int j = __ffs(mb) - 1; mb &= mb - 1; mover[rm++] = w * 32 + j; }
      int th = 0, tm = 0;
      for (int ww = 0; ww < kSelWarps; ++ww) { th += redi[ww]; tm += (int)red64[ww]; }
      __syncthreads();
      base_h += th;
      base_m += tm;
    }
    moves = base_h;
    __syncthreads();
    const int D = s.D;
    const int per_tok = D / 4 + D;               // K words + V bytes per head
    const long long total = (long long)moves * s.Hkv * per_tok;
    for (long long i = threadIdx.x; i < total; i += kSelThreads) {
      const int r = (int)(i / (s.Hkv * per_tok));
      const int rest = (int)(i % (s.Hkv * per_tok));
      const int h = rest / per_tok, e = rest % per_tok;
      const int src = (int)mover[r], dst = (int)hole[r];
      const size_t u = unit_index(s, l, b, h);
      uint8_t* k8u = d.k8 + u * (size_t)s.cap * D;
      uint8_t* v8u = d.v8 + u * (size_t)s.cap * D;
      if (e < D / 4) {
        // one 32-bit word = channels {16kk+2t, +1, +8, +9} of the token
        const int kk = e / 4, tq = e % 4;
        const int c0 = kk * 16 + 2 * tq;
        const uint32_t wv = *reinterpret_cast<const uint32_t*>(
            k8u + (size_t)(src >> 4) * 16 * D + k8_offset(D, src & 15, c0));
        *reinterpret_cast<uint32_t*>(k8u + (size_t)(dst >> 4) * 16 * D + k8_offset(D, dst & 15, c0)) = wv;
      } else {
        const int c = e - D / 4;
        v8u[(size_t)(dst >> 4) * 16 * D + v8_offset(D, dst & 15, c)] =
            v8u[(size_t)(src >> 4) * 16 * D + v8_offset(D, src & 15, c)];
      }
      if (h == 0 && e == 0) {
        pos[dst] = pos[src];
        ema[dst] = ema[src];
      }
    }
  }
  __syncthreads();

  // ------------------------------------------------ 7. requantise the entry leaving the window
  int n8n = n8p;
  const int tl = t - s.W;
  int requant = 0;
  if (tl >= 0) {
    const int rs = tl % s.WR;
    const int rslot = s.cap + rs;
    if (pos[rslot] == tl) {
      if (n8p < s.cap) {
        const int D = s.D;
        const char* k16b = reinterpret_cast<const char*>(d.k16);
        const char* v16b = reinterpret_cast<const char*>(d.v16);
        for (int i = threadIdx.x; i < s.Hkv * D; i += kSelThreads) {
          const int h = i / D, c = i % D;
          const size_t u = unit_index(s, l, b, h);
          const size_t rblk = (u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;
          const float xk = __half2float(*reinterpret_cast<const __half*>(k16b + rblk + k16_offset(D, rs & 15, c)));
          const float xv = __half2float(*reinterpret_cast<const __half*>(v16b + rblk + v16_offset(D, rs & 15, c)));
          const size_t dblk = (u * (size_t)(s.cap / 16) + (n8p >> 4)) * 16 * D;
          d.k8[dblk + k8_offset(D, n8p & 15, c)] = quant_code_sel(xk, d.sK[u * D + c]);
          d.v8[dblk + v8_offset(D, n8p & 15, c)] = quant_code_sel(xv, d.sV[u * D + c]);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
          pos[n8p] = tl;
          ema[n8p] = ema[rslot];
          pos[rslot] = -1;
        }
        n8n = n8p + 1;
        requant = 1;
      } else if (threadIdx.x == 0) {
        atomicOr(d.status, kStatusCapacity);
      }
    }
  }
  if (threadIdx.x == 0) {
    d.n8[lb] = n8n;
    // algorithmic bytes of this (layer, sequence)
    const unsigned long long D = s.D, Hkv = s.Hkv, Hq = s.Hq;
    const unsigned long long nres = (unsigned long long)n8 + nring;   // incl. new token
    const unsigned long long attn = Hkv * D * (2ull * n8 + 4ull * nring) + 2ull * Hkv * D * 4 +
                                    Hq * D * (2 + 4) + Hkv * nres * 4;
    unsigned long long step_b = attn + nres * (4 + 4 + 4 + 4 * Hkv) + 2ull * Hkv * D * 2 * 2 +
                                (unsigned long long)requant * 2 * Hkv * D * 3 +
                                (unsigned long long)moves * (2 * Hkv * D + 8) * 2 +
                                4ull * (cnt + 1);
    if (l == 0) step_b += (unsigned long long)s.V * 4;
    atomicAdd(&d.stats->evicted, (unsigned long long)cnt);
    atomicAdd(&d.stats->moved, (unsigned long long)moves);
    atomicAdd(&d.stats->requant, (unsigned long long)requant);
    atomicAdd(&d.stats->attn_bytes, attn);
    atomicAdd(&d.stats->step_bytes, step_b);
    if (blockIdx.x == 0) atomicAdd(&d.stats->steps, 1ull);
  }
}

int launch_select(const Shape& s, const Dev& d, long long step, int32_t* budget, float* conf_out,
                  int32_t* evicted_pos, int32_t* n_evicted, int k_bound, cudaStream_t stream) {
  int sort_cap = 1;
  while (sort_cap < k_bound) sort_cap <<= 1;
  if (sort_cap > s.max_evict) {
    sort_cap = 1;
    while (sort_cap < s.max_evict) sort_cap <<= 1;
  }
  const size_t smem = (size_t)(s.cap / 32) * 4 + (size_t)sort_cap * 4;
  static size_t configured = 0;
  if (smem > 48 * 1024 && smem > configured) {
    if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return -1;
    configured = smem;
  }
  select_kernel<<<s.L * s.B, kSelThreads, smem, stream>>>(s, d, step, budget, conf_out,
                                                          evicted_pos, n_evicted, sort_cap);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace confkv
