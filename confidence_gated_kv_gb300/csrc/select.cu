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

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kCache = 6;   // slots per thread kept in registers between passes

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

__global__ void __launch_bounds__(kSelThreads, 4) select_kernel(Shape s, Dev d, long long step,
                                                             int32_t* __restrict__ evicted_out,
                                                             int32_t* __restrict__ nevict_out,
                                                             int sort_cap) {
  extern __shared__ __align__(16) uint32_t dsm[];
  uint32_t* bitmap = dsm;                                  // [cap/32] evicted INT8 slots
  int32_t* list = reinterpret_cast<int32_t*>(dsm + s.cap / 32);   // [sort_cap]
  __shared__ unsigned long long red64[kSelWarps];
  __shared__ int redi[kSelWarps];
  __shared__ int hist[256];
  __shared__ int red5i[kSelWarps][3];
  __shared__ float red5f[kSelWarps][2];
  __shared__ int s_cnt, s_k8, s_digit, s_remaining, s_evslot;
  __shared__ unsigned long long s_prefix, s_mask;

  const int l = blockIdx.x / s.B, b = blockIdx.x % s.B;
  const size_t lb = lb_index(s, l, b);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t* pos = d.pos + lb * s.S;
  float* ema = d.ema + lb * s.S;
  uint32_t* keys = d.scratch + lb * s.S;
  const int t = d.T0[b] + (int)step;
  const int n8 = d.n8[lb];
  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_k8 = 0;
    s_evslot = -1;
  }

  // ------------------------------------------------ 1. budget of this layer
  // c was merged once per sequence by the last confidence block of the step.
  const int N = (d.cval[b] >= s.tau) ? d.n_high[l] : d.n_low[l];

  // ------------------------------------------------ 2. EMA update + candidate ranges
  // Virtual index i < n8: INT8 slot i; otherwise ring slot cap + (i - n8).
  // The first kCache slots of every thread stay in registers for pass 3.
  const int nvirt = n8 + s.WR;
  const int thr = t - s.P;               // candidates: pos < t - P
  const float lam = s.lam, inv_hq = 1.0f / (float)s.Hq;
  int nring = 0;
  float amin = FLT_MAX, amax = -FLT_MAX;
  int pmin = INT_MAX, pmax = INT_MIN;
  int cpos[kCache];
  float cema[kCache];
  {
    // The first kCache slots of this thread: every load is issued before any
    // value is used (positions, then the KV-head mass partials and the EMA).
    // positions, EMA and the KV-head mass partials are all loaded in one
    // round (slots that turn out to be empty simply ignore their values)
    float A[kCache], eold[kCache];
#pragma unroll
    for (int c = 0; c < kCache; ++c) {
      const int i = threadIdx.x + c * kSelThreads;
      const int slot = i < n8 ? i : s.cap + (i - n8);
      cpos[c] = -1;
      A[c] = 0.f;
      eold[c] = 0.f;
      if (i < nvirt) {
        cpos[c] = pos[slot];
        eold[c] = ema[slot];
        const float* mp = d.mass + lb * s.Hkv * s.S + slot;
        for (int h = 0; h < s.Hkv; ++h) A[c] += __ldg(mp + (size_t)h * s.S);
      }
    }
#pragma unroll
    for (int c = 0; c < kCache; ++c) {
      const int i = threadIdx.x + c * kSelThreads;
      const int p = cpos[c];
      cema[c] = 0.f;
      if (i < nvirt && p >= 0) {
        const int slot = i < n8 ? i : s.cap + (i - n8);
        nring += (i >= n8);
        const float a = fmaf(lam, eold[c], (1.0f - lam) * (A[c] * inv_hq));
        ema[slot] = a;
        cema[c] = a;
        if (p < thr) {
          amin = fminf(amin, a); amax = fmaxf(amax, a);
          pmin = min(pmin, p); pmax = max(pmax, p);
        }
      }
    }
    // slots beyond the register cache (long caches)
    for (int i = threadIdx.x + kCache * kSelThreads; i < nvirt; i += kSelThreads) {
      const int slot = i < n8 ? i : s.cap + (i - n8);
      const int p = pos[slot];
      if (i >= n8 && p < 0) continue;
      nring += (i >= n8);
      float Ai = 0.f;
      for (int h = 0; h < s.Hkv; ++h) Ai += __ldg(&d.mass[(lb * s.Hkv + h) * s.S + slot]);
      const float a = fmaf(lam, ema[slot], (1.0f - lam) * (Ai * inv_hq));
      ema[slot] = a;
      if (p < thr) {
        amin = fminf(amin, a); amax = fmaxf(amax, a);
        pmin = min(pmin, p); pmax = max(pmax, p);
      }
    }
  }
  // one combined block reduction of (nring, amin, amax, pmin, pmax)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    nring += __shfl_xor_sync(0xffffffffu, nring, o);
    amin = fminf(amin, __shfl_xor_sync(0xffffffffu, amin, o));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
    pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
  }
  if (lane == 0) {
    red5i[warp][0] = nring; red5i[warp][1] = pmin; red5i[warp][2] = pmax;
    red5f[warp][0] = amin; red5f[warp][1] = amax;
  }
  __syncthreads();
  nring = red5i[0][0]; pmin = red5i[0][1]; pmax = red5i[0][2];
  amin = red5f[0][0]; amax = red5f[0][1];
  for (int w = 1; w < kSelWarps; ++w) {
    nring += red5i[w][0];
    pmin = min(pmin, red5i[w][1]); pmax = max(pmax, red5i[w][2]);
    amin = fminf(amin, red5f[w][0]); amax = fmaxf(amax, red5f[w][1]);
  }
  const int n = n8 + nring - 1;          // resident entries, new token excluded
  const int k = max(0, n - N);

  // ------------------------------------------------ 3. rank and select
  if (k > 0) {
    const float arng = amax - amin;
    const float prng = (float)(pmax - pmin);
    const float alpha = s.alpha;
    auto score_key = [&](float a, int p) -> uint32_t {
      const float ah = arng > 0.f ? (a - amin) / arng : 0.f;
      const float rh = prng > 0.f ? (float)(p - pmin) / prng : 0.f;
      return __float_as_uint(alpha * ah + (1.0f - alpha) * rh);   // s >= 0: bits are monotone
    };
    unsigned long long best = ~0ull;
    int bslot = -1;
#pragma unroll
    for (int c = 0; c < kCache; ++c) {
      const int i = threadIdx.x + c * kSelThreads;
      const int p = cpos[c];
      if (i >= nvirt || p < 0 || p >= thr) continue;
      const int slot = i < n8 ? i : s.cap + (i - n8);
      const uint32_t key = score_key(cema[c], p);
      if (k > 1) keys[slot] = key;
      const unsigned long long comp = ((unsigned long long)key << 32) | (uint32_t)p;
      if (comp < best) { best = comp; bslot = slot; }
    }
    for (int i = threadIdx.x + kCache * kSelThreads; i < nvirt; i += kSelThreads) {
      const int slot = i < n8 ? i : s.cap + (i - n8);
      const int p = pos[slot];
      if (p < 0 || p >= thr) continue;
      const uint32_t key = score_key(ema[slot], p);
      if (k > 1) keys[slot] = key;
      const unsigned long long comp = ((unsigned long long)key << 32) | (uint32_t)p;
      if (comp < best) { best = comp; bslot = slot; }
    }
    if (k == 1) {
      // ---------------------------------------------- one eviction: argmin
      const unsigned long long thr1 = block_reduce(best, MinOp(), red64);
      if (best == thr1 && bslot >= 0) s_evslot = bslot;   // composites are unique
      __syncthreads();
      if (threadIdx.x == 0) {
        const int es = s_evslot;
        list[0] = (int)(uint32_t)(thr1 & 0xffffffffu);
        s_cnt = 1;
        if (es < s.cap) {
          s_k8 = 1;
        } else {
          pos[es] = -1;   // evicted ring entry: the slot becomes empty
        }
      }
    } else {
      // ---------------------------------------------- k > 1: 64-bit radix select
      for (int w = threadIdx.x; w < s.cap / 32; w += kSelThreads) bitmap[w] = 0u;
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
      const unsigned long long threshold = s_prefix | ~s_mask;
      // -------------------------------------------- 4. mark the evicted
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
  const int D = s.D;
  const int tl = t - s.W;                      // position leaving the FP16 window
  const int rs = tl >= 0 ? tl % s.WR : 0;
  const int rslot = s.cap + rs;
  // pos[rslot] is final here: a ring eviction of this step already cleared it
  const bool req = tl >= 0 && pos[rslot] == tl;
  if (req && n8p >= s.cap && threadIdx.x == 0) atomicOr(d.status, kStatusCapacity);
  const bool do_req = req && n8p < s.cap;
  if (k <= 1) {
    // ---------------------------------------------- 6+7. at most one move, then requant
    // The move reads slot n8 - 1 and the requant writes slot n8p, which can be
    // the same slot: every thread loads first, the block synchronises, then
    // every thread stores.
    const int dst = s_evslot, src = n8 - 1;
    const bool do_move = k == 1 && k8 == 1 && dst < src;
    moves = do_move ? 1 : 0;
    const int per_tok = D / 4 + D;             // K words + V bytes per head
    constexpr int kMv = 8;                     // move items per thread (Hkv*per_tok <= 8*256)
    constexpr int kRq = 8;                     // requant channels per thread (Hkv*D <= 8*256)
    if (s.Hkv * per_tok > kMv * kSelThreads || s.Hkv * D > kRq * kSelThreads) {
      // many KV heads: move first, then requantise (slot n8 - 1 is read before it is rewritten)
      for (int i = threadIdx.x; do_move && i < s.Hkv * per_tok; i += kSelThreads) {
        const int h = i / per_tok, e = i % per_tok;
        const size_t u = unit_index(s, l, b, h);
        uint8_t* k8u = d.k8 + u * (size_t)s.cstride * D;
        uint8_t* v8u = d.v8 + u * (size_t)s.cstride * D;
        if (e < D / 4) {
          const int c0 = (e / 4) * 16 + 2 * (e % 4);
          *reinterpret_cast<uint32_t*>(k8u + (size_t)(dst >> 4) * 16 * D + k8_offset(D, dst & 15, c0)) =
              *reinterpret_cast<const uint32_t*>(k8u + (size_t)(src >> 4) * 16 * D + k8_offset(D, src & 15, c0));
        } else {
          const int c = e - D / 4;
          v8u[(size_t)(dst >> 4) * 16 * D + v8_offset(D, dst & 15, c)] =
              v8u[(size_t)(src >> 4) * 16 * D + v8_offset(D, src & 15, c)];
        }
      }
      int mpos = 0;
      float mema = 0.f;
      if (threadIdx.x == 0 && do_move) { mpos = pos[src]; mema = ema[src]; }
      __syncthreads();
      if (threadIdx.x == 0 && do_move) { pos[dst] = mpos; ema[dst] = mema; }
      const char* k16b = reinterpret_cast<const char*>(d.k16);
      const char* v16b = reinterpret_cast<const char*>(d.v16);
      for (int i = threadIdx.x; do_req && i < s.Hkv * D; i += kSelThreads) {
        const int h = i / D, c = i % D;
        const size_t u = unit_index(s, l, b, h);
        const size_t rblk = (u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;
        const float xk = __half2float(*reinterpret_cast<const __half*>(k16b + rblk + k16_offset(D, rs & 15, c)));
        const float xv = __half2float(*reinterpret_cast<const __half*>(v16b + rblk + v16_offset(D, rs & 15, c)));
        const size_t dblk = (u * (size_t)(s.cstride / 16) + (n8p >> 4)) * 16 * D;
        d.k8[dblk + k8_offset(D, n8p & 15, c)] = quant_code_sel(xk, d.sK[u * D + c]);
        d.v8[dblk + v8_offset(D, n8p & 15, c)] = quant_code_sel(xv, d.sV[u * D + c]);
      }
      float rema = 0.f;
      if (threadIdx.x == 0 && do_req) rema = ema[rslot];
      __syncthreads();
      if (threadIdx.x == 0 && do_req) { pos[n8p] = tl; ema[n8p] = rema; pos[rslot] = -1; }
    } else {
    // every load of this phase is issued before any value is used
    uint32_t mv[kMv];
    unsigned short xk[kRq], xv[kRq];
    float sk[kRq], sv[kRq];
#pragma unroll
    for (int j = 0; j < kMv; ++j) {
      const int i = threadIdx.x + j * kSelThreads;
      mv[j] = 0u;
      if (do_move && i < s.Hkv * per_tok) {
        const int h = i / per_tok, e = i % per_tok;
        const size_t u = unit_index(s, l, b, h);
        const uint8_t* k8u = d.k8 + u * (size_t)s.cstride * D;
        const uint8_t* v8u = d.v8 + u * (size_t)s.cstride * D;
        if (e < D / 4)
          mv[j] = *reinterpret_cast<const uint32_t*>(k8u + (size_t)(src >> 4) * 16 * D +
                                                     k8_offset(D, src & 15, (e / 4) * 16 + 2 * (e % 4)));
        else
          mv[j] = v8u[(size_t)(src >> 4) * 16 * D + v8_offset(D, src & 15, e - D / 4)];
      }
    }
    const char* k16b = reinterpret_cast<const char*>(d.k16);
    const char* v16b = reinterpret_cast<const char*>(d.v16);
#pragma unroll
    for (int j = 0; j < kRq; ++j) {
      const int i = threadIdx.x + j * kSelThreads;
      xk[j] = xv[j] = 0;
      sk[j] = sv[j] = 1.f;
      if (do_req && i < s.Hkv * D) {
        const int h = i / D, c = i % D;
        const size_t u = unit_index(s, l, b, h);
        const size_t rblk = (u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;
        xk[j] = *reinterpret_cast<const unsigned short*>(k16b + rblk + k16_offset(D, rs & 15, c));
        xv[j] = *reinterpret_cast<const unsigned short*>(v16b + rblk + v16_offset(D, rs & 15, c));
        sk[j] = d.sK[u * D + c];
        sv[j] = d.sV[u * D + c];
      }
    }
    int mpos = 0;
    float mema = 0.f, rema = 0.f;
    if (threadIdx.x == 0) {
      if (do_move) { mpos = pos[src]; mema = ema[src]; }
      if (do_req) rema = ema[rslot];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kMv; ++j) {
      const int i = threadIdx.x + j * kSelThreads;
      if (do_move && i < s.Hkv * per_tok) {
        const int h = i / per_tok, e = i % per_tok;
        const size_t u = unit_index(s, l, b, h);
        uint8_t* k8u = d.k8 + u * (size_t)s.cstride * D;
        uint8_t* v8u = d.v8 + u * (size_t)s.cstride * D;
        if (e < D / 4)
          *reinterpret_cast<uint32_t*>(k8u + (size_t)(dst >> 4) * 16 * D +
                                       k8_offset(D, dst & 15, (e / 4) * 16 + 2 * (e % 4))) = mv[j];
        else
          v8u[(size_t)(dst >> 4) * 16 * D + v8_offset(D, dst & 15, e - D / 4)] = (uint8_t)mv[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kRq; ++j) {
      const int i = threadIdx.x + j * kSelThreads;
      if (do_req && i < s.Hkv * D) {
        const int h = i / D, c = i % D;
        const size_t u = unit_index(s, l, b, h);
        const size_t dblk = (u * (size_t)(s.cstride / 16) + (n8p >> 4)) * 16 * D;
        d.k8[dblk + k8_offset(D, n8p & 15, c)] = quant_code_sel(__half2float(__ushort_as_half(xk[j])), sk[j]);
        d.v8[dblk + v8_offset(D, n8p & 15, c)] = quant_code_sel(__half2float(__ushort_as_half(xv[j])), sv[j]);
      }
    }
    if (threadIdx.x == 0) {
      if (do_move) { pos[dst] = mpos; ema[dst] = mema; }
      if (do_req) { pos[n8p] = tl; ema[n8p] = rema; pos[rslot] = -1; }
    }
    }
  } else {
    // ---------------------------------------------- 6. compaction (tail fill), k > 1
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
      const int per_tok = D / 4 + D;             // K words + V bytes per head
      const long long total = (long long)moves * s.Hkv * per_tok;
      for (long long i = threadIdx.x; i < total; i += kSelThreads) {
        const int r = (int)(i / (s.Hkv * per_tok));
        const int rest = (int)(i % (s.Hkv * per_tok));
        const int h = rest / per_tok, e = rest % per_tok;
        const int src = (int)mover[r], dst = (int)hole[r];
        const size_t u = unit_index(s, l, b, h);
        uint8_t* k8u = d.k8 + u * (size_t)s.cstride * D;
        uint8_t* v8u = d.v8 + u * (size_t)s.cstride * D;
        if (e < D / 4) {
          // one 32-bit word = channels {16kk+2t, +1, +8, +9} of the token
          const int c0 = (e / 4) * 16 + 2 * (e % 4);
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
    // ---------------------------------------------- 7. requantise the entry leaving the window
    if (do_req) {
      const char* k16b = reinterpret_cast<const char*>(d.k16);
      const char* v16b = reinterpret_cast<const char*>(d.v16);
      for (int i = threadIdx.x; i < s.Hkv * D; i += kSelThreads) {
        const int h = i / D, c = i % D;
        const size_t u = unit_index(s, l, b, h);
        const size_t rblk = (u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;
        const float xk = __half2float(*reinterpret_cast<const __half*>(k16b + rblk + k16_offset(D, rs & 15, c)));
        const float xv = __half2float(*reinterpret_cast<const __half*>(v16b + rblk + v16_offset(D, rs & 15, c)));
        const size_t dblk = (u * (size_t)(s.cstride / 16) + (n8p >> 4)) * 16 * D;
        d.k8[dblk + k8_offset(D, n8p & 15, c)] = quant_code_sel(xk, d.sK[u * D + c]);
        d.v8[dblk + v8_offset(D, n8p & 15, c)] = quant_code_sel(xv, d.sV[u * D + c]);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        pos[n8p] = tl;
        ema[n8p] = ema[rslot];
        pos[rslot] = -1;
      }
    }
  }
  const int n8n = n8p + (do_req ? 1 : 0);
  const int requant = do_req ? 1 : 0;
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

int launch_select(const Shape& s, const Dev& d, long long step, int32_t* evicted_pos,
                  int32_t* n_evicted, int k_bound, cudaStream_t stream) {
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
  select_kernel<<<s.L * s.B, kSelThreads, smem, stream>>>(s, d, step, evicted_pos, n_evicted,
                                                          sort_cap);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace confkv
