// The selection of one (layer, sequence) at the end of a decode step: budget,
// EMA update, ranking, bottom-k selection, the sorted evicted positions,
// compaction of the INT8 region and requantisation of the token that leaves
// the FP16 window.  Run by the select kernel (one CTA per (layer, sequence))
// and, for small shapes, by the fused step kernel (attention.cu).
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
//
// Work layout.  The whole CTA walks the slots four at a time (int4 / float4
// loads of pos, EMA and the KV-head mass partials).  Ranking keys and the
// candidate positions go to shared memory (global scratch when a cache is too
// long for it).  One eviction is a block argmin; more use a radix select on
// the 32-bit keys (8-bit digits), with a second pass over positions only when
// keys tie exactly at the cut.  The evicted positions come out sorted from a
// bitmap over the position range.  Token payload work (moves and the
// requantisation) gives each warp one KV head: lane i owns one 32-bit word
// of the token's INT8 K (the four channels of one mma fragment) and the V
// channels i, i + 32, ...; the same lane-to-byte map for a move and the
// requantisation lets one thread read a slot before it rewrites it, so the
// common one-eviction path needs no barrier between them.
#pragma once
#include <cuda_runtime.h>
#include <cfloat>
#include <climits>
#include "confkv_internal.cuh"

namespace confkv {

constexpr int kSelThreads = 256;           // threads of the select kernel
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxWarps = 10;           // warps of any block that runs select_group
constexpr int kPosWords = 2048;            // sorted-output bitmap: 65536 positions per window
constexpr uint32_t kNoKey = 0xffffffffu;   // ranking key of a slot that is not a candidate
constexpr size_t kSelSmemKeysMax = 100 * 1024;

// Byte offsets into the dynamic shared memory of the select kernel.
struct SelSmem {
  int off_posbits;   // [kPosWords] u32
  int off_bm8;       // [cap / 32] u32: evicted INT8 slots
  int off_key;       // [S] u32 keys, then the compaction lists (keys in shared memory only)
  int off_pos;       // [S] i32 candidate positions, INT_MAX elsewhere (keys in shared memory only)
  int off_wpre;      // [cap / 32 + 1] i32 evicted slots before each bitmap word (ordered compaction)
  int off_stage;     // [warps][Hkv][64] u32 one token per warp in flight (ordered compaction)
  int bytes;
};


// Small shared arrays of select_group (in dynamic shared memory: a block
// that runs a selection after other work reuses its shared memory for them).
struct SelShared {
  int red_i[kSelMaxWarps][4];
  float red_f[kSelMaxWarps][2];
  unsigned long long red64[kSelMaxWarps];
  int hist[256];
  int scan_w[kSelMaxWarps];
  int s_digit, s_rem, s_dcnt, s_cnt, s_k8, s_evslot, s_evpos, s_prs;
};

// Order-preserving compaction of the INT8 region (the ablation of tail fill):
// every survivor at slot i moves to i - (evicted slots below i).  Windows of
// (NT / 32) slots in increasing order; warp w stages slot a + w in shared
// memory, the block synchronises, then every warp stores.  A destination is
// always below its source, so a window's stores never touch a later
// window's sources; inside a window a store can hit another warp's source,
// hence the barrier between the loads and the stores.  Windows of NT / 32
// slots, one per warp.  Returns the moves.
template <int D, int NT>
__device__ __forceinline__ int ordered_compaction(const Shape& s, const Dev& d, size_t u0, int n8,
                                                  const uint32_t* bm8, int* wpre, uint32_t* stage,
                                                  int32_t* pos, float* ema, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (n8 + 31) >> 5;
  constexpr int kV = D / 32;
  // exclusive prefix of the evicted counts per bitmap word, and the first hole
  int base = 0, first = INT_MAX;
  for (int w0 = 0; w0 < nw; w0 += NT) {
    const int w = w0 + threadIdx.x;
    const uint32_t bits = w < nw ? bm8[w] : 0u;
    const int c = __popc(bits);
    if (bits) first = min(first, w * 32 + __ffs(bits) - 1);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    __syncthreads();
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    int off = base, tot = 0;
    for (int ww = 0; ww < (NT / 32); ++ww) {
      if (ww < warp) off += red[ww];
      tot += red[ww];
    }
    if (w < nw) wpre[w] = off + incl - c;
    base += tot;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
  __syncthreads();
  if (lane == 0) red[warp] = first;
  __syncthreads();
  for (int ww = 0; ww < (NT / 32); ++ww) first = min(first, red[ww]);
  if (first >= n8) return 0;
  const size_t ustride8 = (size_t)s.cstride * D;
  const int kc0 = 16 * (lane >> 2) + 2 * (lane & 3);
  uint32_t* mine = stage + (size_t)warp * s.Hkv * 64;
  int moved = 0;
  for (int a = first; a < n8; a += (NT / 32)) {
    const int i = a + warp;
    int dst = i;
    int32_t mp = 0;
    float me = 0.f;
    if (i < n8 && !((bm8[i >> 5] >> (i & 31)) & 1u))
      dst = i - (wpre[i >> 5] + __popc(bm8[i >> 5] & ((1u << (i & 31)) - 1u)));
    const bool mv = dst != i;
    if (mv) {
      const size_t sblk = (size_t)(i >> 4) * 16 * D;
      for (int h = 0; h < s.Hkv; ++h) {
        const uint8_t* k8u = d.k8 + (u0 + h) * ustride8 + sblk;
        const uint8_t* v8u = d.v8 + (u0 + h) * ustride8 + sblk;
        if (lane < D / 4) mine[h * 64 + lane] = *reinterpret_cast<const uint32_t*>(k8u + k8_offset(D, i & 15, kc0));
        uint32_t vb = 0u;
#pragma unroll
        for (int c = 0; c < kV; ++c) vb |= (uint32_t)v8u[v8_offset(D, i & 15, lane + 32 * c)] << (8 * c);
        mine[h * 64 + 32 + lane] = vb;
      }
      mp = pos[i];
      me = ema[i];
      ++moved;
    }
    __syncthreads();
    if (mv) {
      const size_t dblk = (size_t)(dst >> 4) * 16 * D;
      for (int h = 0; h < s.Hkv; ++h) {
        uint8_t* k8u = d.k8 + (u0 + h) * ustride8 + dblk;
        uint8_t* v8u = d.v8 + (u0 + h) * ustride8 + dblk;
        if (lane < D / 4) *reinterpret_cast<uint32_t*>(k8u + k8_offset(D, dst & 15, kc0)) = mine[h * 64 + lane];
        const uint32_t vb = mine[h * 64 + 32 + lane];
#pragma unroll
        for (int c = 0; c < kV; ++c) v8u[v8_offset(D, dst & 15, lane + 32 * c)] = (uint8_t)(vb >> (8 * c));
      }
      if (lane == 0) {
        pos[dst] = mp;
        ema[dst] = me;
      }
    }
  }
  __syncthreads();
  // every lane of a moving warp counted the move once per warp: lane 0 reports
  int m = lane == 0 ? moved : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  int total = 0;
  for (int ww = 0; ww < (NT / 32); ++ww) total += red[ww];
  __syncthreads();
  return total;
}

// Stored byte of code = clamp(rint(x / s), -127, 127): the code + 128.
__device__ __forceinline__ uint32_t quant_code_sel(float x, float s) {
  float r = rintf(__fdiv_rn(x, s));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return (uint32_t)((int)r + kCodeBias);
}

// Warp 0 scans a 256-bin histogram for the digit that holds the rem-th
// smallest element; the other threads wait at the caller's barrier.
__device__ __forceinline__ void hist_find(const int* hist, int rem, int lane, int* s_digit,
                                          int* s_rem, int* s_dcnt) {
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
        *s_digit = lane * 8 + j;
        *s_rem = rem - before;
        *s_dcnt = cnt[j];
      }
      before += cnt[j];
    }
  }
}

// The selection of one (layer, sequence) lb = l * B + b, run by a whole
// block of NT threads (a multiple of 32, at most 320): the EMA update, the
// ranking and bottom-k, the sorted evicted positions, compaction and
// requantisation.  dsm is dynamic shared memory laid out as `sm` describes,
// sh the small shared arrays; the caller's block synchronises before and
// after.  The last selection of a step (of the L * B) takes the step's
// resident footprint and, for steps inside a graph reservation, advances the
// device step index.
// kGrid: the select kernel, one CTA per (layer, sequence): lbi is blockIdx.x
// (re-read rather than kept in a register, which the kernel's 64-register
// budget needs).
template <int D, bool kSmemKeys, bool kDevStep, bool kOrdered, int NT, bool kGrid>
__device__ __forceinline__ void select_group(const Shape s, const Dev d, long long step_arg, int lbi_arg,
                                             int32_t* __restrict__ evicted_out, int32_t* __restrict__ nevict_out,
                                             const SelSmem sm, unsigned char* dsm, SelShared& sh) {
  static_assert(NT % 32 == 0 && NT / 32 <= kSelMaxWarps, "select_group block size");
  constexpr int NW = NT / 32;
  uint32_t* posbits = reinterpret_cast<uint32_t*>(dsm + sm.off_posbits);
  uint32_t* bm8 = reinterpret_cast<uint32_t*>(dsm + sm.off_bm8);
  auto& red_i = sh.red_i;
  auto& red_f = sh.red_f;
  auto& red64 = sh.red64;
  int* hist = sh.hist;
  int* scan_w = sh.scan_w;
  int& s_digit = sh.s_digit;
  int& s_rem = sh.s_rem;
  int& s_dcnt = sh.s_dcnt;
  int& s_cnt = sh.s_cnt;
  int& s_k8 = sh.s_k8;
  int& s_evslot = sh.s_evslot;
  int& s_evpos = sh.s_evpos;
  int& s_prs = sh.s_prs;

  // a step inside a graph reservation reads the step index from the device
  const long long step = kDevStep ? __ldcg(d.step_dev) : step_arg;
#define lbi (kGrid ? blockIdx.x : (unsigned)lbi_arg)
  const int l = lbi / s.B, b = lbi % s.B;
  const size_t lb = lb_index(s, l, b);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cap = s.cap, WR = s.WR, S = s.S, Hkv = s.Hkv;
  int32_t* pos = d.pos + lb * S;
  float* ema = d.ema + lb * S;
  const float* mass = d.mass + lb * (size_t)Hkv * S;
  uint32_t* KEY = kSmemKeys ? reinterpret_cast<uint32_t*>(dsm + sm.off_key) : d.scratch + lb * S;
  int32_t* SPOS = kSmemKeys ? reinterpret_cast<int32_t*>(dsm + sm.off_pos) : nullptr;
  const int t = d.T0[b] + (int)step;
  const int n8 = d.n8[lb];
  const int thr = t - s.P;                 // candidates: pos < t - P
  const int tl = t - s.W;                  // position leaving the FP16 window
  const int rs = tl >= 0 ? tl % WR : 0;
  const int rslot = cap + rs;
  const int nvirt = n8 + WR;               // element e: INT8 slot e < n8, else ring slot cap + e - n8
  auto slot_of = [&](int e) { return e < n8 ? e : cap + (e - n8); };

  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_k8 = 0;
    s_evslot = -1;
    s_evpos = -1;
    if (lbi == 0 && step > 0) {
      // the previous step's footprint is complete (its kernels have ended)
      const int pp = (int)((step - 1) & 1);
      const unsigned long long e = d.stats->res_entries_acc[pp], by = d.stats->res_bytes_acc[pp];
      if (e > d.stats->peak_entries) d.stats->peak_entries = e;
      if (by > d.stats->peak_bytes) d.stats->peak_bytes = by;
      d.stats->res_entries_acc[pp] = 0ull;
      d.stats->res_bytes_acc[pp] = 0ull;
    }
  }
  for (int w = threadIdx.x; w < (n8 + 31) / 32; w += NT) bm8[w] = 0u;

  // ------------------------------------------------ 1. budget of this layer
  // c was merged once per sequence earlier in this step (the attention
  // kernel, or a vocabulary CTA of the fused step kernel).  In the fused
  // step another CTA of the same kernel wrote it, and the mass: both are
  // read through L2 there.
  const int N = ((float)(kGrid ? d.cval[b] : __ldcg(d.cval + b)) >= (float)s.tau) ? d.n_high[l] : d.n_low[l];

  // ------------------------------------------------ 2. EMA update, candidate ranges
  const int q8 = (n8 + 3) >> 2;            // INT8 quads (the last one may be partial)
  const int nq = q8 + (WR >> 2);
  const float lam = s.lam, inv_hq = 1.0f / (float)s.Hq;
  int nring = 0, ncand = 0;
  float amin = FLT_MAX, amax = -FLT_MAX;
  int pmin = INT_MAX, pmax = INT_MIN;
  // One quad of slots: the EMA update, the ranking's candidate ranges, the
  // keys in shared memory; the position held by the slot whose token leaves
  // the FP16 window (read here, before any slot of this step changes).
  auto ema_quad = [&](int q, const int4 P4, const float4 E4, const float4 A4) {
    const bool ring = q >= q8;
    const int slot0 = ring ? cap + 4 * (q - q8) : 4 * q;
    const int pv[4] = {P4.x, P4.y, P4.z, P4.w};
    const float ev[4] = {E4.x, E4.y, E4.z, E4.w};
    const float av[4] = {A4.x, A4.y, A4.z, A4.w};
    float nv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int p = pv[j];
      const bool valid = ring ? p >= 0 : 4 * q + j < n8;
      nv[j] = ev[j];
      int cp = INT_MAX;
      if (valid) {
        const float a = fmaf(lam, ev[j], (1.0f - lam) * (av[j] * inv_hq));
        nv[j] = a;
        nring += ring;
        if (p < thr) {
          cp = p;
          ++ncand;
          amin = fminf(amin, a); amax = fmaxf(amax, a);
          pmin = min(pmin, p); pmax = max(pmax, p);
        }
      }
      if (kSmemKeys) {
        KEY[slot0 + j] = __float_as_uint(nv[j]);
        SPOS[slot0 + j] = cp;
      }
      // (rslot lies in exactly one ring quad; s_prs is read only when tl >= 0)
      if (ring && tl >= 0 && slot0 + j == rslot) s_prs = p;
    }
    *reinterpret_cast<float4*>(ema + slot0) = make_float4(nv[0], nv[1], nv[2], nv[3]);
  };
  if constexpr (kGrid) {
    // two quads per thread and pass (a long cache over 256 threads)
    for (int q0 = threadIdx.x; q0 < nq; q0 += 2 * NT) {
      int4 P4[2];
      float4 E4[2], A4[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int q = q0 + r * NT;
        P4[r] = make_int4(-1, -1, -1, -1);
        E4[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        A4[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q < nq) {
          const int slot0 = q < q8 ? 4 * q : cap + 4 * (q - q8);
          P4[r] = *reinterpret_cast<const int4*>(pos + slot0);
          E4[r] = *reinterpret_cast<const float4*>(ema + slot0);
        }
      }
#pragma unroll 4
      for (int h = 0; h < Hkv; ++h) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int q = q0 + r * NT;
          if (q < nq) {
            const int slot0 = q < q8 ? 4 * q : cap + 4 * (q - q8);
            const float4 m = __ldg(reinterpret_cast<const float4*>(mass + (size_t)h * S + slot0));
            A4[r].x += m.x; A4[r].y += m.y; A4[r].z += m.z; A4[r].w += m.w;
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
        if (q0 + r * NT < nq) ema_quad(q0 + r * NT, P4[r], E4[r], A4[r]);
    }
  } else {
    // one quad per thread and pass, the KV heads' mass loads issued eight at
    // a time before they are summed (a short cache: the pass is one round of
    // loads, so what counts is how many are in flight)
    for (int q = threadIdx.x; q < nq; q += NT) {
      const int slot0 = q < q8 ? 4 * q : cap + 4 * (q - q8);
      const int4 P4 = *reinterpret_cast<const int4*>(pos + slot0);
      const float4 E4 = *reinterpret_cast<const float4*>(ema + slot0);
      float4 A4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int h0 = 0; h0 < Hkv; h0 += 8) {
        float4 m[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          m[j] = h0 + j < Hkv ? __ldcg(reinterpret_cast<const float4*>(mass + (size_t)(h0 + j) * S + slot0))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          A4.x += m[j].x; A4.y += m[j].y; A4.z += m[j].z; A4.w += m[j].w;
        }
      }
      ema_quad(q, P4, E4, A4);
    }
  }
  // one combined block reduction of (nring, ncand, amin, amax, pmin, pmax)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    nring += __shfl_xor_sync(0xffffffffu, nring, o);
    ncand += __shfl_xor_sync(0xffffffffu, ncand, o);
    amin = fminf(amin, __shfl_xor_sync(0xffffffffu, amin, o));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
    pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
  }
  if (lane == 0) {
    red_i[warp][0] = nring; red_i[warp][1] = ncand; red_i[warp][2] = pmin; red_i[warp][3] = pmax;
    red_f[warp][0] = amin; red_f[warp][1] = amax;
  }
  __syncthreads();
  nring = red_i[0][0]; ncand = red_i[0][1]; pmin = red_i[0][2]; pmax = red_i[0][3];
  amin = red_f[0][0]; amax = red_f[0][1];
  for (int w = 1; w < NW; ++w) {
    nring += red_i[w][0]; ncand += red_i[w][1];
    pmin = min(pmin, red_i[w][2]); pmax = max(pmax, red_i[w][3]);
    amin = fminf(amin, red_f[w][0]); amax = fmaxf(amax, red_f[w][1]);
  }
  const int n = n8 + nring - 1;            // resident entries, new token excluded
  const int kwant = max(0, n - N);
  const int k = min(kwant, ncand);         // a budget below the protected window is flagged below

  // ------------------------------------------------ 3. rank and select
  // s = alpha a_hat + (1 - alpha) r_hat >= 0, so its float bits order like s.
  const float arng = amax - amin, prng = (float)(pmax - pmin);
  const float ia = arng > 0.f ? 1.0f / arng : 0.f, ip = prng > 0.f ? 1.0f / prng : 0.f;
  const float alpha = s.alpha, beta = 1.0f - s.alpha;
  // candidate position of element e (INT_MAX if none) and its score bits
  auto cand_of = [&](int slot, bool int8) -> int {
    if (kSmemKeys) return SPOS[slot];
    const int p = pos[slot];
    return ((int8 || p >= 0) && p < thr) ? p : INT_MAX;
  };
  auto key_of = [&](int slot, int p) -> uint32_t {
    const float a = kSmemKeys ? __uint_as_float(KEY[slot]) : ema[slot];
    return __float_as_uint(alpha * ((a - amin) * ia) + beta * ((float)(p - pmin) * ip));
  };
  uint32_t kpre = 0u, kmask = 0u, ppre = 0u, pmask = 0u;
  bool kall = true;
  if (k == 1) {
    // ---------------------------------------------- one eviction: argmin of (s, position)
    unsigned long long best = ~0ull;
    int bslot = -1;
    for (int e = threadIdx.x; e < nvirt; e += NT) {
      const int slot = slot_of(e);
      const int p = cand_of(slot, e < n8);
      if (p == INT_MAX) continue;
      const unsigned long long comp = ((unsigned long long)key_of(slot, p) << 32) | (uint32_t)p;
      if (comp < best) { best = comp; bslot = slot; }
    }
    unsigned long long m = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long v = __shfl_xor_sync(0xffffffffu, m, o);
      m = v < m ? v : m;
    }
    if (lane == 0) red64[warp] = m;
    __syncthreads();
    m = red64[0];
    for (int w = 1; w < NW; ++w) m = red64[w] < m ? red64[w] : m;
    if (best == m && bslot >= 0) {   // composites are unique
      s_evslot = bslot;
      s_evpos = (int)(uint32_t)(m & 0xffffffffu);
    }
  } else if (k > 1) {
    // ---------------------------------------------- k > 1: keys, then radix select
    for (int e = threadIdx.x; e < nvirt; e += NT) {
      const int slot = slot_of(e);
      const int p = cand_of(slot, e < n8);
      KEY[slot] = p == INT_MAX ? kNoKey : key_of(slot, p);
    }
    int rem = k;
    kall = false;
    for (int shift = 24; shift >= 0 && !kall; shift -= 8) {
      if constexpr (NT == 256) {
        hist[threadIdx.x] = 0;
      } else {
        for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < nvirt; e += NT) {
        const uint32_t key = KEY[slot_of(e)];
        if ((key & kmask) == kpre) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (warp == 0) hist_find(hist, rem, lane, &s_digit, &s_rem, &s_dcnt);
      __syncthreads();
      kpre |= (uint32_t)s_digit << shift;
      kmask |= 255u << shift;
      rem = s_rem;
      kall = s_dcnt == rem;                  // the whole bucket goes: no finer digit needed
    }
    if (!kall) {
      // keys tie exactly at the cut: the rem oldest of them go
      bool pall = false;
      for (int shift = 24; shift >= 0 && !pall; shift -= 8) {
        if constexpr (NT == 256) {
        hist[threadIdx.x] = 0;
      } else {
        for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
      }
        __syncthreads();
        for (int e = threadIdx.x; e < nvirt; e += NT) {
          const int slot = slot_of(e);
          if (KEY[slot] != kpre) continue;
          const uint32_t p = (uint32_t)cand_of(slot, e < n8);
          if ((p & pmask) == ppre) atomicAdd(&hist[(p >> shift) & 255u], 1);
        }
        __syncthreads();
        if (warp == 0) hist_find(hist, rem, lane, &s_digit, &s_rem, &s_dcnt);
        __syncthreads();
        ppre |= (uint32_t)s_digit << shift;
        pmask |= 255u << shift;
        rem = s_rem;
        pall = s_dcnt == rem;
      }
    }
  }
  // element selected by the radix select (k > 1)
  auto evicted = [&](int slot, bool int8, int& p) -> bool {
    const uint32_t key = KEY[slot];
    if (key == kNoKey) return false;
    const uint32_t mk = key & kmask;
    if (mk > kpre) return false;
    p = cand_of(slot, int8);
    if (mk < kpre || kall) return true;
    return ((uint32_t)p & pmask) <= ppre;
  };

  // ------------------------------------------------ 4. sorted evicted positions
  int32_t* ev = evicted_out + lb * s.max_evict;
  if (k == 1) {
    __syncthreads();
    if (threadIdx.x == 0 && s.max_evict > 0) ev[0] = s_evpos;
  } else if (k > 1) {
    int out_base = 0;
    for (long long wb = pmin; wb < thr; wb += 32ll * kPosWords) {
      const int base = (int)wb;
      const int nwords = (int)min((long long)kPosWords, ((long long)thr - wb + 31) / 32);
      for (int w = threadIdx.x; w < nwords; w += NT) posbits[w] = 0u;
      __syncthreads();
      for (int e = threadIdx.x; e < nvirt; e += NT) {
        const int slot = slot_of(e);
        int p = 0;
        if (!evicted(slot, e < n8, p)) continue;
        const long long off = (long long)p - base;
        if (off >= 0 && off < 32ll * nwords) atomicOr(&posbits[off >> 5], 1u << (off & 31));
      }
      __syncthreads();
      // each thread owns 8 consecutive words; block exclusive scan of their counts
      constexpr int kWpt = (kPosWords + NT - 1) / NT;
      const int w0 = threadIdx.x * kWpt;
      int mine = 0;
#pragma unroll
      for (int j = 0; j < kWpt; ++j) mine += (w0 + j < nwords) ? __popc(posbits[w0 + j]) : 0;
      int incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) scan_w[warp] = incl;
      __syncthreads();
      int off = out_base + incl - mine, total = 0;
      for (int w = 0; w < NW; ++w) {
        if (w < warp) off += scan_w[w];
        total += scan_w[w];
      }
#pragma unroll
      for (int j = 0; j < kWpt; ++j) {
        if (w0 + j >= nwords) break;
        uint32_t bits = posbits[w0 + j];
        while (bits) {
          const int bit = __ffs(bits) - 1;
          bits &= bits - 1;
          if (off < s.max_evict) ev[off] = base + 32 * (w0 + j) + bit;
          ++off;
        }
      }
      out_base += total;
      __syncthreads();
    }
    // apply: INT8 evictions into the bitmap, ring evictions empty their slot
    int mycnt = 0, myk8 = 0;
    for (int e = threadIdx.x; e < nvirt; e += NT) {
      const int slot = slot_of(e);
      int p = 0;
      if (!evicted(slot, e < n8, p)) continue;
      ++mycnt;
      if (e < n8) {
        atomicOr(&bm8[slot >> 5], 1u << (slot & 31));
        ++myk8;
      } else {
        pos[slot] = -1;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mycnt += __shfl_xor_sync(0xffffffffu, mycnt, o);
      myk8 += __shfl_xor_sync(0xffffffffu, myk8, o);
    }
    if (lane == 0 && mycnt) atomicAdd(&s_cnt, mycnt);
    if (lane == 0 && myk8) atomicAdd(&s_k8, myk8);
  }
  if (k == 1 && threadIdx.x == 0) {
    s_cnt = 1;
    s_k8 = s_evslot < cap ? 1 : 0;
  }
  __syncthreads();
  const int cnt = s_cnt;
  const int k8 = s_k8;
  if (threadIdx.x == 0) {
    nevict_out[lb] = cnt;
    if (cnt != kwant) atomicOr(d.status, kStatusBadCount);
    if (cnt > s.max_evict) atomicOr(d.status, kStatusEvictBound);
  }

  // ------------------------------------------------ 5. compaction and requantisation
  const int n8p = n8 - k8;
  int moves = 0;
  constexpr bool ordered = kOrdered;   // order-preserving compaction (ablation instances only)
  if (ordered && k8 > 0) {
    if (k == 1) {
      if (threadIdx.x == 0) bm8[s_evslot >> 5] |= 1u << (s_evslot & 31);
      __syncthreads();
    }
    moves = ordered_compaction<D, NT>(s, d, unit_index(s, l, b, 0), n8, bm8,
                                  reinterpret_cast<int*>(dsm + sm.off_wpre),
                                  reinterpret_cast<uint32_t*>(dsm + sm.off_stage), pos, ema, red_i[0]);
  }
  const size_t u0 = unit_index(s, l, b, 0);
  const size_t ustride8 = (size_t)s.cstride * D;        // INT8 bytes per unit
  const size_t ustride16 = (size_t)WR * D * 2;          // FP16 ring bytes per unit
  bool req;
  if (k <= 1) {
    req = tl >= 0 && s_prs == tl && s_evslot != rslot;
  } else {
    req = tl >= 0 && pos[rslot] == tl;   // a ring eviction of this step already cleared it
  }
  if (req && n8p >= cap && threadIdx.x == 0) atomicOr(d.status, kStatusCapacity);
  const bool do_req = req && n8p < cap;
  const int kw = lane >> 2, kt = lane & 3;   // K word of this lane: channels 16kw + 2kt + {0,1,8,9}
  const int kc0 = 16 * kw + 2 * kt;
  constexpr int kVPerLane = D / 32;

  if (!ordered && k > 1 && k8 > 0) {
    // ---------------------------------------------- tail fill: holes < n8p <- survivors >= n8p
    uint32_t* hole = KEY;                 // [moves]
    uint32_t* mover = KEY + (S >> 1);     // [moves]
    const int nw = (n8 + 31) >> 5;
    int base_h = 0, base_m = 0;
    for (int w0 = 0; w0 < nw; w0 += NT) {
      const int w = w0 + threadIdx.x;
      uint32_t hb = 0u, mb = 0u;
      if (w < nw) {
        const uint32_t bits = bm8[w];
        // slots of this word below n8p (holes are evicted ones) and in [n8p, n8) (movers survive)
        const int lo = w * 32;
        const uint32_t below = n8p <= lo ? 0u : (n8p >= lo + 32 ? 0xffffffffu : ((1u << (n8p - lo)) - 1u));
        const uint32_t inreg = n8 >= lo + 32 ? 0xffffffffu : ((1u << (n8 - lo)) - 1u);
        hb = bits & below;
        mb = ~bits & inreg & ~below;
      }
      const int ch = __popc(hb), cm = __popc(mb);
      int ih = ch, im = cm;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int vh = __shfl_up_sync(0xffffffffu, ih, o);
        const int vm = __shfl_up_sync(0xffffffffu, im, o);
        if (lane >= o) { ih += vh; im += vm; }
      }
      __syncthreads();
      if (lane == 31) { red_i[warp][0] = ih; red_i[warp][1] = im; }
      __syncthreads();
      int offh = base_h, offm = base_m, th = 0, tm = 0;
      for (int ww = 0; ww < NW; ++ww) {
        if (ww < warp) { offh += red_i[ww][0]; offm += red_i[ww][1]; }
        th += red_i[ww][0];
        tm += red_i[ww][1];
      }
      int rh = offh + ih - ch, rm = offm + im - cm;
      while (hb) { const int j = __ffs(hb) - 1; hb &= hb - 1; hole[rh++] = w * 32 + j; }
      while (mb) { const int j = __ffs(mb) - 1; mb &= mb - 1; mover[rm++] = w * 32 + j; }
      base_h += th;
      base_m += tm;
    }
    moves = base_h;
    __syncthreads();
    // one warp per move, four KV heads at a time: every load before any store
    for (int mv = warp; mv < moves; mv += NW) {
      const int src = (int)mover[mv], dst = (int)hole[mv];
      if (lane == 0) {
        pos[dst] = pos[src];
        ema[dst] = ema[src];
      }
      const size_t sblk = (size_t)(src >> 4) * 16 * D, dblk = (size_t)(dst >> 4) * 16 * D;
      const int sk_off = k8_offset(D, src & 15, kc0), dk_off = k8_offset(D, dst & 15, kc0);
      for (int h0 = 0; h0 < Hkv; h0 += 4) {
        uint32_t kwv[4];
        uint8_t vbv[4][kVPerLane];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          if (h0 + hh >= Hkv) break;
          const uint8_t* k8u = d.k8 + (u0 + h0 + hh) * ustride8 + sblk;
          const uint8_t* v8u = d.v8 + (u0 + h0 + hh) * ustride8 + sblk;
          if (lane < D / 4) kwv[hh] = *reinterpret_cast<const uint32_t*>(k8u + sk_off);
#pragma unroll
          for (int i = 0; i < kVPerLane; ++i) vbv[hh][i] = v8u[v8_offset(D, src & 15, lane + 32 * i)];
        }
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          if (h0 + hh >= Hkv) break;
          uint8_t* k8u = d.k8 + (u0 + h0 + hh) * ustride8 + dblk;
          uint8_t* v8u = d.v8 + (u0 + h0 + hh) * ustride8 + dblk;
          if (lane < D / 4) *reinterpret_cast<uint32_t*>(k8u + dk_off) = kwv[hh];
#pragma unroll
          for (int i = 0; i < kVPerLane; ++i) v8u[v8_offset(D, dst & 15, lane + 32 * i)] = vbv[hh][i];
        }
      }
    }
    __syncthreads();   // a mover may sit in slot n8p, which the requantisation rewrites
  }

  // one eviction from the INT8 region: move slot n8 - 1 into the hole (same
  // lanes as the requantisation below, which may rewrite slot n8 - 1)
  const int dst1 = s_evslot, src1 = n8 - 1;
  const bool move1 = !ordered && k == 1 && k8 == 1 && dst1 < src1;
  if (move1) moves = 1;
  const char* k16b = reinterpret_cast<const char*>(d.k16);
  const char* v16b = reinterpret_cast<const char*>(d.v16);
  // metadata of the move and the requantisation, read by thread 0 before
  // any of it is written (slot n8 - 1 can be both a source and a target)
  int mpos = 0;
  float mema = 0.f, rema = 0.f;
  if (threadIdx.x == 0) {
    if (move1) { mpos = pos[src1]; mema = ema[src1]; }
    if (do_req) rema = ema[rslot];
  }
  if (move1 || do_req) {
    const size_t sblk = (size_t)(src1 >> 4) * 16 * D, dblk = (size_t)(dst1 >> 4) * 16 * D;
    const size_t qblk = (size_t)(n8p >> 4) * 16 * D;
    const size_t rblk = (size_t)(rs >> 4) * 16 * D * 2;
    for (int h = warp; h < Hkv; h += NW) {
      const size_t u = u0 + h;
      uint8_t* k8u = d.k8 + u * ustride8;
      uint8_t* v8u = d.v8 + u * ustride8;
      // every load of this KV head (the move's source, the ring entry and
      // the scales) before any store: one round of loads instead of two.  A
      // lane stores only bytes it loaded itself, so the requantisation may
      // rewrite the move's source slot n8 - 1 without a barrier.
      uint32_t kv = 0u;
      uint8_t vb[kVPerLane];
      uint2 xk = make_uint2(0u, 0u);
      float2 s01 = make_float2(1.f, 1.f), s89 = make_float2(1.f, 1.f);
      unsigned short xv[kVPerLane];
      float sv[kVPerLane];
      if (move1) {
        if (lane < D / 4) kv = *reinterpret_cast<const uint32_t*>(k8u + sblk + k8_offset(D, src1 & 15, kc0));
#pragma unroll
        for (int i = 0; i < kVPerLane; ++i) vb[i] = v8u[sblk + v8_offset(D, src1 & 15, lane + 32 * i)];
      }
      if (do_req) {
        const char* rk = k16b + u * ustride16 + rblk;
        const char* rv = v16b + u * ustride16 + rblk;
        const float* sKu = d.sK + u * D;
        const float* sVu = d.sV + u * D;
        if (lane < D / 4) {
          xk = *reinterpret_cast<const uint2*>(rk + k16_offset(D, rs & 15, kc0));
          s01 = *reinterpret_cast<const float2*>(sKu + kc0);
          s89 = *reinterpret_cast<const float2*>(sKu + kc0 + 8);
        }
#pragma unroll
        for (int i = 0; i < kVPerLane; ++i) {
          xv[i] = *reinterpret_cast<const unsigned short*>(rv + v16_offset(D, rs & 15, lane + 32 * i));
          sv[i] = sVu[lane + 32 * i];
        }
      }
      if (move1) {
        if (lane < D / 4) *reinterpret_cast<uint32_t*>(k8u + dblk + k8_offset(D, dst1 & 15, kc0)) = kv;
#pragma unroll
        for (int i = 0; i < kVPerLane; ++i) v8u[dblk + v8_offset(D, dst1 & 15, lane + 32 * i)] = vb[i];
      }
      if (do_req) {
        if (lane < D / 4) {
          const uint32_t w =
              quant_code_sel(__half2float(__ushort_as_half((unsigned short)(xk.x & 0xffffu))), s01.x) |
              quant_code_sel(__half2float(__ushort_as_half((unsigned short)(xk.x >> 16))), s01.y) << 8 |
              quant_code_sel(__half2float(__ushort_as_half((unsigned short)(xk.y & 0xffffu))), s89.x) << 16 |
              quant_code_sel(__half2float(__ushort_as_half((unsigned short)(xk.y >> 16))), s89.y) << 24;
          *reinterpret_cast<uint32_t*>(k8u + qblk + k8_offset(D, n8p & 15, kc0)) = w;
        }
#pragma unroll
        for (int i = 0; i < kVPerLane; ++i)
          v8u[qblk + v8_offset(D, n8p & 15, lane + 32 * i)] =
              (uint8_t)quant_code_sel(__half2float(__ushort_as_half(xv[i])), sv[i]);
      }
    }
  }
  if (threadIdx.x == 0) {
    if (k == 1 && dst1 >= cap) pos[dst1] = -1;   // evicted ring entry: the slot becomes empty
    if (move1) { pos[dst1] = mpos; ema[dst1] = mema; }
    if (do_req) { pos[n8p] = tl; ema[n8p] = rema; pos[rslot] = -1; }
  }
  const int n8n = n8p + (do_req ? 1 : 0);
  const int requant = do_req ? 1 : 0;
  if (threadIdx.x == 0) {
    d.n8[lb] = n8n;
    // algorithmic bytes of this (layer, sequence)
    const unsigned long long Dl = D, Hk = Hkv, Hq = s.Hq;
    const unsigned long long nres = (unsigned long long)n8 + nring;   // incl. new token
    const unsigned long long attn = Hk * Dl * (2ull * n8 + 4ull * nring) + 2ull * Hk * Dl * 4 +
                                    Hq * Dl * (2 + 4) + Hk * nres * 4;
    unsigned long long step_b = attn + nres * (4 + 4 + 4 + 4 * Hk) + 2ull * Hk * Dl * 2 * 2 +
                                (unsigned long long)requant * 2 * Hk * Dl * 3 +
                                (unsigned long long)moves * (2 * Hk * Dl + 8) * 2 +
                                4ull * (cnt + 1);
    if (l == 0) step_b += (unsigned long long)s.V * 4;
    atomicAdd(&d.stats->evicted, (unsigned long long)cnt);
    atomicAdd(&d.stats->moved, (unsigned long long)moves);
    atomicAdd(&d.stats->requant, (unsigned long long)requant);
    atomicAdd(&d.stats->attn_bytes, attn);
    atomicAdd(&d.stats->step_bytes, step_b);
    if (lbi == 0) atomicAdd(&d.stats->steps, 1ull);
    // resident footprint of this (layer, sequence) after the step: the INT8
    // region and the ring entries that neither were evicted nor left for INT8
    const unsigned long long ring_after = (unsigned long long)(nring - (cnt - k8) - requant);
    atomicAdd(&d.stats->res_entries_acc[step & 1], (unsigned long long)n8n + ring_after);
    atomicAdd(&d.stats->res_bytes_acc[step & 1], Hk * Dl * (2ull * (unsigned long long)n8n + 4ull * ring_after));
    const unsigned groups = kGrid ? gridDim.x : (unsigned)(s.L * s.B);
    if (kDevStep) {
      // the last CTA to finish advances the step index (every CTA has read it
      // before its own increment of the counter)
      __threadfence();
      if (atomicAdd(d.sel_done, 1u) == groups - 1u) {
        *d.sel_done = 0u;
        *d.step_dev = step + 1;
        __threadfence();
      }
    }
  }
}
#undef lbi



// Dynamic shared memory of one selection (keys in shared memory when they
// fit under kSelSmemKeysMax, else in the global scratch).
static inline SelSmem plan_select(const Shape& s) {
  SelSmem p{};
  size_t off = 0;
  p.off_posbits = (int)off;
  off += (size_t)kPosWords * 4;
  p.off_bm8 = (int)off;
  off += ((size_t)(s.cap / 32) * 4 + 15) & ~(size_t)15;
  p.off_wpre = p.off_stage = -1;
  if (s.compaction == 1) {
    p.off_wpre = (int)off;
    off += ((size_t)(s.cap / 32 + 1) * 4 + 15) & ~(size_t)15;
    p.off_stage = (int)off;
    off += (size_t)kSelWarps * s.Hkv * 64 * 4;
  }
  const size_t keys = (size_t)s.S * 4;
  if (off + 2 * keys <= kSelSmemKeysMax) {
    p.off_key = (int)off;
    off += keys;
    p.off_pos = (int)off;
    off += keys;
  } else {
    p.off_key = p.off_pos = -1;
  }
  p.bytes = (int)off;
  return p;
}

}  // namespace confkv
