// Mixed-precision single-query decode attention with attention-mass output.
//
// CONF-KV reads a contiguously compacted cache whose newest W tokens are FP16
// and whose older survivors are INT8 per head and channel, with the dequant
// fused into blockwise online-softmax reads (gist.science/de/paper/2605.24786,
// Systemintegration; paper.rainbus.top/paper/2605.24786, 前置知识: blockwise
// online softmax).  Algorithm 1 (same page, 方法步骤详情, steps 1 and 5) also
// needs the attention mass of every cached token to update its EMA; here the
// mass is the softmax probability averaged over the query heads.
//
// Work decomposition: one unit = (layer, sequence, KV head); its G = Hq/Hkv
// query heads share the unit's K/V.  A unit's 16-token blocks (INT8 blocks
// first, then the FP16 ring) are split over `splits` CTAs that form one
// thread-block cluster.
//
// Data movement: a producer warp streams the CTA's blocks into a ring of
// shared-memory stages with cp.async.bulk (1-D TMA) completing on mbarriers;
// an INT8 stage is 4 blocks (K span + V span, contiguous in HBM), an FP16
// stage 2 blocks, both 128*D bytes.  Four consumer warps take one block of a
// stage each and release the stage on an "empty" mbarrier.  Every wait is
// bounded: on time-out the kernel sets a status bit, drains its own copies
// and finishes without hanging.
//
// Per 16-token block a consumer warp issues two tensor-core products with
// mma.sync.m16n8k16 (fp16 in, fp32 accumulate):
//   QK^T: A = the G query rows, as fp16 "hi" parts in rows 0..G-1 and the
//         fp16 remainders q - hi in rows 8..8+G-1 (near-fp32 accuracy for
//         free in the otherwise empty rows); for INT8 blocks the per-channel
//         K scale and log2(e)/sqrt(d) are folded into q, so the B operand is
//         the raw code, converted exactly to fp16 with two byte permutes and
//         one packed subtract.
//   PV:   A = exp2(s - m) as hi/lo fp16 rows, B = V codes (or fp16 values);
//         the per-channel V scale multiplies the accumulator once, when the
//         warp moves from INT8 to FP16 blocks.
// Raw scores stay in shared memory; once the cluster knows every head's
// global max M and normaliser Lsum, each CTA turns its scores into mass:
//   mass_kvh(i) = sum_{g<G} exp2(s_gi - M_g) / Lsum_g
// and writes one fp32 per token (summed over KV heads by the select kernel).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>
#include <cfloat>
#include "confidence_merge.cuh"
#include "select_body.cuh"

namespace cg = cooperative_groups;

namespace confkv {

constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr long long kSpinLimit = 1LL << 22;   // mbarrier polls per wait (a few seconds at most)
constexpr float kQPre = 256.0f;               // q pre-scale before the hi/lo split
constexpr float kQPreInv = 1.0f / 256.0f;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// One poll of an mbarrier phase.  The thread may sleep in it for up to
// kSuspendNs until the phase completes (it wakes when the phase completes):
// waiting warps then take few issue slots from the warps that work.  With
// the hint the Qwen-32B attention kernel ran 0.2600 against 0.2639 ms per
// launch, GPT-2 batch 1 18.3 against 18.6 us per step; 200 ns and 10 us
// measured the same as 1 us.
constexpr uint32_t kSuspendNs = 1000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendNs)
      : "memory");
  return ok != 0;
}
// One poll without the suspend hint: whether the phase has completed now.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait: false after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (long long i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Stored INT8 bytes are code + 128 = u.  The fp16 with bits 0x6400 | u is
// exactly 1024 + u = 1152 + code, so two byte permutes turn four stored bytes
// into two half2 operands {byte0, byte1}, {byte2, byte3}.
//  - K operand: used as is; the constant 1152 contributes 1152 * sum_c q'_c to
//    every score of a query row, which is subtracted once per block in fp32
//    (the QK accumulator restarts at zero every block).
//  - V operand: also used as is; the PV accumulator gathers 1152 * sum p on
//    top of sum p * code.  That bias is subtracted every 16 INT8 blocks of a
//    warp and at the end of its INT8 blocks (ws_flush_v_bias), from the row
//    sum of p that the softmax keeps anyway; left to the end of a long INT8
//    region it would grow the accumulator ~1000-fold above the result and
//    the fp32 tensor-core sums would lose ~3e-3 over 8K tokens per warp.
__device__ __forceinline__ void u8x4_to_h2x2_biased(uint32_t w, uint32_t& b0, uint32_t& b1) {
  b0 = __byte_perm(w, 0x64646464u, 0x5140);
  b1 = __byte_perm(w, 0x64646464u, 0x5342);
}
// 2^x with the hardware approximation (relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_h2(__half a, __half b) {
  __half2 h = __halves2half2(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void split_hi_lo(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
}

// Two floats -> packed hi = fp16(x), lo = fp16(x - hi) pairs.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __float22half2_rn(make_float2(x0, x1));
  const float2 hf = __half22float2(h);
  const __half2 r = __float22half2_rn(make_float2(x0 - hf.x, x1 - hf.y));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float load_q(const void* q, size_t idx, int bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[idx]);
  return __half2float(reinterpret_cast<const __half*>(q)[idx]);
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// A fragments of the G query rows for all D/16 k-steps.  Row g (< G) holds
// hi(q'_g), row g + 8 holds lo(q'_g); q'_g[c] = q_g[c] * scale[c] * qs.
// Returns 1152 * sum_c (hi + lo) of the lane's row (for the K operand offset).
template <int D>
__device__ __forceinline__ float make_q_frag(uint32_t (&aq)[D / 16][4], const void* q, size_t qoff,
                                             int bf16, const float* kscale, float qs, int G,
                                             int g, int t) {
  float sum = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (g < G) {
      const int c0 = kk * 16 + 2 * t;
      const int cs[4] = {c0, c0 + 1, c0 + 8, c0 + 9};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float sc = kscale ? kscale[cs[e]] : 1.0f;
        x[e] = load_q(q, qoff + (size_t)g * D + cs[e], bf16) * sc * qs;
      }
    }
    __half h[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      split_hi_lo(x[e], h[e], lo[e]);
      sum += __half2float(h[e]) + __half2float(lo[e]);
    }
    aq[kk][0] = pack_h2(h[0], h[1]);    // row g,   k = 2t, 2t+1
    aq[kk][1] = pack_h2(lo[0], lo[1]);  // row g+8, k = 2t, 2t+1
    aq[kk][2] = pack_h2(h[2], h[3]);    // row g,   k = 2t+8, 2t+9
    aq[kk][3] = pack_h2(lo[2], lo[3]);  // row g+8, k = 2t+8, 2t+9
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  return 1152.0f * sum;
}

// Online-softmax update for one 16-token block: scores sc4[nt][j] belong to
// tokens 8*nt + 2t + j of row g.  Writes the raw scores to shared memory and
// returns the P fragment (hi rows g, lo rows g+8).  The reference maximum
// m_run only moves when the block maximum exceeds it by more than 8 (log2
// units), so most blocks skip rescaling the accumulator; p = 2^(s - m_run)
// then stays below 2^8, well inside fp16.
template <int D, bool kFlush>
__device__ __forceinline__ void softmax_block(float (&sc4)[2][2], const bool (&valid)[2][2],
                                              int G, int g, float& m_run, float& l_run,
                                              float& l_fl, float (&acc)[D / 8][4], float* sc_dst,
                                              uint32_t (&pa)[4], float* sc_regs) {
  // Rows g >= G (padding) see q = 0, so their scores are 0: they keep a
  // state of their own that nothing reads.
  float mloc = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (!valid[nt][j]) sc4[nt][j] = -INFINITY;
      mloc = fmaxf(mloc, sc4[nt][j]);
    }
  // The row maximum of the four lanes exceeds m_run + 8 exactly when one
  // lane's own maximum does, so the quad reduction runs only then.
  if (__any_sync(0xffffffffu, mloc > m_run + 8.0f)) {
    mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
    mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
    const bool move = mloc > m_run + 8.0f;   // true for the first finite block too
    const float corr = move ? (m_run == -INFINITY ? 0.f : ex2(m_run - mloc)) : 1.0f;
    if (move) m_run = mloc;
    l_run *= corr;
    if (kFlush) l_fl *= corr;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      acc[j][0] *= corr; acc[j][1] *= corr; acc[j][2] *= corr; acc[j][3] *= corr;
    }
  }
  // m_run is -inf only while every score of the row so far is: then any
  // finite reference gives p = 2^(-inf) = 0 as well
  const float m_ref = m_run == -INFINITY ? 0.f : m_run;
  float p[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) p[nt][j] = ex2(sc4[nt][j] - m_ref);
  l_run += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
  if (sc_regs) {
    sc_regs[0] = sc4[0][0]; sc_regs[1] = sc4[0][1]; sc_regs[2] = sc4[1][0]; sc_regs[3] = sc4[1][1];
  } else if (g < G) {
    *reinterpret_cast<float2*>(sc_dst) = make_float2(sc4[0][0], sc4[0][1]);
    *reinterpret_cast<float2*>(sc_dst + 8) = make_float2(sc4[1][0], sc4[1][1]);
  }
  split2(p[0][0], p[0][1], pa[0], pa[1]);   // rows g / g+8, tokens 2t, 2t+1
  split2(p[1][0], p[1][1], pa[2], pa[3]);   // rows g / g+8, tokens 8+2t, 9+2t
}

// Stage schedule of one CTA: INT8 blocks [a0, a1) in groups of 4, then ring
// blocks [r0, r1) in groups of 2.
struct Sched {
  int a0, a1, r0, r1, n8st, nst;
  __device__ void init(int blk0, int blk1, int nb8) {
    a0 = blk0;
    a1 = max(blk0, min(blk1, nb8));
    r0 = max(blk0, nb8) - nb8;
    r1 = max(blk1, nb8) - nb8;
    n8st = (a1 - a0 + 3) / 4;
    nst = n8st + (r1 - r0 + 1) / 2;
  }
  __device__ void first_last(int i, bool& ring, int& first, int& nb) const {
    if (i < n8st) {
      ring = false;
      first = a0 + 4 * i;
      nb = min(4, a1 - first);
    } else {
      ring = true;
      first = r0 + 2 * (i - n8st);
      nb = min(2, r1 - first);
    }
  }
};

// Per-warp attention state of one unit.
template <int D>
struct WarpState {
  uint32_t aq[D / 16][4];   // query A fragments (INT8 version, then FP16 version)
  float acc[D / 8][4];      // PV accumulators: rows g (hi P) and g + 8 (lo P)
  float m_run, l_run;       // reference maximum (log2 units) and lane-partial sum
  float l_flushed;          // part of l_run whose INT8 V bias is already removed
  float qoffset;            // -1152 * sum(q') / kQPre of the row: the INT8 K operand
                            // offset, in score units and negated
  int n8blk;                // INT8 blocks done by this warp in this unit
  bool in_ring;
};

template <int D>
__device__ __forceinline__ void ws_begin(WarpState<D>& w, const void* q, size_t qoff, int bf16,
                                         const float* sKu, float qs, int G, int g, int t) {
  w.qoffset = -kQPreInv * make_q_frag<D>(w.aq, q, qoff, bf16, sKu, qs, G, g, t);
#pragma unroll
  for (int j = 0; j < D / 8; ++j) w.acc[j][0] = w.acc[j][1] = w.acc[j][2] = w.acc[j][3] = 0.f;
  w.m_run = -INFINITY;
  w.l_run = 0.f;
  w.l_flushed = 0.f;
  w.n8blk = 0;
  w.in_ring = false;
}

// Removes the INT8 V bias 1152 * sum p that the accumulator gathered since
// the last flush.  The INT8 V operand enters the products as fp16
// 1152 + code (two byte permutes, no subtraction).  l_run - l_flushed is this
// lane's sum of the p since then (both are rescaled with the accumulator):
// the four lanes of a row add up the row's bias.  The high and low parts of
// P sit in rows g and g + 8; the bias of both is removed from row g, whose
// sum with row g + 8 is the output.
template <int D>
__device__ __forceinline__ void ws_flush_v_bias(WarpState<D>& w) {
  float l = w.l_run - w.l_flushed;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  const float bias = 1152.0f * l;
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    w.acc[j][0] -= bias;
    w.acc[j][1] -= bias;
  }
  w.l_flushed = w.l_run;
}

// Multiply what the INT8 codes accumulated by the per-channel V scale.
template <int D>
__device__ __forceinline__ void ws_scale_v(WarpState<D>& w, const float* sVu, int t) {
  // the bias of the blocks since the last flush (all of them without
  // flushes), then the scale; called once per unit, so l_flushed is left
  float l = w.l_run - w.l_flushed;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  const float bias = 1152.0f * l;
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    const float2 sv = *reinterpret_cast<const float2*>(sVu + j * 8 + 2 * t);
    w.acc[j][0] = (w.acc[j][0] - bias) * sv.x;
    w.acc[j][1] = (w.acc[j][1] - bias) * sv.y;
    w.acc[j][2] *= sv.x;
    w.acc[j][3] *= sv.y;
  }
}

// INT8 -> FP16 transition: unscaled q fragments, V scale applied to the
// accumulator.
template <int D>
__device__ __forceinline__ void ws_to_ring(WarpState<D>& w, const void* q, size_t qoff, int bf16,
                                           float qs, const float* sVu, int G, int g, int t) {
  make_q_frag<D>(w.aq, q, qoff, bf16, nullptr, qs, G, g, t);
  w.qoffset = 0.f;
  ws_scale_v<D>(w, sVu, t);
  w.in_ring = true;
}

// One INT8 block at shared-memory addresses kb / vb (16*D bytes each).
// kFlush: remove the INT8 V bias every 16 blocks of the warp (long INT8
// regions); otherwise it is removed once, when the warp leaves them.
template <int D, bool kFlush>
__device__ __forceinline__ void int8_block(WarpState<D>& w, uint32_t kb, uint32_t vb, int blk,
                                           int n8, int G, int g, int t, int lane, float* sc_dst,
                                           float* sc_regs = nullptr) {
  constexpr int NC = D / 32;
  uint4 kw[NC], vw[NC];
#pragma unroll
  for (int r = 0; r < NC; ++r) kw[r] = lds128(kb + r * 512 + lane * 16);
#pragma unroll
  for (int r = 0; r < NC; ++r) vw[r] = lds128(vb + r * 512 + lane * 16);
  float sc4[2][2];
  bool valid[2][2];
  // tokens of this lane left in the INT8 region from its first (2t)
  const int rem = n8 - blk * 16 - 2 * t;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t b0, b1;
      u8x4_to_h2x2_biased(comp(kw[nt * (NC / 2) + (kk >> 2)], kk & 3), b0, b1);
      mma16816(c, w.aq[kk], b0, b1);
    }
    // kQPreInv is a power of two: the same value as ((c0 + c2) - 1152 sum q') / kQPre
    sc4[nt][0] = fmaf(c[0] + c[2], kQPreInv, w.qoffset);
    sc4[nt][1] = fmaf(c[1] + c[3], kQPreInv, w.qoffset);
    valid[nt][0] = nt * 8 < rem;
    valid[nt][1] = nt * 8 + 1 < rem;
  }
  uint32_t pa[4];
  softmax_block<D, kFlush>(sc4, valid, G, g, w.m_run, w.l_run, w.l_flushed, w.acc, sc_dst, pa,
                           sc_regs);
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    uint32_t b0, b1;
    u8x4_to_h2x2_biased(comp(vw[j >> 2], j & 3), b0, b1);   // 1152 + code: bias flushed below
    mma16816(w.acc[j], pa, b0, b1);
  }
  if (kFlush && (++w.n8blk & 15) == 0) ws_flush_v_bias<D>(w);
}

// One FP16 ring block at kb / vb (32*D bytes each); posb = the block's 16
// slot positions (-1 = empty).
template <int D>
__device__ __forceinline__ void ring_block(WarpState<D>& w, uint32_t kb, uint32_t vb,
                                           const int32_t* posb, int G, int g, int t, int lane,
                                           float* sc_dst, float* sc_regs = nullptr, int live = -1) {
  // live: the block's slot (0-15) that holds a token whatever posb says (a
  // fused step's new token, appended after posb was copied), or -1
  const int2 pv0 = *reinterpret_cast<const int2*>(posb + 2 * t);
  const int2 pv1 = *reinterpret_cast<const int2*>(posb + 8 + 2 * t);
  bool valid[2][2];
  valid[0][0] = pv0.x >= 0 || 2 * t == live; valid[0][1] = pv0.y >= 0 || 2 * t + 1 == live;
  valid[1][0] = pv1.x >= 0 || 8 + 2 * t == live; valid[1][1] = pv1.y >= 0 || 9 + 2 * t == live;
  float sc4[2][2];
  uint32_t pa[4];
  if constexpr (D == 64) {
    // Every K word of the block is loaded before the first product and every
    // V word before the first PV product: the loads are volatile asm, so a
    // load between two products holds back the second one for the full
    // shared-memory latency.  (GPT-2 shapes: batch 1 18.6 against 20.1 us
    // per step, batch 8 46.1 against 48.0 us.)
    uint4 kw[D / 16];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) kw[i] = lds128(kb + i * 512 + lane * 16);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint4 w4 = kw[nt * (D / 32) + (kk >> 1)];
        mma16816(c, w.aq[kk], comp(w4, (kk & 1) * 2), comp(w4, (kk & 1) * 2 + 1));
      }
      sc4[nt][0] = (c[0] + c[2]) * kQPreInv;
      sc4[nt][1] = (c[1] + c[3]) * kQPreInv;
    }
    softmax_block<D, false>(sc4, valid, G, g, w.m_run, w.l_run, w.l_flushed, w.acc, sc_dst, pa, sc_regs);
    uint4 vw[D / 16];
#pragma unroll
    for (int r = 0; r < D / 16; ++r) vw[r] = lds128(vb + r * 512 + lane * 16);
#pragma unroll
    for (int r = 0; r < D / 16; ++r) {
      mma16816(w.acc[2 * r], pa, vw[r].x, vw[r].y);
      mma16816(w.acc[2 * r + 1], pa, vw[r].z, vw[r].w);
    }
  } else {
    // D = 128: loads next to their products.  The preloaded form above
    // needs 32 more registers at the consumers' 168-register limit and ran
    // slower here (Qwen-32B attention 0.266 against 0.263 ms per launch).
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint4 w4 = lds128(kb + (nt * (D / 32) + (kk >> 1)) * 512 + lane * 16);
        mma16816(c, w.aq[kk], comp(w4, (kk & 1) * 2), comp(w4, (kk & 1) * 2 + 1));
      }
      sc4[nt][0] = (c[0] + c[2]) * kQPreInv;
      sc4[nt][1] = (c[1] + c[3]) * kQPreInv;
    }
    softmax_block<D, false>(sc4, valid, G, g, w.m_run, w.l_run, w.l_flushed, w.acc, sc_dst, pa, sc_regs);
#pragma unroll
    for (int r = 0; r < D / 16; ++r) {
      const uint4 w4 = lds128(vb + r * 512 + lane * 16);
      mma16816(w.acc[2 * r], pa, w4.x, w4.y);
      mma16816(w.acc[2 * r + 1], pa, w4.z, w4.w);
    }
  }
}

// End of a warp's blocks: V scale if it never reached the ring, the row sum
// over the row's four lanes, and (m, l, o) to shared memory.
template <int D>
__device__ __forceinline__ void ws_store(WarpState<D>& w, const float* sVu, int G, int g, int t,
                                         float* wm, float* wl, float* wo) {
  if (!w.in_ring) ws_scale_v<D>(w, sVu, t);
  float l = w.l_run;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  if (g < G) {
    float* o = wo + g * D;
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
      *reinterpret_cast<float2*>(o + j * 8 + 2 * t) =
          make_float2(w.acc[j][0] + w.acc[j][2], w.acc[j][1] + w.acc[j][3]);
    if (t == 0) {
      wm[g] = w.m_run;
      wl[g] = l;
    }
  }
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// ===========================================================================
// Split kernel: the blocks of one unit spread over a cluster of `splits`
// CTAs (long caches or few units); merged through distributed shared memory.
// ===========================================================================
template <int D>
__global__ void __launch_bounds__(kAttnThreads) attention_kernel(Shape s, Dev d,
                                                                 const void* __restrict__ q,
                                                                 float* __restrict__ out,
                                                                 int32_t* __restrict__ budget,
                                                                 float* __restrict__ conf_out,
                                                                 int splits, int chunk_blocks,
                                                                 int stages) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  constexpr int kStageBytes = 128 * D;       // 4 INT8 blocks or 2 FP16 blocks (K + V)
  constexpr int kHalf = kStageBytes / 2;     // K span | V span
  const int G = s.G;
  const int chunk_tok = chunk_blocks * 16;
  unsigned char* sbuf = smem_raw;                                   // [stages][kStageBytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + stages * kStageBytes);  // full, empty
  float* sc = reinterpret_cast<float*>(bars + 2 * kMaxStages);      // [G][chunk_tok]
  float* wm = sc + G * chunk_tok;                     // [NW][G]
  float* wl = wm + kConsumerWarps * G;                // [NW][G]
  float* wo = wl + kConsumerWarps * G;                // [NW][G][D]
  float* cm = wo + kConsumerWarps * G * D;            // [G]    CTA max     (read by peers)
  float* cl = cm + kMaxG;                             // [G]    CTA sum     (read by peers)
  float* co = cl + kMaxG;                             // [G][D] CTA output  (read by peers)
  float* gM = co + G * D;                             // [G]
  float* gL = gM + kMaxG;                             // [G]
  int& s_abort = *reinterpret_cast<int*>(gL + kMaxG);  // set when a bounded wait gave up

  cg::cluster_group cluster = cg::this_cluster();
  const int u = blockIdx.x / splits;
  const int rank = blockIdx.x % splits;
  const int h = u % s.Hkv;
  const int b = (u / s.Hkv) % s.B;
  const int l = u / (s.Hkv * s.B);
  const size_t lb = lb_index(s, l, b);
  const int n8 = d.n8[lb];
  const int nb8 = (n8 + 15) >> 4;
  const int nbR = s.WR >> 4;
  const int nbT = nb8 + nbR;
  const int blk0 = min(nbT, rank * chunk_blocks);
  const int blk1 = min(nbT, blk0 + chunk_blocks);
  Sched sch;
  sch.init(blk0, blk1, nb8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const size_t qoff = (lb * s.Hq + (size_t)h * G) * D;
  const float* sKu = d.sK + (size_t)u * D;
  const float* sVu = d.sV + (size_t)u * D;
  const uint8_t* k8u = d.k8 + (size_t)u * s.cstride * D;
  const uint8_t* v8u = d.v8 + (size_t)u * s.cstride * D;
  const char* k16u = reinterpret_cast<const char*>(d.k16) + (size_t)u * s.WR * D * 2;
  const char* v16u = reinterpret_cast<const char*>(d.v16) + (size_t)u * s.WR * D * 2;
  const int32_t* posR = d.pos + lb * s.S + s.cap;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(kMaxStages + i); };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < stages; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------ producer warp
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < sch.nst; ++i) {
        const int slot = i % stages, use = i / stages;
        if (use >= 1 && !mbar_wait(empty_bar(slot), (use - 1) & 1)) {
          atomicOr(d.status, kStatusTimeout);
          s_abort = 1;
          break;
        }
        if (*(volatile int*)&s_abort) break;
        bool ring;
        int first, nb;
        sch.first_last(i, ring, first, nb);
        const uint32_t span = (uint32_t)(nb * 16 * D * (ring ? 2 : 1));
        const char* ksrc = ring ? k16u + (size_t)first * 32 * D
                                : reinterpret_cast<const char*>(k8u) + (size_t)first * 16 * D;
        const char* vsrc = ring ? v16u + (size_t)first * 32 * D
                                : reinterpret_cast<const char*>(v8u) + (size_t)first * 16 * D;
        const uint32_t dst = smem_u32(sbuf + (size_t)slot * kStageBytes);
        mbar_arrive_tx(full_bar(slot), 2 * span);
        bulk_g2s(dst, ksrc, span, full_bar(slot));
        bulk_g2s(dst + kHalf, vsrc, span, full_bar(slot));
        issued = i + 1;
      }
      // drain: every issued copy must have landed before the CTA moves on
      for (int i = max(0, issued - stages); i < issued; ++i) {
        if (!mbar_wait(full_bar(i % stages), (i / stages) & 1)) atomicOr(d.status, kStatusTimeout);
      }
    }
  } else {
    // ------------------------------------------------ consumer warps
    WarpState<D> ws;
    const float qs = kQPre * 1.4426950408889634f * rsqrtf((float)D);
    ws_begin<D>(ws, q, qoff, s.qbf16, sKu, qs, G, g, t);
    for (int i = 0; i < sch.nst; ++i) {
      const int slot = i % stages;
      if (!mbar_wait(full_bar(slot), (i / stages) & 1)) {
        if (lane == 0) atomicOr(d.status, kStatusTimeout);
        s_abort = 1;
        break;
      }
      if (*(volatile int*)&s_abort) break;
      bool ring;
      int first, nb;
      sch.first_last(i, ring, first, nb);
      const uint32_t stage = smem_u32(sbuf + (size_t)slot * kStageBytes);
      if (!ring) {
        if (warp < nb) {
          const int blk = first + warp;
          int8_block<D, true>(ws, stage + warp * 16 * D, stage + kHalf + warp * 16 * D, blk, n8, G, g,
                              t, lane, sc + g * chunk_tok + (blk - blk0) * 16 + 2 * t);
        }
      } else {
        const int jb = warp - 2 * ((i - sch.n8st) & 1);
        if (jb >= 0 && jb < nb) {
          if (!ws.in_ring) ws_to_ring<D>(ws, q, qoff, s.qbf16, qs, sVu, G, g, t);
          const int rb = first + jb;
          ring_block<D>(ws, stage + jb * 32 * D, stage + kHalf + jb * 32 * D, posR + rb * 16, G, g,
                        t, lane, sc + g * chunk_tok + (nb8 + rb - blk0) * 16 + 2 * t);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(slot));
    }
    ws_store<D>(ws, sVu, G, g, t, wm + warp * G, wl + warp * G, wo + warp * G * D);
  }
  __syncthreads();
  const bool aborted = s_abort != 0;
  for (int i = threadIdx.x; i < G * D; i += kAttnThreads) {
    const int gg = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wm[w * G + gg]);
    float o = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = wm[w * G + gg];
      const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      o += wo[(w * G + gg) * D + c] * f;
      L += wl[w * G + gg] * f;
    }
    co[gg * D + c] = o;
    if (c == 0) {
      cm[gg] = M;
      cl[gg] = L;
    }
  }
  // ---------------------------------------------------------------- cluster merge
  cluster.sync();
  if (threadIdx.x < G) {
    const int gg = threadIdx.x;
    float M = -INFINITY;
    for (int r = 0; r < splits; ++r) M = fmaxf(M, cluster.map_shared_rank(cm, r)[gg]);
    float L = 0.f;
    for (int r = 0; r < splits; ++r) {
      const float mr = cluster.map_shared_rank(cm, r)[gg];
      if (mr != -INFINITY) L += cluster.map_shared_rank(cl, r)[gg] * ex2(mr - M);
    }
    gM[gg] = M;
    gL[gg] = L;
  }
  __syncthreads();
  if (!aborted) {
    // attention mass of this CTA's tokens, summed over its G query heads
    float* mass_u = d.mass + (size_t)u * s.S;
    const int ntok = (blk1 - blk0) * 16;
    for (int i = threadIdx.x; i < ntok; i += kAttnThreads) {
      const float s0 = sc[i];
      if (s0 == -INFINITY) continue;   // empty ring slot or tail past n8
      float m = 0.f;
      for (int gg = 0; gg < G; ++gg) m += ex2(sc[gg * chunk_tok + i] - gM[gg]) / gL[gg];
      const int blk = blk0 + (i >> 4);
      const int slot = blk < nb8 ? blk * 16 + (i & 15) : s.cap + (blk - nb8) * 16 + (i & 15);
      mass_u[slot] = m;
    }
    if (rank == 0) {
      float* o = out + qoff;
      for (int i = threadIdx.x; i < G * D; i += kAttnThreads) {
        const int gg = i / D;
        float acc_o = 0.f;
        for (int r = 0; r < splits; ++r) {
          const float mr = cluster.map_shared_rank(cm, r)[gg];
          if (mr != -INFINITY) acc_o += cluster.map_shared_rank(co, r)[i] * ex2(mr - gM[gg]);
        }
        o[i] = acc_o / gL[gg];
      }
    }
  }
  cluster.sync();   // peers keep their shared memory alive until rank 0 has read it
  // confidence and budgets of sequence blockIdx.x (once per sequence)
  if ((int)blockIdx.x < s.B && warp == 0) conf_merge_warp(s, d, blockIdx.x, budget, conf_out);
}

// ===========================================================================
// Persistent kernel: two CTAs per SM walk the units u = blockIdx.x,
// blockIdx.x + gridDim.x, ...  Each CTA has three roles:
//   producer warp   streams, unit after unit without stopping, a small unit
//                   header (query rows, K and V scales, ring positions) and
//                   the unit's K/V blocks into shared memory (1-D TMA bulk
//                   copies completing on mbarriers; K/V with an evict-first
//                   L2 hint);
//   4 consumer warps take one block of every stage and keep the online
//                   softmax state; the raw scores go to this CTA's slot of a
//                   global scratch buffer (evict-last: it is rewritten every
//                   unit and stays in L2);
//   epilogue warp   merges the consumers' partial results of unit u, writes
//                   the output and the per-token attention mass, while the
//                   consumers already work on unit u + 1.
// The per-unit buffers handed to the epilogue (partials, score slot) and the
// unit header are double-buffered.  Every mbarrier wait is bounded.
// ===========================================================================
constexpr int kPConsumers = 4;
constexpr int kPThreads = (kPConsumers + 2) * 32;
constexpr int kPMaxStages = 12;
// mbarriers of the persistent kernel: full and empty per stage, header full
// and empty, done and efree (two each), and the fused step's append; an even
// count keeps the shared ints after them 16-byte aligned
constexpr int kPBars = 2 * kPMaxStages + 10;

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Ring positions are copied into the unit header up to this ring size; longer
// rings (a cache kept entirely in FP16) are read from global memory instead,
// so the header does not crowd out the K/V stages.
constexpr int kHdrRingMax = 1024;

// Shared-memory header of one unit (byte offsets).
struct HeaderLayout {
  int q, sk, sv, pos, bytes;
  bool pos_in;   // ring positions in the header
  __host__ __device__ HeaderLayout(int G, int D, int WR) {
    q = 0;
    sk = (G * D * 2 + 15) / 16 * 16;
    sv = sk + D * 4;
    pos = sv + D * 4;
    pos_in = WR <= kHdrRingMax;
    bytes = (pos + (pos_in ? WR * 4 : 0) + 127) / 128 * 128;
  }
};

// Query A fragments built from the header copy of q (2-byte elements) and,
// for INT8 blocks, the K scales.  Same layout as make_q_frag.
template <int D>
__device__ __forceinline__ float make_q_frag_s(uint32_t (&aq)[D / 16][4], const unsigned char* qh,
                                               int bf16, const float* ksc, float qs, int G, int g,
                                               int t) {
  float sum = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (g < G) {
      const int c0 = kk * 16 + 2 * t;
      const int cs[4] = {c0, c0 + 1, c0 + 8, c0 + 9};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float sc = ksc ? ksc[cs[e]] : 1.0f;
        const unsigned short raw = reinterpret_cast<const unsigned short*>(qh)[g * D + cs[e]];
        const float qv = bf16 ? __uint_as_float((uint32_t)raw << 16)
                              : __half2float(__ushort_as_half(raw));
        x[e] = qv * sc * qs;
      }
    }
    __half h[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      split_hi_lo(x[e], h[e], lo[e]);
      sum += __half2float(h[e]) + __half2float(lo[e]);
    }
    aq[kk][0] = pack_h2(h[0], h[1]);
    aq[kk][1] = pack_h2(lo[0], lo[1]);
    aq[kk][2] = pack_h2(h[2], h[3]);
    aq[kk][3] = pack_h2(lo[2], lo[3]);
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  return 1152.0f * sum;
}

// Ring of `n` slots with a phase bit that flips on every wrap.
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Unit at position p of prestep's order (the (layer, sequence) groups with
// the most INT8 entries first, the KV heads of a group in turn), or -1 past
// the last unit.
__device__ __forceinline__ int unit_of_rank(const Shape& s, const Dev& d, int units, int p) {
  if (p >= units) return -1;
  return __ldcg(d.order + p / s.Hkv) * s.Hkv + p % s.Hkv;
}

// k-th unit of this CTA, or -1 after its last (called by the producer only;
// it hands each unit index to the other warps through shared memory).
//   kSchedQueue       the next position of prestep's sorted order (longest
//                     units first) from a counter that prestep zeroes every
//                     step.  A CTA takes its next unit when it starts
//                     streaming the current one, so the atomic stays off the
//                     stream, and the CTAs that finish early take the
//                     remaining units: the longest-first queue evens out the
//                     CTAs' end times.
//   kSchedRoundRobin  u = blockIdx.x + k * gridDim.x (groups not sorted).
//   fused step        CTA vocab_ctas + i takes unit i, and only that one.
template <bool kFused>
__device__ __forceinline__ int next_unit(const Shape& s, const Dev& d, int units, int k) {
  if (kFused) {
    const int u = (int)blockIdx.x - s.vocab_ctas;
    return (k == 0 && u >= 0 && u < units) ? u : -1;
  }
  if (d.sched == kSchedQueue) return unit_of_rank(s, d, units, (int)atomicAdd(d.queue, 1u));
  const int u = (int)blockIdx.x + k * (int)gridDim.x;
  return u < units ? u : -1;
}

// Fused step: the stage that the producer issues, and the consumers take,
// i-th.  The INT8 stages come first, then the ring stages with the one that
// holds this step's new token (ring stage jnew) moved last: every other
// stage can be issued before the new token is appended, and only the last
// one has to follow the append.
__device__ __forceinline__ int fused_stage(int i, int n8st, int nst, int jnew) {
  if (i < n8st) return i;
  const int k = i - n8st;
  if (k == nst - 1 - n8st) return n8st + jnew;
  return n8st + (k < jnew ? k : k + 1);
}

// Modes of the persistent kernel.
//   kModeAttention    attention and mass only (prestep and select run as
//                     kernels of their own);
//   kModeFused        the whole decode step in one launch for shapes whose
//                     units fit one CTA per SM: the first vocab_ctas CTAs
//                     (SMs the units leave free) reduce the vocabulary
//                     chunks with all their warps; with no SM to spare, the
//                     epilogue warps of the first B * SV unit CTAs take one
//                     chunk each.  The warp that completes a sequence's
//                     chunks merges its confidence and budgets and flags
//                     them (release).  Each unit CTA appends its new token,
//                     streams its unit and counts one arrival on its (layer,
//                     sequence); the CTA that makes a group's last arrival
//                     runs its selection (select_body.cuh) once its own work
//                     is done, after a bounded wait for the sequence's flag.
//                     The CTAs that reduce the vocabulary come first and wait
//                     on nothing, so that wait always ends.
//   kModeFusedDevStep the same, with the step index read from the device (a
//                     step inside a graph reservation);
//   kModeAttentionShared  kModeAttention for launches with few units per CTA:
//                     the warps of a CTA share out its last unit's mass, which
//                     would otherwise be the epilogue warp's loop alone at
//                     the end of the kernel.
enum : int { kModeAttention = 0, kModeFused = 1, kModeFusedDevStep = 2, kModeAttentionShared = 3 };

// What a fused step needs beyond the attention arguments.
struct FusedArgs {
  long long step;                 // step index (kModeFused)
  const __half* k_new;            // [L][B][Hkv][D]
  const __half* v_new;
  int32_t* evicted;               // [L][B][max_evict]
  int32_t* nevict;                // [L][B]
  SelSmem sm;                     // selection layout, at offset kFusedSelOff of the stage area
};

// Shared memory of a selection inside the fused kernel (after the CTA's own
// work, reusing the stage area): SelShared at 0, the selection's dynamic
// layout from kFusedSelOff.
constexpr int kFusedSelOff = 2048;

// Shared ints before the fused step's selection list (s_misc[kFusedMiscInts]).
constexpr int kFusedMiscInts = 26;
// Bytes of the persistent kernel's shared ints (abort flag, unit indices,
// the fused step's selection list of up to L * B + 2 groups), a multiple of
// 16: a fused step's score slot follows them.
__host__ __device__ inline int misc_bytes(const Shape& s) {
  return ((kFusedMiscInts + s.L * s.B + 2) * 4 + 15) / 16 * 16;
}
static_assert(sizeof(SelShared) <= kFusedSelOff, "SelShared fits below the selection area");

// One quad (4 consecutive slots) of a unit's per-token attention mass:
// mass(slot) = sum over the G query heads of 2^(s_g - M_g) / L_g, from the
// raw-score rows scg[g * S + slot].  kStream: the scores are read once with
// streaming loads (evict-first, coherent), so that they do not displace L1
// lines the consumer warps use (plain cached loads here cost the kernel
// ~8 us per launch on the Qwen-32B shape).
template <bool kStream>
__device__ __forceinline__ void mass_quad(float* mass_u, const float* scg, int S, int G, int slot,
                                          const float (&Mg)[kMaxG], const float (&invL)[kMaxG]) {
  float4 sv[kMaxG];
#pragma unroll
  for (int gg = 0; gg < kMaxG; ++gg) {
    if (gg < G) {
      const float4* src = reinterpret_cast<const float4*>(scg + (size_t)gg * S + slot);
      sv[gg] = kStream ? __ldcs(src) : *src;
    }
  }
  float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int gg = 0; gg < kMaxG; ++gg) {
    if (gg < G) {
      m.x += ex2(sv[gg].x - Mg[gg]) * invL[gg];
      m.y += ex2(sv[gg].y - Mg[gg]) * invL[gg];
      m.z += ex2(sv[gg].z - Mg[gg]) * invL[gg];
      m.w += ex2(sv[gg].w - Mg[gg]) * invL[gg];
    }
  }
  *reinterpret_cast<float4*>(mass_u + slot) = m;
}

// The mass quads of one unit (nb8 INT8 blocks, then the ring) in chunks of
// 32, one quad per lane, taken from the shared counter *chunk until none is
// left: the warps that share a unit this way write distinct quads.  stat
// holds the unit's maxima M_g and 1 / L_g (kMaxG each).  The next chunk is
// taken before the current one is written, so that the counter's round trip
// overlaps the score loads.  Out of line: a CTA runs it once, on its last
// unit, and it stays out of the code of the loops that run every unit.
__device__ __noinline__ void mass_chunks_shared(float* mass_u, const float* scg, int S, int cap, int WR,
                                                int nb8, int G, const float* stat, int* chunk) {
  const int lane = threadIdx.x & 31;
  float Mg[kMaxG], invL[kMaxG];
#pragma unroll
  for (int gg = 0; gg < kMaxG; ++gg) {
    Mg[gg] = stat[gg];
    invL[gg] = stat[kMaxG + gg];
  }
  const int nq = (nb8 * 16 + WR) / 4;
  auto take = [&](void) {
    int c = 0;
    if (lane == 0) c = atomicAdd(chunk, 1);
    return __shfl_sync(0xffffffffu, c, 0);
  };
  for (int c = take(); c * 32 < nq;) {
    const int cn = take();
    const int i = c * 32 + lane;
    if (i < nq) {
      const int v = 4 * i;
      mass_quad<true>(mass_u, scg, S, G, v < nb8 * 16 ? v : cap + (v - nb8 * 16), Mg, invL);
    }
    c = cn;
  }
}

template <int D, bool kFlush, int kMode, int NC>
__global__ void __launch_bounds__((NC + 2) * 32, NC == 4 ? 2 : 1) attention_persistent_kernel(
    Shape s, Dev d, const void* __restrict__ q, float* __restrict__ out,
    int32_t* __restrict__ budget, float* __restrict__ conf_out, const float* __restrict__ logits,
    int stages, FusedArgs fa) {
  static_assert(NC == 4 || NC == 8, "consumer warps");
  constexpr int NTH = (NC + 2) * 32;   // threads: NC consumer warps, the producer, the epilogue warp
  constexpr bool kFused = kMode == kModeFused || kMode == kModeFusedDevStep;
  constexpr bool kDevStep = kMode == kModeFusedDevStep;
  constexpr bool kShareLast = kMode == kModeAttentionShared;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  constexpr int kStageBytes = 128 * D;
  constexpr int kHalf = kStageBytes / 2;
  const int G = s.G;
  const HeaderLayout hl(G, D, s.WR);
  unsigned char* sbuf = smem_raw;                                          // [stages][kStageBytes]
  unsigned char* hbuf = smem_raw + (size_t)stages * kStageBytes;           // [2][hl.bytes]
  float* wpart = reinterpret_cast<float*>(hbuf + 2 * hl.bytes);            // [2][4][G][D + 2]
  const int part_floats = NC * G * (D + 2);
  uint64_t* bars = reinterpret_cast<uint64_t*>(wpart + 2 * part_floats);
  int* s_misc = reinterpret_cast<int*>(bars + kPBars);
  int& s_abort = s_misc[0];
  // unit index of header slot hs (set by the producer before its arrival on
  // hfull) and of partials slot ps (set by consumer warp 0 before its arrival
  // on done); -1 ends the CTA's work
  volatile int* s_unit = s_misc + 1;    // [2]
  volatile int* s_eunit = s_misc + 3;   // [2]
  // fused step: the (layer, sequence) groups whose selection falls to this
  // CTA: s_nsel of them in s_sel (room for L * B + 2; each group has one
  // last arrival, so no CTA lists more than L * B)
  volatile int* s_nsel = s_misc + 5;
  volatile int* s_sel = s_misc + kFusedMiscInts;
  // fused step: the ring stage holding the new token's slot (fused_stage),
  // set by the producer before its arrival on header slot 0
  volatile int* s_jnew = s_misc + 6;
  // fused step: the new token's ring slot (0 <= rs < WR)
  volatile int* s_rsnew = s_misc + 7;
  // fused step: the unit's maxima Mg[kMaxG] and 1 / Lg[kMaxG]; attention
  // only: those of the unit whose mass is being written (s_mpub, below)
  float* s_stat = reinterpret_cast<float*>(s_misc + 8);
  // attention only: the mass of the CTA's last unit (k-th) is shared out in
  // chunks of 32 quads from s_mchunk, once the epilogue warp has put the
  // unit's stats in s_stat and set s_mpub = k; the consumer warps, which
  // have no further unit, take chunks beside it.  s_mpub = -2 - k: the
  // epilogue writes unit k's mass alone (it did not see it was the last).
  volatile int* s_mchunk = s_misc + 24;
  volatile int* s_mpub = s_misc + 25;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(kPMaxStages + i); };
  auto hfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * kPMaxStages + i); };
  auto hempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * kPMaxStages + 2 + i); };
  auto done_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * kPMaxStages + 4 + i); };
  auto efree_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * kPMaxStages + 6 + i); };
  // fused step: the new token appended (by the epilogue warp) and made
  // visible to bulk copies
  const uint32_t app_bar = bar0 + 8u * (uint32_t)(2 * kPMaxStages + 8);
  // this CTA's two score slots: [2][G][S] (token index = slot index in the
  // unit); a fused step keeps its one unit's scores in shared memory, after
  // the shared ints
  float* scg_base = kFused ? reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(s_misc) + misc_bytes(s))
                           : d.scores + (size_t)blockIdx.x * 2 * G * s.S;

  const int units = s.L * s.B * s.Hkv;
  const int nbR = s.WR >> 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  pdl_wait();
  // fused step: the step index of the new token and of the selections
  const long long fstep = kDevStep ? __ldcg(d.step_dev) : fa.step;
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_nsel[0] = 0;
    s_mpub[0] = -1;
    for (int i = 0; i < stages; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), NC);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(hfull_bar(i), 1);
      mbar_init(hempty_bar(i), NC);
      mbar_init(done_bar(i), NC);
      mbar_init(efree_bar(i), 1);
    }
    mbar_init(app_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  auto fail = [&](void) {
    atomicOr(d.status, kStatusTimeout);
    s_abort = 1;
  };
  auto aborted = [&](void) { return *(volatile int*)&s_abort != 0; };

  // One unit's arrival on (layer, sequence) lb; the CTA that makes the last
  // of the Hkv runs the group's selection (finish).
  auto arrive_group = [&](int lb) {
    if (atomicAdd(d.arrive + lb, 1u) == (unsigned)s.Hkv - 1u) {
      __threadfence();   // acquire: the other arrivals' writes are visible to this CTA's selection
      s_sel[atomicAdd((int*)s_nsel, 1)] = lb;
    }
  };

  // End of this CTA's work: in a fused step, every warp meets here once its
  // role is done, and the whole CTA runs the selections that fell to it over
  // the stage area (every bulk copy into it has landed: the producer waited
  // for them).
  auto finish = [&](void) {
    if constexpr (kFused) {
      __syncthreads();
      const int n = s_nsel[0];
      if (n > 0 && threadIdx.x == 0 && !aborted()) {
        // the budgets need c of the group's sequence, which the warp that
        // completed its vocabulary chunks flags (release) once written: in
        // the CTAs dispatched first, which wait on nothing, so this wait
        // ends; it is bounded all the same
        const uint32_t tag = (uint32_t)(fstep + 1);
        bool ok = true;
        for (int i = 0; i < n && ok; ++i) {
          const uint32_t* f = d.conf_ready + s_sel[i] % s.B;
          long long it = 0;
          while (ld_acquire_gpu(f) != tag)
            if (++it > kSpinLimit) { ok = false; break; }
        }
        if (!ok) fail();
      }
      __syncthreads();
      if (n > 0 && !aborted()) {
        __threadfence();
        SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
        for (int i = 0; i < n; ++i) {
          const int lb = s_sel[i];
          if (threadIdx.x == 0) d.arrive[lb] = 0u;   // every arrival of this step is in
          select_group<D, true, kDevStep, false, NTH, false>(s, d, fstep, lb, fa.evicted, fa.nevict, fa.sm,
                                                            smem_raw + kFusedSelOff, sh);
          __syncthreads();
        }
      }
    }
  };

  // Per-token attention mass of unit u from its raw scores in score slot
  // scg, over the quads (4 consecutive slots; slot groups never straddle the
  // INT8 / ring boundary) first, first + stride, ...; empty slots get 0
  // (never read).
  auto mass_quads = [&](int u, int nb8, const float* scg, const float (&Mg)[kMaxG], const float (&invL)[kMaxG],
                        int first, int stride) {
    float* mass_u = d.mass + (size_t)u * s.S;
    const int nq = (nb8 * 16 + s.WR) / 4;
    for (int i = first; i < nq; i += stride) {
      const int v = 4 * i;
      mass_quad<!kFused>(mass_u, scg, s.S, G, v < nb8 * 16 ? v : s.cap + (v - nb8 * 16), Mg, invL);
    }
  };

  // Fused step: vocabulary chunk c (sequence c / SV) by this warp.  The
  // warp that completes a sequence's chunks merges its confidence and
  // budgets and flags them (conf_ready = step + 1) for the selections.
  auto vocab_chunk = [&](int c) {
    const int bc = c / s.SV;
    // one round of loads for the chunk sizes of a fused step (<= 768 logits)
    conf_partial_warp<24>(s, d, logits, bc, c % s.SV);
    unsigned int prev = 0;
    if (lane == 0) {
      __threadfence();
      prev = atomicAdd(d.conf_done + bc, 1u);
    }
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev == (unsigned int)s.SV - 1u) {
      __threadfence();
      conf_merge_warp(s, d, bc, budget, conf_out);
      if (lane == 0) d.conf_done[bc] = 0u;   // zero again for the next launch
      __syncwarp();
      __threadfence();   // every lane's budgets and c are visible before the flag
      if (lane == 0) st_release_gpu(d.conf_ready + bc, (uint32_t)(fstep + 1));
    }
  };

  // The work of this warp's role; every role returns here, so that the end
  // of the CTA's work (finish: a fused step's selections) has one call site
  // and its code one copy, fetched once per step for every warp of the CTA.
  auto role = [&](void) {
  if constexpr (kFused) {
    const bool vocab_cta = (int)blockIdx.x < s.vocab_ctas;
    if (!vocab_cta && warp == NC + 1) {
      // The epilogue warp, idle until the unit is streamed, appends the new
      // token to the unit's ring slot; the proxy fence orders those stores
      // before the bulk copy (async proxy) of the ring stage that reads them
      // back, which the producer issues last, after this arrival.
      const int u = (int)blockIdx.x - s.vocab_ctas;
      const int b = (u / s.Hkv) % s.B;
      append_unit_warp<D>(s, d, u, d.T0[b] + (int)fstep, fa.k_new, fa.v_new);
      asm volatile("fence.proxy.async.global;\n" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(app_bar);
    }
    // Vocabulary chunks.  The CTAs before the units (vocab_ctas of them, on
    // SMs the units leave free, dispatched first) reduce them with all their
    // warps, so the confidence is merged while the units stream and no
    // unit's epilogue warp works on it.  With no such CTA, the epilogue warp
    // of unit CTA c < B * SV reduces chunk c while the consumer warps stream
    // the unit (small chunks: 512 logits).
    if (vocab_cta || (warp == NC + 1 && s.vocab_ctas == 0)) {
      const int nw = NTH / 32;
      const int c0 = vocab_cta ? (int)blockIdx.x * nw + warp : (int)blockIdx.x;
      const int stride = vocab_cta ? s.vocab_ctas * nw : s.B * s.SV;
      for (int c = c0; c < s.B * s.SV; c += stride) vocab_chunk(c);
    }
    if (vocab_cta) {
      return;
    }
  }

  if (warp == NC) {
    // ------------------------------------------------ producer warp
    if constexpr (kFused) {
      // Fused step: this CTA's one unit, u = blockIdx.x - vocab_ctas.  The header (q and
      // the scales) and every stage but the ring stage holding the new
      // token's slot do not depend on this step's new token; that stage
      // comes last (fused_stage), once the epilogue warp has appended the
      // token (app_bar).  The header's copy of the ring positions may hold
      // the new token's slot before or after the append (before it, the slot
      // is free: -1); the consumers count that slot as valid either way.
      const uint64_t pol = policy_evict_first();
      const int u = (int)blockIdx.x - s.vocab_ctas;
      const int h = u % s.Hkv, b = (u / s.Hkv) % s.B, l = u / (s.Hkv * s.B);
      const size_t lb = lb_index(s, l, b);
      const int nb8 = (d.n8[lb] + 15) >> 4;
      const int t_new = d.T0[b] + (int)fstep;
      const int jnew = ((t_new % s.WR) >> 4) >> 1;
      Sched sch;
      sch.init(0, nb8 + nbR, nb8);
      const char* k8u = reinterpret_cast<const char*>(d.k8) + (size_t)u * s.cstride * D;
      const char* v8u = reinterpret_cast<const char*>(d.v8) + (size_t)u * s.cstride * D;
      const char* k16u = reinterpret_cast<const char*>(d.k16) + (size_t)u * s.WR * D * 2;
      const char* v16u = reinterpret_cast<const char*>(d.v16) + (size_t)u * s.WR * D * 2;
      RingPos st;
      int issued = 0;
      bool ok = true;
      auto issue = [&](int i) {
        if (issued >= stages && !mbar_wait(empty_bar(st.slot), st.phase ^ 1u)) return false;
        bool ring;
        int first, nb;
        sch.first_last(fused_stage(i, sch.n8st, sch.nst, jnew), ring, first, nb);
        const uint32_t span = (uint32_t)(nb * 16 * D * (ring ? 2 : 1));
        const char* ksrc = ring ? k16u + (size_t)first * 32 * D : k8u + (size_t)first * 16 * D;
        const char* vsrc = ring ? v16u + (size_t)first * 32 * D : v8u + (size_t)first * 16 * D;
        const uint32_t dst = smem_u32(sbuf + (size_t)st.slot * kStageBytes);
        mbar_arrive_tx(full_bar(st.slot), 2 * span);
        bulk_g2s_hint(dst, ksrc, span, full_bar(st.slot), pol);
        bulk_g2s_hint(dst + kHalf, vsrc, span, full_bar(st.slot), pol);
        st.next(stages);
        ++issued;
        return true;
      };
      if (lane == 0) {
        s_unit[0] = u;
        s_jnew[0] = jnew;
        s_rsnew[0] = t_new % s.WR;
        const uint32_t hdst = smem_u32(hbuf);
        const uint32_t qbytes = (uint32_t)(G * D * 2);
        mbar_arrive_tx(hfull_bar(0), qbytes + 2u * D * 4 + (hl.pos_in ? (uint32_t)s.WR * 4 : 0u));
        bulk_g2s(hdst + hl.q, reinterpret_cast<const char*>(q) + (lb * s.Hq + (size_t)h * G) * D * 2, qbytes,
                 hfull_bar(0));
        bulk_g2s(hdst + hl.sk, d.sK + (size_t)u * D, D * 4, hfull_bar(0));
        bulk_g2s(hdst + hl.sv, d.sV + (size_t)u * D, D * 4, hfull_bar(0));
        if (hl.pos_in)
          bulk_g2s(hdst + hl.pos, d.pos + lb * s.S + s.cap, (uint32_t)s.WR * 4, hfull_bar(0));
        for (int i = 0; i < sch.nst && ok; ++i) {
          if (i == sch.nst - 1 && !mbar_wait(app_bar, 0)) ok = false;
          if (ok) ok = issue(i);
        }
        if (!ok) fail();
      }
      if (lane == 0) {
        // wait (bounded) for the last copy of every stage slot
        RingPos dr = st;
        for (int i = 0; i < stages && i < issued; ++i) {
          dr.slot = dr.slot == 0 ? stages - 1 : dr.slot - 1;
          if (dr.slot == stages - 1) dr.phase ^= 1u;
          if (!mbar_wait(full_bar(dr.slot), dr.phase)) atomicOr(d.status, kStatusTimeout);
        }
      }
      return;
    }
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      RingPos st;
      long long issued = 0;
      int u = next_unit<kFused>(s, d, units, 0);
      for (int k = 0; !aborted(); ++k) {
        const int hs = k & 1;
        if (k >= 2 && !mbar_wait(hempty_bar(hs), (uint32_t)(((k >> 1) - 1) & 1))) { fail(); break; }
        if (u < 0) {
          // no more units: the other warps see -1 in this header slot
          s_unit[hs] = -1;
          mbar_arrive(hfull_bar(hs));
          break;
        }
        s_unit[hs] = u;
        const int h = u % s.Hkv, b = (u / s.Hkv) % s.B, l = u / (s.Hkv * s.B);
        const size_t lb = lb_index(s, l, b);
        const int nb8 = (d.n8[lb] + 15) >> 4;
        // unit header
        const uint32_t hdst = smem_u32(hbuf + (size_t)hs * hl.bytes);
        const uint32_t qbytes = (uint32_t)(G * D * 2);
        mbar_arrive_tx(hfull_bar(hs), qbytes + 2u * D * 4 + (hl.pos_in ? (uint32_t)s.WR * 4 : 0u));
        bulk_g2s(hdst + hl.q, reinterpret_cast<const char*>(q) + (lb * s.Hq + (size_t)h * G) * D * 2,
                 qbytes, hfull_bar(hs));
        bulk_g2s(hdst + hl.sk, d.sK + (size_t)u * D, D * 4, hfull_bar(hs));
        bulk_g2s(hdst + hl.sv, d.sV + (size_t)u * D, D * 4, hfull_bar(hs));
        if (hl.pos_in)
          bulk_g2s(hdst + hl.pos, d.pos + lb * s.S + s.cap, (uint32_t)s.WR * 4, hfull_bar(hs));
        // K/V stages
        Sched sch;
        sch.init(0, nb8 + nbR, nb8);
        const char* k8u = reinterpret_cast<const char*>(d.k8) + (size_t)u * s.cstride * D;
        const char* v8u = reinterpret_cast<const char*>(d.v8) + (size_t)u * s.cstride * D;
        const char* k16u = reinterpret_cast<const char*>(d.k16) + (size_t)u * s.WR * D * 2;
        const char* v16u = reinterpret_cast<const char*>(d.v16) + (size_t)u * s.WR * D * 2;
        bool ok = true;
        int u_next = -1;
        for (int i = 0; i < sch.nst; ++i) {
          if (issued >= stages && !mbar_wait(empty_bar(st.slot), st.phase ^ 1u)) { ok = false; break; }
          bool ring;
          int first, nb;
          sch.first_last(i, ring, first, nb);
          const uint32_t span = (uint32_t)(nb * 16 * D * (ring ? 2 : 1));
          const char* ksrc = ring ? k16u + (size_t)first * 32 * D : k8u + (size_t)first * 16 * D;
          const char* vsrc = ring ? v16u + (size_t)first * 32 * D : v8u + (size_t)first * 16 * D;
          const uint32_t dst = smem_u32(sbuf + (size_t)st.slot * kStageBytes);
          mbar_arrive_tx(full_bar(st.slot), 2 * span);
          bulk_g2s_hint(dst, ksrc, span, full_bar(st.slot), pol);
          bulk_g2s_hint(dst + kHalf, vsrc, span, full_bar(st.slot), pol);
          st.next(stages);
          ++issued;
          // the next unit is known early, so a queue's atomic stays off the stream
          if (i == 0) u_next = next_unit<kFused>(s, d, units, k + 1);
        }
        if (!ok) { fail(); break; }
        u = sch.nst > 0 ? u_next : next_unit<kFused>(s, d, units, k + 1);
      }
      // wait (bounded) for the last copy of every stage slot: nothing may be
      // in flight into shared memory when the CTA's threads have all exited
      RingPos dr = st;
      for (int i = 0; i < stages && i < issued; ++i) {
        dr.slot = dr.slot == 0 ? stages - 1 : dr.slot - 1;
        if (dr.slot == stages - 1) dr.phase ^= 1u;
        if (!mbar_wait(full_bar(dr.slot), dr.phase)) atomicOr(d.status, kStatusTimeout);
      }
    }
    return;
  }

  if (warp == NC + 1) {
    // ------------------------------------------------ epilogue warp
    if constexpr (kFused) {
      // fused step: the append and the vocabulary chunk, if any, are done
      // (above); the consumer warps finish the unit themselves
      return;
    }
    // Idle until the first unit is done: the confidence of the step.
    if (logits) {
      // Logits in host memory: this CTA reduces its vocabulary chunks to
      // partials here, so that their transfer overlaps the attention; the
      // CTA that finishes the last chunk of a sequence merges that sequence.
      for (int c = blockIdx.x; c < s.B * s.SV; c += gridDim.x) {
        const int b = c / s.SV;
        conf_partial_warp(s, d, logits, b, c % s.SV);
        unsigned int prev = 0;
        if (lane == 0) {
          __threadfence();
          prev = atomicAdd(d.conf_done + b, 1u);
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == (unsigned int)s.SV - 1u) {
          __threadfence();
          conf_merge_warp(s, d, b, budget, conf_out);
          if (lane == 0) d.conf_done[b] = 0u;   // zero again for the next launch
        }
      }
    } else if (!kFused) {
      // the prestep kernel wrote the partials: merge the sequences this CTA owns
      for (int b = blockIdx.x; b < s.B; b += gridDim.x) conf_merge_warp(s, d, b, budget, conf_out);
    }
    for (int k = 0;; ++k) {
      const int ps = k & 1;
      if (aborted() || !mbar_wait(done_bar(ps), (uint32_t)((k >> 1) & 1))) {
        if (!aborted()) fail();
        break;
      }
      const int u = s_eunit[ps];
      if (u < 0) break;
      const int h = u % s.Hkv, b = (u / s.Hkv) % s.B, l = u / (s.Hkv * s.B);
      const size_t lb = lb_index(s, l, b);
      const int nb8 = (d.n8[lb] + 15) >> 4;
      const float* part = wpart + (size_t)ps * part_floats;   // [4][G][D + 2]: o..., m, l
      float Mg[kMaxG], Lg[kMaxG], fw[NC][kMaxG];
#pragma unroll
      for (int gg = 0; gg < kMaxG; ++gg) {
        Mg[gg] = -INFINITY;
        Lg[gg] = 0.f;
        if (gg < G) {
#pragma unroll
          for (int w = 0; w < NC; ++w) Mg[gg] = fmaxf(Mg[gg], part[(w * G + gg) * (D + 2) + D]);
#pragma unroll
          for (int w = 0; w < NC; ++w) {
            const float mw = part[(w * G + gg) * (D + 2) + D];
            fw[w][gg] = (mw == -INFINITY) ? 0.f : ex2(mw - Mg[gg]);
            Lg[gg] += part[(w * G + gg) * (D + 2) + D + 1] * fw[w][gg];
          }
        }
      }
      // output
      float* o = out + (lb * s.Hq + (size_t)h * G) * D;
#pragma unroll
      for (int gg = 0; gg < kMaxG; ++gg) {
        if (gg < G) {
          const float inv = 1.0f / Lg[gg];
          for (int c = lane; c < D; c += 32) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < NC; ++w) acc += part[(w * G + gg) * (D + 2) + c] * fw[w][gg];
            o[gg * D + c] = acc * inv;
          }
        }
      }
      // attention mass of the unit's tokens.  With kShareLast, the CTA's
      // last unit is the one whose next header the consumer warps have
      // taken (no unit) and arrived on its done barrier (that phase cannot
      // move on before this warp frees the slot): they share its mass.
      const float* scg = scg_base + (size_t)ps * G * s.S;
      float invL[kMaxG];
#pragma unroll
      for (int gg = 0; gg < kMaxG; ++gg) invL[gg] = gg < G ? 1.0f / Lg[gg] : 0.f;
      int last = 0;
      if constexpr (kShareLast) {
        const int kn = k + 1;
        if (lane == 0) last = mbar_test(done_bar(kn & 1), (uint32_t)((kn >> 1) & 1)) && s_eunit[kn & 1] < 0;
        last = __shfl_sync(0xffffffffu, last, 0);
      }
      if (kShareLast && last) {
        if (lane == 0) {
          s_mchunk[0] = 0;
#pragma unroll
          for (int gg = 0; gg < kMaxG; ++gg) {
            s_stat[gg] = Mg[gg];
            s_stat[kMaxG + gg] = invL[gg];
          }
          __threadfence_block();
          s_mpub[0] = k;
        }
        __syncwarp();
        mass_chunks_shared(d.mass + (size_t)u * s.S, scg, s.S, s.cap, s.WR, nb8, G, s_stat, (int*)s_mchunk);
      } else {
        if (kShareLast && lane == 0) s_mpub[0] = -2 - k;
        mass_quads(u, nb8, scg, Mg, invL, lane, 32);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(efree_bar(ps));
    }
    return;
  }

  // -------------------------------------------------- consumer warps
  const float qs = kQPre * 1.4426950408889634f * rsqrtf((float)D);
  const uint64_t keep = policy_evict_last();
  RingPos st;
  int fused_nb8 = 0;   // fused step: INT8 blocks of the CTA's unit
  // k: the CTA's units so far; the loop ends on the header without a unit
  // (every other exit aborts the CTA)
  int k = 0;
  for (;; ++k) {
    const int hs = k & 1;
    if (aborted() || !mbar_wait(hfull_bar(hs), (uint32_t)((k >> 1) & 1))) {
      if (!aborted()) fail();
      break;
    }
    const int u = s_unit[hs];
    if (k >= 2 && !mbar_wait(efree_bar(hs), (uint32_t)(((k >> 1) - 1) & 1))) {
      fail();
      break;
    }
    // the epilogue takes the unit index with this unit's partials
    if (warp == 0 && lane == 0) s_eunit[hs] = u;
    if (u < 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(done_bar(hs));
      break;
    }
    const int b = (u / s.Hkv) % s.B, l = u / (s.Hkv * s.B);
    const size_t lb = lb_index(s, l, b);
    const int n8 = d.n8[lb];
    const int nb8 = (n8 + 15) >> 4;
    fused_nb8 = nb8;
    const unsigned char* hdr = hbuf + (size_t)hs * hl.bytes;
    const float* sKh = reinterpret_cast<const float*>(hdr + hl.sk);
    const float* sVh = reinterpret_cast<const float*>(hdr + hl.sv);
    const int32_t* posh = hl.pos_in ? reinterpret_cast<const int32_t*>(hdr + hl.pos) : d.pos + lb * s.S + s.cap;
    float* scg = scg_base + (size_t)hs * G * s.S;
    Sched sch;
    sch.init(0, nb8 + nbR, nb8);
    WarpState<D> ws;
    ws.qoffset = -kQPreInv * make_q_frag_s<D>(ws.aq, hdr + hl.q, s.qbf16, sKh, qs, G, g, t);
#pragma unroll
    for (int j = 0; j < D / 8; ++j) ws.acc[j][0] = ws.acc[j][1] = ws.acc[j][2] = ws.acc[j][3] = 0.f;
    ws.m_run = -INFINITY;
    ws.l_run = 0.f;
    ws.l_flushed = 0.f;
    ws.n8blk = 0;
    ws.in_ring = false;
    float sc4buf[4];
    bool ok = true;
    // raw scores of tokens tok0 + {2t, 2t+1, 8+2t, 9+2t} of head g (the
    // lane's four, in sc4buf) to the unit's score slot
    auto store_scores = [&](int tok0) {
      float* dst = scg + (size_t)g * s.S + tok0 + 2 * t;
      if constexpr (kFused) {
        // the unit's score slot in shared memory
        *reinterpret_cast<float2*>(dst) = make_float2(sc4buf[0], sc4buf[1]);
        *reinterpret_cast<float2*>(dst + 8) = make_float2(sc4buf[2], sc4buf[3]);
      } else {
        asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;\n" ::"l"(dst),
                     "f"(sc4buf[0]), "f"(sc4buf[1]), "l"(keep) : "memory");
        asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;\n" ::"l"(dst + 8),
                     "f"(sc4buf[2]), "f"(sc4buf[3]), "l"(keep) : "memory");
      }
    };
    // INT8 stages: stage i holds blocks 4i .. 4i + 3; with 8 consumer warps,
    // warps 0-3 take the even INT8 stages and warps 4-7 the odd ones
    for (int i = 0; i < sch.n8st; ++i) {
      if (!mbar_wait(full_bar(st.slot), st.phase)) { ok = false; break; }
      const uint32_t stage = smem_u32(sbuf + (size_t)st.slot * kStageBytes);
      const int wi = warp & 3;
      const int blk = 4 * i + wi;
      const bool mine = (warp >> 2) == i % (NC / 4) && blk < nb8;
      if (mine)
        int8_block<D, kFlush>(ws, stage + wi * 16 * D, stage + kHalf + wi * 16 * D, blk, n8, G, g, t, lane,
                              nullptr, sc4buf);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st.slot));
      st.next(stages);
      if (mine && g < G) store_scores(blk * 16);
    }
    // ring stages: ring stage r holds ring blocks 2r, 2r + 1; the warp
    // pairs (0-1, 2-3, ...) take the ring stages in turn, so every pair
    // works at once (a fused step streams the new token's stage last)
    for (int i = sch.n8st; ok && i < sch.nst; ++i) {
      if (!mbar_wait(full_bar(st.slot), st.phase)) { ok = false; break; }
      const int r = (kFused ? fused_stage(i, sch.n8st, sch.nst, s_jnew[0]) : i) - sch.n8st;
      const uint32_t stage = smem_u32(sbuf + (size_t)st.slot * kStageBytes);
      const int jb = warp - 2 * ((i - sch.n8st) % (NC / 2));
      const int rb = 2 * r + jb;
      const bool mine = jb >= 0 && jb < 2 && rb < nbR;
      if (mine) {
        if (!ws.in_ring) {
          make_q_frag_s<D>(ws.aq, hdr + hl.q, s.qbf16, nullptr, qs, G, g, t);
          ws.qoffset = 0.f;
          ws_scale_v<D>(ws, sVh, t);
          ws.in_ring = true;
        }
        const int live = (kFused && rb == (s_rsnew[0] >> 4)) ? (s_rsnew[0] & 15) : -1;
        ring_block<D>(ws, stage + jb * 32 * D, stage + kHalf + jb * 32 * D, posh + rb * 16, G, g, t, lane,
                      nullptr, sc4buf, live);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st.slot));
      st.next(stages);
      if (mine && g < G) store_scores(s.cap + rb * 16);
    }
    if (!ok) {
      fail();
      break;
    }
    // partials of this warp -> the epilogue warp: [4][G][D + 2] = o..., m, l
    if (!ws.in_ring) ws_scale_v<D>(ws, sVh, t);
    float lsum = ws.l_run;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    if (g < G) {
      float* pw = wpart + (size_t)hs * part_floats + (size_t)(warp * G + g) * (D + 2);
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        pw[j * 8 + 2 * t] = ws.acc[j][0] + ws.acc[j][2];
        pw[j * 8 + 2 * t + 1] = ws.acc[j][1] + ws.acc[j][3];
      }
      if (t == 0) {
        pw[D] = ws.m_run;
        pw[D + 1] = lsum;
      }
    }
    // fused step: one unit only; the consumer warps finish it below
    if constexpr (kFused) break;
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(done_bar(hs));
      mbar_arrive(hempty_bar(hs));
    }
  }
  if constexpr (kShareLast) {
    // No further unit: take chunks of the last unit's mass beside the
    // epilogue warp, so that the CTA's tail is not one warp's loop.  The
    // epilogue publishes the unit's stats once the unit is done, or that it
    // writes the mass alone (bounded wait; an aborted CTA skips this).
    const int k_last = k - 1;
    if (k_last >= 0 && !aborted()) {
      int pub = 0;   // 1: help, -1: the epilogue has it
      for (long long it = 0; it < kSpinLimit && !aborted(); ++it) {
        const int m = s_mpub[0];
        if (m == k_last) { pub = 1; break; }
        if (m == -2 - k_last) { pub = -1; break; }
        __nanosleep(64);
      }
      if (pub > 0) {
        __threadfence_block();
        // the unit and its INT8 length, as the epilogue has them
        const int ul = s_eunit[k_last & 1];
        const int bl = (ul / s.Hkv) % s.B, ll = ul / (s.Hkv * s.B);
        const int nb8l = (d.n8[lb_index(s, ll, bl)] + 15) >> 4;
        mass_chunks_shared(d.mass + (size_t)ul * s.S, scg_base + (size_t)(k_last & 1) * G * s.S, s.S, s.cap,
                           s.WR, nb8l, G, s_stat, (int*)s_mchunk);
      } else if (pub == 0 && !aborted()) {
        fail();
      }
    }
  }
  if constexpr (kFused) {
    // Fused step: the consumer warps finish this CTA's only unit, u =
    // blockIdx.x - vocab_ctas: merge their partials, write the output and the tokens'
    // attention mass (scores in shared memory), and count the unit's arrival
    // on its (layer, sequence).  Every consumer warp reaches both named
    // barriers, whether or not a bounded wait above gave up.
    // The code here runs once per launch, so it is kept short (loops, not
    // unrolled copies): its instructions are fetched cold every step.
    named_sync(1, NC * 32);
    const int u = (int)blockIdx.x - s.vocab_ctas;
    const int h = u % s.Hkv, b = (u / s.Hkv) % s.B, l = u / (s.Hkv * s.B);
    const size_t lb = lb_index(s, l, b);
    const int tid = threadIdx.x;
    const float* part = wpart;   // slot 0: [NC][G][D + 2] = o..., m, l
    if (!aborted() && warp < G) {
      // head warp: the maximum and normaliser over the NC partials
      const float mw = lane < NC ? part[(lane * G + warp) * (D + 2) + D] : -INFINITY;
      const float lw = lane < NC ? part[(lane * G + warp) * (D + 2) + D + 1] : 0.f;
      float m = mw;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float lsum = mw == -INFINITY ? 0.f : lw * ex2(mw - m);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
      if (lane == 0) {
        s_stat[warp] = m;
        s_stat[kMaxG + warp] = 1.0f / lsum;
      }
    }
    named_sync(1, NC * 32);
    if (!aborted()) {
      float* o = out + (lb * s.Hq + (size_t)h * G) * D;
#pragma unroll 1
      for (int idx = tid; idx < G * D; idx += NC * 32) {
        const int gg = idx / D, c = idx - gg * D;
        const float M = s_stat[gg];
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < NC; ++w) {
          const float mw = part[(w * G + gg) * (D + 2) + D];
          if (mw != -INFINITY) acc += part[(w * G + gg) * (D + 2) + c] * ex2(mw - M);
        }
        o[idx] = acc * s_stat[kMaxG + gg];
      }
      // attention mass of the unit's tokens from the scores in shared memory
      float* mass_u = d.mass + (size_t)u * s.S;
      const int nq = (fused_nb8 * 16 + s.WR) / 4;
#pragma unroll 1
      for (int i = tid; i < nq; i += NC * 32) {
        const int v = 4 * i;
        const int slot = v < fused_nb8 * 16 ? v : s.cap + (v - fused_nb8 * 16);
        float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int gg = 0; gg < G; ++gg) {
          const float4 sv = *reinterpret_cast<const float4*>(scg_base + (size_t)gg * s.S + slot);
          const float M = s_stat[gg], iL = s_stat[kMaxG + gg];
          m.x += ex2(sv.x - M) * iL;
          m.y += ex2(sv.y - M) * iL;
          m.z += ex2(sv.z - M) * iL;
          m.w += ex2(sv.w - M) * iL;
        }
        *reinterpret_cast<float4*>(mass_u + slot) = m;
      }
    }
    named_sync(1, NC * 32);
    // every consumer thread's mass stores come before the barrier; this
    // fence (cumulative) makes them visible at GPU scope before the group
    // arrival that may start the group's selection in another CTA
    if (threadIdx.x == 0 && !aborted()) {
      __threadfence();
      arrive_group((int)lb);
    }
  }
  };
  role();
  finish();
}

// ---------------------------------------------------------------------------
// Launch shapes
// ---------------------------------------------------------------------------
static int stage_bytes(int D) { return 128 * D; }

static int chunk_of(int splits, int max_tokens) {
  const int nbT = (max_tokens + 15) / 16;
  return (nbT + splits - 1) / splits;
}

static int fixed_bytes_split(const Shape& s, int splits, int max_tokens) {
  const int chunk = chunk_of(splits, max_tokens);
  const int G = s.G, D = s.D;
  size_t f = (size_t)G * chunk * 16 + 2 * kConsumerWarps * G + (size_t)kConsumerWarps * G * D +
             2 * kMaxG + (size_t)G * D + 2 * kMaxG + 4;
  return (int)(f * sizeof(float)) + 2 * kMaxStages * 8;
}

// Fused steps run the persistent kernel with kFusedConsumers (8) consumer
// warps, one CTA per SM (every unit on an SM of its own); the
// attention-only launch with 4, two CTAs per SM.

// Shared memory besides the stages: two headers, two partials slots, the
// mbarriers, the shared ints and, in a fused step (nc = kFusedConsumers),
// the unit's score slot G x S.
static int fixed_bytes_persistent(const Shape& s, int nc = kPConsumers) {
  const HeaderLayout hl(s.G, s.D, s.WR);
  const int part = nc * s.G * (s.D + 2) * 4;
  const int scores = nc == kFusedConsumers ? (s.G * s.S * 4 + 15) / 16 * 16 : 0;
  return 2 * hl.bytes + 2 * part + kPBars * 8 + misc_bytes(s) + scores;
}

int attention_max_smem() { return 225 * 1024; }

// Split kernel: as many stages as fit while two CTAs share an SM.
static int stages_split(const Shape& s, int splits, int max_tokens) {
  int st = (113 * 1024 - fixed_bytes_split(s, splits, max_tokens)) / stage_bytes(s.D);
  return st > kMaxStages ? kMaxStages : (st < 2 ? 2 : st);
}

// Persistent kernel: as many stages as fit while two CTAs share an SM (4
// consumer warps), or in the whole SM (8).
static int stages_persistent(const Shape& s, int nc = kPConsumers) {
  const int budget = nc == kPConsumers ? 113 * 1024 : 225 * 1024;
  int st = (budget - fixed_bytes_persistent(s, nc)) / stage_bytes(s.D);
  return st > kPMaxStages ? kPMaxStages : (st < 2 ? 2 : st);
}

int attention_smem_bytes(const Shape& s, int splits, int max_tokens) {
  if (splits == 1) return stages_persistent(s) * stage_bytes(s.D) + fixed_bytes_persistent(s);
  return stages_split(s, splits, max_tokens) * stage_bytes(s.D) +
         fixed_bytes_split(s, splits, max_tokens);
}

int attention_persistent_ctas();

// SMs of the current device (152 on GB300), recorded per device
static int num_sms() {
  static int sms[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool known = dev >= 0 && dev < kMaxDevices;
  if (known && sms[dev] > 0) return sms[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  if (known) sms[dev] = n;
  return n;
}

int attention_persistent_ctas() { return 2 * num_sms(); }

void attention_grid(const Shape& s, const Dev& d, int splits, int* grid_out, int* cluster_out) {
  const int units = s.L * s.B * s.Hkv;
  if (splits > 1) {
    *grid_out = units * splits;
    *cluster_out = splits;
    return;
  }
  // one unit per CTA, or two CTAs per SM; when the units fill between one
  // and two such rounds, half of them per round (both rounds full: the
  // 512 units of 4K tokens took 0.118 ms on 256 CTAs, 0.123 ms on 304)
  const int full = 2 * num_sms();
  int grid = units <= full ? units : units < 2 * full ? (units + 1) / 2 : full;
  if (grid > d.score_ctas) grid = d.score_ctas;
  if (d.attn_ctas > 0 && grid > d.attn_ctas) grid = d.attn_ctas;
  *grid_out = grid;
  *cluster_out = 1;
}

// Self-test of the bounded-wait path: one CTA waits on an mbarrier that no
// thread ever arrives on, with a short poll limit, then reports the time-out
// through the device status word exactly as the decode kernels do.  Nothing
// faults and the context stays usable.
__global__ void selftest_wait_kernel(Dev d, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool done = false;
    for (long long i = 0; i < limit && !done; ++i) done = mbar_try_wait(b, 0);
    if (!done) atomicOr(d.status, kStatusTimeout);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(b) : "memory");
  }
}

int launch_selftest_timeout(const Dev& d, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(d, 4096);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// INT8 tokens per unit above which the persistent kernel flushes the INT8 V
// bias as it goes (see launch_d)
constexpr int kFlushTokens = 8192;
// Units per CTA below which the attention-only launch shares out each CTA's
// last unit's mass (see launch_d)
constexpr int kShareUnits = 8;

template <int D>
static int launch_d(const Shape& s, const Dev& d, const void* q, float* out, int32_t* budget,
                    float* conf_out, const float* logits, int splits, int max_tokens,
                    cudaStream_t stream) {
  const int chunk = chunk_of(splits, max_tokens);
  const int smem = attention_smem_bytes(s, splits, max_tokens);
  if (smem > attention_max_smem()) return -1;
  const int units = s.L * s.B * s.Hkv;
  if (splits == 1) {
    // Units whose INT8 region can exceed 8192 tokens take the instance that
    // removes the INT8 V bias every 16 blocks of a warp.  The error that
    // this avoids grows with a warp's INT8 blocks: 2.7e-3 max-abs at ~500
    // blocks per warp (32K-token units), below 7e-4 up to 128.  Shorter
    // units keep the other instance: the flush state costs 2 % of a kernel
    // at its register limit (0.292 against 0.285 ms on the Qwen-32B shape).
    // With fewer than kShareUnits units per CTA, the instance whose warps
    // share out a CTA's last unit's mass: there the epilogue warp's loop
    // over that unit is a large part of the kernel's end (4K-token units, 2
    // per CTA: 0.1118 against 0.1178 ms per launch).  With more units per
    // CTA the last ones are the queue's shortest and the sharing code cost
    // the kernel 1.6 % (Qwen-32B shape, 13.5 units per CTA).
    static int configured[3][kMaxDevices] = {};
    int grid = 0, cluster = 0;
    attention_grid(s, d, 1, &grid, &cluster);
    const bool flush = max_tokens - s.WR > kFlushTokens;
    const bool share = !flush && units < kShareUnits * grid;
    auto kern = flush   ? attention_persistent_kernel<D, true, kModeAttention, kPConsumers>
                : share ? attention_persistent_kernel<D, false, kModeAttentionShared, kPConsumers>
                        : attention_persistent_kernel<D, false, kModeAttention, kPConsumers>;
    if (ensure_smem(kern, attention_max_smem(), configured[flush ? 1 : share ? 2 : 0]) != cudaSuccess) return -1;
    return launch_pdl(kern, dim3(grid), dim3(kPThreads), (size_t)smem, stream, s, d, q, out, budget,
                      conf_out, logits, stages_persistent(s), FusedArgs{}) == cudaSuccess
               ? 0
               : -1;
  }
  static int configured_split[kMaxDevices] = {};
  if (ensure_smem(attention_kernel<D>, attention_max_smem(), configured_split) != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)units * splits);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attention_kernel<D>, s, d, q, out, budget, conf_out,
                                     splits, chunk, stages_split(s, splits, max_tokens));
  return e == cudaSuccess ? 0 : -1;
}

// A fused step: every unit on a CTA of its own and one CTA per SM (8
// consumer warps), at most one vocabulary chunk per CTA; units short enough
// for the instance without the INT8 V bias flush; tail-fill compaction; and
// the selection's keys and bitmaps inside the stage area.
bool fused_step_fits(const Shape& s, const Dev& d, int splits, int max_tokens) {
  const long long units = (long long)s.L * s.B * s.Hkv;
  if (splits != 1 || s.compaction != 0) return false;
  if (units + s.vocab_ctas > attention_persistent_ctas() / 2) return false;
  // without vocabulary CTAs each unit CTA's epilogue warp reduces at most
  // one vocabulary chunk
  if (s.vocab_ctas == 0 && (long long)s.B * s.SV > units) return false;
  if (d.attn_ctas > 0 && units > d.attn_ctas) return false;
  if (units > d.score_ctas) return false;
  if (max_tokens - s.WR > kFlushTokens) return false;
  // two stages at least beside the unit's score slot and the rest
  if (fixed_bytes_persistent(s, kFusedConsumers) + 2 * stage_bytes(s.D) > attention_max_smem()) return false;
  const SelSmem sm = plan_select(s);
  if (sm.off_key < 0) return false;
  const long long need = kFusedSelOff + ((sm.bytes + 127) & ~127);
  return need <= (long long)stages_persistent(s, kFusedConsumers) * stage_bytes(s.D);
}

template <int D>
static int launch_fused_d(const Shape& s, const Dev& d, long long step, const void* q, const void* k_new,
                          const void* v_new, const float* logits, float* out, int32_t* budget, float* conf_out,
                          int32_t* evicted_pos, int32_t* n_evicted, cudaStream_t stream) {
  static int configured[2][kMaxDevices] = {};
  const bool dev = step < 0;
  auto kern = dev ? attention_persistent_kernel<D, false, kModeFusedDevStep, kFusedConsumers>
                  : attention_persistent_kernel<D, false, kModeFused, kFusedConsumers>;
  if (ensure_smem(kern, attention_max_smem(), configured[dev]) != cudaSuccess) return -1;
  const int stages = stages_persistent(s, kFusedConsumers);
  const int smem = stages * stage_bytes(D) + fixed_bytes_persistent(s, kFusedConsumers);
  const int grid = s.L * s.B * s.Hkv + s.vocab_ctas;
  FusedArgs fa{};
  fa.step = step;
  fa.k_new = static_cast<const __half*>(k_new);
  fa.v_new = static_cast<const __half*>(v_new);
  fa.evicted = evicted_pos;
  fa.nevict = n_evicted;
  fa.sm = plan_select(s);
  return launch_pdl(kern, dim3(grid), dim3((kFusedConsumers + 2) * 32), (size_t)smem, stream, s, d, q, out,
                    budget, conf_out, logits, stages, fa) == cudaSuccess
             ? 0
             : -1;
}

int launch_fused_step(const Shape& s, const Dev& d, long long step, const void* q, const void* k_new,
                      const void* v_new, const float* logits, float* out, int32_t* budget, float* conf_out,
                      int32_t* evicted_pos, int32_t* n_evicted, int max_tokens, cudaStream_t stream) {
  if (!fused_step_fits(s, d, 1, max_tokens)) return -1;
  if (s.D == 128)
    return launch_fused_d<128>(s, d, step, q, k_new, v_new, logits, out, budget, conf_out, evicted_pos,
                               n_evicted, stream);
  if (s.D == 64)
    return launch_fused_d<64>(s, d, step, q, k_new, v_new, logits, out, budget, conf_out, evicted_pos,
                              n_evicted, stream);
  return -1;
}

int launch_attention(const Shape& s, const Dev& d, const void* q, float* out, int32_t* budget,
                     float* conf_out, const float* logits, int splits, int max_tokens,
                     cudaStream_t stream) {
  if (splits > 1 && logits) return -1;   // the split-K kernel merges partials of the prestep kernel
  if (s.D == 128) return launch_d<128>(s, d, q, out, budget, conf_out, logits, splits, max_tokens, stream);
  if (s.D == 64) return launch_d<64>(s, d, q, out, budget, conf_out, logits, splits, max_tokens, stream);
  return -1;
}

}  // namespace confkv
