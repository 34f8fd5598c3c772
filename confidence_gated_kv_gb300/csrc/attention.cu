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
// query heads share the unit's K/V.  A unit's token blocks (INT8 blocks first,
// then the FP16 ring) are split over `splits` CTAs that form one thread-block
// cluster; inside a CTA each warp takes every NW-th block.
//
// Per 16-token block a warp issues two tensor-core products with
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
#include "confkv_internal.cuh"

namespace cg = cooperative_groups;

namespace confkv {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr float kQPre = 256.0f;         // q pre-scale before the hi/lo split
constexpr float kQPreInv = 1.0f / 256.0f;

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four signed int8 (bytes 0..3 of w) -> two half2 {byte0, byte1}, {byte2,
// byte3}, exactly: byte ^ 0x80 = code + 128 = u; the fp16 with bits
// 0x6400 | u is 1024 + u; subtracting 1152 leaves the code.
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& b0, uint32_t& b1) {
  const uint32_t x = w ^ 0x80808080u;
  uint32_t lo = __byte_perm(x, 0x64646464u, 0x5140);
  uint32_t hi = __byte_perm(x, 0x64646464u, 0x5342);
  const __half2 bias = __float2half2_rn(1152.0f);
  __half2 hl = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
  __half2 hh = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
  b0 = *reinterpret_cast<uint32_t*>(&hl);
  b1 = *reinterpret_cast<uint32_t*>(&hh);
}

__device__ __forceinline__ uint32_t pack_h2(__half a, __half b) {
  __half2 h = __halves2half2(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void split_hi_lo(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
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
template <int D>
__device__ __forceinline__ void make_q_frag(uint32_t (&aq)[D / 16][4], const void* q, size_t qoff,
                                            int bf16, const float* kscale, float qs, int G,
                                            int g, int t) {
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
    for (int e = 0; e < 4; ++e) split_hi_lo(x[e], h[e], lo[e]);
    aq[kk][0] = pack_h2(h[0], h[1]);    // row g,   k = 2t, 2t+1
    aq[kk][1] = pack_h2(lo[0], lo[1]);  // row g+8, k = 2t, 2t+1
    aq[kk][2] = pack_h2(h[2], h[3]);    // row g,   k = 2t+8, 2t+9
    aq[kk][3] = pack_h2(lo[2], lo[3]);  // row g+8, k = 2t+8, 2t+9
  }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) attention_kernel(Shape s, Dev d,
                                                                 const void* __restrict__ q,
                                                                 float* __restrict__ out,
                                                                 int splits, int chunk_blocks) {
  extern __shared__ __align__(16) float smem[];
  const int G = s.G;
  const int chunk_tok = chunk_blocks * 16;
  float* sc = smem;                                   // [G][chunk_tok] raw scores (log2 units)
  float* wm = sc + G * chunk_tok;                     // [NW][G]
  float* wl = wm + kAttnWarps * G;                    // [NW][G]
  float* wo = wl + kAttnWarps * G;                    // [NW][G][D]
  float* cm = wo + kAttnWarps * G * D;                // [G]    CTA max     (read by peers)
  float* cl = cm + kMaxG;                             // [G]    CTA sum     (read by peers)
  float* co = cl + kMaxG;                             // [G][D] CTA output  (read by peers)
  float* gM = co + G * D;                             // [G]
  float* gL = gM + kMaxG;                             // [G]

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
  const int blk0 = rank * chunk_blocks;
  const int blk1 = min(nbT, blk0 + chunk_blocks);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const size_t qoff = (lb * s.Hq + (size_t)h * G) * D;
  const float qs = kQPre * 1.4426950408889634f * rsqrtf((float)D);
  const float* sKu = d.sK + (size_t)u * D;
  const float* sVu = d.sV + (size_t)u * D;
  const int8_t* k8u = d.k8 + (size_t)u * s.cap * D;
  const int8_t* v8u = d.v8 + (size_t)u * s.cap * D;
  const char* k16u = reinterpret_cast<const char*>(d.k16) + (size_t)u * s.WR * D * 2;
  const char* v16u = reinterpret_cast<const char*>(d.v16) + (size_t)u * s.WR * D * 2;
  const int32_t* posR = d.pos + lb * s.S + s.cap;

  uint32_t aq[D / 16][4];
  make_q_frag<D>(aq, q, qoff, s.qbf16, sKu, qs, G, g, t);
  float acc[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  bool in_ring = false;

  for (int blk = blk0 + warp; blk < blk1; blk += kAttnWarps) {
    const bool ring = blk >= nb8;
    if (ring && !in_ring) {
      // INT8 -> FP16 transition: unscaled q, and apply the V scale to what
      // has been accumulated from codes so far.
      make_q_frag<D>(aq, q, qoff, s.qbf16, nullptr, qs, G, g, t);
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        const float2 sv = *reinterpret_cast<const float2*>(sVu + j * 8 + 2 * t);
        acc[j][0] *= sv.x; acc[j][1] *= sv.y; acc[j][2] *= sv.x; acc[j][3] *= sv.y;
      }
      in_ring = true;
    }
    float sc4[2][2];
    bool valid[2][2];
    if (!ring) {
      // ------------------------------------------------ INT8 block
      constexpr int NC = D / 32;
      const uint4* kb = reinterpret_cast<const uint4*>(k8u + (size_t)blk * 16 * D);
      const uint4* vb = reinterpret_cast<const uint4*>(v8u + (size_t)blk * 16 * D);
      uint4 kw[NC], vw[NC];
#pragma unroll
      for (int r = 0; r < NC; ++r) kw[r] = __ldg(kb + r * 32 + lane);
#pragma unroll
      for (int r = 0; r < NC; ++r) vw[r] = __ldg(vb + r * 32 + lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t b0, b1;
          i8x4_to_h2x2(comp(kw[nt * (NC / 2) + (kk >> 2)], kk & 3), b0, b1);
          mma16816(c, aq[kk], b0, b1);
        }
        sc4[nt][0] = (c[0] + c[2]) * kQPreInv;
        sc4[nt][1] = (c[1] + c[3]) * kQPreInv;
        const int tok = blk * 16 + nt * 8 + 2 * t;
        valid[nt][0] = tok < n8;
        valid[nt][1] = tok + 1 < n8;
      }
      // softmax + PV below uses vw
      float p[2][2];
      {
        float mloc = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (!valid[nt][j] || g >= G) sc4[nt][j] = -INFINITY;
            mloc = fmaxf(mloc, sc4[nt][j]);
          }
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
        const float m_new = fmaxf(m_run, mloc);
        const float corr = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
        float ps = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            p[nt][j] = (sc4[nt][j] == -INFINITY) ? 0.f : exp2f(sc4[nt][j] - m_new);
            ps += p[nt][j];
          }
        l_run = l_run * corr + ps;
        m_run = m_new;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          acc[j][0] *= corr; acc[j][1] *= corr; acc[j][2] *= corr; acc[j][3] *= corr;
        }
      }
      if (g < G) {
        float* dst = sc + g * chunk_tok + (blk - blk0) * 16 + 2 * t;
        *reinterpret_cast<float2*>(dst) = make_float2(sc4[0][0], sc4[0][1]);
        *reinterpret_cast<float2*>(dst + 8) = make_float2(sc4[1][0], sc4[1][1]);
      }
      uint32_t pa[4];
      {
        __half hi[2][2], lo[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) split_hi_lo(p[nt][j], hi[nt][j], lo[nt][j]);
        pa[0] = pack_h2(hi[0][0], hi[0][1]);
        pa[1] = pack_h2(lo[0][0], lo[0][1]);
        pa[2] = pack_h2(hi[1][0], hi[1][1]);
        pa[3] = pack_h2(lo[1][0], lo[1][1]);
      }
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        uint32_t b0, b1;
        i8x4_to_h2x2(comp(vw[j >> 2], j & 3), b0, b1);
        mma16816(acc[j], pa, b0, b1);
      }
    } else {
      // ------------------------------------------------ FP16 ring block
      constexpr int NC = D / 16;
      const int rb = blk - nb8;
      const uint4* kb = reinterpret_cast<const uint4*>(k16u + (size_t)rb * 32 * D);
      const uint4* vb = reinterpret_cast<const uint4*>(v16u + (size_t)rb * 32 * D);
      const int2 pv0 = *reinterpret_cast<const int2*>(posR + rb * 16 + 2 * t);
      const int2 pv1 = *reinterpret_cast<const int2*>(posR + rb * 16 + 8 + 2 * t);
      valid[0][0] = pv0.x >= 0; valid[0][1] = pv0.y >= 0;
      valid[1][0] = pv1.x >= 0; valid[1][1] = pv1.y >= 0;
      uint4 kw[NC];
#pragma unroll
      for (int r = 0; r < NC; ++r) kw[r] = __ldg(kb + r * 32 + lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint4& w4 = kw[nt * (D / 32) + (kk >> 1)];
          mma16816(c, aq[kk], comp(w4, (kk & 1) * 2), comp(w4, (kk & 1) * 2 + 1));
        }
        sc4[nt][0] = (c[0] + c[2]) * kQPreInv;
        sc4[nt][1] = (c[1] + c[3]) * kQPreInv;
      }
      float p[2][2];
      {
        float mloc = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (!valid[nt][j] || g >= G) sc4[nt][j] = -INFINITY;
            mloc = fmaxf(mloc, sc4[nt][j]);
          }
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
        const float m_new = fmaxf(m_run, mloc);
        const float corr = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
        float ps = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            p[nt][j] = (sc4[nt][j] == -INFINITY) ? 0.f : exp2f(sc4[nt][j] - m_new);
            ps += p[nt][j];
          }
        l_run = l_run * corr + ps;
        m_run = m_new;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          acc[j][0] *= corr; acc[j][1] *= corr; acc[j][2] *= corr; acc[j][3] *= corr;
        }
      }
      if (g < G) {
        float* dst = sc + g * chunk_tok + (blk - blk0) * 16 + 2 * t;
        *reinterpret_cast<float2*>(dst) = make_float2(sc4[0][0], sc4[0][1]);
        *reinterpret_cast<float2*>(dst + 8) = make_float2(sc4[1][0], sc4[1][1]);
      }
      uint32_t pa[4];
      {
        __half hi[2][2], lo[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) split_hi_lo(p[nt][j], hi[nt][j], lo[nt][j]);
        pa[0] = pack_h2(hi[0][0], hi[0][1]);
        pa[1] = pack_h2(lo[0][0], lo[0][1]);
        pa[2] = pack_h2(hi[1][0], hi[1][1]);
        pa[3] = pack_h2(lo[1][0], lo[1][1]);
      }
      uint4 vw[NC];
#pragma unroll
      for (int r = 0; r < NC; ++r) vw[r] = __ldg(vb + r * 32 + lane);
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        const uint4& w4 = vw[j >> 1];
        mma16816(acc[j], pa, comp(w4, (j & 1) * 2), comp(w4, (j & 1) * 2 + 1));
      }
    }
  }
  if (!in_ring) {
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      const float2 sv = *reinterpret_cast<const float2*>(sVu + j * 8 + 2 * t);
      acc[j][0] *= sv.x; acc[j][1] *= sv.y; acc[j][2] *= sv.x; acc[j][3] *= sv.y;
    }
  }
  // ---------------------------------------------------------------- warp -> CTA
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  if (g < G) {
    float* o = wo + (warp * G + g) * D;
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
      *reinterpret_cast<float2*>(o + j * 8 + 2 * t) =
          make_float2(acc[j][0] + acc[j][2], acc[j][1] + acc[j][3]);
    if (t == 0) {
      wm[warp * G + g] = m_run;
      wl[warp * G + g] = l_run;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += kAttnThreads) {
    const int gg = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w * G + gg]);
    float o = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float mw = wm[w * G + gg];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
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
      if (mr != -INFINITY) L += cluster.map_shared_rank(cl, r)[gg] * exp2f(mr - M);
    }
    gM[gg] = M;
    gL[gg] = L;
  }
  __syncthreads();
  // attention mass of this CTA's tokens, summed over its G query heads
  float* mass_u = d.mass + (size_t)u * s.S;
  const int ntok = (blk1 - blk0) * 16;
  for (int i = threadIdx.x; i < ntok; i += kAttnThreads) {
    const float s0 = sc[i];
    if (s0 == -INFINITY) continue;   // empty ring slot or tail past n8
    float m = 0.f;
    for (int gg = 0; gg < G; ++gg) m += exp2f(sc[gg * chunk_tok + i] - gM[gg]) / gL[gg];
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
        if (mr != -INFINITY) acc_o += cluster.map_shared_rank(co, r)[i] * exp2f(mr - gM[gg]);
      }
      o[i] = acc_o / gL[gg];
    }
  }
  cluster.sync();   // peers keep their shared memory alive until rank 0 has read it
}

int attention_smem_bytes(const Shape& s, int splits, int max_tokens) {
  const int nbT = (max_tokens + 15) / 16;
  const int chunk = (nbT + splits - 1) / splits;
  const int G = s.G, D = s.D;
  size_t f = (size_t)G * chunk * 16 + 2 * kAttnWarps * G + (size_t)kAttnWarps * G * D + 2 * kMaxG +
             (size_t)G * D + 2 * kMaxG;
  return (int)(f * sizeof(float));
}

int attention_max_smem() { return 200 * 1024; }

template <int D>
static int launch_d(const Shape& s, const Dev& d, const void* q, float* out, int splits,
                    int max_tokens, cudaStream_t stream) {
  const int nbT = (max_tokens + 15) / 16;
  const int chunk = (nbT + splits - 1) / splits;
  const int smem = attention_smem_bytes(s, splits, max_tokens);
  static int configured = 0;
  if (smem > configured) {
    if (cudaFuncSetAttribute(attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attention_max_smem()) != cudaSuccess)
      return -1;
    configured = attention_max_smem();
  }
  const unsigned units = (unsigned)(s.L * s.B * s.Hkv);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * splits);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, attention_kernel<D>, s, d, q, out, splits, chunk);
  return e == cudaSuccess ? 0 : -1;
}

int launch_attention(const Shape& s, const Dev& d, const void* q, float* out, int splits,
                     int max_tokens, cudaStream_t stream) {
  if (s.D == 128) return launch_d<128>(s, d, q, out, splits, max_tokens, stream);
  if (s.D == 64) return launch_d<64>(s, d, q, out, splits, max_tokens, stream);
  return -1;
}

}  // namespace confkv
