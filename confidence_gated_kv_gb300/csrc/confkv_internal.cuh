// Internal definitions shared by the CONF-KV kernels and the host runtime.
//
// Data layout in HBM (all carved from one caller-allocated workspace):
//
//   Slot space of one (layer l, sequence b): S = cap + WR slots.
//     slots [0, cap)       INT8 region, dense: slots [0, n8) are resident.
//     slots [cap, cap+WR)  FP16 ring of WR = W + 16 slots; a token at
//                          position p lives in ring slot p mod WR; a slot
//                          whose pos is -1 is empty.
//   Per-slot metadata [l][b][S]: pos (int32), ema (fp32).
//   Attention-mass partials [l][b][kvh][S] (fp32, one per KV head).
//
//   K/V payload per unit u = (l, b, kvh), in 16-token blocks:
//     INT8:  k8, v8  [u][cstride/16][16*D bytes], each byte the code + 128;
//                    cstride = cap + 16 slots (only the first cap are used)
//                    (code in [-127, 127], stored biased as uint8)
//     FP16:  k16,v16 [u][WR/16][16*D halves]
//   Inside a block the bytes are interleaved so that lane `lane` of a warp
//   reading 16 contiguous bytes at  r*512 + lane*16  receives exactly its
//   B-operand fragments of mma.m16n8k16 (QK^T for K, PV for V).  The
//   offset functions below are the single definition of that interleave.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace confkv {

constexpr int kRingExtra = 16;      // WR = W + kRingExtra
constexpr int kMaxG = 8;            // query heads per KV head supported
constexpr int kMaxSV = 1024;        // confidence partial blocks per sequence
constexpr int kCodeBias = 128;      // stored INT8 byte = code + 128

// ---------------------------------------------------------------------------
// Block interleave (host and device).  tau in [0,16) is the token within the
// block, c in [0,D) the channel.  Returns a byte offset inside the block.
// ---------------------------------------------------------------------------

// INT8 K: token tau = 8*nt + g pairs with mma column g of n-tile nt; channel
// c = 16*kk + {2t, 2t+1, 2t+8, 2t+9}[bsel] pairs with k-step kk, lane 4g+t.
__host__ __device__ inline int k8_offset(int D, int tau, int c) {
  int nt = tau >> 3, g = tau & 7;
  int kk = c >> 4, cc = c & 15;
  int t = (cc & 7) >> 1, bsel = ((cc >> 3) << 1) | (cc & 1);
  int nc = D >> 5;                                // 16-byte chunks per lane
  int r = nt * (nc >> 1) + (kk >> 2), w = kk & 3;
  return r * 512 + ((g << 2) | t) * 16 + w * 4 + bsel;
}

// INT8 V: channel c = 8*j + g pairs with mma column g of n-tile j; token
// tau = {2t, 2t+1, 2t+8, 2t+9}[bsel] pairs with the k index of lane 4g+t.
__host__ __device__ inline int v8_offset(int D, int tau, int c) {
  int j = c >> 3, g = c & 7;
  int t = (tau & 7) >> 1, bsel = ((tau >> 3) << 1) | (tau & 1);
  int r = j >> 2, w = j & 3;
  (void)D;
  return r * 512 + ((g << 2) | t) * 16 + w * 4 + bsel;
}

// FP16 K (offset in bytes): token tau = 8*nt + g; channel
// c = 16*kk + 8*reg + 2t + half.
__host__ __device__ inline int k16_offset(int D, int tau, int c) {
  int nt = tau >> 3, g = tau & 7;
  int kk = c >> 4, cc = c & 15;
  int t = (cc & 7) >> 1, reg = cc >> 3, half = cc & 1;
  int r = nt * (D >> 5) + (kk >> 1);
  return r * 512 + ((g << 2) | t) * 16 + (kk & 1) * 8 + reg * 4 + half * 2;
}

// FP16 V (offset in bytes): channel c = 8*j + g; token
// tau = 8*reg + 2t + half.
__host__ __device__ inline int v16_offset(int D, int tau, int c) {
  int j = c >> 3, g = c & 7;
  int t = (tau & 7) >> 1, reg = tau >> 3, half = tau & 1;
  int r = j >> 1;
  (void)D;
  return r * 512 + ((g << 2) | t) * 16 + (j & 1) * 8 + reg * 4 + half * 2;
}

// ---------------------------------------------------------------------------
// Shapes, device pointers and counters passed to every kernel by value.
// ---------------------------------------------------------------------------

struct ConfPartial {     // one vocab chunk of one sequence
  float M;               // chunk maximum
  float z1, z2;          // largest and second largest logit of the chunk
  int i1;                // index of z1 (lowest index on ties)
  float S, Se;           // sum exp(z - M) as an unevaluated sum S + Se
  float T, Te;           // sum (z - M) exp(z - M) as T + Te
};

struct DevStats {        // cumulative counters, updated with atomics
  unsigned long long steps;
  unsigned long long evicted;
  unsigned long long moved;
  unsigned long long requant;
  unsigned long long attn_bytes;   // algorithmic bytes of the attention kernel
  unsigned long long step_bytes;   // algorithmic bytes of the whole step
  // resident footprint after each step: every selection adds its (layer,
  // sequence)'s entries and K/V bytes to the accumulators of the step's
  // parity; the first selection of the next step (group 0) folds them into
  // the peaks and zeroes them, and confkv_get_stats folds the latest step's
  // on the host, so no selection waits on another
  unsigned long long res_entries_acc[2], res_bytes_acc[2];
  unsigned long long peak_entries, peak_bytes;
};

struct Shape {
  int L, B, Hq, Hkv, G, D, V;
  int cap, W, WR, P, S;      // S = cap + WR slots per (l, b)
  int cstride;               // INT8 slots between consecutive units in memory (cap + 16):
                             // unit bases do not all share one power-of-two alignment
  int SV;                    // confidence partial blocks per sequence
  int qbf16;                 // query dtype: 0 fp16, 1 bf16
  int max_evict;             // rows of evicted_pos per (l, b)
  double tau, wH, wm, wp;     // confidence weights and threshold (float64 math)
  float alpha, lam;           // rank weight and EMA decay (float32 math)
  int compaction;             // 0 tail fill, 1 order preserving (ablation)
  int vocab_ctas;             // fused step: CTAs after the units that only reduce vocabulary
                              // chunks (0: the units' epilogue warps reduce one chunk each)
};

struct Dev {
  uint8_t* k8; uint8_t* v8;        // biased INT8 codes (code + 128)
  __half* k16; __half* v16;
  float* sK;   float* sV;          // [l][b][kvh][D]
  int32_t* pos; float* ema;        // [l][b][S]
  float* mass;                     // [l][b][kvh][S]
  int32_t* n8;                     // [l][b]
  int32_t* T0;                     // [b]
  int32_t* n_high; int32_t* n_low; // [l]
  ConfPartial* conf;               // [b][SV]
  double* cval;                    // [b] confidence of the current step
  uint32_t* conf_done;             // [b] chunk partials of b done in the attention kernel (0 between steps)
  uint32_t* scratch;               // [l][b][S] selection keys / compaction pairs
  DevStats* stats;
  int32_t* status;                 // device status word (0 = ok)
  uint32_t* absmax;                // [2][l][b][kvh][D] prefill scratch
  float* scores;                   // [persistent CTAs][2][G][S] attention score scratch
  int score_ctas;                  // persistent attention CTAs the score scratch holds
  int attn_ctas;                   // cap on the persistent attention grid (0 = none)
  long long* step_dev;             // decode steps done since prefill (read by prestep and select)
  uint32_t* sel_done;              // select CTAs finished in the current step (0 between steps)
  int32_t* order;                  // [l*b] (layer, sequence) groups, most INT8 entries first
                                   // (written by prestep when `sorted`)
  int sorted;                      // prestep sorts the groups every step
  int sched;                       // how the persistent attention kernel deals its units
  uint32_t* queue;                 // next sorted position to hand out (kSchedQueue; zeroed by prestep)
  uint32_t* arrive;                // [l*b] fused steps: units of (l, b) done this step
  uint32_t* conf_ready;            // [b] fused steps: step index + 1 once c and the budgets of b are written
};

enum : int { kSchedRoundRobin = 0, kSchedQueue = 1 };

// Groups (layer, sequence) that prestep can sort by INT8 length in one block.
constexpr int kSortMaxGroups = 1024;

// Status bits written by kernels (never trap; the host reads them lazily).
enum : int32_t {
  kStatusOk = 0,
  kStatusCapacity = 1,     // an INT8 region would overflow
  kStatusEvictBound = 2,   // more evictions than the evicted_pos rows hold
  kStatusBadCount = 4,     // inconsistent eviction count (selection failed)
  kStatusTimeout = 8,      // a bounded mbarrier wait gave up
};

__host__ __device__ inline size_t unit_index(const Shape& s, int l, int b, int h) {
  return ((size_t)l * s.B + b) * s.Hkv + h;
}
__host__ __device__ inline size_t lb_index(const Shape& s, int l, int b) {
  return (size_t)l * s.B + b;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The three kernels of a step (and the first
// kernel of the next step) are launched with programmatic stream
// serialisation, and each waits (griddepcontrol.wait) before its first global
// memory access until the previous kernel has completed and its writes are
// visible.  No kernel triggers its dependents early: the next grid is
// launched as the CTAs of the current one exit, which saves part of the
// launch gap (triggering at kernel entry instead measured about 5% slower per
// step).  The data order is exactly the stream order; without the launch
// attribute the wait does nothing.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Devices a process can use with the per-device records below.
constexpr int kMaxDevices = 64;

// Raises `kernel`'s dynamic shared memory limit to at least `bytes` on the
// current device.  cudaFuncSetAttribute acts on the current device only, so
// each launcher keeps its own record `done` of the limit set per device.
template <typename... KArgs>
inline cudaError_t ensure_smem(void (*kernel)(KArgs...), int bytes, int (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool known = dev >= 0 && dev < kMaxDevices;
  if (known && done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && known) done[dev] = bytes;
  return e;
}
#endif

#ifdef __CUDACC__
// Append the new token of unit u = (l, b, kvh) at position t to its FP16 ring
// slot t mod WR (rainbus Algorithm 1 step 13), by one whole warp: lane i
// writes the 8 bytes of K that hold channels 16(i/4) + 2(i%4) + {0, 1, 8, 9}
// of the interleaved block and V channels i, i + 32, ...; lane 0 writes the
// slot's position and a zero EMA (the same values for every KV head of the
// group).
template <int D>
__device__ __forceinline__ void append_unit_warp(const Shape& s, const Dev& d, int u, int t,
                                                 const __half* __restrict__ k_new,
                                                 const __half* __restrict__ v_new) {
  const int lane = threadIdx.x & 31;
  const int kc0 = 16 * (lane >> 2) + 2 * (lane & 3);
  const int lbi = u / s.Hkv;
  const int rs = t % s.WR;
  const size_t blk = ((size_t)u * (s.WR / 16) + (rs >> 4)) * 16 * D * 2;
  const unsigned short* kn = reinterpret_cast<const unsigned short*>(k_new) + (size_t)u * D;
  const unsigned short* vn = reinterpret_cast<const unsigned short*>(v_new) + (size_t)u * D;
  char* k16b = reinterpret_cast<char*>(d.k16);
  char* v16b = reinterpret_cast<char*>(d.v16);
  if (lane < D / 4) {
    uint2 kx;
    kx.x = *reinterpret_cast<const uint32_t*>(kn + kc0);
    kx.y = *reinterpret_cast<const uint32_t*>(kn + kc0 + 8);
    *reinterpret_cast<uint2*>(k16b + blk + k16_offset(D, rs & 15, kc0)) = kx;
  }
#pragma unroll
  for (int i = 0; i < D / 32; ++i)
    *reinterpret_cast<unsigned short*>(v16b + blk + v16_offset(D, rs & 15, lane + 32 * i)) = vn[lane + 32 * i];
  if (lane == 0) {
    d.pos[(size_t)lbi * s.S + s.cap + rs] = t;
    d.ema[(size_t)lbi * s.S + s.cap + rs] = 0.f;
  }
}
#endif

// ---------------------------------------------------------------------------
// Kernel launchers (defined in the .cu files; all asynchronous on `stream`).
// ---------------------------------------------------------------------------
int launch_prefill(const Shape& s, const Dev& d, const void* k, const void* v, long long t_max,
                   const int32_t* T0_host, cudaStream_t stream);
// step: the index of this decode step, or -1 for a step that takes it from
// d.step_dev (a step captured into a graph, and every step while replays are
// reserved); the select kernel of such a step advances d.step_dev.
// conf: whether its blocks also reduce the logits to confidence partials
// (otherwise the persistent attention kernel does).
int launch_prestep(const Shape& s, const Dev& d, long long step, const float* logits,
                   const void* k_new, const void* v_new, bool conf, cudaStream_t stream);
// Writes out, and budget and conf_out (may be null) from the confidence
// partials.  logits: null when the prestep kernel wrote the partials; else
// (persistent kernel only) the epilogue warps reduce these logits to the
// partials first and the last CTA to finish them merges.
int launch_attention(const Shape& s, const Dev& d, const void* q, float* out, int32_t* budget,
                     float* conf_out, const float* logits, int splits, int max_tokens,
                     cudaStream_t stream);
// Grid and cluster size of the attention launch for `splits` CTAs per unit
// (the persistent kernel when 1, whose CTAs are not clustered).
void attention_grid(const Shape& s, const Dev& d, int splits, int* grid, int* cluster);
int launch_select(const Shape& s, const Dev& d, long long step, int32_t* evicted_pos,
                  int32_t* n_evicted, cudaStream_t stream);
int attention_smem_bytes(const Shape& s, int splits, int max_tokens);
// Fused step: one launch for the whole decode step (append, vocabulary
// reduction and confidence, attention with mass, and every selection) when
// fused_step_fits: one CTA per unit and per SM, each CTA's epilogue warp
// reducing a vocabulary chunk while the unit streams; step as for
// launch_prestep.
bool fused_step_fits(const Shape& s, const Dev& d, int splits, int max_tokens);
int launch_fused_step(const Shape& s, const Dev& d, long long step, const void* q, const void* k_new,
                      const void* v_new, const float* logits, float* out, int32_t* budget, float* conf_out,
                      int32_t* evicted_pos, int32_t* n_evicted, int max_tokens, cudaStream_t stream);
int attention_max_smem();
int attention_persistent_ctas();   // persistent CTAs per launch (2 per SM)
// Warps of a fused-step CTA: 8 consumer warps, the producer and the epilogue warp.
constexpr int kFusedConsumers = 8;
constexpr int kFusedWarps = kFusedConsumers + 2;
int launch_selftest_timeout(const Dev& d, cudaStream_t stream);

}  // namespace confkv
