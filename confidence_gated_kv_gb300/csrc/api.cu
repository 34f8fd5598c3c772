// C ABI of the CONF-KV decode-step cache manager: configuration checks,
// workspace layout, host-side bounds that size each launch, state export /
// import, counters and per-kernel timing.  The arithmetic of the method lives
// in the kernels (prestep.cu, attention.cu, select.cu, prefill.cu).
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/confkv.h"
#include "confkv_internal.cuh"

using namespace confkv;

namespace {

constexpr int kNumSMs = 152;          // GB300: 2 dies x 76 SMs
constexpr int kMaxSplits = 8;         // portable thread-block cluster size

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Carve {
  size_t off = 0;
  char* base = nullptr;
  template <typename T>
  T* take(size_t count) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

struct Staging {
  void* q; void* k_new; void* v_new; float* logits;
  float* out; int32_t* budget; float* conf; int32_t* evicted; int32_t* nevict;
};

bool valid_config(const confkv_config* c) {
  if (!c || !c->n_high || !c->n_low) return false;
  if (c->L < 1 || c->B < 1 || c->Hq < 1 || c->Hkv < 1 || c->V < 2 || c->W < 1 || c->P < 0)
    return false;
  if ((long long)c->V > 4096LL * kMaxSV) return false;   // vocabulary chunks of <= 4096 logits
  if (c->compaction != CONFKV_COMPACT_TAIL_FILL && c->compaction != CONFKV_COMPACT_ORDERED) return false;
  if (c->Hq % c->Hkv != 0 || c->Hq / c->Hkv > kMaxG) return false;
  if (c->d != 64 && c->d != 128) return false;
  if (c->cap < 16 || c->max_evict < 0) return false;
  if (c->q_dtype != CONFKV_Q_FP16 && c->q_dtype != CONFKV_Q_BF16) return false;
  if (!std::isfinite(c->tau) || !std::isfinite(c->w_H) || !std::isfinite(c->w_m) ||
      !std::isfinite(c->w_p))
    return false;
  if (!(c->alpha >= 0.f && c->alpha <= 1.f) || !(c->lam >= 0.f && c->lam <= 1.f)) return false;
  for (int l = 0; l < c->L; ++l) {
    if (c->n_high[l] < 1 || c->n_low[l] < 1) return false;
    if (c->n_high[l] < c->P || c->n_low[l] < c->P) return false;
  }
  // 32-bit slot and element indexing inside kernels
  const long long cap = align_up(c->cap, 16);
  if (cap + c->W + kRingExtra > (1ll << 30)) return false;
  return true;
}

Shape make_shape(const confkv_config* c) {
  Shape s{};
  s.L = c->L; s.B = c->B; s.Hq = c->Hq; s.Hkv = c->Hkv; s.G = c->Hq / c->Hkv; s.D = c->d;
  s.V = c->V;
  s.cap = (int)align_up(c->cap, 16);
  s.W = c->W;
  s.WR = (int)align_up(c->W + kRingExtra, 16);
  s.P = c->P;
  s.S = s.cap + s.WR;
  s.cstride = s.cap + 16;
  // vocabulary chunks per sequence: at most 4096 logits each (16 per thread
  // of a 256-thread prestep block).  Shapes whose every (layer, sequence,
  // KV head) unit can have an SM of its own (the fused step):
  //   - with SMs left over, enough of them to reduce the vocabulary with
  //     about one warp per 1024 logits or fewer, those SMs take vocabulary
  //     CTAs, and the chunks are cut to one per warp of those CTAs (at
  //     least 256 logits each): each warp loads its chunk in one round, and
  //     the confidence is merged long before the units' attention ends;
  //   - otherwise the smallest chunks from 512 logits up that leave at most
  //     one chunk per unit: the epilogue warp of a unit's CTA reduces one
  //     while the unit streams.
  // Wider vocabularies than kMaxSV chunks are rejected.
  const long long units = (long long)c->L * c->B * c->Hkv;
  const long long sms = attention_persistent_ctas() / 2;
  const long long min_sv = (c->V + 4095) / 4096;
  long long sv = min_sv;
  s.vocab_ctas = 0;
  if (units <= sms) {
    const long long spare = sms - units;
    if (spare > 0 && spare * kFusedWarps >= (long long)c->B * ((c->V + 1023) / 1024)) {
      // no more CTAs than give every warp a chunk of 256 logits or more
      const long long want = ((long long)c->B * ((c->V + 255) / 256) + kFusedWarps - 1) / kFusedWarps;
      s.vocab_ctas = (int)std::min(spare, want);
      sv = std::max(min_sv, std::min((long long)s.vocab_ctas * kFusedWarps / c->B, ((long long)c->V + 255) / 256));
    } else {
      int chunk = 512;
      while (chunk < 4096 && (long long)c->B * ((c->V + chunk - 1) / chunk) > units) chunk *= 2;
      sv = (c->V + chunk - 1) / chunk;
    }
  }
  sv = std::min<long long>(std::max<long long>(sv, 1), kMaxSV);
  // chunks of ceil(V / SV) logits: the count that leaves no chunk empty
  const long long chunk = (c->V + sv - 1) / sv;
  s.SV = (int)((c->V + chunk - 1) / chunk);
  s.qbf16 = c->q_dtype == CONFKV_Q_BF16;
  s.max_evict = c->max_evict > 0 ? c->max_evict : s.cap + s.WR;
  s.tau = c->tau; s.wH = c->w_H; s.wm = c->w_m; s.wp = c->w_p;
  s.alpha = c->alpha; s.lam = c->lam;
  s.compaction = c->compaction;
  return s;
}

size_t layout(const Shape& s, char* base, Dev* d, Staging* st) {
  Carve cv;
  cv.base = base;
  const size_t units = (size_t)s.L * s.B * s.Hkv;
  const size_t lbs = (size_t)s.L * s.B;
  Dev dd{};
  dd.k8 = cv.take<uint8_t>(units * s.cstride * s.D);
  dd.v8 = cv.take<uint8_t>(units * s.cstride * s.D);
  dd.k16 = cv.take<__half>(units * s.WR * s.D);
  dd.v16 = cv.take<__half>(units * s.WR * s.D);
  dd.sK = cv.take<float>(units * s.D);
  dd.sV = cv.take<float>(units * s.D);
  dd.pos = cv.take<int32_t>(lbs * s.S);
  dd.ema = cv.take<float>(lbs * s.S);
  dd.mass = cv.take<float>(units * s.S);
  dd.n8 = cv.take<int32_t>(lbs);
  dd.T0 = cv.take<int32_t>(s.B);
  dd.n_high = cv.take<int32_t>(s.L);
  dd.n_low = cv.take<int32_t>(s.L);
  dd.conf = cv.take<ConfPartial>((size_t)s.B * s.SV);
  dd.cval = cv.take<double>(s.B);
  dd.conf_done = cv.take<uint32_t>(s.B);
  dd.scratch = cv.take<uint32_t>(lbs * s.S);
  dd.stats = cv.take<DevStats>(1);
  dd.status = cv.take<int32_t>(1);
  dd.absmax = cv.take<uint32_t>(2 * units * s.D);
  dd.score_ctas = attention_persistent_ctas();
  dd.attn_ctas = 0;
  dd.scores = cv.take<float>((size_t)dd.score_ctas * 2 * s.G * s.S);
  dd.step_dev = cv.take<long long>(1);
  dd.sel_done = cv.take<uint32_t>(1);
  dd.order = cv.take<int32_t>(lbs);
  dd.queue = cv.take<uint32_t>(1);
  dd.arrive = cv.take<uint32_t>(lbs);
  dd.conf_ready = cv.take<uint32_t>(s.B);
  // the persistent attention kernel takes its units longest first from a
  // queue over prestep's sorted order (round robin when there are too many
  // groups to sort in one prestep launch)
  dd.sorted = lbs <= (size_t)kSortMaxGroups ? 1 : 0;
  dd.sched = dd.sorted ? kSchedQueue : kSchedRoundRobin;
  Staging sg{};
  sg.q = cv.take<uint16_t>(lbs * s.Hq * s.D);
  sg.k_new = cv.take<uint16_t>(units * s.D);
  sg.v_new = cv.take<uint16_t>(units * s.D);
  sg.logits = cv.take<float>((size_t)s.B * s.V);
  sg.out = cv.take<float>(lbs * s.Hq * s.D);
  sg.budget = cv.take<int32_t>(lbs);
  sg.conf = cv.take<float>(s.B);
  sg.evicted = cv.take<int32_t>(lbs * s.max_evict);
  sg.nevict = cv.take<int32_t>(lbs);
  if (d) *d = dd;
  if (st) *st = sg;
  return align_up(cv.off, 256);
}

}  // namespace

struct confkv_ctx {
  confkv_config cfg;
  std::vector<int32_t> n_high, n_low;
  Shape s;
  Dev d;
  Staging st;
  char* ws = nullptr;
  size_t ws_bytes = 0;
  int device = 0;
  bool prefilled = false;
  std::vector<int32_t> T0;
  long long steps = 0;
  long long n_bound = 0;    // max resident entries of any (l, b), new token excluded
  long long n8_bound = 0;   // max INT8 entries of any (l, b)
  int minN = 0, maxN = 0;
  long long host_h2d = 0, host_d2h = 0;   // bytes of the last confkv_step_host
  long long launches = 0;                  // kernels launched by decode steps
  bool fused_ok = true;                    // small shapes may run a step as one launch
  // confkv_step_host: a second stream copies the attention output back while
  // the select kernel runs (created on first use)
  cudaStream_t aux = nullptr;
  cudaEvent_t ev_attn = nullptr, ev_aux = nullptr, ev_in = nullptr, ev_q = nullptr;
  // profiling
  bool prof_on = false;
  int prof_max = 0, prof_count = 0;
  int prof_every = 1;        // record every prof_every-th step
  long long prof_tick = 0;   // steps seen while profiling is on
  std::vector<cudaEvent_t> ev;
  // graph replays: steps reserved and the attention plan pinned for them
  long long pin_left = 0;
  int pin_splits = 0, pin_max_tokens = 0;
};

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? CONFKV_OK : CONFKV_ECUDA; }
static bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// Alignment the decode kernels rely on: q is read with bulk copies (16-byte
// source addresses), k_new / v_new as 32-bit words, every other buffer as
// 4-byte elements.
static bool step_args_aligned(const void* q, const void* k_new, const void* v_new, const float* logits,
                              const float* out, const int32_t* budget, const float* confidence,
                              const int32_t* evicted_pos, const int32_t* n_evicted) {
  return aligned(q, 16) && aligned(k_new, 4) && aligned(v_new, 4) && aligned(logits, 4) && aligned(out, 4) &&
         aligned(budget, 4) && (!confidence || aligned(confidence, 4)) && aligned(evicted_pos, 4) &&
         aligned(n_evicted, 4);
}
static cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

extern "C" {

int confkv_workspace_bytes(const confkv_config* cfg, size_t* bytes) {
  if (!bytes || !valid_config(cfg)) return CONFKV_EINVAL;
  *bytes = layout(make_shape(cfg), nullptr, nullptr, nullptr);
  return CONFKV_OK;
}

int confkv_create(const confkv_config* cfg, void* workspace, size_t workspace_bytes,
                  confkv_ctx** out) {
  if (!out || !valid_config(cfg) || !workspace) return CONFKV_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return CONFKV_EINVAL;
  const Shape s = make_shape(cfg);
  const size_t need = layout(s, nullptr, nullptr, nullptr);
  if (workspace_bytes < need) return CONFKV_ECAPACITY;
  confkv_ctx* c = new (std::nothrow) confkv_ctx();
  if (!c) return CONFKV_ECAPACITY;
  c->cfg = *cfg;
  c->n_high.assign(cfg->n_high, cfg->n_high + cfg->L);
  c->n_low.assign(cfg->n_low, cfg->n_low + cfg->L);
  c->cfg.n_high = c->n_high.data();
  c->cfg.n_low = c->n_low.data();
  c->s = s;
  c->ws = static_cast<char*>(workspace);
  c->ws_bytes = workspace_bytes;
  layout(s, c->ws, &c->d, &c->st);
  cudaGetDevice(&c->device);
  c->minN = c->maxN = c->n_high[0];
  for (int l = 0; l < s.L; ++l) {
    c->minN = std::min({c->minN, c->n_high[l], c->n_low[l]});
    c->maxN = std::max({c->maxN, c->n_high[l], c->n_low[l]});
  }
  cudaError_t e = cudaMemcpy(c->d.n_high, c->n_high.data(), s.L * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(c->d.n_low, c->n_low.data(), s.L * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(c->d.stats, 0, sizeof(DevStats));
  if (e == cudaSuccess) e = cudaMemset(c->d.status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(c->d.step_dev, 0, sizeof(long long));
  if (e == cudaSuccess) e = cudaMemset(c->d.sel_done, 0, sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->d.conf_done, 0, s.B * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->d.arrive, 0, (size_t)s.L * s.B * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->d.conf_ready, 0, s.B * sizeof(uint32_t));
  if (e != cudaSuccess) {
    delete c;
    return CONFKV_ECUDA;
  }
  c->T0.assign(s.B, 0);
  *out = c;
  return CONFKV_OK;
}

void confkv_destroy(confkv_ctx* ctx) {
  if (!ctx) return;
  for (cudaEvent_t e : ctx->ev) cudaEventDestroy(e);
  if (ctx->ev_attn) cudaEventDestroy(ctx->ev_attn);
  if (ctx->ev_aux) cudaEventDestroy(ctx->ev_aux);
  if (ctx->ev_in) cudaEventDestroy(ctx->ev_in);
  if (ctx->ev_q) cudaEventDestroy(ctx->ev_q);
  if (ctx->aux) cudaStreamDestroy(ctx->aux);
  delete ctx;
}

int confkv_prefill(confkv_ctx* ctx, const int32_t* prefill_len, const void* k, const void* v,
                   int64_t t_max, void* stream) {
  if (!ctx || !prefill_len || t_max < 0) return CONFKV_EINVAL;
  const Shape& s = ctx->s;
  long long tmax0 = 0;
  for (int b = 0; b < s.B; ++b) {
    if (prefill_len[b] < 0 || prefill_len[b] > t_max) return CONFKV_EINVAL;
    tmax0 = std::max<long long>(tmax0, prefill_len[b]);
  }
  if (tmax0 > 0 && (!k || !v)) return CONFKV_EINVAL;
  if (tmax0 > 0 && (!aligned(k, 2) || !aligned(v, 2))) return CONFKV_EINVAL;
  if (tmax0 - s.W > s.cap) return CONFKV_ECAPACITY;
  cudaStream_t st = as_stream(stream);
  ctx->T0.assign(prefill_len, prefill_len + s.B);
  cudaError_t e = cudaMemcpyAsync(ctx->d.T0, ctx->T0.data(), s.B * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d.stats, 0, sizeof(DevStats), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d.status, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d.step_dev, 0, sizeof(long long), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d.sel_done, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d.conf_done, 0, s.B * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d.arrive, 0, (size_t)s.L * s.B * sizeof(uint32_t), st);
  // the step indices start again from 0: no flag of the earlier steps may match
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d.conf_ready, 0, s.B * sizeof(uint32_t), st);
  if (e != cudaSuccess) return CONFKV_ECUDA;
  if (launch_prefill(s, ctx->d, k, v, t_max, ctx->T0.data(), st) != 0) return CONFKV_ECUDA;
  // the host copy of T0 is pageable: make sure it has been consumed
  if (cudaStreamSynchronize(st) != cudaSuccess) return CONFKV_ECUDA;
  ctx->prefilled = true;
  ctx->steps = 0;
  ctx->pin_left = 0;
  ctx->n_bound = tmax0;
  ctx->n8_bound = std::max<long long>(0, tmax0 - s.W);
  return CONFKV_OK;
}

// Launch shape of the attention kernel for an INT8 bound.
// Attention launch for shape s, a bound n8_bound on the INT8 entries of any
// (layer, sequence) and a cap on the persistent grid (0 = none).
static int plan_attention_shape(const Shape& s, long long attn_ctas, long long n8_bound, int* splits_out,
                                int* max_tokens_out) {
  const int max_tokens = (int)align_up((size_t)n8_bound, 16) + s.WR;
  const long long units = (long long)s.L * s.B * s.Hkv;
  const int nbT = max_tokens / 16;
  int splits = 1;
  // Units split over CTA clusters only while there are fewer units than
  // persistent CTAs (two per SM) and each CTA keeps at least 64 blocks
  // (1024 tokens); then enough CTAs to fill the GPU a few times over, and no
  // more CTAs than the caller's cap on the attention grid.  Below that, the
  // cluster's launch and merge cost more than the shorter stream saves:
  // 144 units of ~500 tokens took 0.0165 ms as whole units against 0.025 ms
  // on 8-CTA clusters, and from one unit per persistent CTA upwards whole
  // units are faster too (512 units of 4K tokens: 0.123 against 0.176 ms on
  // 2-CTA clusters).
  const long long cap = attn_ctas;
  const bool few = units < 2LL * kNumSMs;
  while (few && splits < kMaxSplits && units * splits < 4LL * kNumSMs && nbT / (splits * 2) >= 64 &&
         (cap == 0 || units * splits * 2 <= cap))
    splits *= 2;
  while (splits < kMaxSplits && attention_smem_bytes(s, splits, max_tokens) > attention_max_smem())
    splits *= 2;
  if (attention_smem_bytes(s, splits, max_tokens) > attention_max_smem()) return CONFKV_ECAPACITY;
  *splits_out = splits;
  *max_tokens_out = max_tokens;
  return CONFKV_OK;
}

static int plan_attention_for(const confkv_ctx* ctx, long long n8_bound, int* splits_out,
                              int* max_tokens_out) {
  return plan_attention_shape(ctx->s, ctx->d.attn_ctas, n8_bound, splits_out, max_tokens_out);
}

int confkv_launch_plan(const confkv_config* cfg, int64_t n8_bound, int32_t attn_ctas, int32_t* splits,
                       int32_t* ctas, int32_t* cluster) {
  if (!splits || !ctas || !cluster || !valid_config(cfg) || n8_bound < 0 || attn_ctas < 0)
    return CONFKV_EINVAL;
  const Shape s = make_shape(cfg);
  if (n8_bound > s.cap) return CONFKV_EINVAL;
  int sp = 0, mt = 0;
  const int r = plan_attention_shape(s, attn_ctas, n8_bound, &sp, &mt);
  if (r != CONFKV_OK) return r;
  Dev d{};
  d.score_ctas = attention_persistent_ctas();
  d.attn_ctas = attn_ctas;
  int g = 0, c = 0;
  attention_grid(s, d, sp, &g, &c);
  *splits = sp;
  *ctas = g;
  *cluster = c;
  return CONFKV_OK;
}

// Launch shape for the current bounds (the pinned one while steps are reserved).
static int plan_attention(const confkv_ctx* ctx, int* splits_out, int* max_tokens_out) {
  if (ctx->pin_left > 0) {
    *splits_out = ctx->pin_splits;
    *max_tokens_out = ctx->pin_max_tokens;
    return CONFKV_OK;
  }
  return plan_attention_for(ctx, ctx->n8_bound, splits_out, max_tokens_out);
}

// Checks of one step taken with host bounds (steps, n_bound, n8_bound) and the
// bounds after it: worst cases, decided on the host before anything launches.
static int step_bounds(const confkv_ctx* ctx, long long steps, long long n_bound, long long n8_bound,
                       long long* n_after, long long* n8_after) {
  const Shape& s = ctx->s;
  const long long k_bound = std::max(0LL, n_bound - ctx->minN);
  *n_after = std::min<long long>(n_bound, ctx->maxN) + 1;
  // a token leaves the FP16 window this step only if position t - W >= 0 for
  // some sequence; otherwise the INT8 region cannot grow
  long long t_max = 0;
  for (int b = 0; b < s.B; ++b) t_max = std::max<long long>(t_max, (long long)ctx->T0[b] + steps);
  const long long req_bound = t_max - s.W >= 0 ? 1 : 0;
  *n8_after = std::min(n8_bound + req_bound, *n_after - 1);
  if (k_bound > s.max_evict) return CONFKV_ECAPACITY;
  if (*n8_after > s.cap) return CONFKV_ECAPACITY;
  // positions stay in int32
  if (t_max >= (1LL << 31) - 1) return CONFKV_ECAPACITY;
  return CONFKV_OK;
}

int confkv_attention_plan(confkv_ctx* ctx, int32_t* splits, int32_t* smem_bytes) {
  if (!ctx || !splits || !smem_bytes) return CONFKV_EINVAL;
  int sp = 0, mt = 0;
  const int r = plan_attention(ctx, &sp, &mt);
  if (r != CONFKV_OK) return r;
  *splits = sp;
  *smem_bytes = attention_smem_bytes(ctx->s, sp, mt);
  return CONFKV_OK;
}

int confkv_set_step_mode(confkv_ctx* ctx, int32_t mode) {
  if (!ctx || (mode != CONFKV_STEP_AUTO && mode != CONFKV_STEP_SEPARATE)) return CONFKV_EINVAL;
  ctx->fused_ok = mode == CONFKV_STEP_AUTO;
  return CONFKV_OK;
}

int confkv_step_launches(confkv_ctx* ctx, int32_t* launches) {
  if (!ctx || !launches) return CONFKV_EINVAL;
  int splits = 0, max_tokens = 0;
  const int r = plan_attention(ctx, &splits, &max_tokens);
  if (r != CONFKV_OK) return r;
  *launches = ctx->fused_ok && fused_step_fits(ctx->s, ctx->d, splits, max_tokens) ? 1 : 3;
  return CONFKV_OK;
}

int confkv_set_attention_ctas(confkv_ctx* ctx, int32_t ctas) {
  if (!ctx || ctas < 0) return CONFKV_EINVAL;
  ctx->d.attn_ctas = ctas;
  return CONFKV_OK;
}

int confkv_attention_grid(confkv_ctx* ctx, int32_t* ctas, int32_t* cluster) {
  if (!ctx || !ctas || !cluster) return CONFKV_EINVAL;
  int sp = 0, mt = 0;
  const int r = plan_attention(ctx, &sp, &mt);
  if (r != CONFKV_OK) return r;
  int g = 0, c = 0;
  attention_grid(ctx->s, ctx->d, sp, &g, &c);
  *ctas = g;
  *cluster = c;
  return CONFKV_OK;
}

static int step_impl(confkv_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                     const float* logits, float* out, int32_t* budget, float* confidence,
                     int32_t* evicted_pos, int32_t* n_evicted, void* stream, cudaEvent_t after_attention,
                     cudaEvent_t before_attention = nullptr, bool conf_in_attention = false);

int confkv_step(confkv_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                const float* logits, float* out, int32_t* budget, float* confidence,
                int32_t* evicted_pos, int32_t* n_evicted, void* stream) {
  return step_impl(ctx, q, k_new, v_new, logits, out, budget, confidence, evicted_pos, n_evicted, stream,
                   nullptr);
}

// after_attention: recorded on `stream` once the attention kernel (the last
// writer of `out`) has been launched, when not null; before_attention: waited
// for on `stream` before the attention kernel is launched, when not null;
// conf_in_attention: reduce the logits to confidence partials in the
// persistent attention kernel rather than in the prestep kernel (logits in
// host memory: their transfer then overlaps the attention).
static int step_impl(confkv_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                     const float* logits, float* out, int32_t* budget, float* confidence,
                     int32_t* evicted_pos, int32_t* n_evicted, void* stream, cudaEvent_t after_attention,
                     cudaEvent_t before_attention, bool conf_in_attention) {
  if (!ctx) return CONFKV_EINVAL;
  if (!ctx->prefilled) return CONFKV_ESTATE;
  if (!q || !k_new || !v_new || !logits || !out || !budget || !evicted_pos || !n_evicted)
    return CONFKV_EINVAL;
  if (!step_args_aligned(q, k_new, v_new, logits, out, budget, confidence, evicted_pos, n_evicted))
    return CONFKV_EINVAL;
  const Shape& s = ctx->s;
  cudaStream_t st = as_stream(stream);
  // Under stream capture nothing runs now: the launches go into a graph
  // whose replays the caller accounts for with confkv_graph_advance, inside
  // a reservation made with confkv_graph_reserve.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return CONFKV_ECUDA;
  const bool capturing = cs != cudaStreamCaptureStatusNone;
  if (capturing && ctx->pin_left <= 0) return CONFKV_ESTATE;
  long long n_after = 0, n8_after = 0;
  int r = step_bounds(ctx, ctx->steps, ctx->n_bound, ctx->n8_bound, &n_after, &n8_after);
  if (r != CONFKV_OK) return r;
  int splits = 0, max_tokens = 0;
  r = plan_attention(ctx, &splits, &max_tokens);
  if (r != CONFKV_OK) return r;

  const bool prof = !capturing && ctx->prof_on && ctx->prof_count < ctx->prof_max &&
                    (ctx->prof_tick++ % ctx->prof_every) == 0;
  cudaEvent_t* ev = prof ? &ctx->ev[4 * ctx->prof_count] : nullptr;
  if (prof) cudaEventRecord(ev[0], st);
  // inside a graph reservation every step (captured or not) takes its index
  // from the device counter, which the reservation set and each step advances
  const long long step_arg = (capturing || ctx->pin_left > 0) ? -1 : ctx->steps;
  const bool attn_conf = conf_in_attention && splits == 1;
  // Small shapes: the whole step in one launch (attention.cu, fused mode),
  // when every unit and vocabulary chunk gets a CTA of its own in one wave.
  if (!conf_in_attention && !before_attention && ctx->fused_ok && fused_step_fits(s, ctx->d, splits, max_tokens)) {
    if (prof) cudaEventRecord(ev[1], st);
    if (launch_fused_step(s, ctx->d, step_arg, q, k_new, v_new, logits, out, budget, confidence, evicted_pos,
                          n_evicted, max_tokens, st) != 0)
      return CONFKV_ECUDA;
    if (prof) {
      cudaEventRecord(ev[2], st);
      cudaEventRecord(ev[3], st);
      ctx->prof_count++;
    }
    if (after_attention && cudaEventRecord(after_attention, st) != cudaSuccess) return CONFKV_ECUDA;
    if (!capturing) {
      ctx->launches += 1;
      ctx->steps++;
      ctx->n_bound = n_after;
      ctx->n8_bound = n8_after;
      if (ctx->pin_left > 0) ctx->pin_left--;
    }
    return CONFKV_OK;
  }
  if (launch_prestep(s, ctx->d, step_arg, logits, k_new, v_new, !attn_conf, st) != 0) return CONFKV_ECUDA;
  if (prof) cudaEventRecord(ev[1], st);
  if (before_attention && cudaStreamWaitEvent(st, before_attention, 0) != cudaSuccess) return CONFKV_ECUDA;
  if (launch_attention(s, ctx->d, q, out, budget, confidence, attn_conf ? logits : nullptr, splits,
                       max_tokens, st) != 0)
    return CONFKV_ECUDA;
  if (prof) cudaEventRecord(ev[2], st);
  if (after_attention && cudaEventRecord(after_attention, st) != cudaSuccess) return CONFKV_ECUDA;
  if (launch_select(s, ctx->d, step_arg, evicted_pos, n_evicted, st) != 0) return CONFKV_ECUDA;
  if (!capturing) ctx->launches += 3;
  if (prof) {
    cudaEventRecord(ev[3], st);
    ctx->prof_count++;
  }
  if (!capturing) {
    ctx->steps++;
    ctx->n_bound = n_after;
    ctx->n8_bound = n8_after;
    if (ctx->pin_left > 0) ctx->pin_left--;
  }
  return CONFKV_OK;
}

int confkv_graph_reserve(confkv_ctx* ctx, int64_t steps) {
  if (!ctx || steps < 1) return CONFKV_EINVAL;
  if (!ctx->prefilled) return CONFKV_ESTATE;
  long long n_bound = ctx->n_bound, n8_bound = ctx->n8_bound, n8_max = n8_bound;
  for (long long i = 0; i < steps; ++i) {
    long long na = 0, n8a = 0;
    const int r = step_bounds(ctx, ctx->steps + i, n_bound, n8_bound, &na, &n8a);
    if (r != CONFKV_OK) return r;
    n8_max = std::max(n8_max, n8_bound);
    n_bound = na;
    n8_bound = n8a;
  }
  int splits = 0, max_tokens = 0;
  const int r = plan_attention_for(ctx, n8_max, &splits, &max_tokens);
  if (r != CONFKV_OK) return r;
  // the device step counter starts from the host's count (steps outside a
  // reservation pass their index as an argument and leave it alone)
  if (cudaMemcpy(ctx->d.step_dev, &ctx->steps, sizeof(long long), cudaMemcpyHostToDevice) != cudaSuccess)
    return CONFKV_ECUDA;
  ctx->pin_left = steps;
  ctx->pin_splits = splits;
  ctx->pin_max_tokens = max_tokens;
  return CONFKV_OK;
}

int confkv_graph_advance(confkv_ctx* ctx, int64_t steps) {
  if (!ctx || steps < 0) return CONFKV_EINVAL;
  if (steps > ctx->pin_left) return CONFKV_ESTATE;
  for (long long i = 0; i < steps; ++i) {
    long long na = 0, n8a = 0;
    const int r = step_bounds(ctx, ctx->steps, ctx->n_bound, ctx->n8_bound, &na, &n8a);
    if (r != CONFKV_OK) return r;   // cannot happen inside a reservation
    ctx->steps++;
    ctx->n_bound = na;
    ctx->n8_bound = n8a;
  }
  ctx->pin_left -= steps;
  return CONFKV_OK;
}

int confkv_selftest_timeout(confkv_ctx* ctx, void* stream) {
  if (!ctx) return CONFKV_EINVAL;
  return launch_selftest_timeout(ctx->d, as_stream(stream)) == 0 ? CONFKV_OK : CONFKV_ECUDA;
}

int confkv_graph_release(confkv_ctx* ctx) {
  if (!ctx) return CONFKV_EINVAL;
  ctx->pin_left = 0;
  return CONFKV_OK;
}

// Device address of page-locked host memory, if `p` lies in such memory (an
// allocation of cudaHostAlloc / cudaMallocHost or a cudaHostRegister range)
// and the device can address it; false for pageable or device memory.
static bool device_view(const void* p, void** dev) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return false;
  *dev = a.devicePointer;
  return true;
}

int confkv_step_host(confkv_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                     const float* logits, float* out, int32_t* budget, float* confidence,
                     int32_t* evicted_pos, int32_t* n_evicted, void* stream) {
  if (!ctx) return CONFKV_EINVAL;
  if (!q || !k_new || !v_new || !logits || !out || !budget || !evicted_pos || !n_evicted)
    return CONFKV_EINVAL;
  const Shape& s = ctx->s;
  const Staging& g = ctx->st;
  cudaStream_t st = as_stream(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return CONFKV_ECUDA;
  if (cs != cudaStreamCaptureStatusNone) return CONFKV_ESTATE;   // host copies stay outside graphs
  const size_t lbs = (size_t)s.L * s.B;
  const size_t nq = lbs * s.Hq * s.D * 2, nkv = lbs * s.Hkv * s.D * 2;
  if (!ctx->aux) {
    if (cudaStreamCreateWithFlags(&ctx->aux, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ctx->ev_attn, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ctx->ev_aux, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ctx->ev_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ctx->ev_q, cudaEventDisableTiming) != cudaSuccess)
      return CONFKV_ECUDA;
  }
  // Mapped mode: when every buffer but q is page-locked host memory that the
  // device can address, the kernels read logits and the new K/V and write
  // every output in place over the host link, and only q (read by the bulk
  // copies of the attention kernel) is staged, on the second stream while
  // the first kernel runs.
  void *mk = nullptr, *mv = nullptr, *ml = nullptr, *mo = nullptr, *mb = nullptr, *mc = nullptr,
       *me = nullptr, *mn = nullptr;
  const bool mapped = device_view(k_new, &mk) && device_view(v_new, &mv) && device_view(logits, &ml) &&
                      device_view(out, &mo) && device_view(budget, &mb) &&
                      (!confidence || device_view(confidence, &mc)) && device_view(evicted_pos, &me) &&
                      device_view(n_evicted, &mn) &&
                      step_args_aligned(ctx->st.q, mk, mv, static_cast<const float*>(ml),
                                        static_cast<const float*>(mo), static_cast<const int32_t*>(mb),
                                        confidence ? static_cast<const float*>(mc) : nullptr,
                                        static_cast<const int32_t*>(me), static_cast<const int32_t*>(mn));
  if (mapped) {
    cudaError_t e = cudaEventRecord(ctx->ev_in, st);   // g.q is free once earlier work on `stream` is
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->aux, ctx->ev_in, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(g.q, q, nq, cudaMemcpyHostToDevice, ctx->aux);
    if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_q, ctx->aux);
    if (e != cudaSuccess) return CONFKV_ECUDA;
    const int r = step_impl(ctx, g.q, mk, mv, static_cast<const float*>(ml), static_cast<float*>(mo),
                            static_cast<int32_t*>(mb), confidence ? static_cast<float*>(mc) : nullptr,
                            static_cast<int32_t*>(me), static_cast<int32_t*>(mn), stream, nullptr, ctx->ev_q,
                            true);
    if (r != CONFKV_OK) return r;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    long long written = 0;
    for (size_t i = 0; i < lbs; ++i) written += n_evicted[i] > 0 ? n_evicted[i] : 0;
    ctx->host_h2d = (long long)(nq + 2 * nkv + (size_t)s.B * s.V * 4);
    ctx->host_d2h = (long long)(lbs * s.Hq * s.D * 4 + lbs * 4 + (confidence ? (size_t)s.B * 4 : 0) +
                                (size_t)written * 4 + lbs * 4);
    return CONFKV_OK;
  }
  cudaError_t e = cudaMemcpyAsync(g.q, q, nq, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(g.k_new, k_new, nkv, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(g.v_new, v_new, nkv, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(g.logits, logits, (size_t)s.B * s.V * 4, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return CONFKV_ECUDA;
  // no row of evicted positions can hold more than this step's eviction bound
  const long long k_bound =
      std::min<long long>(s.max_evict, std::max(0LL, ctx->n_bound - ctx->minN));
  const int r = step_impl(ctx, g.q, g.k_new, g.v_new, g.logits, g.out, g.budget,
                          confidence ? g.conf : nullptr, g.evicted, g.nevict, stream, ctx->ev_attn);
  if (r != CONFKV_OK) return r;
  // the attention output is final once the attention kernel is done: copy it
  // back on the second stream while the select kernel runs
  e = cudaStreamWaitEvent(ctx->aux, ctx->ev_attn, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out, g.out, lbs * s.Hq * s.D * 4, cudaMemcpyDeviceToHost, ctx->aux);
  if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_aux, ctx->aux);
  if (e == cudaSuccess) e = cudaMemcpyAsync(budget, g.budget, lbs * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && confidence)
    e = cudaMemcpyAsync(confidence, g.conf, (size_t)s.B * 4, cudaMemcpyDeviceToHost, st);
  // the first k_bound entries of every row: the rest is never written
  if (e == cudaSuccess && k_bound > 0)
    e = cudaMemcpy2DAsync(evicted_pos, (size_t)s.max_evict * 4, g.evicted, (size_t)s.max_evict * 4,
                          (size_t)k_bound * 4, lbs, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(n_evicted, g.nevict, lbs * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ctx->ev_aux, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  ctx->host_h2d = (long long)(nq + 2 * nkv + (size_t)s.B * s.V * 4);
  ctx->host_d2h = (long long)(lbs * s.Hq * s.D * 4 + lbs * 4 + (confidence ? (size_t)s.B * 4 : 0) +
                              lbs * (size_t)k_bound * 4 + lbs * 4);
  return cuda_status(e);
}

// ------------------------------------------------------------------ export / import

static int copy_unit_raw(confkv_ctx* ctx, int b, int l, std::vector<uint8_t>& k8, std::vector<uint8_t>& v8,
                         std::vector<uint16_t>& k16, std::vector<uint16_t>& v16, std::vector<int32_t>& pos,
                         std::vector<float>& ema, std::vector<float>& sK, std::vector<float>& sV, int32_t& n8,
                         cudaStream_t st) {
  const Shape& s = ctx->s;
  const int D = s.D;
  k8.resize((size_t)s.Hkv * s.cstride * D);
  v8.resize(k8.size());
  k16.resize((size_t)s.Hkv * s.WR * D);
  v16.resize(k16.size());
  pos.resize(s.S);
  ema.resize(s.S);
  sK.resize((size_t)s.Hkv * D);
  sV.resize(sK.size());
  const size_t u0 = unit_index(s, l, b, 0), lb = lb_index(s, l, b);
  cudaError_t e = cudaMemcpyAsync(k8.data(), ctx->d.k8 + u0 * s.cstride * D, k8.size(), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v8.data(), ctx->d.v8 + u0 * s.cstride * D, v8.size(), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(k16.data(), ctx->d.k16 + u0 * s.WR * D, k16.size() * 2, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v16.data(), ctx->d.v16 + u0 * s.WR * D, v16.size() * 2, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(pos.data(), ctx->d.pos + lb * s.S, s.S * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ema.data(), ctx->d.ema + lb * s.S, s.S * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(sK.data(), ctx->d.sK + u0 * D, sK.size() * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(sV.data(), ctx->d.sV + u0 * D, sV.size() * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&n8, ctx->d.n8 + lb, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(e);
}

int confkv_export_unit(confkv_ctx* ctx, int32_t b, int32_t l, confkv_unit_host* o, void* stream) {
  if (!ctx || !o || b < 0 || l < 0 || b >= ctx->s.B || l >= ctx->s.L) return CONFKV_EINVAL;
  if (!o->pos8 || !o->ema8 || !o->k8 || !o->v8 || !o->posR || !o->emaR || !o->k16 || !o->v16 ||
      !o->sK || !o->sV)
    return CONFKV_EINVAL;
  const Shape& s = ctx->s;
  const int D = s.D, Hkv = s.Hkv;
  std::vector<uint8_t> k8, v8;
  std::vector<uint16_t> k16, v16;
  std::vector<int32_t> pos;
  std::vector<float> ema, sK, sV;
  int32_t n8 = 0;
  const int r = copy_unit_raw(ctx, b, l, k8, v8, k16, v16, pos, ema, sK, sV, n8, as_stream(stream));
  if (r != CONFKV_OK) return r;
  o->n8 = n8;
  for (int i = 0; i < n8; ++i) {
    o->pos8[i] = pos[i];
    o->ema8[i] = ema[i];
    for (int h = 0; h < Hkv; ++h) {
      const size_t blk = ((size_t)h * s.cstride + (i & ~15)) * D;
      for (int c = 0; c < D; ++c) {
        o->k8[((size_t)i * Hkv + h) * D + c] = (int8_t)((int)k8[blk + k8_offset(D, i & 15, c)] - kCodeBias);
        o->v8[((size_t)i * Hkv + h) * D + c] = (int8_t)((int)v8[blk + v8_offset(D, i & 15, c)] - kCodeBias);
      }
    }
  }
  int nR = 0;
  for (int rs = 0; rs < s.WR; ++rs) {
    const int p = pos[s.cap + rs];
    if (p < 0) continue;
    o->posR[nR] = p;
    o->emaR[nR] = ema[s.cap + rs];
    for (int h = 0; h < Hkv; ++h) {
      const size_t blk = ((size_t)h * s.WR + (rs & ~15)) * D;   // in halves
      for (int c = 0; c < D; ++c) {
        o->k16[((size_t)nR * Hkv + h) * D + c] = k16[blk + k16_offset(D, rs & 15, c) / 2];
        o->v16[((size_t)nR * Hkv + h) * D + c] = v16[blk + v16_offset(D, rs & 15, c) / 2];
      }
    }
    ++nR;
  }
  o->nR = nR;
  for (int i = 0; i < Hkv * D; ++i) {
    o->sK[i] = sK[i];
    o->sV[i] = sV[i];
  }
  return CONFKV_OK;
}

int confkv_import_unit(confkv_ctx* ctx, int32_t b, int32_t l, const confkv_unit_host* in,
                       void* stream) {
  if (!ctx || !in || b < 0 || l < 0 || b >= ctx->s.B || l >= ctx->s.L) return CONFKV_EINVAL;
  const Shape& s = ctx->s;
  const int D = s.D, Hkv = s.Hkv;
  if (in->n8 < 0 || in->n8 > s.cap || in->nR < 0 || in->nR > s.WR) return CONFKV_EINVAL;
  if ((in->n8 && (!in->pos8 || !in->ema8 || !in->k8 || !in->v8)) ||
      (in->nR && (!in->posR || !in->emaR || !in->k16 || !in->v16)) || !in->sK || !in->sV)
    return CONFKV_EINVAL;
  std::vector<uint8_t> k8((size_t)Hkv * s.cstride * D, kCodeBias), v8(k8.size(), kCodeBias);
  std::vector<uint16_t> k16((size_t)Hkv * s.WR * D, 0), v16(k16.size(), 0);
  std::vector<int32_t> pos(s.S, -1);
  std::vector<float> ema(s.S, 0.f);
  for (int i = 0; i < in->n8; ++i) {
    if (in->pos8[i] < 0) return CONFKV_EINVAL;
    pos[i] = in->pos8[i];
    ema[i] = in->ema8[i];
    for (int h = 0; h < Hkv; ++h) {
      const size_t blk = ((size_t)h * s.cstride + (i & ~15)) * D;
      for (int c = 0; c < D; ++c) {
        const int ck = in->k8[((size_t)i * Hkv + h) * D + c], cv = in->v8[((size_t)i * Hkv + h) * D + c];
        if (ck < -127 || cv < -127) return CONFKV_EINVAL;   // codes are symmetric
        k8[blk + k8_offset(D, i & 15, c)] = (uint8_t)(ck + kCodeBias);
        v8[blk + v8_offset(D, i & 15, c)] = (uint8_t)(cv + kCodeBias);
      }
    }
  }
  for (int j = 0; j < in->nR; ++j) {
    const int p = in->posR[j];
    if (p < 0) return CONFKV_EINVAL;
    const int rs = p % s.WR;
    if (pos[s.cap + rs] >= 0) return CONFKV_EINVAL;   // two entries in one ring slot
    pos[s.cap + rs] = p;
    ema[s.cap + rs] = in->emaR[j];
    for (int h = 0; h < Hkv; ++h) {
      const size_t blk = ((size_t)h * s.WR + (rs & ~15)) * D;
      for (int c = 0; c < D; ++c) {
        k16[blk + k16_offset(D, rs & 15, c) / 2] = in->k16[((size_t)j * Hkv + h) * D + c];
        v16[blk + v16_offset(D, rs & 15, c) / 2] = in->v16[((size_t)j * Hkv + h) * D + c];
      }
    }
  }
  cudaStream_t st = as_stream(stream);
  const size_t u0 = unit_index(s, l, b, 0), lb = lb_index(s, l, b);
  int32_t n8 = in->n8;
  cudaError_t e = cudaMemcpyAsync(ctx->d.k8 + u0 * s.cstride * D, k8.data(), k8.size(), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.v8 + u0 * s.cstride * D, v8.data(), v8.size(), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.k16 + u0 * s.WR * D, k16.data(), k16.size() * 2, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.v16 + u0 * s.WR * D, v16.data(), v16.size() * 2, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.pos + lb * s.S, pos.data(), s.S * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.ema + lb * s.S, ema.data(), s.S * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.sK + u0 * D, in->sK, (size_t)Hkv * D * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.sV + u0 * D, in->sV, (size_t)Hkv * D * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->d.n8 + lb, &n8, 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return CONFKV_ECUDA;
  ctx->prefilled = true;
  ctx->pin_left = 0;   // bounds may have grown: a pinned plan no longer holds
  ctx->n_bound = std::max<long long>(ctx->n_bound, (long long)in->n8 + in->nR);
  ctx->n8_bound = std::max<long long>(ctx->n8_bound, in->n8);
  return CONFKV_OK;
}

int confkv_get_clock(confkv_ctx* ctx, int32_t* prefill_len, int64_t* steps) {
  if (!ctx || !prefill_len || !steps) return CONFKV_EINVAL;
  for (int b = 0; b < ctx->s.B; ++b) prefill_len[b] = ctx->T0[b];
  *steps = ctx->steps;
  return CONFKV_OK;
}

int confkv_set_clock(confkv_ctx* ctx, const int32_t* prefill_len, int64_t steps, void* stream) {
  if (!ctx || !prefill_len || steps < 0) return CONFKV_EINVAL;
  for (int b = 0; b < ctx->s.B; ++b)
    if (prefill_len[b] < 0) return CONFKV_EINVAL;
  ctx->T0.assign(prefill_len, prefill_len + ctx->s.B);
  ctx->steps = steps;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(ctx->d.T0, ctx->T0.data(), ctx->s.B * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ctx->d.step_dev, &ctx->steps, sizeof(long long), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(e);
}

// ------------------------------------------------------------------ stats / profiling

int confkv_get_stats(confkv_ctx* ctx, confkv_stats* out, void* stream) {
  if (!ctx || !out) return CONFKV_EINVAL;
  const Shape& s = ctx->s;
  cudaStream_t st = as_stream(stream);
  DevStats ds{};
  int32_t status = 0;
  const size_t lbs = (size_t)s.L * s.B;
  std::vector<int32_t> n8(lbs), pos(lbs * s.S);
  cudaError_t e = cudaMemcpyAsync(&ds, ctx->d.stats, sizeof(ds), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&status, ctx->d.status, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(n8.data(), ctx->d.n8, lbs * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(pos.data(), ctx->d.pos, pos.size() * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return CONFKV_ECUDA;
  long long res = 0, res_bytes = 0;
  for (size_t i = 0; i < lbs; ++i) {
    long long nr = 0;
    for (int rs = 0; rs < s.WR; ++rs) nr += pos[i * s.S + s.cap + rs] >= 0;
    res += n8[i] + nr;
    res_bytes += (long long)s.Hkv * s.D * (2LL * n8[i] + 4LL * nr);
  }
  out->steps = (int64_t)ds.steps;
  out->evicted = (int64_t)ds.evicted;
  out->moved = (int64_t)ds.moved;
  out->requantised = (int64_t)ds.requant;
  out->attn_bytes = (double)ds.attn_bytes;
  out->step_bytes = (double)ds.step_bytes;
  out->resident = res;
  out->resident_bytes = res_bytes;
  out->device_status = status;
  out->host_h2d_bytes = ctx->host_h2d;
  out->host_d2h_bytes = ctx->host_d2h;
  // the latest step's footprint is still in its accumulators (the next
  // step folds it on the device)
  const int last = (int)((ctx->steps + 1) & 1);
  out->peak_resident = (int64_t)std::max(ds.peak_entries, ctx->steps > 0 ? ds.res_entries_acc[last] : 0ull);
  out->peak_resident_bytes = (int64_t)std::max(ds.peak_bytes, ctx->steps > 0 ? ds.res_bytes_acc[last] : 0ull);
  out->workspace_bytes = (int64_t)ctx->ws_bytes;
  out->launches = ctx->launches;
  return status ? CONFKV_EDEVICE : CONFKV_OK;
}

int confkv_profile_enable(confkv_ctx* ctx, int32_t max_steps, int32_t every) {
  if (!ctx || max_steps < 1 || every < 1) return CONFKV_EINVAL;
  ctx->prof_every = every;
  ctx->prof_tick = 0;
  for (cudaEvent_t e : ctx->ev) cudaEventDestroy(e);
  ctx->ev.assign(4 * (size_t)max_steps, nullptr);
  for (auto& e : ctx->ev)
    if (cudaEventCreate(&e) != cudaSuccess) return CONFKV_ECUDA;
  ctx->prof_max = max_steps;
  ctx->prof_count = 0;
  ctx->prof_on = true;
  return CONFKV_OK;
}

int confkv_profile_disable(confkv_ctx* ctx) {
  if (!ctx) return CONFKV_EINVAL;
  ctx->prof_on = false;
  return CONFKV_OK;
}

int confkv_profile_read(confkv_ctx* ctx, double* ms_prestep, double* ms_attention, double* ms_select,
                        int32_t* steps) {
  if (!ctx || !ms_prestep || !ms_attention || !ms_select || !steps) return CONFKV_EINVAL;
  double a = 0, b = 0, c = 0;
  for (int i = 0; i < ctx->prof_count; ++i) {
    cudaEvent_t* e = &ctx->ev[4 * i];
    if (cudaEventSynchronize(e[3]) != cudaSuccess) return CONFKV_ECUDA;
    float x = 0, y = 0, z = 0;
    cudaEventElapsedTime(&x, e[0], e[1]);
    cudaEventElapsedTime(&y, e[1], e[2]);
    cudaEventElapsedTime(&z, e[2], e[3]);
    a += x; b += y; c += z;
  }
  *ms_prestep = a;
  *ms_attention = b;
  *ms_select = c;
  *steps = ctx->prof_count;
  ctx->prof_count = 0;
  return CONFKV_OK;
}

int32_t confkv_block_offset(int32_t kind, int32_t d, int32_t tau, int32_t c) {
  if ((d != 64 && d != 128) || tau < 0 || tau > 15 || c < 0 || c >= d) return -1;
  switch (kind) {
    case 0: return k8_offset(d, tau, c);
    case 1: return v8_offset(d, tau, c);
    case 2: return k16_offset(d, tau, c);
    case 3: return v16_offset(d, tau, c);
    default: return -1;
  }
}

const char* confkv_status_string(int status) {
  switch (status) {
    case CONFKV_OK: return "ok";
    case CONFKV_EINVAL: return "invalid argument or configuration";
    case CONFKV_ECAPACITY: return "capacity exceeded";
    case CONFKV_ECUDA: return "CUDA runtime error";
    case CONFKV_ETIMEOUT: return "bounded device wait timed out";
    case CONFKV_ENOTIMPL: return "not implemented for this shape";
    case CONFKV_EDEVICE: return "device status word reports an error";
    case CONFKV_ESTATE: return "call out of order";
    default: return "unknown status";
  }
}

int32_t confkv_version(void) { return 100; }

}  // extern "C"
