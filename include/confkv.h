/*
 * confkv.h -- C ABI of the CONF-KV per-decode-step cache manager for one
 * NVIDIA GB300 (sm_103a).
 *
 * The method: CONF-KV, "Confidence-Aware KV Cache Eviction with
 * Mixed-Precision Storage for Long-Horizon LLM".  Citations name the page and
 * the section they come from:
 *   [rainbus]  paper.rainbus.top/paper/2605.24786 -- sections 核心方法 (core
 *              method), 方法步骤详情 (Algorithm 1, steps 1-13), 前置知识
 *              (prerequisites: EMA, blockwise online softmax), 复现评估
 *              (reproducibility: hyper-parameters).
 *   [gist-de]  gist.science/de/paper/2605.24786 -- Technischer
 *              Zusammenfassung, Methodik: Konfidenzschätzung, Adaptive
 *              Budgetauswahl, Token-Ranking und Eviktion, Systemintegration.
 *
 * Conventions
 *   - Every function returns a status: CONFKV_OK (0) or a negative code below.
 *     Nothing aborts, traps or exits the process.
 *   - All tensor arguments of confkv_prefill / confkv_step are DEVICE
 *     pointers owned by the caller; the library reads inputs and writes
 *     outputs and keeps no reference after the call returns.  The only device
 *     memory the library uses is the caller-allocated workspace (see
 *     confkv_workspace_bytes); it never calls cudaMalloc itself.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued on it and the call returns without
 *     synchronising, except where a function says it synchronises.
 *   - Device-side anomalies (an INT8 region that would overflow, an
 *     inconsistent eviction count) set bits of a device status word; they are
 *     reported as CONFKV_EDEVICE by the next confkv_get_stats.
 *   - Layouts are row-major, outermost index first.  L layers, B sequences,
 *     Hq query heads, Hkv KV heads, d head dim (64 or 128), V vocabulary.
 */
#ifndef CONFKV_H
#define CONFKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CONFKV_OK 0
#define CONFKV_EINVAL (-1)     /* bad argument or configuration */
#define CONFKV_ECAPACITY (-2)  /* a cache region or output buffer is too small */
#define CONFKV_ECUDA (-3)      /* a CUDA runtime call failed */
#define CONFKV_ETIMEOUT (-4)   /* a bounded device wait gave up */
#define CONFKV_ENOTIMPL (-5)   /* shape not supported by the compiled kernels */
#define CONFKV_EDEVICE (-6)    /* the device status word reports an error */
#define CONFKV_ESTATE (-7)     /* call out of order (e.g. step before prefill) */

#define CONFKV_Q_FP16 0
#define CONFKV_Q_BF16 1

/*
 * Configuration.  Defaults on the pages: w = (0.4, 0.3, 0.3) and tau = 0.7
 * ([gist-de] Konfidenzschätzung; [rainbus] 核心方法), alpha = 0.65
 * ([rainbus] 核心方法), lambda = 0.9 ([rainbus] 前置知识, EMA), P = 32 or 64,
 * W = 128 ([rainbus] 复现评估).
 */
typedef struct confkv_config {
  int32_t L, Hq, Hkv, d, V;   /* layers, query heads, KV heads, head dim, vocab */
  int32_t B;                  /* sequences stepped together */
  int32_t cap;                /* INT8 slots per (layer, sequence): must hold the
                                 prefill older than W and every budget + 1;
                                 rounded up to a multiple of 16 */
  int32_t W;                  /* FP16 window: the newest W tokens stay FP16 */
  int32_t P;                  /* protected window: the newest P tokens are never
                                 evicted ([gist-de] Token-Ranking und Eviktion) */
  int32_t q_dtype;            /* CONFKV_Q_FP16 or CONFKV_Q_BF16 */
  int32_t max_evict;          /* rows of evicted_pos per (layer, sequence);
                                 0 selects cap + W + 16 */
  double tau;                 /* budget threshold: N = n_high if c >= tau */
  double w_H, w_m, w_p;       /* confidence weights */
  float alpha;                /* rank weight of the EMA mass */
  float lam;                  /* EMA decay */
  const int32_t* n_high;      /* host [L]: tight budget per layer (c >= tau) */
  const int32_t* n_low;       /* host [L]: loose budget per layer (c < tau);
                                 per-layer values give the pyramidal variant
                                 ([gist-de] Systemintegration) */
  int32_t compaction;         /* CONFKV_COMPACT_TAIL_FILL (0, default): each
                                 evicted INT8 slot below the new length takes a
                                 survivor from above it (at most k moves);
                                 CONFKV_COMPACT_ORDERED (1): survivors keep
                                 position order (every survivor above the first
                                 hole moves), the contiguous compaction of
                                 [gist-de] Systemintegration, kept as an
                                 ablation of the layout */
} confkv_config;

enum { CONFKV_COMPACT_TAIL_FILL = 0, CONFKV_COMPACT_ORDERED = 1 };

typedef struct confkv_ctx confkv_ctx;

/* Bytes of device workspace the context needs (state + scratch).  Returns
 * CONFKV_EINVAL for an invalid configuration: d not 64/128, Hq % Hkv != 0,
 * Hq / Hkv > 8, V < 2 or V > 4096 * 1024, some budget < P or < 1, cap < 16,
 * W < 1, compaction not 0 or 1. */
int confkv_workspace_bytes(const confkv_config* cfg, size_t* bytes);

/* Create a context over `workspace` (device memory, >= the size above, 256-byte
 * aligned, owned by the caller and kept alive until confkv_destroy).  The
 * context copies the configuration, including n_high / n_low.  Synchronous. */
int confkv_create(const confkv_config* cfg, void* workspace, size_t workspace_bytes,
                  confkv_ctx** out);

/* Free the host-side context (the workspace stays the caller's). */
void confkv_destroy(confkv_ctx* ctx);

/*
 * Ingest the prefill and reset the cache.  k, v: device fp16
 * [L][B][Hkv][t_max][d]; sequence b uses its first prefill_len[b] tokens
 * (prefill_len is a HOST array of B values, 0 <= prefill_len[b] <= t_max).
 * Scales per (layer, sequence, KV head, channel) from the absmax over the
 * prefill: s = absmax / 127 in float32 (1 if the channel is zero).  Positions
 * >= prefill_len - W stay FP16; older positions are stored as INT8 codes
 * clamp(rint(x / s), -127, 127) ([gist-de] Systemintegration; the pages do
 * not describe prefill, this rule follows their per-head per-channel INT8).
 * EMA mass starts at 0.  Returns CONFKV_ECAPACITY if prefill_len - W > cap,
 * CONFKV_EINVAL if k or v is not 2-byte aligned.
 */
int confkv_prefill(confkv_ctx* ctx, const int32_t* prefill_len, const void* k, const void* v,
                   int64_t t_max, void* stream);

/*
 * One decode step for all B sequences: the token at position
 * t_b = prefill_len[b] + (steps done since prefill) ([rainbus] 方法步骤详情,
 * Algorithm 1):
 *   q      [L][B][Hq][d]  fp16 or bf16 (q_dtype): the decode query
 *   k_new  [L][B][Hkv][d] fp16, v_new likewise: the new token's K/V
 *   logits [B][V] fp32: next-token logits (temperature 1)
 * Outputs (device):
 *   out         [L][B][Hq][d] fp32: attention of q over the cache plus the new
 *               token, before any eviction of this step
 *   budget      [B][L] int32: N chosen for (sequence, layer)
 *   confidence  [B] fp32 or NULL: c of each sequence
 *   evicted_pos [L][B][max_evict] int32: absolute positions evicted by this
 *               step, ascending; only the first n_evicted[l][b] entries of a
 *               row are written
 *   n_evicted   [L][B] int32
 * The step computes c = w_H(1 - H/log V) + w_m sigmoid(log p1 - log p2) +
 * w_p p1, N = n_high if c >= tau else n_low, attention with the per-token
 * attention mass averaged over query heads, the EMA a <- lam a + (1 - lam) A,
 * and, if the cache holds more than N entries (the new token not counted),
 * evicts the n - N lowest s = alpha a_hat + (1 - alpha) r_hat among entries
 * older than the newest P, compacts the INT8 region, requantises the entry
 * that leaves the FP16 window and appends the new token.
 * Alignment: q must be 16-byte aligned (the attention kernel copies query
 * rows with bulk copies), k_new and v_new 4-byte aligned (read as 32-bit
 * words), logits, out, budget, confidence, evicted_pos and n_evicted 4-byte
 * aligned; otherwise CONFKV_EINVAL, before anything is launched.  Tensors
 * from a torch allocation or a contiguous slice at a multiple of 8 elements
 * satisfy all of these.
 * Returns CONFKV_ECAPACITY (before launching anything) if the worst case of
 * this step could overflow cap or max_evict.
 */
int confkv_step(confkv_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                const float* logits, float* out, int32_t* budget, float* confidence,
                int32_t* evicted_pos, int32_t* n_evicted, void* stream);

/*
 * confkv_step with HOST buffers (same shapes); returns once the outputs are
 * in the host buffers.  Two modes, chosen per call, with identical results:
 *  - mapped: when k_new, v_new, logits and every output buffer lie in
 *    page-locked host memory the device can address (cudaHostAlloc,
 *    cudaMallocHost or cudaHostRegister), the kernels read those inputs and
 *    write those outputs in place over the host link.  Only q is copied, to
 *    a staging buffer inside the workspace, on a second library-owned
 *    stream (created on the first call) while the first kernel runs.
 *  - staged: otherwise every input is copied to staging buffers inside the
 *    workspace first, and the outputs are copied back (the attention output
 *    on the second stream while the last kernel runs).  Pinned memory makes
 *    these copies asynchronous DMA.
 * Mapped mode also needs k_new and v_new 4-byte aligned and every other
 * buffer but q 4-byte aligned; misaligned pinned buffers take the staged
 * mode.  q has no alignment requirement here (it is always staged).
 * confidence may be NULL.  Of each row of evicted_pos only the first
 * n_evicted entries are meaningful; in mapped mode only those are written,
 * in staged mode as many as the step's worst-case eviction count are copied
 * back.  The rest of the row is untouched.
 */
int confkv_step_host(confkv_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                     const float* logits, float* out, int32_t* budget, float* confidence,
                     int32_t* evicted_pos, int32_t* n_evicted, void* stream);

/* CUDA graphs.  The step index lives in device memory, so the three kernels
 * of a confkv_step captured into a CUDA graph (stream capture on `stream`)
 * replay correctly step after step.  The host still keeps worst-case bounds
 * (capacity, eviction rows, attention launch shape), so replays go inside a
 * reservation:
 *   confkv_graph_reserve(ctx, n)  checks that n more steps fit under the
 *       worst-case bounds and pins one attention launch shape valid for all
 *       of them.  CONFKV_ECAPACITY if they do not fit, CONFKV_ESTATE before
 *       prefill, CONFKV_EINVAL if n < 1.
 *   confkv_step under capture then records a step without running it and
 *       without advancing the host state; under capture without a
 *       reservation it returns CONFKV_ESTATE.  confkv_step_host is never
 *       captured (CONFKV_ESTATE).
 *   confkv_graph_advance(ctx, k)  accounts for k executed replays (k at most
 *       the steps left in the reservation, else CONFKV_ESTATE).  Plain
 *       confkv_step calls inside a reservation use the pinned shape and
 *       count against it as well.
 *   confkv_graph_release(ctx)  drops the reservation (prefill and
 *       confkv_import_unit drop it too).
 * The pages have no counterpart of these calls: they serve callers that put
 * the cache manager into their own decode graph. */
int confkv_graph_reserve(confkv_ctx* ctx, int64_t steps);
/* Self-test of failure detection: launches one CTA that waits on an mbarrier
 * nothing ever arrives on, with the decode kernels' polling loop but a short
 * limit (4096 polls).  The wait runs out and sets the time-out bit
 * (CONFKV_STATUS_TIMEOUT) of the device status word, which the next
 * confkv_get_stats reports as CONFKV_EDEVICE; nothing faults and the context
 * stays usable (confkv_prefill clears the word).  Asynchronous on `stream`.
 * The pages have no counterpart: it tests this library's own bounded waits. */
int confkv_selftest_timeout(confkv_ctx* ctx, void* stream);
int confkv_graph_advance(confkv_ctx* ctx, int64_t steps);
int confkv_graph_release(confkv_ctx* ctx);

/* Cache of one (sequence b, layer l) in a plain host layout.  Caller-owned
 * buffers sized for cap INT8 entries and W + 16 FP16 entries:
 *   pos8[cap], ema8[cap], k8/v8[cap][Hkv][d] int8 codes,
 *   posR[W+16], emaR[W+16], k16/v16[W+16][Hkv][d] fp16 bit patterns,
 *   sK, sV [Hkv][d] fp32 scales.
 * INT8 entries are listed in slot order, FP16 entries in ring-slot order. */
typedef struct confkv_unit_host {
  int32_t n8, nR;
  int32_t* pos8;
  float* ema8;
  int8_t* k8;
  int8_t* v8;
  int32_t* posR;
  float* emaR;
  uint16_t* k16;
  uint16_t* v16;
  float* sK;
  float* sV;
} confkv_unit_host;

/* Copy the cache of (b, l) to host (synchronises `stream`). */
int confkv_export_unit(confkv_ctx* ctx, int32_t b, int32_t l, confkv_unit_host* out, void* stream);

/* Overwrite the cache of (b, l) from host buffers in the export layout
 * (synchronises `stream`).  FP16 entries go to ring slot pos mod (W + 16);
 * two entries must not share a slot.  Used to resume from a checkpoint or to
 * load a crafted state. */
int confkv_import_unit(confkv_ctx* ctx, int32_t b, int32_t l, const confkv_unit_host* in,
                       void* stream);

/* Position clock: prefill_len[B] (host) and the number of steps done since
 * prefill.  confkv_set_clock restores it with a checkpoint. */
int confkv_get_clock(confkv_ctx* ctx, int32_t* prefill_len, int64_t* steps);
int confkv_set_clock(confkv_ctx* ctx, const int32_t* prefill_len, int64_t steps, void* stream);

/* Bits of the device status word (confkv_stats.device_status). */
enum {
  CONFKV_STATUS_CAPACITY = 1,     /* an INT8 region would have overflowed cap */
  CONFKV_STATUS_EVICT_BOUND = 2,  /* more evictions than evicted_pos rows hold */
  CONFKV_STATUS_BAD_COUNT = 4,    /* eviction count differs from n - N */
  CONFKV_STATUS_TIMEOUT = 8       /* a bounded wait inside a kernel gave up */
};

typedef struct confkv_stats {
  int64_t steps;             /* steps since prefill */
  int64_t evicted;           /* entries evicted since prefill */
  int64_t moved;             /* entries moved by compaction */
  int64_t requantised;       /* entries moved from FP16 to INT8 */
  double attn_bytes;         /* algorithmic bytes of the attention kernel, summed */
  double step_bytes;         /* algorithmic bytes of whole steps, summed */
  int64_t resident;          /* cache entries resident now, all units */
  int64_t resident_bytes;    /* K/V bytes resident now at stored widths */
  int32_t device_status;     /* raw device status bits (0 = ok) */
  int64_t host_h2d_bytes;    /* bytes the last confkv_step_host moved host -> device */
  int64_t host_d2h_bytes;    /* bytes the last confkv_step_host moved device -> host */
  int64_t peak_resident;     /* largest `resident` seen at the end of any step since
                                prefill (exact: summed on the device every step) */
  int64_t peak_resident_bytes; /* largest `resident_bytes` at the end of any step
                                since prefill (the pages' peak KV memory, [rainbus]
                                results table) */
  int64_t workspace_bytes;   /* device bytes the context holds: the caller's
                                workspace (the allocator footprint; fixed at create) */
  int64_t launches;          /* kernels this context has launched for decode steps
                                since it was created (host count) */
} confkv_stats;

/* Read the counters and the device status word (synchronises `stream`).
 * Returns CONFKV_EDEVICE if the status word is non-zero. */
int confkv_get_stats(confkv_ctx* ctx, confkv_stats* out, void* stream);

/* Per-kernel timing with CUDA events on the launching stream.  While enabled,
 * every `every`-th confkv_step (the first one included) records events
 * around its three kernels (confidence and append / attention /
 * select-compact-requant); the others run without events, since each event
 * record between kernels costs the stream about two microseconds.
 * confkv_profile_read synchronises and returns the summed milliseconds of
 * each kernel and the number of steps recorded, then clears them.  At most
 * `max_steps` recorded steps are kept.  CONFKV_EINVAL if max_steps < 1 or
 * every < 1. */
int confkv_profile_enable(confkv_ctx* ctx, int32_t max_steps, int32_t every);
int confkv_profile_disable(confkv_ctx* ctx);
int confkv_profile_read(confkv_ctx* ctx, double* ms_prestep, double* ms_attention,
                        double* ms_select, int32_t* steps);

/* Attention launch shape chosen for the next step: CTAs per (layer, sequence,
 * KV head) unit and dynamic shared memory per CTA.  Units go to the split-K
 * kernel (2-8 CTAs per unit in one cluster) only when there are fewer units
 * than persistent CTAs (two per SM) and every CTA of a cluster still streams
 * at least 64 16-token blocks; otherwise each unit runs whole on the
 * persistent kernel (splits = 1).  confkv_launch_plan does the same planning
 * without a context. */
int confkv_attention_plan(confkv_ctx* ctx, int32_t* splits, int32_t* smem_bytes);

/* How confkv_step runs a step on the device (results do not depend on it):
 *   CONFKV_STEP_AUTO (default)  one kernel launch for the whole step when
 *       every (layer, sequence, KV head) unit can have an SM of its own
 *       (one CTA per unit; the SMs left over reduce the vocabulary, or with
 *       none left the units' epilogue warps take one chunk of at most 4096
 *       logits each), the INT8 region of a unit stays within 8192 tokens,
 *       compaction is tail fill, the selection's working set and the
 *       unit's scores fit the kernel's shared memory and the logits are in
 *       device memory; otherwise three launches;
 *   CONFKV_STEP_SEPARATE  always three launches (confidence reduction and
 *       append; attention; selection).
 * The fused launch removes two kernel launches and their gaps from steps of
 * small shapes (the pages' per-step profile, [rainbus] 复现评估, is
 * dominated by such fixed costs there).  confkv_step_launches gives the
 * launches the next step would take.  CONFKV_EINVAL for a null ctx or an
 * unknown mode.  The pages give no counterpart: these are launch controls of
 * this library. */
enum { CONFKV_STEP_AUTO = 0, CONFKV_STEP_SEPARATE = 1 };
int confkv_set_step_mode(confkv_ctx* ctx, int32_t mode);
int confkv_step_launches(confkv_ctx* ctx, int32_t* launches);

/* Caps the attention grid at `ctas` CTAs; 0 (the default) lets the
 * persistent kernel use two CTAs per SM.  The split-K kernel is chosen only
 * while units x splits stays within the cap, otherwise the persistent kernel
 * runs on at most `ctas` CTAs.  A smaller grid leaves SMs to work on other
 * streams, at a proportional cost in attention time.  Takes effect at the
 * next launch (a captured graph keeps the grid it was captured with; steps
 * inside a graph reservation keep the reserved plan).  Results do not depend
 * on it.  The pages give no counterpart: it is a
 * launch-shape control of this library.  CONFKV_EINVAL for a null ctx or a
 * negative count. */
int confkv_set_attention_ctas(confkv_ctx* ctx, int32_t ctas);

/* Grid of the attention launch chosen for the next step: `ctas` CTAs in
 * clusters of `cluster`.  The persistent kernel (one CTA per unit in
 * confkv_attention_plan) runs unclustered CTAs that each walk whole
 * (layer, sequence, KV head) units; the split-K kernel runs one cluster of
 * `splits` CTAs per unit. */
int confkv_attention_grid(confkv_ctx* ctx, int32_t* ctas, int32_t* cluster);

/* The attention launch a step would take, planned on the host alone (no
 * context; nothing runs on a GPU): for configuration `cfg`, a bound
 * `n8_bound` on the INT8 entries of any (layer, sequence) and a cap
 * `attn_ctas` on the persistent grid (0 = none, as confkv_set_attention_ctas),
 * `splits` CTAs per (layer, sequence, KV head) unit (1 = the persistent
 * kernel) and a grid of `ctas` CTAs in clusters of `cluster`.  A context
 * plans each step the same way with its own host bound on n8 (the largest
 * prefill minus W, then at most the largest budget).  The SM count is the
 * current device's, 152 (GB300) when none can be queried.  CONFKV_EINVAL
 * for a null argument, an invalid configuration, a negative bound or cap,
 * or a bound above cap; CONFKV_ECAPACITY when no launch fits in shared
 * memory.  The pages give no counterpart: it exposes this library's launch
 * planning. */
int confkv_launch_plan(const confkv_config* cfg, int64_t n8_bound, int32_t attn_ctas, int32_t* splits,
                       int32_t* ctas, int32_t* cluster);

/* Byte offset of (token tau in [0,16), channel c) inside one 16-token block of
 * the device layout: kind 0 = INT8 K, 1 = INT8 V, 2 = FP16 K, 3 = FP16 V.
 * Host-only helper for tests of the interleave; -1 for bad arguments. */
int32_t confkv_block_offset(int32_t kind, int32_t d, int32_t tau, int32_t c);

/* Largest number of per-chunk partial results confkv_confidence_noalloc can
 * hold: B * ceil(V / 4096) must not exceed it.  The library reserves this
 * scratch (32 bytes per partial, 128 KiB) on every GPU that loads it, for as
 * long as the process runs. */
#define CONFKV_NOALLOC_MAX_PARTIALS 4096

/*
 * Confidence c of B next-token distributions, computed without allocating
 * any device memory.  The paper has no counterpart of this call: it exists
 * for callers that cannot allocate where they need the score -- a plug-in
 * whose host process owns every device buffer through its own pool, a
 * real-time loop that forbids allocation after start-up, or code that must
 * not risk the implicit synchronisation an allocation can cause.  The caller
 * passes only its input and output:
 *   logits      device fp32 [B][V] (temperature 1)
 *   confidence  device fp32 [B], written: the same c as the `confidence`
 *               output of confkv_step, c = w_H (1 - H / log V) +
 *               w_m sigmoid(log p1 - log p2) + w_p p1
 * The partial results of the vocabulary reduction go to one fixed scratch
 * array owned by the library (CONFKV_NOALLOC_MAX_PARTIALS entries per GPU).
 * Every call uses that same array and leaves its last contents there, so
 * calls whose kernels overlap on the GPU (streams without ordering between
 * them) race and give wrong results; order them on one stream.  The first
 * call on a device looks up the array's device address (once per device,
 * with that device current); make that first call before any stream capture.
 * Returns CONFKV_ECAPACITY, without launching anything, if
 * B * ceil(V / 4096) > CONFKV_NOALLOC_MAX_PARTIALS; CONFKV_EINVAL for null
 * pointers, logits or confidence not 4-byte aligned, B < 1, V < 2 or
 * non-finite weights.  Asynchronous on `stream`.
 */
int confkv_confidence_noalloc(const float* logits, int32_t B, int32_t V, double w_H, double w_m,
                              double w_p, float* confidence, void* stream);

/* Human-readable text of a status code. */
const char* confkv_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t confkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CONFKV_H */
