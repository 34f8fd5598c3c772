"""Decode-step benchmark of the CONF-KV cache manager on GB300.

One step = the whole decode-step path for all sequences and layers:
confidence reduction + ring append, mixed FP16/INT8 attention with attention
mass, and select / compact / requantise.  The default workload is the
Qwen-32B-shaped one (64 layers, 40/8 heads, d 128, vocab 152064, batch 8,
4096-token prefill, N_high 1024 / N_low 2048, P 64, W 256).

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload (sequences are independent: no collective on the
data path); `value` is the whole-job step rate.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference   # the float64 CPU oracle on host cores
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CONF-KV decode steps/s (all layers) + achieved HBM GB/s vs GB300 peak, 1 GPU"
PROFILE_EVERY = 7   # at least this many timed steps per step that records per-kernel CUDA events
PROFILE_EVERY_LONG = 31   # the same for windows of more than PROFILE_LONG_STEPS steps
PROFILE_LONG_STEPS = 200


def profile_stride(pool: int, steps: int = 0) -> int:
    """Sampling stride for the per-kernel events: the smallest k >= PROFILE_EVERY
    (PROFILE_EVERY_LONG for windows longer than PROFILE_LONG_STEPS steps)
    coprime with the input pool size, so that the sampled steps visit every
    pool entry instead of a fixed subset of them.  A step that records the
    events runs ~2-4 us longer (each event ends the launch overlap of the
    kernels around it): 1 % of a Qwen-sized step, 10 % of an 18 us one, so
    long windows sample more sparsely."""
    import math
    k = PROFILE_EVERY_LONG if steps > PROFILE_LONG_STEPS else PROFILE_EVERY
    while math.gcd(k, max(pool, 1)) != 1:
        k += 1
    return k
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _traffic_ratio_from_profiles(kernel_tag: str):
    """DRAM bytes per algorithmic byte of a kernel, from the machine-readable
    ncu record profiles/<kernel_tag>.json (key
    `dram_bytes_per_algorithmic_byte`), or None if there is none or it does
    not describe the kernel now built (`stale`: true).  Each unit streams its
    own K/V once, so traffic grows in proportion to the algorithmic bytes and
    a launch's traffic is this ratio times its algorithmic bytes."""
    p = os.path.join(ROOT, "profiles", kernel_tag + ".json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p))
    except (OSError, ValueError):
        return None
    if rec.get("stale"):
        return None
    r = rec.get("dram_bytes_per_algorithmic_byte")
    return float(r) if isinstance(r, (int, float)) else None


def blas_threads() -> dict:
    """Threads the BLAS behind numpy may use: threadpoolctl where installed,
    else the thread count reported by the OpenBLAS library numpy has loaded
    (its exported get_num_threads call), else the environment."""
    try:
        from threadpoolctl import threadpool_info
        info = [x for x in threadpool_info() if x.get("user_api") == "blas"]
        if info:
            return {"threads": max(int(x["num_threads"]) for x in info),
                    "library": str(info[0].get("internal_api")), "how": "threadpoolctl"}
    except Exception:
        pass
    try:
        import ctypes
        import numpy  # noqa: F401  (loads its BLAS)
        libs = sorted({ln.split()[-1] for ln in open("/proc/self/maps") if "openblas" in ln.lower()})
        for path in libs:
            lib = ctypes.CDLL(path)
            for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                         "scipy_openblas_get_num_threads", "openblas_get_num_threads"):
                f = getattr(lib, name, None)
                if f is not None:
                    f.restype = ctypes.c_int
                    return {"threads": int(f()), "library": os.path.basename(path), "how": name}
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return {"threads": int(os.environ[var]), "library": None, "how": var}
    return {"threads": None, "library": None, "how": "unknown"}


def untimed_steps(warmup: int, pool: int) -> int:
    """Decode steps run before the timed window: at least the W warm-up
    steps, and at least the first step (which cuts the prefill down to the
    budget) plus one full cycle of the R-entry step-input pool.  The cache
    length then follows its periodic regime, in which the pool's confident
    entries flip the budget at fixed points of every cycle, so a short timed
    window sees the same cache sizes as a long one."""
    return max(int(warmup), int(pool) + 1)


def spin_cycles(steps: int, clock_ghz: float = 2.07) -> int:
    """GPU clock cycles of the device delay queued before the first timed
    event: long enough for the host to queue the window's first steps behind
    it (about 60 us of host time per step, at most 50 ms), so that neither
    the host's launch latency nor an idle GPU's clock ramp falls inside the
    timed window."""
    ms = min(50.0, 2.0 + 0.06 * max(int(steps), 1))
    return int(ms * 1e-3 * clock_ghz * 1e9)


def l2_note(w) -> str:
    """How the timed window relates to the 129 MB L2, from the workload's
    steady-state K/V bytes per step (each cache at its loose budget)."""
    n = min(max(w.n_low), w.T0 + w.steps)
    n8 = max(0, n - w.W)
    nr = min(n, w.W + 16)
    kv = w.L * w.B * w.Hkv * w.d * (2 * n8 + 4 * nr)
    if kv > 129e6:
        return "inputs larger than L2: ~%.2f GB of K/V streamed per step > 129 MB L2, no flush" % (kv / 1e9)
    return ("K/V of ~%.1f MB per step fits the 129 MB L2 and stays resident between steps "
            "(not flushed)" % (kv / 1e6))


def bench_config(w, args, ws: int) -> dict:
    """The `config` object of the JSON line: the same dict for both arms."""
    return {"workload": w.name, "compaction": args.compaction, "global_batch": w.B * ws,
            "seq_len": w.T0, "layers": w.L, "heads": [w.Hq, w.Hkv], "head_dim": w.d, "vocab": w.V,
            "budgets": [w.n_high[0], w.n_low[0]], "budgets_last_layer": [w.n_high[-1], w.n_low[-1]],
            "P": w.P, "W": w.W, "query_dtype": w.q_dtype,
            "parallelism": "replicas (dp%d over sequences)" % ws, "l2": l2_note(w)}


class ClockSampler:
    """nvidia-smi clocks, utilisation and throttle reasons sampled every
    200 ms.  `stop` reports the median SM clock over the samples taken under
    load (GPU utilisation >= 50 %; all samples if none was), and every
    throttle reason seen while sampling."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 10:
                rows.append(f)
        os.unlink(self.path)
        return summarise_clocks(rows)


def _num(x):
    try:
        return float(x)
    except ValueError:
        return None


def summarise_clocks(rows):
    """Summary of nvidia-smi rows in ClockSampler.FIELDS order."""
    if not rows:
        return None
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    loaded = [r for r in rows if (_num(r[9]) or 0.0) >= 50.0]
    use = loaded or rows
    sm = sorted(v for v in (_num(r[1]) for r in use) if v is not None)
    mx = [v for v in (_num(r[2]) for r in rows) if v is not None]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
    return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class OracleSample:
    """The float64 oracle over a bounded sample of the workload: `units`
    (sequence, layer) units, each prefilled and stepped once during set-up
    (the first step evicts the prefill down to the budget), then stepped at
    steady-state cache size by `run`."""

    def __init__(self, w, seed: int, units: int):
        import numpy as np
        from oracle import confkv_oracle as orc
        from workload import prefill_unit
        self.w, self.seed, self.orc = w, seed, orc
        self.prm = orc.Params.from_workload(w)
        rng = np.random.default_rng(seed)
        self.picks = [(int(rng.integers(w.B)), int(rng.integers(w.L))) for _ in range(units)]
        self.states = []
        self.s = 0
        for b, l in self.picks:
            k, v = prefill_unit(w, seed, b, l)
            self.states.append(orc.prefill_unit(k, v, w.W))
        self.run(1)

    def run(self, steps: int):
        from workload import step_unit, step_logits
        orc, w = self.orc, self.w
        done = 0
        wall0, cpu0 = time.perf_counter(), time.process_time()
        for _ in range(steps):
            for i, (b, l) in enumerate(self.picks):
                q, kn, vn = step_unit(w, self.seed, self.s, b, l)
                c = orc.confidence(step_logits(w, self.seed, self.s, b)).c
                N = orc.budget(c, w.tau, w.n_high[l], w.n_low[l])
                self.states[i] = orc.step_unit(self.prm, self.states[i], w.T0 + self.s,
                                               q.float().numpy(), kn, vn, N).state
                done += 1
            self.s += 1
        return done, time.perf_counter() - wall0, time.process_time() - cpu0

    def steps_per_s(self, done: int, wall: float) -> float:
        return 1.0 / (wall / max(done, 1) * self.w.L * self.w.B)


def cpu_baseline(w, seed: int, units: int = 8, steps: int = 120):
    """Oracle steps/s of the whole workload, extrapolated from a bounded
    sample of unit-steps timed on the host cores (about 10 s of oracle work
    on the Qwen-32B shape)."""
    smp = OracleSample(w, seed, units)
    done, wall, cpu = smp.run(steps)
    return {
        "value": smp.steps_per_s(done, wall),
        "unit": "steps/s",
        "cores": max(1, int(round(cpu / wall))) if wall > 0 else 1,
        "cores_available": len(os.sched_getaffinity(0)),
        "blas": blas_threads(),
        "kind": "oracle",
        "sample": "%d (sequence, layer) unit-steps of %s at steady-state cache size (confidence "
                  "over the full vocabulary, attention, EMA, ranking, eviction, requantisation), "
                  "%.1f s wall; steps/s = 1 / (time per unit-step x L x B)" % (done, w.name, wall),
    }


def run_reference(args):
    """The reference arm: the float64 oracle timed on the host cores, on the
    GPU arm's workload and config.  Each timed step runs a bounded sample of
    the workload (2 (sequence, layer) unit-steps at steady-state cache size);
    `value` extrapolates it to whole steps (all L x B units), `ms_per_step` is
    the measured wall time of one timed step."""
    from workload import get_workload
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    w = get_workload(args.workload)
    if args.batch:
        w = w.replace(B=args.batch)
    units = 2
    smp = OracleSample(w, args.seed, units=units)
    for _ in range(args.warmup):
        smp.run(1)
    vals = []
    tot_done, tot_wall, tot_cpu = 0, 0.0, 0.0
    for _ in range(args.steps):
        done, wall, cpu = smp.run(1)
        vals.append(smp.steps_per_s(done, wall))
        tot_done += done
        tot_wall += wall
        tot_cpu += cpu
    vals.sort()
    v = vals[len(vals) // 2]
    cpu_line = {"value": v, "unit": "steps/s",
                "cores": max(1, int(round(tot_cpu / tot_wall))) if tot_wall > 0 else 1,
                "cores_available": len(os.sched_getaffinity(0)), "blas": blas_threads(), "kind": "oracle",
                "sample": "each timed step: %d (sequence, layer) unit-steps of %s at steady-state size; "
                          "steps/s = 1 / (time per unit-step x L x B), median over steps" % (units, w.name)}
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot_wall / max(args.steps, 1),
        "extrapolated": {"ms_per_whole_step": 1000.0 / v, "unit_steps_per_timed_step": units,
                         "unit_steps_per_whole_step": w.L * w.B,
                         "how": "value = whole-step rate extrapolated from the timed unit-steps; "
                                "ms_per_step = measured wall time of one timed step"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(w, args, ws),
        "cpu_baseline": cpu_line,
        "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def replica_seed(base: int, i: int, rank: int) -> int:
    """Seed of the i-th timed instance on `rank`: replicas on different ranks
    draw different prefills and step inputs."""
    return base + i + 7919 * rank


def reduce_timing(ms: float, steps: int, world_size: int, device):
    """Max of the per-rank timed milliseconds over all ranks, and the
    whole-job rate: every rank ran `steps` steps of its own replica."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world_size > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, world_size * steps / (ms_max / 1000.0)


def run_ours(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import confidence_gated_kv_gb300 as ck
    if not os.path.exists(ck.binding.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    from workload import get_workload, prefill_batch_fast, step_pool_fast

    w = get_workload(args.workload)
    if args.batch:
        w = w.replace(B=args.batch)
    cfg = ck.config_from_workload(w, compaction=1 if args.compaction == "ordered" else 0)
    R = args.pool
    stream = torch.cuda.current_stream()
    every = profile_stride(R, args.steps)

    pre = untimed_steps(args.warmup, R)
    clocks = ClockSampler(local)
    clocks.start()

    def timed_seed(seed):
        """Prefill, the untimed steps (at least W warm-up steps), then exactly
        K timed steps of one seeded instance of the workload."""
        cache = ck.Cache(cfg, device=dev)
        cache.set_step_mode(ck.binding.STEP_SEPARATE if args.step_mode == "separate" else ck.binding.STEP_AUTO)
        k, v = prefill_batch_fast(w, seed, dev)
        cache.prefill(k, v, [w.T0] * w.B)
        torch.cuda.synchronize()
        del k, v
        torch.cuda.empty_cache()
        pool = step_pool_fast(w, seed, R, dev)
        q, kn, vn, lg = pool
        outs = cache.new_outputs()
        for s in range(pre):
            cache.step(q[s % R], kn[s % R], vn[s % R], lg[s % R], outs)
        torch.cuda.synchronize()
        st0 = cache.stats()
        # per-kernel events on every `every`-th timed step: an event record
        # between kernels costs the stream ~2 us, so recording all four on
        # every step would slow the very steps it times
        cache.profile_enable((args.steps + every - 1) // every, every)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # a device delay ahead of the first event: the host queues the
        # window's first steps behind it, so the window measures the GPU
        # running the steps back to back, not the host's first launches
        # the same confkv_step call per step, with its arguments prepared
        # once per pool entry (host time per call stays well below a step)
        run = cache.prepared_steps([(q[j], kn[j], vn[j], lg[j]) for j in range(R)], outs)
        torch.cuda._sleep(spin_cycles(args.steps))
        ev0.record(stream)
        for s in range(args.steps):
            run((pre + s) % R)
        ev1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        ms = ev0.elapsed_time(ev1)
        prof = cache.profile_read()
        cache.profile_disable()
        st1 = cache.stats()
        ms_max, sps = reduce_timing(ms, args.steps, ws, dev)
        return dict(seed=seed, cache=cache, pool=pool, outs=outs, st0=st0, st1=st1, prof=prof,
                    ms_max=ms_max, sps=sps)

    # The pages report the median of three seeds: each seed is its own
    # prefill and step-input pool, timed over exactly K steps; the reported
    # rate and every per-kernel figure come from the median seed.
    runs = []
    for i in range(max(1, args.seeds)):
        r = timed_seed(replica_seed(args.seed, i, rank))
        if runs:   # only the last seed's cache stays for the e2e and graph runs
            for key in ("cache", "pool", "outs"):
                runs[-1].pop(key, None)
            torch.cuda.empty_cache()
        runs.append(r)
    clk = clocks.stop()
    med = sorted(runs, key=lambda r: r["sps"])[len(runs) // 2]
    cache, outs = runs[-1]["cache"], runs[-1]["outs"]
    q, kn, vn, lg = runs[-1]["pool"]
    st0, st1, prof, ms_max, steps_per_s = med["st0"], med["st1"], med["prof"], med["ms_max"], med["sps"]
    seeds = {"values": [r["sps"] for r in runs], "seeds": [r["seed"] for r in runs],
             "attention_ms": [r["prof"]["attention_ms"] / max(r["prof"]["steps"], 1) for r in runs],
             "attention_bytes": [(r["st1"]["attn_bytes"] - r["st0"]["attn_bytes"]) / args.steps for r in runs],
             "reported": "median" if len(runs) > 1 else "single"}

    attn_bytes = (st1["attn_bytes"] - st0["attn_bytes"]) / args.steps
    step_bytes = (st1["step_bytes"] - st0["step_bytes"]) / args.steps
    attn_ms = prof["attention_ms"] / max(prof["steps"], 1)
    peak, peak_kind = _peaks()
    achieved = attn_bytes / (attn_ms / 1000.0) / 1e9
    ratio = _traffic_ratio_from_profiles("attention_kernel_" + w.name)
    traffic = ratio * attn_bytes if ratio is not None else None

    # attention + compaction chain: everything but the logits reduction and the
    # append of the new token (attention, EMA, ranking, eviction, compaction,
    # requantisation), over the time of the attention and select kernels
    prestep_bytes = w.B * w.V * 4 + w.L * w.B * w.Hkv * w.d * 2 * 2 * 2
    chain_bytes = step_bytes - prestep_bytes
    chain_ms = (prof["attention_ms"] + prof["select_ms"]) / max(prof["steps"], 1)
    chain_gbs = chain_bytes / (chain_ms / 1000.0) / 1e9
    chain = {"what": "attention + EMA/rank/evict/compact/requant", "algorithmic_bytes_per_step": chain_bytes,
             "ms_per_step": chain_ms, "achieved_gbs": chain_gbs, "peak_gbs": peak, "frac": chain_gbs / peak}

    # ------------------------------------------------ end to end, host buffers
    e2e = None
    if args.e2e_steps > 0:
        hq = [q[j].cpu().pin_memory() for j in range(R)]
        hk = [kn[j].cpu().pin_memory() for j in range(R)]
        hv = [vn[j].cpu().pin_memory() for j in range(R)]
        hl = [lg[j].cpu().pin_memory() for j in range(R)]
        hout = cache.host_outputs()
        h2d = hq[0].numel() * hq[0].element_size() + 2 * hk[0].numel() * 2 + hl[0].numel() * 4
        d2h = sum(x.numel() * x.element_size() for x in hout.values())
        for s in range(4):   # untimed: first calls create the library's second stream
            cache.step_host(hq[s % R], hk[s % R], hv[s % R], hl[s % R], hout)
        torch.cuda.synchronize()
        e0 = time.perf_counter()
        for s in range(args.e2e_steps):
            j = s % R
            cache.step_host(hq[j], hk[j], hv[j], hl[j], hout)
        e_el = time.perf_counter() - e0
        hst = cache.stats()
        # pinned buffers: the library's mapped mode (kernels read and write the
        # host buffers in place, q staged); it reports the bytes that crossed
        h2d, d2h = hst["host_h2d_bytes"] or h2d, hst["host_d2h_bytes"] or d2h
        e2e = {"value": ws * args.e2e_steps / e_el, "unit": "steps/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "api": "confkv_step_host", "steps": args.e2e_steps}

    # ------------------------------------------------ CUDA-graph replays (optional)
    graph = None
    if args.graph:
        splits_g, _ = cache.attention_plan()
        cache.graph_reserve(args.steps)
        graphs = [cache.capture_step(q[j], kn[j], vn[j], lg[j], outs) for j in range(R)]
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(spin_cycles(args.steps))
        g0.record(stream)
        done = 0
        for s in range(args.steps):
            graphs[(pre + s) % R].replay()
            if (s + 1) % 64 == 0:
                cache.graph_advance(s + 1 - done)
                done = s + 1
        g1.record(stream)
        torch.cuda.synchronize()
        cache.graph_advance(args.steps - done)
        cache.graph_release()
        gms = g0.elapsed_time(g1)
        graph = {"value": args.steps / (gms / 1000.0), "unit": "steps/s", "ms_per_step": gms / args.steps,
                 "how": "one captured step per pool entry, replayed; device-side step index",
                 "ctas_per_unit": splits_g}
        del graphs

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.seed)

    splits, smem = cache.attention_plan()
    st = cache.stats()
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": steps_per_s,
            "unit": "steps/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "seeds": seeds,
            "ms_per_step": ms_max / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "fp16/int8 storage, fp16 tensor-core products, fp32 accumulate",
            "data": "synthetic",
            "config": bench_config(w, args, ws),
            "untimed_steps": {"count": pre, "warmup": args.warmup,
                              "why": "at least W warm-up steps, and at least the first step plus one "
                                     "cycle of the %d-entry step-input pool, so the timed window starts "
                                     "in the cache's periodic regime" % R},
            "timed_window": "CUDA events on the launching stream around exactly K steps, queued behind "
                            "a device delay so that host launch latency stays outside the window",
            "hbm": {"achieved_gbs": step_bytes / (ms_max / args.steps / 1000.0) / 1e9,
                    "algorithmic_bytes_per_step": step_bytes, "peak_gbs": peak, "peak_kind": peak_kind,
                    "frac": step_bytes / (ms_max / args.steps / 1000.0) / 1e9 / peak},
            "roofline": {"kernel": "attention_kernel", "bound": "hbm", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "algorithmic_bytes_per_launch": attn_bytes,
                         "avg_launch_ms": attn_ms, "peak_kind": peak_kind},
            "chain": chain,
            "breakdown_ms_per_step": {k: prof[k + "_ms"] / max(prof["steps"], 1)
                                      for k in ("prestep", "attention", "select")},
            "kernel_timing": "CUDA events around each kernel on every %dth timed step (%d steps sampled)"
                             % (every, prof["steps"]),
            "attention_launch": {"ctas_per_unit": splits, "smem_bytes": smem},
            "step_launches": cache.step_launches(), "step_mode": args.step_mode,
            "gpu_launches": int(st1["launches"] - st0["launches"]),
            "clocks": clk,
            "e2e": e2e,
            "graph": graph,
            "cpu_baseline": cpu,
            "state": {"resident_entries": st["resident"], "resident_kv_bytes": st["resident_bytes"],
                      "evicted_total": st["evicted"], "moved_total": st["moved"]},
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# --compare: CONF-KV against full KV and a 512-token sliding window on the
# same kernels (the pages' baselines; they publish the ratios only)
# ---------------------------------------------------------------------------
COMPARE_KINDS = ("confkv", "fullkv", "sliding512")


def variant_workload(w, kind: str, steps_total: int):
    """The workload's shape and data under one cache policy.

    confkv      the workload's own budgets, window and weights;
    fullkv      no eviction (budgets above any cache length) and an FP16
                window covering the prefill and every generated token, so
                nothing is ever quantised;
    sliding512  recency only (alpha = 0) with N_high = N_low = 512, every
                resident entry inside a 512-token FP16 window."""
    L = w.L
    if kind == "confkv":
        return w
    if kind == "fullkv":
        W = (w.T0 + steps_total + 16 + 15) // 16 * 16
        return w.replace(n_high=(1 << 30,) * L, n_low=(1 << 30,) * L, W=W, cap=16)
    if kind == "sliding512":
        return w.replace(n_high=(512,) * L, n_low=(512,) * L, alpha=0.0, W=512)
    raise ValueError(kind)


def prefill_kv_bytes(w, T0: int) -> int:
    """K/V bytes at stored widths right after a prefill of T0 tokens per
    sequence: positions older than the W newest in INT8, the rest in FP16."""
    n8 = max(0, T0 - w.W)
    return w.L * w.B * w.Hkv * w.d * (2 * n8 + 4 * (T0 - n8))


def run_compare(args):
    """One JSON line: per-step latency (CUDA events around every step), the
    step rate and the peak resident KV bytes of each policy over the same
    trajectory (same prefill, same step inputs), and the ratios the pages
    quote (p50 latency and throughput of full KV over CONF-KV)."""
    import numpy as np
    import torch
    import confidence_gated_kv_gb300 as ck
    if not os.path.exists(ck.binding.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    from workload import get_workload, prefill_batch_fast, step_pool_fast

    dev = torch.device("cuda", 0)
    w0 = get_workload(args.workload)
    if args.batch:
        w0 = w0.replace(B=args.batch)
    gen = args.compare_steps
    R = args.pool
    q, kn, vn, lg = step_pool_fast(w0, args.seed, R, dev)
    stream = torch.cuda.current_stream()
    res = {}
    for kind in COMPARE_KINDS:
        w = variant_workload(w0, kind, args.warmup + gen)
        cache = ck.Cache(ck.config_from_workload(w), device=dev)
        k, v = prefill_batch_fast(w0, args.seed, dev)
        cache.prefill(k, v, [w0.T0] * w0.B)
        del k, v
        outs = cache.new_outputs()
        for s in range(args.warmup):
            cache.step(q[s % R], kn[s % R], vn[s % R], lg[s % R], outs)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(gen)]
        for s in range(gen):
            j = (args.warmup + s) % R
            evs[s][0].record(stream)
            cache.step(q[j], kn[j], vn[j], lg[j], outs)
            evs[s][1].record(stream)
        torch.cuda.synchronize()
        ms = np.array([a.elapsed_time(b) for a, b in evs])
        st = cache.stats()
        # peak K/V bytes at stored widths: the exact maximum over the ends of
        # all steps since prefill, kept on the device; the workspace is the
        # allocator footprint (all device memory the context holds)
        res[kind] = {"p50_ms": float(np.median(ms)), "mean_ms": float(ms.mean()),
                     "p90_ms": float(np.percentile(ms, 90)), "steps_per_s": 1000.0 / float(ms.mean()),
                     "peak_kv_bytes": int(st["peak_resident_bytes"]), "peak_entries": int(st["peak_resident"]),
                     "prefill_kv_bytes": int(prefill_kv_bytes(w, w0.T0)),
                     "workspace_bytes": int(st["workspace_bytes"]),
                     "final_resident_entries": int(st["resident"]),
                     "W": w.W, "budgets": [w.n_high[0], w.n_low[0]], "alpha": w.alpha}
        del cache, outs
        torch.cuda.empty_cache()
    c, f, sl = res["confkv"], res["fullkv"], res["sliding512"]
    line = {"metric": "CONF-KV vs full KV and sliding-512 on the same kernels, 1 GPU",
            "workload": w0.name, "batch": w0.B, "prefill": w0.T0, "generated_steps": gen,
            "warmup": args.warmup, "data": "synthetic", "timing": "CUDA events around every step",
            "variants": res,
            "ratios": {"p50_latency_fullkv_over_confkv": f["p50_ms"] / c["p50_ms"],
                       "throughput_confkv_over_fullkv": f["mean_ms"] / c["mean_ms"],
                       "throughput_sliding512_over_fullkv": f["mean_ms"] / sl["mean_ms"],
                       "peak_kv_fullkv_over_confkv": f["peak_kv_bytes"] / max(c["peak_kv_bytes"], 1),
                       "workspace_fullkv_over_confkv": f["workspace_bytes"] / max(c["workspace_bytes"], 1)},
            "pages": {"p50_latency_fullkv_over_confkv": 1.8, "throughput_confkv_over_fullkv_batch8": 2.06,
                      "note": "GPT-2 / Qwen-32B at 2048 generated tokens on the pages' GPU; context only"}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--workload", default="qwen32b")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (small captures)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=4003)
    ap.add_argument("--seeds", type=int, default=3, help="seeded instances timed; the median is reported")
    ap.add_argument("--pool", type=int, default=16)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--compaction", default="tailfill", choices=["tailfill", "ordered"],
                    help="INT8 compaction: tail fill (default) or the order-preserving ablation")
    ap.add_argument("--step-mode", default="auto", choices=["auto", "separate"],
                    help="auto: one fused launch per step where the shape allows it; separate: three kernels")
    ap.add_argument("--graph", action="store_true",
                    help="also time CUDA-graph replays of captured steps (extra 'graph' key)")
    ap.add_argument("--compare", action="store_true",
                    help="CONF-KV vs full KV vs sliding-512 on the same kernels (one JSON line)")
    ap.add_argument("--compare-steps", type=int, default=2048, help="generated tokens per policy in --compare")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.compare:
        return run_compare(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
