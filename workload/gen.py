"""Seeded synthetic inputs with the shapes of the CONF-KV evaluation workloads.

The pages evaluate CONF-KV on GPT-2, Qwen-14B/32B and a needle-in-a-haystack
retrieval setup (CONF-KV, paper.rainbus.top/paper/2605.24786, sections
"实验结果" and "复现评估"; gist.science/de/paper/2605.24786, section
"Experimentelle Ergebnisse").  No model weights or datasets are used: the
workloads below reproduce only their geometry (layers, heads, head dim,
vocabulary, batch, prefill and decode lengths) and the budget / window
hyper-parameters, with random K/V, queries and logits.

Two generator back-ends draw the same distributions:

* ``prefill_unit`` / ``step_unit`` / ``step_logits`` (numpy, CPU): every
  (sequence, layer) unit and every pooled step input has its own Philox
  stream keyed by (seed, tag, indices), so any single unit can be regenerated
  on the CPU without drawing the rest.  ``prefill_batch`` / ``step_pool``
  assemble whole batches from these streams (threaded) and upload them.
* ``prefill_batch_fast`` / ``step_pool_fast`` (torch, on the device): the same
  distributions drawn with a device generator.  Fast, but not reproducible on
  the CPU; used only where no CPU-side comparison of the values is needed.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

# Stream tags: one independent random stream per (seed, tag, indices).
_TAG_PREFILL = 1
_TAG_HEAVY = 2
_TAG_NEEDLE = 3
_TAG_QDIR = 4
_TAG_STEP = 5
_TAG_LOGITS = 6


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and hyper-parameters of one synthetic decode workload."""

    name: str
    B: int            # batch (independent sequences)
    L: int            # layers
    Hq: int           # query heads
    Hkv: int          # KV heads
    d: int            # head dim
    V: int            # vocabulary size
    T0: int           # prefill length (tokens per sequence)
    steps: int        # decode steps of the workload
    n_high: tuple     # per-layer tight budget (chosen when c >= tau)
    n_low: tuple      # per-layer loose budget (chosen when c < tau)
    P: int            # protected newest tokens
    W: int            # FP16 window (newest tokens kept in fp16)
    tau: float = 0.7
    alpha: float = 0.65
    lam: float = 0.9
    w_H: float = 0.4
    w_m: float = 0.3
    w_p: float = 0.3
    q_dtype: str = "f16"          # "f16" or "bf16"
    heavy_count: int = 0          # prefill positions whose key is scaled
    heavy_factor: float = 1.0
    logit_sigma: float = 1.0      # logits ~ N(0, sigma) ...
    spike_hi: float = 12.0        # ... plus U[0, spike_hi] at one random index
    needle: bool = False          # plant a key aligned with the queries
    needle_scale: float = 6.0
    needle_depth: tuple = (0.1, 0.9)
    q_noise: float = 0.3          # needle queries: q_dir + N(0, q_noise^2)
    cap: int = 0                  # INT8 capacity per (sequence, layer); 0 -> derived

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def capacity(self) -> int:
        """INT8 slots per (sequence, layer): room for the prefill and the
        largest budget plus one, rounded up to a multiple of 16."""
        c = self.cap if self.cap > 0 else max(self.T0, max(max(self.n_high), max(self.n_low)) + 1)
        return (c + 15) // 16 * 16

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _uniform(L: int, n: int) -> tuple:
    return tuple([int(n)] * L)


def _pyramid(L: int, top: int, bottom: int) -> tuple:
    # Linear interpolation from the first to the last layer, rounded half to
    # even (Python's round).
    if L == 1:
        return (int(top),)
    return tuple(int(round(top - (top - bottom) * l / (L - 1))) for l in range(L))


WORKLOADS = {
    # GPT-2-small geometry, batch 1, 600-token prefill, 64 decode steps.
    "gpt2_b1": Workload(
        name="gpt2_b1", B=1, L=12, Hq=12, Hkv=12, d=64, V=50257, T0=600, steps=64,
        n_high=_uniform(12, 256), n_low=_uniform(12, 512), P=32, W=64,
        q_dtype="f16", heavy_count=8, heavy_factor=4.0, logit_sigma=1.0, spike_hi=12.0),
    # GPT-2-small geometry, batch 8, 128-token prefill, 2048 decode steps,
    # pyramidal per-layer budgets (768 -> 256 loose, 384 -> 128 tight).
    "gpt2_b8_pyramid": Workload(
        name="gpt2_b8_pyramid", B=8, L=12, Hq=12, Hkv=12, d=64, V=50257, T0=128, steps=2048,
        n_high=_pyramid(12, 384, 128), n_low=_pyramid(12, 768, 256), P=64, W=128,
        q_dtype="f16", heavy_count=1, heavy_factor=4.0, logit_sigma=1.0, spike_hi=12.0),
    # Qwen-14B shape: 48 layers, 40/8 heads (GQA 5), d128, batch 4, 8192 prefill.
    "qwen14b": Workload(
        name="qwen14b", B=4, L=48, Hq=40, Hkv=8, d=128, V=152064, T0=8192, steps=256,
        n_high=_uniform(48, 1024), n_low=_uniform(48, 2048), P=64, W=256,
        q_dtype="bf16", heavy_count=0, logit_sigma=1.5, spike_hi=14.0),
    # Qwen-32B shape: 64 layers, 40/8 heads, d128, batch 8, 4096 prefill,
    # 0.5% heavy keys (x3).
    "qwen32b": Workload(
        name="qwen32b", B=8, L=64, Hq=40, Hkv=8, d=128, V=152064, T0=4096, steps=4096,
        n_high=_uniform(64, 1024), n_low=_uniform(64, 2048), P=64, W=256,
        q_dtype="bf16", heavy_count=20, heavy_factor=3.0, logit_sigma=1.5, spike_hi=14.0),
    # Planted-key long-context retrieval shape: 32768-token prefill with one
    # needle key per layer, queries aligned with the needle direction,
    # low-confidence logits.
    "needle32k": Workload(
        name="needle32k", B=1, L=64, Hq=40, Hkv=8, d=128, V=152064, T0=32768, steps=128,
        n_high=_uniform(64, 2048), n_low=_uniform(64, 4096), P=64, W=256,
        q_dtype="bf16", needle=True, logit_sigma=1.5, spike_hi=4.0),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


def _rng(seed: int, tag: int, *idx: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(seed), tag, *map(int, idx)])))


# ----------------------------------------------------------------------------
# Per-unit CPU generators (reproducible per (sequence, layer) / pooled step)
# ----------------------------------------------------------------------------

def heavy_positions(w: Workload, seed: int, b: int, T0: Optional[int] = None) -> np.ndarray:
    """Prefill positions of sequence b whose key is scaled by heavy_factor (in
    every layer and KV head)."""
    T0 = w.T0 if T0 is None else T0
    n = min(w.heavy_count, T0)
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(seed, _TAG_HEAVY, b).choice(T0, size=n, replace=False)).astype(np.int64)


def needle_position(w: Workload, seed: int, b: int, T0: Optional[int] = None) -> int:
    T0 = w.T0 if T0 is None else T0
    lo, hi = w.needle_depth
    u = _rng(seed, _TAG_NEEDLE, b).uniform(lo, hi)
    return int(min(T0 - 1, max(0, math.floor(u * T0))))


def q_direction(w: Workload, seed: int, l: int) -> np.ndarray:
    """Unit query direction per KV head of layer l (needle workload), float32
    [Hkv][d]."""
    x = _rng(seed, _TAG_QDIR, l).standard_normal((w.Hkv, w.d))
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    return x.astype(np.float32)


def prefill_unit(w: Workload, seed: int, b: int, l: int, T0: Optional[int] = None):
    """Prefill K, V of (sequence b, layer l): float16 [Hkv][T0][d] each."""
    T0 = w.T0 if T0 is None else T0
    g = _rng(seed, _TAG_PREFILL, b, l)
    kv = np.empty((2, w.Hkv, T0, w.d), dtype=np.float32)
    g.standard_normal(out=kv, dtype=np.float32)
    if w.heavy_count > 0 and T0 > 0:
        kv[0][:, heavy_positions(w, seed, b, T0), :] *= np.float32(w.heavy_factor)
    if w.needle and T0 > 0:
        p = needle_position(w, seed, b, T0)
        kv[0][:, p, :] = np.float32(w.needle_scale) * q_direction(w, seed, l)
    return kv[0].astype(np.float16), kv[1].astype(np.float16)


def _to_qdtype(x: np.ndarray, q_dtype: str):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16 if q_dtype == "bf16" else torch.float16)


def step_unit(w: Workload, seed: int, r: int, b: int, l: int):
    """Pooled decode-step input r of (sequence b, layer l).

    Returns (q, k_new, v_new): q is a CPU torch tensor [Hq][d] of the
    workload's query dtype; k_new, v_new are float16 numpy [Hkv][d]."""
    g = _rng(seed, _TAG_STEP, r, b, l)
    x = g.standard_normal((w.Hq + 2 * w.Hkv, w.d), dtype=np.float32)
    q = x[: w.Hq]
    if w.needle:
        qd = q_direction(w, seed, l)
        q = np.repeat(qd, w.g, axis=0) + np.float32(w.q_noise) * q
    k_new = x[w.Hq: w.Hq + w.Hkv].astype(np.float16)
    v_new = x[w.Hq + w.Hkv:].astype(np.float16)
    return _to_qdtype(q, w.q_dtype), k_new, v_new


def step_logits(w: Workload, seed: int, r: int, b: int) -> np.ndarray:
    """Pooled logits r of sequence b: float32 [V], N(0, sigma) plus a spike
    U[0, spike_hi] added at one uniform-random index."""
    g = _rng(seed, _TAG_LOGITS, r, b)
    z = g.standard_normal(w.V, dtype=np.float32) * np.float32(w.logit_sigma)
    idx = int(g.integers(w.V))
    z[idx] += np.float32(g.uniform(0.0, w.spike_hi))
    return z


# ----------------------------------------------------------------------------
# Batch assembly (threaded CPU draws, uploaded to `device`)
# ----------------------------------------------------------------------------

def prefill_batch(w: Workload, seed: int, device="cpu", T0: Optional[int] = None, threads: int = 0):
    """K, V as torch float16 [L][B][Hkv][T0][d] built from the per-unit CPU
    streams."""
    import os
    import torch
    T0 = w.T0 if T0 is None else T0
    k = torch.empty((w.L, w.B, w.Hkv, T0, w.d), dtype=torch.float16)
    v = torch.empty_like(k)
    kn, vn = k.numpy(), v.numpy()

    def fill(job):
        b, l = job
        kk, vv = prefill_unit(w, seed, b, l, T0)
        kn[l, b] = kk
        vn[l, b] = vv

    jobs = [(b, l) for b in range(w.B) for l in range(w.L)]
    nthr = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(nthr) as ex:
        list(ex.map(fill, jobs))
    if str(device) != "cpu":
        k = k.to(device)
        v = v.to(device)
    return k, v


def step_pool(w: Workload, seed: int, R: int, device="cpu", threads: int = 0):
    """R pooled step inputs from the per-unit CPU streams:
    q [R][L][B][Hq][d] (query dtype), k_new, v_new [R][L][B][Hkv][d] fp16,
    logits [R][B][V] fp32 (torch tensors on `device`)."""
    import os
    import torch
    qdt = torch.bfloat16 if w.q_dtype == "bf16" else torch.float16
    q = torch.empty((R, w.L, w.B, w.Hq, w.d), dtype=qdt)
    kn = torch.empty((R, w.L, w.B, w.Hkv, w.d), dtype=torch.float16)
    vn = torch.empty_like(kn)
    lg = torch.empty((R, w.B, w.V), dtype=torch.float32)

    def fill(job):
        r, b, l = job
        qq, kk, vv = step_unit(w, seed, r, b, l)
        q[r, l, b] = qq
        kn[r, l, b] = torch.from_numpy(kk)
        vn[r, l, b] = torch.from_numpy(vv)
        if l == 0:
            lg[r, b] = torch.from_numpy(step_logits(w, seed, r, b))

    jobs = [(r, b, l) for r in range(R) for b in range(w.B) for l in range(w.L)]
    nthr = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(nthr) as ex:
        list(ex.map(fill, jobs))
    if str(device) != "cpu":
        q, kn, vn, lg = (t.to(device) for t in (q, kn, vn, lg))
    return q, kn, vn, lg


# ----------------------------------------------------------------------------
# Device generators (same distributions, drawn on the GPU)
# ----------------------------------------------------------------------------

def prefill_batch_fast(w: Workload, seed: int, device, T0: Optional[int] = None):
    """K, V float16 [L][B][Hkv][T0][d] drawn on `device` with a torch device
    generator (same distributions as prefill_batch; different values)."""
    import torch
    T0 = w.T0 if T0 is None else T0
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 7919 + 17)
    k = torch.empty((w.L, w.B, w.Hkv, T0, w.d), dtype=torch.float16, device=device)
    v = torch.empty_like(k)
    for l in range(w.L):
        k[l].normal_(generator=gen)
        v[l].normal_(generator=gen)
    for b in range(w.B):
        if w.heavy_count > 0 and T0 > 0:
            hp = torch.from_numpy(heavy_positions(w, seed, b, T0)).to(device)
            k[:, b, :, hp, :] *= w.heavy_factor
        if w.needle and T0 > 0:
            p = needle_position(w, seed, b, T0)
            for l in range(w.L):
                qd = torch.from_numpy(q_direction(w, seed, l)).to(device)
                k[l, b, :, p, :] = (w.needle_scale * qd).to(torch.float16)
    return k, v


def step_pool_fast(w: Workload, seed: int, R: int, device):
    """R pooled step inputs drawn on `device` (same distributions as
    step_pool; different values)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 104729 + 3)
    qdt = torch.bfloat16 if w.q_dtype == "bf16" else torch.float16
    q = torch.randn((R, w.L, w.B, w.Hq, w.d), generator=gen, device=device)
    if w.needle:
        qd = torch.stack([torch.from_numpy(q_direction(w, seed, l)) for l in range(w.L)]).to(device)
        qd = qd.repeat_interleave(w.g, dim=1)  # [L][Hq][d]
        q = qd[None, :, None] + w.q_noise * q
    q = q.to(qdt)
    kn = torch.randn((R, w.L, w.B, w.Hkv, w.d), generator=gen, device=device).to(torch.float16)
    vn = torch.randn((R, w.L, w.B, w.Hkv, w.d), generator=gen, device=device).to(torch.float16)
    lg = torch.randn((R, w.B, w.V), generator=gen, device=device) * w.logit_sigma
    idx = torch.randint(0, w.V, (R, w.B), generator=gen, device=device)
    spike = torch.rand((R, w.B), generator=gen, device=device) * w.spike_hi
    lg.scatter_add_(2, idx[..., None], spike[..., None])
    return q, kn, vn, lg.contiguous()
