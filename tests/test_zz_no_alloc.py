"""The allocation-free confidence call (confkv_confidence_noalloc) against the
decode step's own confidence output and against the float64 oracle.

That call exists for callers that cannot allocate device memory where they
need the score (a plug-in whose host owns every buffer, a real-time loop
that forbids allocation, code that must not synchronise): its scratch is a
fixed array inside the library, 4096 vocabulary-chunk partials per GPU, so
B * ceil(V / 4096) may not exceed 4096.  This file is collected last so that
a run stopping at its first failure has already run every other test; it
also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import confidence_gated_kv_gb300 as ck
from confidence_gated_kv_gb300 import binding
from oracle import confkv_oracle as orc
from workload import Workload, prefill_batch

from _parity import C_TOL, confident_logits, step_inputs

pytestmark = pytest.mark.gpu

V_QWEN = 152064
MAX_PARTIALS = 4096


def _noalloc(lg_dev, out, w_H=0.4, w_m=0.3, w_p=0.3):
    B, V = int(lg_dev.shape[0]), int(lg_dev.shape[1])
    return ck.lib().confkv_confidence_noalloc(
        ctypes.c_void_p(lg_dev.data_ptr()), B, V, w_H, w_m, w_p, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_confidence_matches_the_step_output_on_consecutive_calls():
    w = Workload(name="noalloc", B=3, L=2, Hq=8, Hkv=2, d=128, V=50257, T0=64, steps=2,
                 n_high=(32, 32), n_low=(48, 48), P=8, W=16, q_dtype="bf16")
    k, v = prefill_batch(w, 31, "cpu")
    cache = ck.Cache(ck.config_from_workload(w))
    cache.prefill(k.cuda(), v.cuda(), [w.T0] * w.B)
    got = torch.empty(w.B, dtype=torch.float32, device="cuda")
    for call in range(2):
        q, kn, vn, lg = step_inputs(w, 31, call)
        if call == 1:
            lg = confident_logits(w.V, w.B, 77)   # a very different distribution
        lg = lg.cuda()
        ref = cache.step(q.cuda(), kn.cuda(), vn.cuda(), lg)["confidence"]
        got.fill_(float("nan"))
        assert _noalloc(lg, got, w.w_H, w.w_m, w.w_p) == binding.OK
        torch.cuda.synchronize()
        err = float((got - ref).abs().max())
        assert np.isfinite(err) and err <= C_TOL, "call %d: |c - c_step| = %g" % (call, err)


def _rows(V: int, B: int, seed: int) -> np.ndarray:
    """Uniform, one-hot and spiked rows (the closed-form limits of
    gist.science/de/paper/2605.24786, Konfidenzschätzung, and the workloads'
    generator), cycled over B rows."""
    g = np.random.default_rng(seed)
    lg = g.normal(0.0, 1.5, size=(B, V)).astype(np.float32)
    for b in range(B):
        kind = b % 4
        if kind == 0:
            lg[b] = 0.5
        elif kind == 1:
            lg[b] = 0.0
            lg[b, g.integers(V)] = 1e4
        elif kind == 2:
            lg[b, g.integers(V)] += g.uniform(0.0, 14.0)
        else:
            lg[b, [0, V - 1]] = 20.0        # duplicated maximum at both ends
    return lg


def test_noalloc_confidence_matches_the_oracle_at_the_capacity_edge():
    # V = 152064 needs 38 partials per row: 107 rows (4066 partials) fit the
    # library's scratch, 108 (4104) do not.  Two calls in a row with
    # different rows: the shared scratch keeps the first call's partials,
    # which the second call must fully overwrite.
    V = V_QWEN
    parts = (V + 4095) // 4096
    B_fit = MAX_PARTIALS // parts
    assert B_fit == 107 and (B_fit + 1) * parts > MAX_PARTIALS
    for call, seed in enumerate((41, 42)):
        lg = _rows(V, B_fit, seed)
        kind = np.arange(B_fit) % 4
        if call == 1:
            lg, kind = lg[::-1].copy(), kind[::-1].copy()
        dev = torch.from_numpy(lg).cuda()
        got = torch.full((B_fit,), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(dev, got) == binding.OK
        torch.cuda.synchronize()
        c = got.cpu().numpy().astype(np.float64)
        ref = np.array([orc.confidence(lg[b]).c for b in range(B_fit)])
        err = np.abs(c - ref)
        assert np.all(np.isfinite(c)) and err.max() <= C_TOL, \
            "call %d: max |c - oracle| = %g at row %d" % (call, err.max(), int(err.argmax()))
        # the closed forms of the uniform and one-hot rows
        assert np.all(np.abs(c[kind == 0] - (0.15 + 0.3 / V)) <= C_TOL)
        assert np.all(np.abs(c[kind == 1] - 1.0) <= C_TOL)
    lg = torch.zeros((B_fit + 1, V), dtype=torch.float32, device="cuda")
    out = torch.empty(B_fit + 1, dtype=torch.float32, device="cuda")
    assert _noalloc(lg, out) == binding.ECAPACITY


def test_noalloc_confidence_rejects_sizes_beyond_its_scratch():
    lg = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    out = torch.empty(2, dtype=torch.float32, device="cuda")
    L = ck.lib()
    # 4097 rows of up to 4096 logits need 4097 partials > 4096
    assert L.confkv_confidence_noalloc(ctypes.c_void_p(lg.data_ptr()), 4097, 8, 0.4, 0.3, 0.3,
                                       ctypes.c_void_p(out.data_ptr()), None) == binding.ECAPACITY
    assert L.confkv_confidence_noalloc(ctypes.c_void_p(lg.data_ptr()), 2, 8 * 4096 * 1024, 0.4, 0.3, 0.3,
                                       ctypes.c_void_p(out.data_ptr()), None) == binding.ECAPACITY
    assert L.confkv_confidence_noalloc(None, 2, 8, 0.4, 0.3, 0.3,
                                       ctypes.c_void_p(out.data_ptr()), None) == binding.EINVAL
