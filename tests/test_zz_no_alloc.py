"""The allocation-free confidence call (confkv_confidence_noalloc) against the
decode step's own confidence output.

That call exists for callers that cannot allocate device memory where they
need the score (a plug-in whose host owns every buffer, a real-time loop
that forbids allocation, code that must not synchronise): its scratch is a
fixed array inside the library.  This file is collected last so that a run
stopping at its first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import confidence_gated_kv_gb300 as ck
from confidence_gated_kv_gb300 import binding
from workload import Workload, prefill_batch

from _parity import C_TOL, confident_logits, step_inputs

pytestmark = pytest.mark.gpu


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
        status = ck.lib().confkv_confidence_noalloc(
            ctypes.c_void_p(lg.data_ptr()), w.B, w.V, w.w_H, w.w_m, w.w_p,
            ctypes.c_void_p(got.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert status == binding.OK
        torch.cuda.synchronize()
        err = float((got - ref).abs().max())
        assert np.isfinite(err) and err <= C_TOL, "call %d: |c - c_step| = %g" % (call, err)


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
