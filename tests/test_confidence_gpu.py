"""The confidence reduction on the GPU at the limits the pages fix, against
the float64 oracle.

CONF-KV's confidence (gist.science/de/paper/2605.24786, Konfidenzschätzung;
paper.rainbus.top/paper/2605.24786, 核心方法) is
c = 0.4 (1 - H/log V) + 0.3 sigmoid(log p1 - log p2) + 0.3 p1.  Its limits:
uniform logits give H/log V = 1, a zero margin and p1 = 1/V, so
c = 0.15 + 0.3/V; a one-hot distribution gives c = 1; two tokens give the
binary-entropy closed form; a duplicated maximum gives a zero margin (R10);
a constant shift of every logit changes nothing.  Each case runs through
confkv_step (one sequence per case, the budget of every layer checked
exactly) at the full Qwen vocabulary, so the duplicated maxima land inside
one vocabulary chunk, on both sides of a chunk boundary and in the ragged
last chunk of the device reduction.
"""
import numpy as np
import pytest
import torch

import confidence_gated_kv_gb300 as ck
from oracle import confkv_oracle as orc
from workload import Workload, prefill_batch

from _parity import C_TOL, TAU_BAND, step_inputs

pytestmark = pytest.mark.gpu

V_QWEN = 152064


def _cache(V: int, B: int):
    w = Workload(name="t_conf", B=B, L=2, Hq=4, Hkv=2, d=64, V=V, T0=40, steps=1,
                 n_high=(24, 24), n_low=(32, 32), P=4, W=16, q_dtype="f16")
    k, v = prefill_batch(w, 5, "cpu")
    cache = ck.Cache(ck.config_from_workload(w))
    cache.prefill(k.cuda(), v.cuda(), [w.T0] * w.B)
    return w, cache


def _check_rows(lg: np.ndarray, labels, closed=None):
    """One decode step with these logits rows, c and budgets against the
    oracle; also confkv_confidence_noalloc on the same rows."""
    B, V = lg.shape
    w, cache = _cache(V, B)
    q, kn, vn, _ = step_inputs(w, 5, 0)
    dev = torch.from_numpy(lg).cuda()
    o = cache.step(q.cuda(), kn.cuda(), vn.cuda(), dev)
    c_na = torch.full((B,), float("nan"), dtype=torch.float32, device="cuda")
    ck.binding.confidence_noalloc(dev, c_na)
    torch.cuda.synchronize()
    c_gpu = o["confidence"].cpu().numpy().astype(np.float64)
    c_noalloc = c_na.cpu().numpy().astype(np.float64)
    bud = o["budget"].cpu().numpy()
    for b in range(B):
        ref = orc.confidence(lg[b]).c
        if closed is not None and closed[b] is not None:
            assert abs(ref - closed[b]) <= 1e-12, "%s: oracle %r vs closed form %r" % (labels[b], ref, closed[b])
        assert abs(c_gpu[b] - ref) <= C_TOL, "%s: step c %r vs oracle %r" % (labels[b], c_gpu[b], ref)
        assert abs(c_noalloc[b] - ref) <= C_TOL, "%s: noalloc c %r vs oracle %r" % (labels[b], c_noalloc[b], ref)
        if abs(ref - w.tau) >= TAU_BAND:
            want = [orc.budget(ref, w.tau, w.n_high[l], w.n_low[l]) for l in range(w.L)]
            assert list(bud[b]) == want, "%s: budgets %r vs %r" % (labels[b], list(bud[b]), want)
    return c_gpu


def test_limits_at_the_full_qwen_vocabulary():
    V = V_QWEN
    g = np.random.default_rng(2024)
    rows, labels, closed = [], [], []

    def add(z, label, c=None):
        rows.append(np.asarray(z, dtype=np.float32))
        labels.append(label)
        closed.append(c)

    add(np.full(V, 0.25), "uniform", 0.15 + 0.3 / V)
    z = np.zeros(V)
    z[12345] = 1e4
    add(z, "one-hot", 1.0)
    # the whole distribution shifted far below zero: c depends on differences only
    z = g.normal(0.0, 1.5, V)
    z[g.integers(V)] += g.uniform(0.0, 14.0)
    add(z, "spiked")
    add(z - 1e4, "spiked, shifted by -1e4")
    # duplicated maxima (R10: zero margin) in several places of the reduction
    for label, idx in [("dup max inside one 4096-logit chunk", (100, 3000)),
                       ("dup max across 4095 / 4096", (4095, 4096)),
                       ("dup max across 4001 / 4002", (4001, 4002)),
                       ("dup max in the ragged last chunk", (V - 2, V - 1)),
                       ("dup max first and last logit", (0, V - 1))]:
        z = g.normal(0.0, 1.0, V)
        z[list(idx)] = 25.0
        add(z, label)
    # a maximum in the last logit alone
    z = g.normal(0.0, 1.0, V)
    z[V - 1] = 30.0
    add(z, "max in the last logit")
    c = _check_rows(np.stack(rows), labels, closed)
    assert abs(c[0] - (0.15 + 0.3 / V)) <= C_TOL and abs(c[1] - 1.0) <= C_TOL


def test_two_token_vocabulary_closed_form():
    # V = 2, logits (z, 0): p1 = sigmoid(|z|), margin |z|, H/log 2 = h_b(p1)/log 2
    zs = [-30.0, -8.0, -2.0, -0.5, 0.0, 0.3, 1.0, 3.0, 8.0, 15.0, 30.0]
    lg = np.array([[z, 0.0] for z in zs], dtype=np.float32)
    closed = []
    for z in zs:
        z = float(np.float32(z))           # the logit the kernels see
        p1 = 1.0 / (1.0 + np.exp(-abs(z)))
        p2 = 1.0 - p1
        h = -(p1 * np.log(p1) + (p2 * np.log(p2) if p2 > 0 else 0.0))
        closed.append(0.4 * (1.0 - h / np.log(2.0)) + 0.3 * p1 + 0.3 * p1)
    _check_rows(lg, ["V=2, z=%g" % z for z in zs], closed)


def test_uniform_and_one_hot_at_the_gpt2_vocabulary():
    V = 50257
    z1 = np.zeros(V, np.float32)
    z1[V - 1] = 1e4
    _check_rows(np.stack([np.full(V, -3.0, np.float32), z1]), ["uniform", "one-hot last"],
                [0.15 + 0.3 / V, 1.0])
