"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: a closed
form, a library routine (scipy, torch), an invariant the pages state, brute
force on tiny inputs, or a step derived by hand.  A plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, the
wrong eviction order) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

from oracle import confkv_oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _prm(**kw):
    base = dict(L=1, Hq=4, Hkv=2, d=16, V=100, W=8, P=2, n_high=(6,), n_low=(12,))
    base.update(kw)
    return orc.Params(**base)


# ---------------------------------------------------------------- confidence

@pytest.mark.parametrize("V", [2, 7, 50257, 152064])
def test_uniform_logits_closed_form(V):
    # p uniform: H = log V so H_hat = 1, m = 0, p(1) = 1/V -> c = 0.3*0.5 + 0.3/V
    r = orc.confidence(np.full(V, 0.25, dtype=np.float32))
    assert abs(r.H_hat - 1.0) < 1e-12
    assert r.m == 0.0
    assert abs(r.c - (0.15 + 0.3 / V)) < 1e-12


def test_one_hot_limit():
    z = np.zeros(50257, dtype=np.float32)
    z[123] = 1e4
    r = orc.confidence(z)
    assert abs(r.c - 1.0) < 1e-12
    assert r.H_hat < 1e-12
    assert abs(r.p1 - 1.0) < 1e-12


@pytest.mark.parametrize("z", list(np.linspace(-20, 20, 81)))
def test_two_token_closed_form(z):
    # V = 2, logits (z, 0): p(1) = sigmoid(|z|), m = |z|,
    # H = binary entropy (scipy), H_hat = H / log 2.
    r = orc.confidence(np.array([z, 0.0]))
    p1 = scipy.special.expit(abs(z))
    H = scipy.stats.entropy([scipy.special.expit(z), scipy.special.expit(-z)])
    want = 0.4 * (1 - H / math.log(2)) + 0.3 * scipy.special.expit(abs(z)) + 0.3 * p1
    assert abs(r.c - want) < 1e-12
    assert abs(r.m - abs(z)) < 1e-12


def test_entropy_margin_top1_against_scipy():
    rng = np.random.default_rng(5)
    for trial in range(20):
        V = int(rng.integers(2, 3000))
        z = rng.normal(0, rng.uniform(0.1, 4), V)
        z[rng.integers(V)] += rng.uniform(0, 14)
        r = orc.confidence(z)
        p = scipy.special.softmax(z)
        lp = np.sort(scipy.special.log_softmax(z))
        assert abs(r.H_hat - scipy.stats.entropy(p) / math.log(V)) < 1e-10
        assert abs(r.m - (lp[-1] - lp[-2])) < 1e-10
        assert abs(r.p1 - p.max()) < 1e-12
        assert 0.0 <= r.c <= 1.0


def test_duplicated_maximum_gives_zero_margin():
    z = np.array([0.1, 3.0, -2.0, 3.0, 1.0])
    assert orc.confidence(z).m == 0.0


def test_confidence_range_extremes():
    rng = np.random.default_rng(1)
    for scale in [1e-6, 1e-2, 1, 30, 1e3]:
        z = rng.normal(0, scale, 500)
        c = orc.confidence(z).c
        assert 0.0 <= c <= 1.0


def test_weights_and_hyperparameters_match_pages():
    g = json.load(open(os.path.join(GOLD, "page_constants.json")))
    p = _prm()
    assert (p.w_H, p.w_m, p.w_p) == (g["w_H"], g["w_m"], g["w_p"])
    assert p.tau == g["tau"] and p.alpha == g["alpha"] and p.lam == g["lambda"]
    # a confident one-hot step picks the tight budget, a uniform one the loose
    c_hi = orc.confidence(np.eye(1, 1000, 3)[0] * 1e4).c
    c_lo = orc.confidence(np.zeros(1000)).c
    w = g["wikitext"]
    assert orc.budget(c_hi, g["tau"], w["N_high"], w["N_low"]) == w["N_high"]
    assert orc.budget(c_lo, g["tau"], w["N_high"], w["N_low"]) == w["N_low"]


def test_budget_threshold_is_inclusive():
    # [gist-de] Adaptive Budgetauswahl: c >= tau takes the tight budget; R9:
    # exactly at tau counts, the next float64 below does not
    assert orc.budget(0.7, 0.7, 10, 20) == 10
    below = float(np.nextafter(0.7, 0.0))
    assert orc.budget(below, 0.7, 10, 20) == 20
    above = float(np.nextafter(0.7, 1.0))
    assert orc.budget(above, 0.7, 10, 20) == 10


def test_budget_decides_in_float64():
    # R9 fixes no narrower precision: a c one float64 step below tau that
    # would round up to float32(tau) still takes the loose budget
    c = float(np.nextafter(0.7, 0.0))
    assert np.float32(c) == np.float32(0.7)
    assert orc.budget(c, 0.7, 10, 20) == 20
    assert orc.budget(0.5, 0.7, 10, 20) == 20 and orc.budget(0.9, 0.7, 10, 20) == 10


# ---------------------------------------------------------------- attention

def _sdpa(q, K, V):
    """torch's scaled-dot-product attention in float64, KV heads expanded to
    the query heads (query head h reads KV head h // g)."""
    Hq, d = q.shape
    n, Hkv, _ = K.shape
    g = Hq // Hkv
    qt = torch.tensor(q, dtype=torch.float64)[:, None, :]            # [Hq][1][d]
    kt = torch.tensor(K, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(g, 0)
    vt = torch.tensor(V, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(g, 0)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0, :].numpy()


@pytest.mark.parametrize("Hq,Hkv,n", [(1, 1, 1), (4, 4, 9), (10, 2, 37), (40, 8, 130)])
def test_attention_matches_torch_sdpa(Hq, Hkv, n):
    rng = np.random.default_rng(n)
    d = 16
    q = rng.normal(size=(Hq, d))
    K = rng.normal(size=(n, Hkv, d)) * 2
    V = rng.normal(size=(n, Hkv, d))
    o, p = orc.attention(q, K, V)
    np.testing.assert_allclose(o, _sdpa(q, K, V), atol=1e-12)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert abs(orc.attention_mass(p).sum() - 1.0) < 1e-12


@pytest.mark.parametrize("block", [1, 3, 16, 128, 1000])
def test_online_softmax_equals_two_pass(block):
    rng = np.random.default_rng(block)
    q = rng.normal(size=(10, 32))
    K = rng.normal(size=(301, 2, 32)) * 3
    V = rng.normal(size=(301, 2, 32))
    o2, _ = orc.attention(q, K, V)
    np.testing.assert_allclose(orc.attention_online(q, K, V, block), o2, atol=1e-12)


def test_mass_is_head_average():
    # Two query heads over one KV head with hand-chosen scores
    # head 0 scores (0, log 3) * sqrt(d)^-1 ... use d = 1 and q = (1), (-1)
    q = np.array([[1.0], [-1.0]])
    K = np.array([[[0.0]], [[math.log(3.0)]]])
    V = np.array([[[1.0]], [[0.0]]])
    o, p = orc.attention(q, K, V)
    # head 0: p = (1/4, 3/4); head 1: p = (3/4, 1/4)
    np.testing.assert_allclose(p, [[0.25, 0.75], [0.75, 0.25]], atol=1e-15)
    np.testing.assert_allclose(orc.attention_mass(p), [0.5, 0.5], atol=1e-15)
    np.testing.assert_allclose(o[:, 0], [0.25, 0.75], atol=1e-15)


# ---------------------------------------------------------------- EMA

def test_ema_closed_form():
    A = 0.37
    a = np.zeros(3)
    for k in range(1, 60):
        a = orc.ema(a, np.full(3, A), 0.9)
        np.testing.assert_allclose(a, (1 - 0.9 ** k) * A, rtol=1e-14, atol=1e-16)


# ---------------------------------------------------------------- INT8

def test_int8_round_trip_bound_and_absmax():
    rng = np.random.default_rng(2)
    x = (rng.normal(size=(500, 3, 64)) * rng.uniform(0.01, 5, size=(1, 3, 64))).astype(np.float16)
    xf = x.astype(np.float32)
    amax = np.abs(xf).max(axis=0)
    s = orc.quant_scale(amax)
    code = orc.quantize(xf, s[None])
    assert np.abs(code.astype(int)).max() <= 127
    err = np.abs(xf - orc.dequantize(code, s[None]))
    # |x - x_hat| <= s/2, plus one float32 rounding of code * s
    assert np.all(err <= s[None] * 0.5 + np.abs(xf) * 2.0 ** -23)
    # the absmax element of every (head, channel) maps to +-127
    idx = np.abs(xf).argmax(axis=0)
    hit = np.take_along_axis(code, idx[None], 0)[0]
    assert np.all(np.abs(hit.astype(int)) == 127)
    # out-of-range values clamp
    big = orc.quantize(np.full((3, 64), 1e4, np.float32), s)
    assert np.all(big == 127)
    assert np.all(orc.quantize(-np.full((3, 64), 1e4, np.float32), s) == -127)


def test_int8_scale_of_zero_channel_and_half_even():
    assert orc.quant_scale(np.float32(0.0)) == np.float32(1.0)
    s = orc.quant_scale(np.float32(127.0))   # s = 1 exactly
    assert s == np.float32(1.0)
    np.testing.assert_array_equal(orc.quantize(np.array([2.5, 3.5, -2.5, -0.5], np.float32), s),
                                  [2, 4, -2, 0])


# ---------------------------------------------------------------- ranking

def test_bottom_k_brute_force():
    rng = np.random.default_rng(3)
    for trial in range(300):
        n = int(rng.integers(2, 13))
        t = 100
        pos = np.sort(rng.choice(np.arange(t - 30, t), size=n, replace=False))
        a = rng.uniform(0, 1, n)
        P = int(rng.integers(0, 6))
        cand = np.nonzero(pos < t - P)[0]
        N = int(rng.integers(max(0, n - cand.size), n + 2))
        ev = orc.select_evictions(a, pos, t, P, N, 0.65)
        k = max(0, n - N)
        assert ev.size == k
        if k == 0:
            continue
        s = 0.65 * (a[cand] - a[cand].min()) / (np.ptp(a[cand]) or 1) + \
            0.35 * (pos[cand] - pos[cand].min()) / (np.ptp(pos[cand]) or 1)
        best = min(itertools.combinations(range(cand.size), k), key=lambda c: s[list(c)].sum())
        assert set(cand[list(best)]) == set(ev)
        assert np.all(pos[ev] < t - P)


def test_ties_break_to_older_position():
    pos = np.array([3, 4, 5, 6, 7, 8])
    a = np.array([0.5, 0.2, 0.2, 0.2, 0.9, 0.1])
    # alpha = 1: pure EMA mass, three exact ties at 0.2; t = 9, P = 1 protects 8
    ev = orc.select_evictions(a, pos, 9, 1, 4, 1.0)
    assert sorted(pos[ev]) == [4, 5]


def test_hand_derived_step():
    g = json.load(open(os.path.join(GOLD, "hand_step.json")))
    prm = orc.Params(L=1, Hq=g["Hq"], Hkv=g["Hkv"], d=g["d"], V=2, W=g["W"], P=g["P"],
                     n_high=(g["N"],), n_low=(g["N"],), alpha=g["alpha"], lam=g["lambda"])
    n = len(g["pos"])
    vals = np.array(g["values"], np.float16)[:, None, :]
    st = orc.UnitState(pos=np.array(g["pos"]), a=np.array(g["a"]), is8=np.zeros(n, bool),
                       kc=np.zeros((n, 1, 2), np.int8), vc=np.zeros((n, 1, 2), np.int8),
                       kh=np.zeros((n, 1, 2), np.float16), vh=vals,
                       sK=np.ones((1, 2), np.float32), sV=np.ones((1, 2), np.float32))
    r = orc.step_unit(prm, st, g["t"], np.array(g["q"]), np.zeros((1, 2), np.float16),
                      np.array([g["v_new"]], np.float16), g["N"])
    np.testing.assert_allclose(r.o[0], g["expected_o"], atol=1e-14)
    assert list(r.evicted) == g["expected_evicted"]
    assert list(r.state.pos) == g["expected_pos_after"]
    np.testing.assert_allclose(r.state.a, g["expected_a_after"], atol=1e-15)
    np.testing.assert_allclose(r.scores, g["expected_scores"], atol=1e-14)


# ---------------------------------------------------------------- trajectories

def _random_inputs(rng, prm, B, T0):
    k = rng.normal(size=(prm.L, B, prm.Hkv, T0, prm.d)).astype(np.float16)
    v = rng.normal(size=(prm.L, B, prm.Hkv, T0, prm.d)).astype(np.float16)
    return k, v


def _step_inputs(rng, prm, B, confident):
    q = rng.normal(size=(prm.L, B, prm.Hq, prm.d))
    kn = rng.normal(size=(prm.L, B, prm.Hkv, prm.d)).astype(np.float16)
    vn = rng.normal(size=(prm.L, B, prm.Hkv, prm.d)).astype(np.float16)
    lg = np.zeros((B, prm.V), np.float32)
    for b in range(B):
        if confident[b]:
            lg[b, rng.integers(prm.V)] = 1e4
        else:
            lg[b] = rng.normal(size=prm.V)
    return q, kn, vn, lg


def test_noop_limit_equals_full_fp16_attention():
    # N and W beyond every cache length: nothing is evicted or quantised and
    # the output is plain attention over the whole fp16 history.
    prm = _prm(L=2, W=10 ** 6, P=2, n_high=(10 ** 6,) * 2, n_low=(10 ** 6,) * 2)
    rng = np.random.default_rng(7)
    B, T0 = 2, 20
    k, v = _random_inputs(rng, prm, B, T0)
    o = orc.Oracle(prm)
    o.prefill(k, v, [T0, 13])
    hist_k = [[list(np.transpose(k[l, b, :, :o.T0[b]], (1, 0, 2))) for b in range(B)] for l in range(prm.L)]
    hist_v = [[list(np.transpose(v[l, b, :, :o.T0[b]], (1, 0, 2))) for b in range(B)] for l in range(prm.L)]
    for step in range(6):
        q, kn, vn, lg = _step_inputs(rng, prm, B, [step % 2 == 0, True])
        res = o.step(q, kn, vn, lg)
        assert res.n_evicted.sum() == 0
        for l in range(prm.L):
            for b in range(B):
                hist_k[l][b].append(kn[l, b])
                hist_v[l][b].append(vn[l, b])
                K = np.array(hist_k[l][b], np.float64)
                Vv = np.array(hist_v[l][b], np.float64)
                np.testing.assert_allclose(res.out[l, b], _sdpa(q[l, b], K, Vv), atol=1e-12)


def test_noop_limit_with_int8_history():
    # No eviction, small W: positions older than the window are read back as
    # dequantised INT8 with the prefill absmax scales.
    W = 4
    prm = _prm(L=1, W=W, P=2, n_high=(10 ** 6,), n_low=(10 ** 6,))
    rng = np.random.default_rng(11)
    B, T0 = 1, 12
    k, v = _random_inputs(rng, prm, B, T0)
    o = orc.Oracle(prm)
    o.prefill(k, v, [T0])
    sK = orc.quant_scale(np.abs(k[0, 0].astype(np.float32)).max(axis=1))
    sV = orc.quant_scale(np.abs(v[0, 0].astype(np.float32)).max(axis=1))
    allk = list(np.transpose(k[0, 0], (1, 0, 2)))
    allv = list(np.transpose(v[0, 0], (1, 0, 2)))
    for step in range(8):
        t = T0 + step
        q, kn, vn, lg = _step_inputs(rng, prm, B, [False])
        res = o.step(q, kn, vn, lg)
        allk.append(kn[0, 0])
        allv.append(vn[0, 0])
        Ks, Vs = [], []
        for p in range(t + 1):
            if p < t - W:
                Ks.append(orc.dequantize(orc.quantize(allk[p].astype(np.float32), sK), sK))
                Vs.append(orc.dequantize(orc.quantize(allv[p].astype(np.float32), sV), sV))
            else:
                Ks.append(allk[p].astype(np.float32))
                Vs.append(allv[p].astype(np.float32))
        np.testing.assert_allclose(res.out[0, 0], _sdpa(q[0, 0], np.array(Ks, np.float64),
                                                        np.array(Vs, np.float64)), atol=1e-12)
        st = o.states[0][0]
        assert np.array_equal(st.is8, st.pos <= t - W)


def test_trajectory_invariants_protected_window_and_length_law():
    prm = _prm(L=2, W=6, P=3, n_high=(5, 4), n_low=(9, 7))
    rng = np.random.default_rng(13)
    B, T0 = 3, 15
    k, v = _random_inputs(rng, prm, B, T0)
    o = orc.Oracle(prm)
    o.prefill(k, v, [T0, 2, 9])
    n_prev = [[o.states[l][b].n for b in range(B)] for l in range(prm.L)]
    for step in range(30):
        conf = [bool(rng.integers(2)) for _ in range(B)]
        q, kn, vn, lg = _step_inputs(rng, prm, B, conf)
        res = o.step(q, kn, vn, lg)
        for b in range(B):
            t = o.T0[b] + step
            assert (res.c[b] >= prm.tau) == conf[b]
            for l in range(prm.L):
                N = res.budget[b, l]
                assert N == (prm.n_high[l] if conf[b] else prm.n_low[l])
                ev = res.evicted[l][b]
                assert np.all(ev < t - prm.P)                    # protected window
                assert list(ev) == sorted(ev)
                assert res.n_evicted[l, b] == max(0, n_prev[l][b] - N)
                st = o.states[l][b]
                assert st.n == min(n_prev[l][b], N) + 1          # length law
                assert np.array_equal(st.is8, st.pos <= t - prm.W)  # FP16 window
                # the newest P positions are all still resident
                assert set(range(max(0, t - prm.P), t + 1)) <= set(st.pos.tolist())
                n_prev[l][b] = st.n
