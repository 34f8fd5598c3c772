"""The oracle's pins catch plausible mistakes in it.

Each case plants one slip in the CPU oracle (a dropped term, a wrong sign or
index, a swapped weight, an off-by-one window, the wrong tie order, a wrong
scale) by replacing one oracle function for the duration of the case, then
runs the pins of test_oracle_pins.py: at least one of them must fail.  The
unmodified oracle passes them all (checked first).  Nothing here touches the
CUDA path."""
import math

import numpy as np
import pytest

import test_oracle_pins as pins
from oracle import confkv_oracle as orc

F32 = np.float32


def _run_pins():
    """{pin name: exception type name} of the pins that fail (with
    representative parameters)."""
    runs = {
        "uniform": lambda: [pins.test_uniform_logits_closed_form(V) for V in (2, 7, 50257)],
        "one_hot": pins.test_one_hot_limit,
        "two_token": lambda: [pins.test_two_token_closed_form(z) for z in (-7.5, -0.5, 0.0, 2.0, 9.0)],
        "scipy": pins.test_entropy_margin_top1_against_scipy,
        "dup_max": pins.test_duplicated_maximum_gives_zero_margin,
        "range": pins.test_confidence_range_extremes,
        "constants": pins.test_weights_and_hyperparameters_match_pages,
        "tau_inclusive": pins.test_budget_threshold_is_inclusive,
        "tau_f64": pins.test_budget_decides_in_float64,
        "sdpa": lambda: [pins.test_attention_matches_torch_sdpa(*a) for a in ((4, 4, 9), (10, 2, 37))],
        "online": lambda: [pins.test_online_softmax_equals_two_pass(b) for b in (1, 16, 1000)],
        "mass": pins.test_mass_is_head_average,
        "ema": pins.test_ema_closed_form,
        "int8": pins.test_int8_round_trip_bound_and_absmax,
        "int8_edge": pins.test_int8_scale_of_zero_channel_and_half_even,
        "brute_force": pins.test_bottom_k_brute_force,
        "ties": pins.test_ties_break_to_older_position,
        "hand_step": pins.test_hand_derived_step,
        "noop": pins.test_noop_limit_equals_full_fp16_attention,
        "noop_int8": pins.test_noop_limit_with_int8_history,
        "trajectory": pins.test_trajectory_invariants_protected_window_and_length_law,
    }
    failed = {}
    for name, fn in runs.items():
        try:
            fn()
        except Exception as e:   # an assertion, or the slip breaking the oracle outright
            failed[name] = type(e).__name__
    return failed


# ------------------------------------------------------------ planted slips

def _conf_variant(kind):
    def f(logits, w_H=0.4, w_m=0.3, w_p=0.3):
        z = np.asarray(logits, dtype=np.float64).ravel()
        V = z.size
        zmax = z.max()
        logp = z - (zmax + math.log(np.exp(z - zmax).sum()))
        p = np.exp(logp)
        nz = p > 0
        H = float(-(p[nz] * logp[nz]).sum())
        H_hat = H if kind == "entropy_not_normalised" else H / math.log(V)
        i1 = int(np.argmax(logp))
        m = float(logp[i1] - np.delete(logp, i1).max())
        if kind == "margin_sign":
            m = -m
        p1 = float(p[i1])
        if kind == "p1_second":
            p1 = float(np.sort(p)[-2])
        sig = 1.0 / (1.0 + math.exp(-m))
        if kind == "drop_entropy":
            c = w_H + w_m * sig + w_p * p1
        elif kind == "weights_swapped":
            c = w_m * (1.0 - H_hat) + w_H * sig + w_p * p1
        else:
            c = w_H * (1.0 - H_hat) + w_m * sig + w_p * p1
        return orc.Confidence(c=float(c), H_hat=float(H_hat), m=m, p1=p1)
    return f


def _attention_variant(kind):
    def f(q, K, V):
        q = np.asarray(q, dtype=np.float64)
        K = np.asarray(K, dtype=np.float64)
        Vv = np.asarray(V, dtype=np.float64)
        Hq, d = q.shape
        n, Hkv, _ = K.shape
        g = Hq // Hkv
        o = np.zeros((Hq, d))
        p = np.zeros((Hq, n))
        for h in range(Hq):
            hk = h % Hkv if kind == "kv_head_index" else h // g
            s = K[:, hk, :] @ q[h]
            if kind != "no_sqrt_d":
                s = s / math.sqrt(d)
            e = np.exp(s - s.max())
            pp = e / e.sum()
            p[h] = pp
            o[h] = (Vv[:, hk, :].T @ pp) if kind != "values_are_keys" else (K[:, hk, :].T @ pp)
        return o, p
    return f


def _select_variant(kind):
    def f(a, pos, t, P, N, alpha):
        pos = np.asarray(pos, dtype=np.int64)
        k = max(0, pos.size - int(N))
        if k == 0:
            return np.zeros(0, dtype=np.int64)
        lim = t - P + 1 if kind == "protect_off_by_one" else t - P
        cand = np.nonzero(pos < lim)[0]
        if cand.size < k:
            raise ValueError("budget below the protected window")
        s = orc.rank_scores(np.asarray(a)[cand], pos[cand], alpha)
        tie = -pos[cand] if kind == "ties_to_newer" else pos[cand]
        order = np.lexsort((tie, s))
        if kind == "evict_largest":
            order = order[::-1]
        return cand[order[:k]]
    return f


_prefill_unit = orc.prefill_unit
_step_unit = orc.step_unit

SLIPS = {
    # confidence (c and the budget)
    "c: entropy term dropped": ("confidence", _conf_variant("drop_entropy")),
    "c: entropy not divided by log V": ("confidence", _conf_variant("entropy_not_normalised")),
    "c: margin sign flipped": ("confidence", _conf_variant("margin_sign")),
    "c: p(1) taken from the second token": ("confidence", _conf_variant("p1_second")),
    "c: entropy and margin weights swapped": ("confidence", _conf_variant("weights_swapped")),
    "budget: c > tau instead of c >= tau": (
        "budget", lambda c, tau, nh, nl: int(nh) if float(c) > float(tau) else int(nl)),
    "budget: tight and loose swapped": (
        "budget", lambda c, tau, nh, nl: int(nl) if float(c) >= float(tau) else int(nh)),
    "budget: compared in float32": (
        "budget", lambda c, tau, nh, nl: int(nh) if np.float32(c) >= np.float32(tau) else int(nl)),
    # attention and mass
    "attention: no 1/sqrt(d)": ("attention", _attention_variant("no_sqrt_d")),
    "attention: KV head h % Hkv instead of h // G": ("attention", _attention_variant("kv_head_index")),
    "attention: keys used as values": ("attention", _attention_variant("values_are_keys")),
    "mass: sum over heads instead of mean": (
        "attention_mass", lambda p: np.asarray(p, dtype=np.float64).sum(axis=0)),
    "mass: first head only": ("attention_mass", lambda p: np.asarray(p, dtype=np.float64)[0]),
    # EMA, ranking, bottom-k
    "ema: lambda and 1 - lambda swapped": (
        "ema", lambda a, A, lam: (1.0 - lam) * np.asarray(a, float) + lam * np.asarray(A, float)),
    "ema: new mass ignored": ("ema", lambda a, A, lam: lam * np.asarray(a, float) + 0.0 * np.asarray(A, float)),
    "rank: alpha on recency": (
        "rank_scores", lambda a, pos, alpha: (1 - alpha) * orc._minmax(a) + alpha * orc._minmax(pos)),
    "rank: recency reversed": (
        "rank_scores", lambda a, pos, alpha: alpha * orc._minmax(a) + (1 - alpha) * orc._minmax(-np.asarray(pos))),
    "evict: protected window one short": ("select_evictions", _select_variant("protect_off_by_one")),
    "evict: ties go to the newer position": ("select_evictions", _select_variant("ties_to_newer")),
    "evict: largest scores evicted": ("select_evictions", _select_variant("evict_largest")),
    # INT8 storage
    "int8: scale absmax / 128": (
        "quant_scale", lambda m: np.where(np.asarray(m, F32) > 0, np.asarray(m, F32) / F32(128.0), F32(1.0)).astype(F32)),
    "int8: floor instead of round": (
        "quantize", lambda x, s: np.clip(np.floor(np.asarray(x, F32) / np.asarray(s, F32)), -127, 127).astype(np.int8)),
    "int8: codes clamped to 126": (
        "quantize", lambda x, s: np.clip(np.rint(np.asarray(x, F32) / np.asarray(s, F32)), -126, 126).astype(np.int8)),
    "int8: dequantised without the scale": ("dequantize", lambda code, s: np.asarray(code).astype(F32)),
    # FP16 window and positions
    "window: one entry too many in FP16 at prefill": (
        "prefill_unit", lambda k, v, W: _prefill_unit(k, v, W + 1)),
    "step: the new token at position t + 1": (
        "step_unit", lambda prm, st, t, q, kn, vn, N: _step_unit(prm, st, t + 1, q, kn, vn, N)),
}


def test_unmodified_oracle_passes_every_pin():
    assert _run_pins() == {}


@pytest.mark.parametrize("slip", sorted(SLIPS))
def test_planted_slip_fails_a_pin(slip, monkeypatch):
    attr, fn = SLIPS[slip]
    monkeypatch.setattr(orc, attr, fn)
    failed = _run_pins()
    # caught by a pin's own check, not only by the slip crashing the oracle
    assert "AssertionError" in failed.values(), "no pin caught %r: %r" % (slip, failed)
