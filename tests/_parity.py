"""Shared helpers of the GPU parity tests: run the CUDA path (through the C
ABI binding) and the CPU oracle on the same seeded inputs and compare.

Tolerances: attention output <= 2e-3 max-abs, EMA <= 1e-5, confidence <= 1e-6;
budgets, evicted positions, INT8 codes, FP16 values, scales and positions
exact; the per-token attention mass (recovered from the GPU's EMA update) to
1e-4 relative plus the fp32 rounding of the EMA it is recovered from.  Two
floating-point decisions may legitimately differ between the float64 oracle
and the GPU's fp32: a budget when |c - tau| < 1e-6, and an eviction among
candidates whose oracle score lies within 1e-5 of the k-th score.  When a
sequence's budget differs, the GPU's evictions of every layer of that
sequence are checked against the oracle's eviction rule applied with the
GPU's budget to the pre-step state (same count, same set up to the tie
band); when an eviction differs inside the tie band it is checked for
validity the same way.  The units concerned are then re-synchronised to the
oracle's state by importing it (inputs only ever flow oracle -> GPU, never
the other way); every other unit is compared as usual.
"""
from __future__ import annotations

import dataclasses
import types

import numpy as np
import torch

from oracle import confkv_oracle as orc
import confidence_gated_kv_gb300 as ck

OUT_TOL = 2e-3
EMA_TOL = 1e-5
C_TOL = 1e-6
TAU_BAND = 1e-6
TIE_BAND = 1e-5
MASS_RTOL = 1e-3
F32_EPS = float(np.finfo(np.float32).eps)


@dataclasses.dataclass
class Flags:
    budget: int = 0
    ties: int = 0
    steps: int = 0
    evictions: int = 0
    max_out_err: float = 0.0
    max_ema_err: float = 0.0
    max_mass_rel_err: float = 0.0
    mass_checked: int = 0
    alt_checked: int = 0


def unit_to_host(st: orc.UnitState) -> dict:
    """Oracle state of one (sequence, layer) in the library's import layout."""
    i8 = st.is8
    return dict(pos8=st.pos[i8].astype(np.int32), ema8=st.a[i8].astype(np.float32),
                k8=st.kc[i8], v8=st.vc[i8], posR=st.pos[~i8].astype(np.int32),
                emaR=st.a[~i8].astype(np.float32), k16=st.kh[~i8], v16=st.vh[~i8],
                sK=st.sK, sV=st.sV)


def compare_unit(gpu: dict, st: orc.UnitState, where: str, ema_tol: float = EMA_TOL) -> float:
    """Exported GPU unit vs oracle unit.  Returns the max EMA error."""
    gpos = np.concatenate([gpu["pos8"], gpu["posR"]]).astype(np.int64)
    assert np.array_equal(np.sort(gpos), np.sort(st.pos)), where + ": resident positions differ"
    np.testing.assert_array_equal(gpu["sK"], st.sK, err_msg=where + ": K scales")
    np.testing.assert_array_equal(gpu["sV"], st.sV, err_msg=where + ": V scales")
    idx = {int(p): i for i, p in enumerate(st.pos)}
    i8 = np.array([idx[int(p)] for p in gpu["pos8"]], dtype=np.int64)
    iR = np.array([idx[int(p)] for p in gpu["posR"]], dtype=np.int64)
    assert np.all(st.is8[i8]) and not np.any(st.is8[iR]), where + ": FP16 / INT8 membership"
    np.testing.assert_array_equal(gpu["k8"], st.kc[i8], err_msg=where + ": K codes")
    np.testing.assert_array_equal(gpu["v8"], st.vc[i8], err_msg=where + ": V codes")
    np.testing.assert_array_equal(gpu["k16"], st.kh[iR], err_msg=where + ": K fp16")
    np.testing.assert_array_equal(gpu["v16"], st.vh[iR], err_msg=where + ": V fp16")
    err = 0.0
    if i8.size:
        err = max(err, float(np.abs(gpu["ema8"].astype(np.float64) - st.a[i8]).max()))
    if iR.size:
        err = max(err, float(np.abs(gpu["emaR"].astype(np.float64) - st.a[iR]).max()))
    assert err <= ema_tol, "%s: EMA error %.3g" % (where, err)
    return err


def check_evictions(gpu_ev: np.ndarray, r: orc.UnitStepResult, where: str) -> bool:
    """True if the GPU evicted exactly the oracle's set; False for an allowed
    difference inside the tie band (raises otherwise)."""
    want = np.asarray(r.evicted)
    got = np.asarray(gpu_ev)
    assert got.size == want.size, "%s: evicted %d, oracle %d" % (where, got.size, want.size)
    assert np.all(np.diff(got) > 0) if got.size > 1 else True, where + ": not ascending"
    if np.array_equal(got, want):
        return True
    # only candidates inside the tie band of the k-th score may differ
    order = np.lexsort((r.cand_pos, r.scores))
    kth = r.scores[order[r.k - 1]]
    amb = set(r.cand_pos[np.abs(r.scores - kth) < TIE_BAND].tolist())
    cand = set(r.cand_pos.tolist())
    assert set(got.tolist()) <= cand, where + ": evicted a non-candidate"
    assert set(got.tolist()) - amb == set(want.tolist()) - amb, where + ": eviction outside the tie band"
    return False


def oracle_selection(pre: orc.UnitState, a_upd, t: int, prm: orc.Params, N: int):
    """The oracle's eviction rule (R1-R3, R8; [rainbus] Algorithm 1 steps
    6-9) applied with budget N to the pre-step state `pre`, whose EMA after
    this step's update is a_upd[:n].  Same fields as the ones check_evictions
    reads from a UnitStepResult."""
    n = pre.n
    ev = orc.select_evictions(np.asarray(a_upd)[:n], pre.pos, t, prm.P, N, prm.alpha)
    scores = cand_pos = None
    if ev.size:
        cand = np.nonzero(pre.pos < t - prm.P)[0]
        cand_pos = pre.pos[cand]
        scores = orc.rank_scores(np.asarray(a_upd)[cand], cand_pos, prm.alpha)
    return types.SimpleNamespace(evicted=np.sort(pre.pos[ev]), scores=scores, cand_pos=cand_pos,
                                 k=int(ev.size))


def check_mass(gpu_pre: dict, gpu_post: dict, r: orc.UnitStepResult, pre: orc.UnitState, t: int,
               lam: float, where: str) -> tuple:
    """Per-token attention mass of the GPU against the oracle's, recovered
    from the GPU's own EMA update a' = lam a + (1 - lam) A of every entry that
    survived the step (and of the new token, whose a starts at 0).  The GPU
    updates in fp32 with lam rounded to fp32, so A = (a' - lam32 a) /
    (1 - lam32) from its fp32 a and a'; the bound adds the fp32 rounding of
    a' (amplified by 1 / (1 - lam)) to MASS_RTOL relative.  Returns (entries
    checked, max relative error)."""
    lam32 = float(np.float32(lam))
    a_pre = {int(p): float(a) for p, a in zip(np.concatenate([gpu_pre["pos8"], gpu_pre["posR"]]),
                                              np.concatenate([gpu_pre["ema8"], gpu_pre["emaR"]]))}
    a_post = {int(p): float(a) for p, a in zip(np.concatenate([gpu_post["pos8"], gpu_post["posR"]]),
                                               np.concatenate([gpu_post["ema8"], gpu_post["emaR"]]))}
    want = {int(p): float(m) for p, m in zip(pre.pos, r.mass[:pre.n])}
    want[int(t)] = float(r.mass[pre.n])
    worst, count = 0.0, 0
    for p, a1 in a_post.items():
        a0 = 0.0 if p == t else a_pre.get(p)
        if a0 is None or p not in want:
            continue
        got = (a1 - lam32 * a0) / (1.0 - lam32)
        tol = MASS_RTOL * abs(want[p]) + 2.0 * F32_EPS * abs(a1) / (1.0 - lam32) + 1e-30
        err = abs(got - want[p])
        assert err <= tol, "%s: mass of position %d: %.9g vs oracle %.9g" % (where, p, got, want[p])
        if want[p] > 0:
            worst = max(worst, err / want[p])
        count += 1
    return count, worst


class Pair:
    """CUDA cache + oracle driven by the same inputs."""

    def __init__(self, w, seed: int, prefill_len=None, cap=None, max_evict=0, k=None, v=None,
                 compaction=0, mode=0):
        self.w = w
        self.seed = seed
        self.prm = orc.Params.from_workload(w)
        self.T0 = list(prefill_len) if prefill_len is not None else [w.T0] * w.B
        if k is None:
            from workload import prefill_batch
            k, v = prefill_batch(w, seed, "cpu", T0=max(self.T0) if self.T0 else 0)
        self.oracle = orc.Oracle(self.prm)
        self.oracle.prefill(k, v, self.T0)
        self.cache = ck.Cache(ck.config_from_workload(w, cap=cap, max_evict=max_evict, compaction=compaction))
        self.cache.prefill(k.cuda(), v.cuda(), self.T0)
        self.cache.set_step_mode(mode)
        self.flags = Flags()
        self.launches = 0          # kernel launches the plain steps took (the library's count)
        self.exports = {}          # (b, l) -> last GPU export that matched the oracle
        self.peak_entries = 0      # largest oracle resident count after a step
        self.peak_bytes = 0
        self.peak_exact = True     # false once a budget decision differed

    def resync(self, units=None):
        units = units if units is not None else [(b, l) for b in range(self.w.B) for l in range(self.w.L)]
        for b, l in units:
            self.cache.import_unit(b, l, unit_to_host(self.oracle.states[l][b]))
            self.exports.pop((b, l), None)

    def compare_states(self, units=None):
        units = units if units is not None else [(b, l) for b in range(self.w.B) for l in range(self.w.L)]
        for b, l in units:
            g = self.cache.export_unit(b, l)
            e = compare_unit(g, self.oracle.states[l][b], "unit b%d l%d" % (b, l))
            self.flags.max_ema_err = max(self.flags.max_ema_err, e)
            self.exports[(b, l)] = g
        return units

    def oracle_footprint(self):
        """Resident entries and K/V bytes at stored widths, over all units."""
        w = self.w
        ent = byt = 0
        for l in range(w.L):
            for b in range(w.B):
                st = self.oracle.states[l][b]
                n8 = int(st.is8.sum())
                ent += st.n
                byt += w.Hkv * w.d * (2 * n8 + 4 * (st.n - n8))
        return ent, byt

    def compare_footprint(self):
        """The library's resident counters against the oracle's state."""
        ent, byt = self.oracle_footprint()
        st = self.cache.stats()
        assert st["resident"] == ent, "resident entries %d vs oracle %d" % (st["resident"], ent)
        assert st["resident_bytes"] == byt, "resident bytes %d vs oracle %d" % (st["resident_bytes"], byt)
        if self.peak_exact:
            assert st["peak_resident"] == self.peak_entries, \
                "peak resident %d vs oracle %d" % (st["peak_resident"], self.peak_entries)
            assert st["peak_resident_bytes"] == self.peak_bytes, \
                "peak resident bytes %d vs oracle %d" % (st["peak_resident_bytes"], self.peak_bytes)
        assert st["steps"] == self.flags.steps, "steps %d vs %d" % (st["steps"], self.flags.steps)
        return st

    def step(self, q, kn, vn, lg, check_state=True, gpu_step=None):
        """One step on both sides; `gpu_step(q, kn, vn, lg)` replaces the
        plain cache.step call (graph replays) and returns the output dict."""
        w = self.w
        if gpu_step is None:
            self.launches += self.cache.step_launches()
            o = self.cache.step(q.cuda(), kn.cuda(), vn.cuda(), lg.cuda())
        else:
            o = gpu_step(q, kn, vn, lg)
        torch.cuda.synchronize()
        pre = [row[:] for row in self.oracle.states]          # states are replaced, never mutated
        t_of = [self.oracle.position(b) for b in range(w.B)]
        res = self.oracle.step(q, kn, vn, lg)
        self.flags.steps += 1
        out = o["out"].cpu().numpy()
        bud = o["budget"].cpu().numpy()
        conf = o["confidence"].cpu().numpy()
        nev = o["n_evicted"].cpu().numpy()
        ev = o["evicted"].cpu().numpy()
        div_seq = set()
        for b in range(w.B):
            assert abs(conf[b] - res.c[b]) <= C_TOL, "c of seq %d: %r vs %r" % (b, conf[b], res.c[b])
            if not np.array_equal(bud[b], res.budget[b]):
                assert abs(res.c[b] - w.tau) < TAU_BAND, "budget of seq %d differs with c = %r" % (b, res.c[b])
                self.flags.budget += 1
                div_seq.add(b)
                self.peak_exact = False
        err = float(np.abs(out - res.out).max())
        self.flags.max_out_err = max(self.flags.max_out_err, err)
        assert err <= OUT_TOL, "attention output error %.3g" % err
        resync = set()
        for l in range(w.L):
            for b in range(w.B):
                where = "step %d l%d b%d" % (self.oracle.step_idx - 1, l, b)
                k = int(nev[l, b])
                r = res.units[l][b]
                if b in div_seq:
                    # the GPU decided the other budget inside the tau band:
                    # its evictions must follow the rule with that budget
                    r = oracle_selection(pre[l][b], res.units[l][b].a_updated, t_of[b], self.prm, int(bud[b, l]))
                    self.flags.alt_checked += 1
                    resync.add((b, l))
                assert k == r.k, "%s: n_evicted %d vs %d" % (where, k, r.k)
                self.flags.evictions += k
                if k and not check_evictions(ev[l, b, :k], r, where):
                    self.flags.ties += 1
                    resync.add((b, l))
        if check_state:
            keep = [(b, l) for b in range(w.B) for l in range(w.L) if (b, l) not in resync]
            before = {u: self.exports.get(u) for u in keep}
            self.compare_states(keep)
            for b, l in keep:
                if before[(b, l)] is not None:
                    c, e = check_mass(before[(b, l)], self.exports[(b, l)], res.units[l][b], pre[l][b],
                                      t_of[b], w.lam, "step %d l%d b%d" % (self.oracle.step_idx - 1, l, b))
                    self.flags.mass_checked += c
                    self.flags.max_mass_rel_err = max(self.flags.max_mass_rel_err, e)
        else:
            self.exports.clear()
        if resync:
            self.resync(sorted(resync))
        ent, byt = self.oracle_footprint()
        self.peak_entries = max(self.peak_entries, ent)
        self.peak_bytes = max(self.peak_bytes, byt)
        if check_state:
            self.compare_footprint()
        st = self.cache.stats()
        assert st["device_status"] == 0
        return o, res


def step_inputs(w, seed: int, r: int):
    """Pooled step inputs r of the whole batch (CPU torch tensors)."""
    from workload import step_unit, step_logits
    qdt = torch.bfloat16 if w.q_dtype == "bf16" else torch.float16
    q = torch.empty((w.L, w.B, w.Hq, w.d), dtype=qdt)
    kn = torch.empty((w.L, w.B, w.Hkv, w.d), dtype=torch.float16)
    vn = torch.empty_like(kn)
    lg = torch.empty((w.B, w.V), dtype=torch.float32)
    for b in range(w.B):
        lg[b] = torch.from_numpy(step_logits(w, seed, r, b))
        for l in range(w.L):
            qq, kk, vv = step_unit(w, seed, r, b, l)
            q[l, b] = qq
            kn[l, b] = torch.from_numpy(kk)
            vn[l, b] = torch.from_numpy(vv)
    return q, kn, vn, lg


def confident_logits(V: int, B: int, seed: int) -> torch.Tensor:
    """Logits with one overwhelming token: c close to 1 (tight budget)."""
    g = np.random.default_rng(seed)
    lg = g.normal(size=(B, V)).astype(np.float32)
    lg[np.arange(B), g.integers(0, V, B)] += 40.0
    return torch.from_numpy(lg)
