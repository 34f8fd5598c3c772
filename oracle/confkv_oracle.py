"""CPU oracle of the CONF-KV per-decode-step cache manager (float64, numpy).

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline / reference leg import this module.  The library's
decode path never calls it, and it shares no code with the CUDA path: it is a
plain, slow restatement of the method, written to be checked by eye.

Sources (cited by page title and section):

* [rainbus] "CONF-KV: Confidence-Aware KV Cache Eviction with Mixed-Precision
  Storage for Long-Horizon LLM", paper.rainbus.top/paper/2605.24786:
  section 前置知识 (prerequisites: EMA, blockwise online softmax),
  核心方法 (core method: c, budget, rank s_i), 方法步骤详情 (Algorithm 1,
  steps 1-13), 复现评估 (hyper-parameters).
* [gist-de] the same paper summarised at gist.science/de/paper/2605.24786,
  "Technischer Zusammenfassung": Methodik -- Konfidenzschätzung (c and its
  weights), Adaptive Budgetauswahl (N_high / N_low), Token-Ranking und
  Eviktion (EMA mass + recency, protected window P), Systemintegration (FP16
  window W, per-head per-channel INT8, pyramidal budgets, contiguous
  compaction).  gist.science/ja and /es carry the same summary and formula.

What the oracle computes, per sequence b and decode step at position t
(Algorithm 1 of [rainbus], 方法步骤详情):

1. p = softmax(logits); c = w_H (1 - H(p)/log V) + w_m sigmoid(log p(1) -
   log p(2)) + w_p p(1)                                      -> `confidence`
2. N_l = N_high[l] if c >= tau else N_low[l]                 -> `budget`
3. per layer l: attention of the decode query over the cache plus the new
   token (two-pass softmax), attention mass A_i               -> `attention`
4. EMA a_i <- lam a_i + (1 - lam) A_i                         -> `ema`
5. if |C_l| > N_l: rank the non-protected entries by
   s_i = alpha a_hat_i + (1 - alpha) r_hat_i, evict the |C_l| - N_l lowest
                                                             -> `select_evictions`
6. append the new K/V in FP16; entries older than the newest W go to INT8
   with per-(head, channel) scales                           -> `step_unit`

Readings where the pages leave a step open (the plainest one the rest of the
pages supports):

R1  Attention covers C plus the new token; eviction acts on C without it; the
    new token is appended afterwards, so |C| after a step is min(|C|, N) + 1.
R2  a_hat and r_hat are min-max normalised over the candidate set; r uses the
    absolute token position; a constant term normalises to 0.
R3  Protected = the P newest resident entries = positions >= t - P; the
    candidates are the entries with position < t - P.
R4  A_i = softmax probability of the single decode query, averaged over all
    Hq query heads; the new token takes part in the normalisation.
R5  An entry is FP16 iff its position is > t - W after appending token t;
    prefill positions >= T0 - W start in FP16.  INT8 entries stay INT8.
R6  INT8 scales per (sequence, layer, KV head, channel), K and V separately,
    fixed at prefill: s = absmax / 127 in float32 (s = 1 if absmax = 0);
    code = clamp(rint(x / s), -127, 127) in float32, round half to even;
    dequantised value = float32(code) * s.
R7  Prefill entries start with a = 0; a new token's EMA starts from 0, so
    after its first update a = (1 - lam) A_self.
R8  Eviction order: (s ascending, position ascending).
R9  The budget test is c >= tau, exactly, in float64 (the pages fix no
    precision).  A c within 1e-6 of tau may be decided the other way by an
    implementation that forms c in fp32; the parity harness flags such steps
    and checks the result against this rule applied with the other budget.
R10 A duplicated maximum gives p(2) = p(1), m = 0.
R12 Raw logits (temperature 1), natural logarithm.
R13 Evicted entries are reported as absolute positions, ascending.

Pins (tests/test_oracle_pins.py): uniform and one-hot logits, the V = 2 closed
form, scipy's entropy / softmax, torch's scaled-dot-product attention, the
online-softmax recurrence, sum of mass = 1, the no-op limit = full attention,
the EMA closed form, the protected window, the length law, the INT8 error
bound, brute-force bottom-k on tiny caches, and a hand-derived step.
Parity unpinned: the readings R2, R4 and R7 themselves (no printed value on
the pages tells them apart from other readings).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

F32 = np.float32


# ----------------------------------------------------------------------------
# Hyper-parameters
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Params:
    """Shape and hyper-parameters.  Defaults follow [rainbus] 核心方法 and
    复现评估: weights (0.4, 0.3, 0.3), tau = 0.7, alpha = 0.65; lam = 0.9
    from [rainbus] 前置知识 (EMA)."""

    L: int
    Hq: int
    Hkv: int
    d: int
    V: int
    W: int
    P: int
    n_high: tuple
    n_low: tuple
    tau: float = 0.7
    alpha: float = 0.65
    lam: float = 0.9
    w_H: float = 0.4
    w_m: float = 0.3
    w_p: float = 0.3

    @classmethod
    def from_workload(cls, w) -> "Params":
        return cls(L=w.L, Hq=w.Hq, Hkv=w.Hkv, d=w.d, V=w.V, W=w.W, P=w.P,
                   n_high=tuple(w.n_high), n_low=tuple(w.n_low), tau=w.tau,
                   alpha=w.alpha, lam=w.lam, w_H=w.w_H, w_m=w.w_m, w_p=w.w_p)


# ----------------------------------------------------------------------------
# Step 1-2: confidence and budget
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Confidence:
    c: float
    H_hat: float
    m: float
    p1: float


def confidence(logits, w_H=0.4, w_m=0.3, w_p=0.3) -> Confidence:
    """c = w_H (1 - H_hat) + w_m sigmoid(m) + w_p p(1).

    H_hat = H(p) / log V is the normalised entropy of p = softmax(logits),
    m = log p(1) - log p(2) the log-probability margin between the two most
    likely tokens and p(1) the top probability ([gist-de] Konfidenzschätzung;
    [rainbus] 核心方法 and Algorithm 1 steps 2-3).  0 log 0 is taken as 0."""
    z = np.asarray(logits, dtype=np.float64).ravel()
    V = z.size
    if V < 2:
        raise ValueError("the normalised entropy needs V >= 2")
    zmax = z.max()
    log_z = zmax + math.log(np.exp(z - zmax).sum())
    logp = z - log_z
    p = np.exp(logp)
    nz = p > 0
    H = float(-(p[nz] * logp[nz]).sum())
    H_hat = H / math.log(V)
    i1 = int(np.argmax(logp))
    rest = np.delete(logp, i1)
    m = float(logp[i1] - rest.max())
    p1 = float(p[i1])
    sig = 1.0 / (1.0 + math.exp(-m))
    c = w_H * (1.0 - H_hat) + w_m * sig + w_p * p1
    return Confidence(c=float(c), H_hat=float(H_hat), m=m, p1=p1)


def budget(c: float, tau: float, n_high: int, n_low: int) -> int:
    """N = N_high if c >= tau else N_low ([gist-de] Adaptive Budgetauswahl;
    [rainbus] Algorithm 1 step 4).  N_high is the tight budget.  The
    comparison is exact, in float64 (R9)."""
    return int(n_high) if float(c) >= float(tau) else int(n_low)


# ----------------------------------------------------------------------------
# INT8 storage (R6)
# ----------------------------------------------------------------------------

def quant_scale(absmax) -> np.ndarray:
    """Per-(head, channel) scale s = absmax / 127 in float32, 1 where absmax
    is 0 ([gist-de] Systemintegration: INT8 per head and channel)."""
    a = np.asarray(absmax, dtype=F32)
    s = a / F32(127.0)
    return np.where(a > 0, s, F32(1.0)).astype(F32)


def quantize(x, s) -> np.ndarray:
    """code = clamp(rint(x / s), -127, 127); x / s in float32, rint rounds
    half to even."""
    q = np.asarray(x, dtype=F32) / np.asarray(s, dtype=F32)
    return np.clip(np.rint(q), -127, 127).astype(np.int8)


def dequantize(code, s) -> np.ndarray:
    """float32(code) * s."""
    return np.asarray(code).astype(F32) * np.asarray(s, dtype=F32)


# ----------------------------------------------------------------------------
# Step 3: attention and attention mass
# ----------------------------------------------------------------------------

def attention(q, K, V):
    """Single-query attention, two-pass softmax, float64.

    q [Hq][d]; K, V [n][Hkv][d] (already dequantised).  Query head h reads
    KV head h // (Hq / Hkv).  Returns (o [Hq][d], p [Hq][n]) with
    p[h, i] = exp(s_hi - max_i s_hi) / sum_i exp(...), s_hi = q_h . k_i / sqrt(d)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    Vv = np.asarray(V, dtype=np.float64)
    Hq, d = q.shape
    n, Hkv, _ = K.shape
    g = Hq // Hkv
    o = np.zeros((Hq, d))
    p = np.zeros((Hq, n))
    for hk in range(Hkv):
        qh = q[hk * g:(hk + 1) * g]                    # [g][d]
        s = (qh @ K[:, hk, :].T) / math.sqrt(d)        # [g][n]
        mx = s.max(axis=1, keepdims=True)              # pass 1: max
        e = np.exp(s - mx)
        pp = e / e.sum(axis=1, keepdims=True)          # pass 2: normalise
        p[hk * g:(hk + 1) * g] = pp
        o[hk * g:(hk + 1) * g] = pp @ Vv[:, hk, :]
    return o, p


def attention_online(q, K, V, block: int = 128):
    """The same attention with the blockwise online-softmax recurrence
    ([rainbus] 前置知识: blockwise online softmax keeps a running maximum and
    normaliser while walking the blocks and gives the exact softmax result).
    Used only to pin `attention` against an independent formulation."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    Vv = np.asarray(V, dtype=np.float64)
    Hq, d = q.shape
    n, Hkv, _ = K.shape
    g = Hq // Hkv
    out = np.zeros((Hq, d))
    for h in range(Hq):
        hk = h // g
        m_run, l_run, acc = -np.inf, 0.0, np.zeros(d)
        for j0 in range(0, n, block):
            s = K[j0:j0 + block, hk, :] @ q[h] / math.sqrt(d)
            m_new = max(m_run, float(s.max()))
            scale = math.exp(m_run - m_new) if m_run > -np.inf else 0.0
            e = np.exp(s - m_new)
            l_run = l_run * scale + float(e.sum())
            acc = acc * scale + e @ Vv[j0:j0 + block, hk, :]
            m_run = m_new
        out[h] = acc / l_run
    return out


def attention_mass(p) -> np.ndarray:
    """A_i = (1 / Hq) sum_h p[h, i] (reading R4)."""
    return np.asarray(p, dtype=np.float64).mean(axis=0)


# ----------------------------------------------------------------------------
# Steps 4-5: EMA, ranking, bottom-k
# ----------------------------------------------------------------------------

def ema(a, A, lam: float):
    """a <- lam a + (1 - lam) A ([rainbus] 前置知识: EMA with lam = 0.9)."""
    return lam * np.asarray(a, dtype=np.float64) + (1.0 - lam) * np.asarray(A, dtype=np.float64)


def _minmax(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    lo, hi = x.min(), x.max()
    if hi > lo:
        return (x - lo) / (hi - lo)
    return np.zeros_like(x)


def rank_scores(a, pos, alpha: float) -> np.ndarray:
    """s_i = alpha a_hat_i + (1 - alpha) r_hat_i over the candidate set
    ([rainbus] 核心方法, alpha = 0.65; normalisation per reading R2)."""
    return alpha * _minmax(a) + (1.0 - alpha) * _minmax(pos)


def select_evictions(a, pos, t: int, P: int, N: int, alpha: float) -> np.ndarray:
    """Indices of the entries to evict from a cache of n = len(pos) entries
    (the new token excluded, R1).  Nothing happens unless n > N; then the
    n - N candidates (position < t - P, R3) with the smallest (s, position)
    go ([rainbus] Algorithm 1 steps 6-9; [gist-de] Token-Ranking und
    Eviktion)."""
    pos = np.asarray(pos, dtype=np.int64)
    n = pos.size
    k = max(0, n - int(N))
    if k == 0:
        return np.zeros(0, dtype=np.int64)
    cand = np.nonzero(pos < t - P)[0]
    if cand.size < k:
        raise ValueError("budget below the protected window: cannot evict %d of %d candidates" % (k, cand.size))
    s = rank_scores(np.asarray(a)[cand], pos[cand], alpha)
    order = np.lexsort((pos[cand], s))   # primary key s, then position (R8)
    return cand[order[:k]]


# ----------------------------------------------------------------------------
# Cache state of one (sequence, layer)
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class UnitState:
    """Resident entries of one (sequence, layer), in position order.

    pos [n] int64; a [n] float64 (EMA mass); is8 [n] bool.  Stored values:
    INT8 entries keep their codes in kc / vc (int8 [n][Hkv][d]); FP16 entries
    keep their fp16 values in kh / vh (float16 [n][Hkv][d]).  sK, sV float32
    [Hkv][d] are the fixed scales."""

    pos: np.ndarray
    a: np.ndarray
    is8: np.ndarray
    kc: np.ndarray
    vc: np.ndarray
    kh: np.ndarray
    vh: np.ndarray
    sK: np.ndarray
    sV: np.ndarray

    @property
    def n(self) -> int:
        return int(self.pos.size)

    def keys(self) -> np.ndarray:
        return np.where(self.is8[:, None, None], dequantize(self.kc, self.sK[None]),
                        self.kh.astype(F32)).astype(np.float64)

    def values(self) -> np.ndarray:
        return np.where(self.is8[:, None, None], dequantize(self.vc, self.sV[None]),
                        self.vh.astype(F32)).astype(np.float64)

    def copy(self) -> "UnitState":
        return UnitState(*(np.array(getattr(self, f.name), copy=True) for f in dataclasses.fields(self)))


def prefill_unit(k, v, W: int) -> UnitState:
    """Cache of one (sequence, layer) after a prefill of T0 tokens.

    k, v: float16 [Hkv][T0][d].  Scales from the absmax over all T0 tokens
    (R6); positions >= T0 - W stay FP16, older ones are stored as INT8 (R5);
    a = 0 (R7)."""
    k = np.asarray(k, dtype=np.float16)
    v = np.asarray(v, dtype=np.float16)
    Hkv, T0, d = k.shape
    if T0 > 0:
        sK = quant_scale(np.abs(k.astype(F32)).max(axis=1))
        sV = quant_scale(np.abs(v.astype(F32)).max(axis=1))
    else:
        sK = np.ones((Hkv, d), F32)
        sV = np.ones((Hkv, d), F32)
    pos = np.arange(T0, dtype=np.int64)
    is8 = pos < T0 - W
    kt = np.transpose(k, (1, 0, 2))   # [T0][Hkv][d]
    vt = np.transpose(v, (1, 0, 2))
    kc = np.where(is8[:, None, None], quantize(kt.astype(F32), sK[None]), 0).astype(np.int8)
    vc = np.where(is8[:, None, None], quantize(vt.astype(F32), sV[None]), 0).astype(np.int8)
    kh = np.where(is8[:, None, None], np.float16(0), kt).astype(np.float16)
    vh = np.where(is8[:, None, None], np.float16(0), vt).astype(np.float16)
    return UnitState(pos=pos, a=np.zeros(T0), is8=is8, kc=kc, vc=vc, kh=kh, vh=vh, sK=sK, sV=sV)


@dataclasses.dataclass
class UnitStepResult:
    o: np.ndarray            # [Hq][d] attention output
    evicted: np.ndarray      # absolute positions, ascending
    mass: np.ndarray         # [n + 1] attention mass of the entries (new token last)
    a_updated: np.ndarray    # [n + 1] EMA after the update, before eviction
    scores: Optional[np.ndarray]   # s_i of the candidates (None if no eviction)
    cand_pos: Optional[np.ndarray]  # positions of the candidates
    k: int                   # number of evicted entries
    state: UnitState         # cache after the step


def step_unit(prm: Params, st: UnitState, t: int, q, k_new, v_new, N: int) -> UnitStepResult:
    """One decode step of one (sequence, layer) at position t with budget N
    ([rainbus] Algorithm 1 steps 1 and 5-13, readings R1-R8)."""
    k_new = np.asarray(k_new, dtype=np.float16)
    v_new = np.asarray(v_new, dtype=np.float16)
    n = st.n
    K = np.concatenate([st.keys(), k_new.astype(F32).astype(np.float64)[None]], axis=0)
    Vv = np.concatenate([st.values(), v_new.astype(F32).astype(np.float64)[None]], axis=0)
    o, p = attention(q, K, Vv)
    A = attention_mass(p)                                   # [n + 1]
    a_upd = ema(np.concatenate([st.a, [0.0]]), A, prm.lam)  # new token starts at 0 (R7)

    ev = select_evictions(a_upd[:n], st.pos, t, prm.P, N, prm.alpha)
    scores = cand_pos = None
    if ev.size:
        cand = np.nonzero(st.pos < t - prm.P)[0]
        cand_pos = st.pos[cand]
        scores = rank_scores(a_upd[cand], cand_pos, prm.alpha)
    keep = np.ones(n, dtype=bool)
    keep[ev] = False

    Hkv, d = st.sK.shape
    new = UnitState(
        pos=np.concatenate([st.pos[keep], [t]]).astype(np.int64),
        a=np.concatenate([a_upd[:n][keep], [a_upd[n]]]),
        is8=np.concatenate([st.is8[keep], [False]]),
        kc=np.concatenate([st.kc[keep], np.zeros((1, Hkv, d), np.int8)]),
        vc=np.concatenate([st.vc[keep], np.zeros((1, Hkv, d), np.int8)]),
        kh=np.concatenate([st.kh[keep], k_new[None]]),
        vh=np.concatenate([st.vh[keep], v_new[None]]),
        sK=st.sK.copy(), sV=st.sV.copy())
    # The entry at position t - W leaves the FP16 window (R5).
    leave = np.nonzero((new.pos == t - prm.W) & ~new.is8)[0]
    for i in leave:
        new.kc[i] = quantize(new.kh[i].astype(F32), new.sK)
        new.vc[i] = quantize(new.vh[i].astype(F32), new.sV)
        new.kh[i] = 0
        new.vh[i] = 0
        new.is8[i] = True
    return UnitStepResult(o=o, evicted=np.sort(st.pos[ev]), mass=A, a_updated=a_upd,
                          scores=scores, cand_pos=cand_pos, k=int(ev.size), state=new)


# ----------------------------------------------------------------------------
# Whole batch
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class StepOutput:
    out: np.ndarray                 # [L][B][Hq][d]
    budget: np.ndarray              # [B][L] int
    c: np.ndarray                   # [B]
    evicted: List[List[np.ndarray]]  # [L][B] ascending positions
    n_evicted: np.ndarray           # [L][B]
    units: List[List[UnitStepResult]]  # [L][B]


class Oracle:
    """Whole-batch oracle: B sequences x L layers of UnitState."""

    def __init__(self, prm: Params):
        self.prm = prm
        self.states: List[List[UnitState]] = []
        self.T0: List[int] = []
        self.step_idx = 0

    def prefill(self, k, v, prefill_len: Sequence[int]):
        """k, v: float16 [L][B][Hkv][Tmax][d] (numpy or torch); sequence b
        uses its first prefill_len[b] tokens."""
        k = _np(k)
        v = _np(v)
        L, B = k.shape[0], k.shape[1]
        self.T0 = [int(x) for x in prefill_len]
        self.states = [[prefill_unit(k[l, b, :, :self.T0[b]], v[l, b, :, :self.T0[b]], self.prm.W)
                        for b in range(B)] for l in range(L)]
        self.step_idx = 0

    def position(self, b: int) -> int:
        return self.T0[b] + self.step_idx

    def step(self, q, k_new, v_new, logits) -> StepOutput:
        """q [L][B][Hq][d]; k_new, v_new [L][B][Hkv][d] fp16; logits [B][V]."""
        prm = self.prm
        q = _np(q).astype(np.float64)
        k_new = _np(k_new)
        v_new = _np(v_new)
        logits = _np(logits)
        L, B = q.shape[0], q.shape[1]
        out = np.zeros((L, B, prm.Hq, prm.d))
        bud = np.zeros((B, L), dtype=np.int64)
        cs = np.zeros(B)
        ev = [[None] * B for _ in range(L)]
        nev = np.zeros((L, B), dtype=np.int64)
        units = [[None] * B for _ in range(L)]
        for b in range(B):
            cs[b] = confidence(logits[b], prm.w_H, prm.w_m, prm.w_p).c
            t = self.position(b)
            for l in range(L):
                N = budget(cs[b], prm.tau, prm.n_high[l], prm.n_low[l])
                bud[b, l] = N
                r = step_unit(prm, self.states[l][b], t, q[l, b], k_new[l, b], v_new[l, b], N)
                self.states[l][b] = r.state
                out[l, b] = r.o
                ev[l][b] = r.evicted
                nev[l, b] = r.k
                units[l][b] = r
        self.step_idx += 1
        return StepOutput(out=out, budget=bud, c=cs, evicted=ev, n_evicted=nev, units=units)


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        return x.numpy()
    return np.asarray(x)
