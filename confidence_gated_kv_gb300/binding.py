"""ctypes binding of libconfkv (include/confkv.h).

Argument marshalling only: every step of the decode path runs in the CUDA
library.  PyTorch provides device memory (the workspace and the output
tensors) and the current stream.  If the library has not been built, loading
fails with an error: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libconfkv.so")

OK, EINVAL, ECAPACITY, ECUDA, ETIMEOUT, ENOTIMPL, EDEVICE, ESTATE = 0, -1, -2, -3, -4, -5, -6, -7
Q_FP16, Q_BF16 = 0, 1


class ConfkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (%d)" % (what, status_string(status), status))
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32), ("V", ctypes.c_int32), ("B", ctypes.c_int32),
        ("cap", ctypes.c_int32), ("W", ctypes.c_int32), ("P", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32), ("max_evict", ctypes.c_int32),
        ("tau", ctypes.c_double), ("w_H", ctypes.c_double), ("w_m", ctypes.c_double),
        ("w_p", ctypes.c_double), ("alpha", ctypes.c_float), ("lam", ctypes.c_float),
        ("n_high", ctypes.POINTER(ctypes.c_int32)), ("n_low", ctypes.POINTER(ctypes.c_int32)),
        ("compaction", ctypes.c_int32),
    ]

COMPACT_TAIL_FILL, COMPACT_ORDERED = 0, 1
STEP_AUTO, STEP_SEPARATE = 0, 1
STATUS_CAPACITY, STATUS_EVICT_BOUND, STATUS_BAD_COUNT, STATUS_TIMEOUT = 1, 2, 4, 8


class UnitHost(ctypes.Structure):
    _fields_ = [
        ("n8", ctypes.c_int32), ("nR", ctypes.c_int32),
        ("pos8", ctypes.c_void_p), ("ema8", ctypes.c_void_p),
        ("k8", ctypes.c_void_p), ("v8", ctypes.c_void_p),
        ("posR", ctypes.c_void_p), ("emaR", ctypes.c_void_p),
        ("k16", ctypes.c_void_p), ("v16", ctypes.c_void_p),
        ("sK", ctypes.c_void_p), ("sV", ctypes.c_void_p),
    ]


class Stats(ctypes.Structure):
    _fields_ = [
        ("steps", ctypes.c_int64), ("evicted", ctypes.c_int64), ("moved", ctypes.c_int64),
        ("requantised", ctypes.c_int64), ("attn_bytes", ctypes.c_double),
        ("step_bytes", ctypes.c_double), ("resident", ctypes.c_int64),
        ("resident_bytes", ctypes.c_int64), ("device_status", ctypes.c_int32),
        ("host_h2d_bytes", ctypes.c_int64), ("host_d2h_bytes", ctypes.c_int64),
        ("peak_resident", ctypes.c_int64), ("peak_resident_bytes", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64), ("launches", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libconfkv.so (built in-tree by confidence_gated_kv_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libconfkv.so is not built (%s); run `python -m "
                              "confidence_gated_kv_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sigs = {
            "confkv_workspace_bytes": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(sz)]),
            "confkv_launch_plan": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.c_int64, i32,
                                                  ctypes.POINTER(i32), ctypes.POINTER(i32),
                                                  ctypes.POINTER(i32)]),
            "confkv_create": (ctypes.c_int, [ctypes.POINTER(Config), vp, sz, ctypes.POINTER(vp)]),
            "confkv_destroy": (None, [vp]),
            "confkv_prefill": (ctypes.c_int, [vp, vp, vp, vp, i64, vp]),
            "confkv_step": (ctypes.c_int, [vp] + [vp] * 9 + [vp]),
            "confkv_step_host": (ctypes.c_int, [vp] + [vp] * 9 + [vp]),
            "confkv_export_unit": (ctypes.c_int, [vp, i32, i32, ctypes.POINTER(UnitHost), vp]),
            "confkv_import_unit": (ctypes.c_int, [vp, i32, i32, ctypes.POINTER(UnitHost), vp]),
            "confkv_get_clock": (ctypes.c_int, [vp, vp, ctypes.POINTER(i64)]),
            "confkv_set_clock": (ctypes.c_int, [vp, vp, i64, vp]),
            "confkv_get_stats": (ctypes.c_int, [vp, ctypes.POINTER(Stats), vp]),
            "confkv_profile_enable": (ctypes.c_int, [vp, i32, i32]),
            "confkv_profile_disable": (ctypes.c_int, [vp]),
            "confkv_profile_read": (ctypes.c_int, [vp] + [ctypes.POINTER(ctypes.c_double)] * 3 +
                                    [ctypes.POINTER(i32)]),
            "confkv_attention_plan": (ctypes.c_int, [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
            "confkv_set_attention_ctas": (ctypes.c_int, [vp, i32]),
            "confkv_set_step_mode": (ctypes.c_int, [vp, i32]),
            "confkv_step_launches": (ctypes.c_int, [vp, ctypes.POINTER(i32)]),
            "confkv_attention_grid": (ctypes.c_int, [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
            "confkv_graph_reserve": (ctypes.c_int, [vp, i64]),
            "confkv_graph_advance": (ctypes.c_int, [vp, i64]),
            "confkv_graph_release": (ctypes.c_int, [vp]),
            "confkv_selftest_timeout": (ctypes.c_int, [vp, vp]),
            "confkv_block_offset": (i32, [i32, i32, i32, i32]),
            "confkv_confidence_noalloc": (ctypes.c_int, [vp, i32, i32, ctypes.c_double, ctypes.c_double,
                                                         ctypes.c_double, vp, vp]),
            "confkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "confkv_version": (i32, []),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().confkv_status_string(int(status)).decode()


def block_offset(kind: int, d: int, tau: int, c: int) -> int:
    return int(lib().confkv_block_offset(kind, d, tau, c))


def confidence_noalloc(logits, out, w_H: float = 0.4, w_m: float = 0.3, w_p: float = 0.3,
                       stream=None):
    """Confidence of each row of `logits` (device fp32 [B][V]) into `out`
    (device fp32 [B]) through confkv_confidence_noalloc, which allocates no
    device memory (see include/confkv.h)."""
    B, V = int(logits.shape[0]), int(logits.shape[1])
    _check(lib().confkv_confidence_noalloc(_ptr(logits), B, V, w_H, w_m, w_p, _ptr(out),
                                           _stream(stream)), "confkv_confidence_noalloc")
    return out


def _check(status: int, what: str):
    if status != OK:
        raise ConfkvError(status, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


_raw_stream_fn = None


def _stream(stream, device_index: int = -1) -> int:
    """Raw cudaStream_t of `stream`, or of the current torch stream of the
    device when None.  The current stream is read through torch's raw-stream
    accessor when it has one: building a torch Stream object on every decode
    step costs more host time than the step's three kernel launches."""
    global _raw_stream_fn
    import torch
    if stream is None:
        if device_index >= 0:
            if _raw_stream_fn is None:
                _raw_stream_fn = getattr(torch._C, "_cuda_getCurrentRawStream", False)
            if _raw_stream_fn:
                return _raw_stream_fn(device_index)
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def make_config(L, Hq, Hkv, d, V, B, cap, W, P, n_high, n_low, q_dtype="f16", tau=0.7, alpha=0.65,
                lam=0.9, w_H=0.4, w_m=0.3, w_p=0.3, max_evict=0, compaction=COMPACT_TAIL_FILL):
    """Build a Config; keeps the budget arrays alive on the returned object."""
    nh = (ctypes.c_int32 * L)(*[int(x) for x in n_high])
    nl = (ctypes.c_int32 * L)(*[int(x) for x in n_low])
    c = Config(L=L, Hq=Hq, Hkv=Hkv, d=d, V=V, B=B, cap=cap, W=W, P=P,
               q_dtype=Q_BF16 if q_dtype in ("bf16", Q_BF16) else Q_FP16,
               max_evict=max_evict, tau=tau, w_H=w_H, w_m=w_m, w_p=w_p, alpha=alpha, lam=lam,
               n_high=nh, n_low=nl, compaction=int(compaction))
    c._keep = (nh, nl)
    return c


def config_from_workload(w, B: Optional[int] = None, cap: Optional[int] = None, max_evict: int = 0,
                         compaction: int = COMPACT_TAIL_FILL):
    return make_config(L=w.L, Hq=w.Hq, Hkv=w.Hkv, d=w.d, V=w.V, B=w.B if B is None else B,
                       cap=w.capacity if cap is None else cap, W=w.W, P=w.P, n_high=w.n_high,
                       n_low=w.n_low, q_dtype=w.q_dtype, tau=w.tau, alpha=w.alpha, lam=w.lam,
                       w_H=w.w_H, w_m=w.w_m, w_p=w.w_p, max_evict=max_evict, compaction=compaction)


def workspace_bytes(cfg: Config) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().confkv_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "confkv_workspace_bytes")
    return int(n.value)


def launch_plan(cfg: Config, n8_bound: int, attn_ctas: int = 0):
    """(CTAs per unit, grid CTAs, cluster size) of the attention launch for a
    bound `n8_bound` on the INT8 entries per (layer, sequence); host only."""
    sp, g, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().confkv_launch_plan(ctypes.byref(cfg), int(n8_bound), int(attn_ctas), ctypes.byref(sp),
                                    ctypes.byref(g), ctypes.byref(c)), "confkv_launch_plan")
    return int(sp.value), int(g.value), int(c.value)


class Cache:
    """A CONF-KV cache manager on the current CUDA device.

    The workspace is one torch uint8 tensor; outputs of `step` are torch
    tensors on the same device."""

    def __init__(self, cfg: Config, device=None):
        import torch
        self.cfg = cfg
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        nbytes = workspace_bytes(cfg)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        h = ctypes.c_void_p()
        _check(lib().confkv_create(ctypes.byref(cfg), self.workspace.data_ptr(), nbytes, ctypes.byref(h)),
               "confkv_create")
        self._h = h
        self._fn_step = lib().confkv_step
        self._dev_index = self.device.index if self.device.index is not None else torch.cuda.current_device()
        self.L, self.B, self.Hq, self.Hkv, self.d, self.V = cfg.L, cfg.B, cfg.Hq, cfg.Hkv, cfg.d, cfg.V
        self.cap = (cfg.cap + 15) // 16 * 16
        self.WR = (cfg.W + 16 + 15) // 16 * 16
        self.max_evict = cfg.max_evict if cfg.max_evict > 0 else self.cap + self.WR

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().confkv_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # ------------------------------------------------------------ decode path
    def prefill(self, k, v, prefill_len: Sequence[int], stream=None):
        """k, v: device fp16 [L][B][Hkv][t_max][d]."""
        t_max = int(k.shape[3])
        pl = (ctypes.c_int32 * self.B)(*[int(x) for x in prefill_len])
        _check(lib().confkv_prefill(self._h, pl, _ptr(k), _ptr(v), t_max, _stream(stream)),
               "confkv_prefill")

    def new_outputs(self):
        import torch
        dev = self.device
        return dict(
            out=torch.empty((self.L, self.B, self.Hq, self.d), dtype=torch.float32, device=dev),
            budget=torch.empty((self.B, self.L), dtype=torch.int32, device=dev),
            confidence=torch.empty((self.B,), dtype=torch.float32, device=dev),
            evicted=torch.empty((self.L, self.B, self.max_evict), dtype=torch.int32, device=dev),
            n_evicted=torch.empty((self.L, self.B), dtype=torch.int32, device=dev),
        )

    def step(self, q, k_new, v_new, logits, outs=None, stream=None):
        """One decode step; returns the dict of output tensors."""
        o = self.new_outputs() if outs is None else outs
        conf = o.get("confidence")
        st = self._fn_step(self._h, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), logits.data_ptr(),
                           o["out"].data_ptr(), o["budget"].data_ptr(),
                           None if conf is None else conf.data_ptr(), o["evicted"].data_ptr(),
                           o["n_evicted"].data_ptr(), _stream(stream, self._dev_index))
        if st != OK:
            raise ConfkvError(st, "confkv_step")
        return o

    def prepared_steps(self, inputs, outs=None, stream=None):
        """A decode loop over fixed device buffers: `inputs` is a list of
        (q, k_new, v_new, logits) tensors, kept alive by the caller.  Returns
        run(i), which makes the confkv_step call for inputs[i] with argument
        values prepared once (no tensor indexing or pointer lookups per
        step, which for small shapes cost more host time than the step's
        launches)."""
        o = self.new_outputs() if outs is None else outs
        conf = o.get("confidence")
        tail = (o["out"].data_ptr(), o["budget"].data_ptr(), None if conf is None else conf.data_ptr(),
                o["evicted"].data_ptr(), o["n_evicted"].data_ptr(), _stream(stream, self._dev_index))
        args = [(self._h, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), lg.data_ptr()) + tail
                for (q, kn, vn, lg) in inputs]
        fn = self._fn_step

        def run(i):
            st = fn(*args[i])
            if st != OK:
                raise ConfkvError(st, "confkv_step")
        return run

    def step_host(self, q, k_new, v_new, logits, outs, stream=None):
        """One decode step from HOST tensors (pinned for asynchronous DMA);
        outputs land in the host tensors of `outs`."""
        _check(lib().confkv_step_host(self._h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(logits),
                                      _ptr(outs["out"]), _ptr(outs["budget"]),
                                      _ptr(outs.get("confidence")), _ptr(outs["evicted"]),
                                      _ptr(outs["n_evicted"]), _stream(stream)),
               "confkv_step_host")
        return outs

    def host_outputs(self, pin: bool = True):
        import torch
        def e(shape, dt):
            return torch.empty(shape, dtype=dt, pin_memory=pin)
        return dict(out=e((self.L, self.B, self.Hq, self.d), torch.float32),
                    budget=e((self.B, self.L), torch.int32),
                    confidence=e((self.B,), torch.float32),
                    evicted=e((self.L, self.B, self.max_evict), torch.int32),
                    n_evicted=e((self.L, self.B), torch.int32))

    # ------------------------------------------------------------ state
    def export_unit(self, b: int, l: int, stream=None) -> dict:
        cap, WR, H, d = self.cap, self.WR, self.Hkv, self.d
        a = dict(pos8=np.zeros(cap, np.int32), ema8=np.zeros(cap, np.float32),
                 k8=np.zeros((cap, H, d), np.int8), v8=np.zeros((cap, H, d), np.int8),
                 posR=np.zeros(WR, np.int32), emaR=np.zeros(WR, np.float32),
                 k16=np.zeros((WR, H, d), np.uint16), v16=np.zeros((WR, H, d), np.uint16),
                 sK=np.zeros((H, d), np.float32), sV=np.zeros((H, d), np.float32))
        u = UnitHost(0, 0, *[a[k].ctypes.data for k in
                             ("pos8", "ema8", "k8", "v8", "posR", "emaR", "k16", "v16", "sK", "sV")])
        _check(lib().confkv_export_unit(self._h, b, l, ctypes.byref(u), _stream(stream)), "confkv_export_unit")
        n8, nR = u.n8, u.nR
        return dict(n8=n8, nR=nR, pos8=a["pos8"][:n8].copy(), ema8=a["ema8"][:n8].copy(),
                    k8=a["k8"][:n8].copy(), v8=a["v8"][:n8].copy(), posR=a["posR"][:nR].copy(),
                    emaR=a["emaR"][:nR].copy(), k16=a["k16"][:nR].view(np.float16).copy(),
                    v16=a["v16"][:nR].view(np.float16).copy(), sK=a["sK"], sV=a["sV"])

    def import_unit(self, b: int, l: int, st: dict, stream=None):
        arrs = dict(pos8=np.ascontiguousarray(st["pos8"], np.int32),
                    ema8=np.ascontiguousarray(st["ema8"], np.float32),
                    k8=np.ascontiguousarray(st["k8"], np.int8), v8=np.ascontiguousarray(st["v8"], np.int8),
                    posR=np.ascontiguousarray(st["posR"], np.int32),
                    emaR=np.ascontiguousarray(st["emaR"], np.float32),
                    k16=np.ascontiguousarray(np.asarray(st["k16"], np.float16)).view(np.uint16),
                    v16=np.ascontiguousarray(np.asarray(st["v16"], np.float16)).view(np.uint16),
                    sK=np.ascontiguousarray(st["sK"], np.float32), sV=np.ascontiguousarray(st["sV"], np.float32))
        u = UnitHost(len(arrs["pos8"]), len(arrs["posR"]),
                     *[arrs[k].ctypes.data for k in
                       ("pos8", "ema8", "k8", "v8", "posR", "emaR", "k16", "v16", "sK", "sV")])
        _check(lib().confkv_import_unit(self._h, b, l, ctypes.byref(u), _stream(stream)), "confkv_import_unit")

    def get_clock(self):
        pl = (ctypes.c_int32 * self.B)()
        st = ctypes.c_int64()
        _check(lib().confkv_get_clock(self._h, pl, ctypes.byref(st)), "confkv_get_clock")
        return list(pl), int(st.value)

    def set_clock(self, prefill_len, steps: int, stream=None):
        pl = (ctypes.c_int32 * self.B)(*[int(x) for x in prefill_len])
        _check(lib().confkv_set_clock(self._h, pl, int(steps), _stream(stream)), "confkv_set_clock")

    def stats(self, stream=None, check: bool = True) -> dict:
        s = Stats()
        r = lib().confkv_get_stats(self._h, ctypes.byref(s), _stream(stream))
        if check:
            _check(r, "confkv_get_stats")
        return {f: getattr(s, f) for f, _ in Stats._fields_}

    def profile_enable(self, max_steps: int, every: int = 1):
        """Record per-kernel CUDA events on every `every`-th step (at most
        `max_steps` recorded steps)."""
        _check(lib().confkv_profile_enable(self._h, int(max_steps), int(every)), "confkv_profile_enable")

    def profile_disable(self):
        _check(lib().confkv_profile_disable(self._h), "confkv_profile_disable")

    def profile_read(self):
        a, b, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        n = ctypes.c_int32()
        _check(lib().confkv_profile_read(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                         ctypes.byref(n)), "confkv_profile_read")
        return dict(prestep_ms=a.value, attention_ms=b.value, select_ms=c.value, steps=n.value)

    def graph_reserve(self, steps: int):
        """Check that `steps` more steps fit and pin one attention launch
        shape for them (required before capturing a step into a graph)."""
        _check(lib().confkv_graph_reserve(self._h, int(steps)), "confkv_graph_reserve")

    def graph_advance(self, steps: int):
        """Account for `steps` executed replays of a captured step."""
        _check(lib().confkv_graph_advance(self._h, int(steps)), "confkv_graph_advance")

    def selftest_timeout(self, stream=None):
        """Run the bounded-wait self-test: sets the time-out status bit."""
        _check(lib().confkv_selftest_timeout(self._h, _stream(stream)), "confkv_selftest_timeout")

    def graph_release(self):
        _check(lib().confkv_graph_release(self._h), "confkv_graph_release")

    def capture_step(self, q, k_new, v_new, logits, outs):
        """Capture one decode step reading these device tensors and writing
        `outs` into a torch.cuda.CUDAGraph.  Call graph_reserve first; after
        each g.replay() call graph_advance(1) (or advance several at once)."""
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            self.step(q, k_new, v_new, logits, outs)
        return g

    def attention_plan(self):
        sp, sm = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().confkv_attention_plan(self._h, ctypes.byref(sp), ctypes.byref(sm)),
               "confkv_attention_plan")
        return int(sp.value), int(sm.value)

    def set_step_mode(self, mode):
        """STEP_AUTO (one launch per step where it fits) or STEP_SEPARATE."""
        _check(lib().confkv_set_step_mode(self._h, int(mode)), "confkv_set_step_mode")

    def step_launches(self) -> int:
        """Kernel launches the next step takes (1: the fused step, 3 otherwise)."""
        n = ctypes.c_int32()
        _check(lib().confkv_step_launches(self._h, ctypes.byref(n)), "confkv_step_launches")
        return int(n.value)

    def set_attention_ctas(self, ctas):
        """Cap the persistent attention grid at `ctas` CTAs (0: two per SM)."""
        _check(lib().confkv_set_attention_ctas(self._h, int(ctas)), "confkv_set_attention_ctas")

    def attention_grid(self):
        """(CTAs, cluster size) of the next attention launch."""
        g, c = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().confkv_attention_grid(self._h, ctypes.byref(g), ctypes.byref(c)),
               "confkv_attention_grid")
        return int(g.value), int(c.value)
