"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/confkv.h declares, validates configurations, and the
16-token block interleave is a bijection whose mma fragments are contiguous."""
import ctypes
import os
import re

import numpy as np
import pytest

import confidence_gated_kv_gb300 as ck
from confidence_gated_kv_gb300 import binding
from workload import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "confkv.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(confkv_[a-z0-9_]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 15
    L = ck.lib()
    for n in names:
        assert hasattr(L, n), n
    assert ck.lib().confkv_version() >= 100


def test_status_strings():
    for code in range(-7, 1):
        assert ck.status_string(code) not in ("", "unknown status")
    assert ck.status_string(-99) == "unknown status"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kind", [0, 1, 2, 3])
def test_block_interleave_is_a_bijection(kind, d):
    elem = 1 if kind < 2 else 2
    offs = np.array([[ck.block_offset(kind, d, tau, c) for c in range(d)] for tau in range(16)])
    assert offs.min() >= 0
    assert np.all(offs % elem == 0)
    flat = np.sort(offs.ravel())
    np.testing.assert_array_equal(flat, np.arange(16 * d) * elem)


@pytest.mark.parametrize("d", [64, 128])
def test_block_interleave_matches_mma_fragments(d):
    # Lane 4g+t reads 16 contiguous bytes at r*512 + lane*16.  For INT8 K the
    # four bytes of word w of chunk r hold token 8*nt+g, channels
    # 16*kk + {2t, 2t+1, 2t+8, 2t+9} (the B fragment of one m16n8k16 QK^T).
    nc = d // 32
    for tau in range(16):
        nt, g = divmod(tau, 8)
        for kk in range(d // 16):
            for t in range(4):
                base = ck.block_offset(0, d, tau, 16 * kk + 2 * t)
                assert base == (nt * (nc // 2) + kk // 4) * 512 + (4 * g + t) * 16 + (kk % 4) * 4
                got = [ck.block_offset(0, d, tau, 16 * kk + c) for c in (2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9)]
                assert got == [base, base + 1, base + 2, base + 3]
    # INT8 V: the word of lane 4g+t for n-tile j holds channel 8j+g of tokens
    # 2t, 2t+1, 2t+8, 2t+9 (the B fragment of one m16n8k16 PV).
    for j in range(d // 8):
        for g in range(8):
            for t in range(4):
                got = [ck.block_offset(1, d, tau, 8 * j + g) for tau in (2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9)]
                base = (j // 4) * 512 + (4 * g + t) * 16 + (j % 4) * 4
                assert got == [base, base + 1, base + 2, base + 3]


def test_bad_arguments_of_offset_helper():
    assert ck.block_offset(0, 96, 0, 0) == -1
    assert ck.block_offset(0, 128, 16, 0) == -1
    assert ck.block_offset(5, 128, 0, 0) == -1


def _cfg(**kw):
    base = dict(L=2, Hq=8, Hkv=2, d=128, V=1000, B=2, cap=256, W=32, P=8,
                n_high=[40, 40], n_low=[80, 80])
    base.update(kw)
    base["n_high"] = list(base["n_high"])[:max(base["L"], 0)]
    base["n_low"] = list(base["n_low"])[:max(base["L"], 0)]
    return ck.make_config(**base)


@pytest.mark.parametrize("bad", [
    dict(d=96), dict(Hq=6, Hkv=4), dict(Hq=18, Hkv=2), dict(V=1), dict(V=4096 * 1024 + 1), dict(W=0),
    dict(n_high=[4, 40]), dict(n_low=[80, 0]), dict(cap=8), dict(L=0), dict(B=0),
    dict(alpha=1.5), dict(lam=-0.1), dict(q_dtype=7), dict(P=-1), dict(compaction=2),
])
def test_invalid_configurations_rejected(bad):
    c = _cfg(**bad)
    if "q_dtype" in bad:
        c.q_dtype = 7
    n = ctypes.c_size_t()
    assert ck.lib().confkv_workspace_bytes(ctypes.byref(c), ctypes.byref(n)) == binding.EINVAL


def test_workspace_grows_with_capacity_and_covers_kv():
    small = ck.workspace_bytes(_cfg(cap=256))
    big = ck.workspace_bytes(_cfg(cap=4096))
    assert big > small
    # INT8 K and V for every (layer, sequence, KV head, slot, channel)
    assert big >= 2 * 2 * 2 * 2 * 4096 * 128


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_every_workload_has_a_valid_configuration(name):
    w = WORKLOADS[name]
    assert ck.workspace_bytes(ck.config_from_workload(w)) > 0


def test_null_handles_are_rejected():
    L = ck.lib()
    assert L.confkv_step(None, *([None] * 9), None) == binding.EINVAL
    assert L.confkv_prefill(None, None, None, None, 0, None) == binding.EINVAL
    assert L.confkv_get_stats(None, None, None) == binding.EINVAL
    assert L.confkv_set_attention_ctas(None, 0) == binding.EINVAL
    assert L.confkv_attention_grid(None, None, None) == binding.EINVAL
    L.confkv_destroy(None)


def test_status_bits_match_the_kernels():
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hdr = open(os.path.join(root, "include", "confkv.h")).read()
    internal = open(os.path.join(root, "confidence_gated_kv_gb300", "csrc", "confkv_internal.cuh")).read()
    pub = {m.group(1): int(m.group(2)) for m in re.finditer(r"CONFKV_STATUS_(\w+) = (\d+)", hdr)}
    dev = {m.group(1): int(m.group(2)) for m in re.finditer(r"kStatus(\w+) = (\d+)", internal)}
    want = {"CAPACITY": "Capacity", "EVICT_BOUND": "EvictBound", "BAD_COUNT": "BadCount", "TIMEOUT": "Timeout"}
    for k, v in want.items():
        assert pub[k] == dev[v]


def test_both_compaction_layouts_are_valid():
    for c in (binding.COMPACT_TAIL_FILL, binding.COMPACT_ORDERED):
        assert ck.workspace_bytes(_cfg(compaction=c)) > 0


# ------------------------------------------------------------ launch planning

@pytest.mark.parametrize("name, n8, expect", [
    # 4096 / 1536 / 1152 units: the persistent kernel, two CTAs per SM
    ("qwen32b", 2048, (1, 304, 1)),
    ("qwen14b", 8192 - 256, (1, 304, 1)),
    ("gpt2_b8_pyramid", 768, (1, 304, 1)),
    # 512 units: two rounds of 256 CTAs, at the 32K-token first step too
    ("needle32k", 32768 - 256, (1, 256, 1)),
    ("needle32k", 4096 - 256, (1, 256, 1)),
    # 144 units of ~600 tokens: one whole unit per CTA, no clusters
    ("gpt2_b1", 600 - 64, (1, 144, 1)),
])
def test_launch_plan_of_each_workload(name, n8, expect):
    w = WORKLOADS[name]
    assert ck.launch_plan(ck.config_from_workload(w), n8) == expect


def test_launch_plan_splits_only_long_units_of_few_sequences():
    from workload import Workload
    w = Workload(name="t", B=1, L=1, Hq=8, Hkv=2, d=128, V=4000, T0=4000, steps=1,
                 n_high=(1500,), n_low=(3000,), P=16, W=64)
    cfg = ck.config_from_workload(w)
    # 2 units of ~4000 tokens: 2-CTA clusters keep 1024+ tokens per CTA
    assert ck.launch_plan(cfg, 4000 - 64) == (2, 4, 2)
    # ~1500 tokens: too short to split
    assert ck.launch_plan(cfg, 1500) == (1, 2, 1)
    # a cap of 2 CTAs keeps whole units on the persistent kernel
    assert ck.launch_plan(cfg, 4000 - 64, attn_ctas=2) == (1, 2, 1)


def test_launch_plan_cap_and_bad_arguments():
    cfg = ck.config_from_workload(WORKLOADS["qwen32b"])
    assert ck.launch_plan(cfg, 2048, attn_ctas=100) == (1, 100, 1)
    L = ck.lib()
    out = [ctypes.c_int32() for _ in range(3)]
    refs = [ctypes.byref(x) for x in out]
    assert L.confkv_launch_plan(ctypes.byref(cfg), -1, 0, *refs) == binding.EINVAL
    assert L.confkv_launch_plan(ctypes.byref(cfg), 2048, -1, *refs) == binding.EINVAL
    assert L.confkv_launch_plan(ctypes.byref(cfg), cfg.cap + 1, 0, *refs) == binding.EINVAL
    assert L.confkv_launch_plan(None, 2048, 0, *refs) == binding.EINVAL
