"""Host-side logic of bench.py that needs no GPU."""
import math
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_profile_stride_is_coprime_with_the_pool():
    # sampled steps must visit every entry of the input pool
    for pool in range(1, 130):
        k = bench.profile_stride(pool)
        assert k >= bench.PROFILE_EVERY
        assert math.gcd(k, pool) == 1
        assert sorted({(s * k) % pool for s in range(pool)}) == list(range(pool))


def test_compare_policies_are_the_pages_baselines():
    from workload import get_workload
    w = get_workload("qwen32b")
    assert bench.variant_workload(w, "confkv", 100) == w
    full = bench.variant_workload(w, "fullkv", 2056)
    # no eviction, and every token of the trajectory inside the FP16 window
    assert min(full.n_high) >= 1 << 30 and min(full.n_low) >= 1 << 30
    assert full.W >= w.T0 + 2056 and full.W % 16 == 0
    slide = bench.variant_workload(w, "sliding512", 2056)
    assert slide.alpha == 0.0 and set(slide.n_high) == {512} and set(slide.n_low) == {512}
    assert slide.W == 512
    import pytest
    with pytest.raises(ValueError):
        bench.variant_workload(w, "h2o", 10)


def test_attention_traffic_ratio_is_read_from_the_summary():
    # `traffic` = this ratio x the timed launches' own algorithmic bytes
    r = bench._traffic_ratio_from_profiles("attention_kernel_qwen32b")
    assert r is not None and 1.0 <= r < 1.2
    assert bench._traffic_ratio_from_profiles("attention_kernel_no_such_workload") is None
