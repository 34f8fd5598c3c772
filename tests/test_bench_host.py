"""Host-side logic of bench.py that needs no GPU."""
import math
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_profile_stride_is_coprime_with_the_pool():
    # sampled steps must visit every entry of the input pool, for short and
    # long timed windows
    for steps, least in ((20, bench.PROFILE_EVERY), (2000, bench.PROFILE_EVERY_LONG)):
        for pool in range(1, 130):
            k = bench.profile_stride(pool, steps)
            assert k >= least
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


def test_attention_traffic_ratio_is_read_from_the_json_record(tmp_path, monkeypatch):
    # `traffic` = this ratio x the timed launches' own algorithmic bytes; the
    # ratio comes from the machine-readable record next to the ncu summary
    import json
    with open(os.path.join(bench.ROOT, "profiles", "attention_kernel_qwen32b.json")) as f:
        rec = json.load(f)
    assert 1.0 <= rec["dram_bytes_per_algorithmic_byte"] < 1.2
    r = bench._traffic_ratio_from_profiles("attention_kernel_qwen32b")
    assert r == (None if rec.get("stale") else rec["dram_bytes_per_algorithmic_byte"])
    assert bench._traffic_ratio_from_profiles("attention_kernel_no_such_workload") is None
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles" / "attention_kernel_x.json").write_text(
        json.dumps({"dram_bytes_per_algorithmic_byte": 1.05, "stale": False}))
    assert bench._traffic_ratio_from_profiles("attention_kernel_x") == 1.05
    # a record marked stale (taken on a kernel that has changed since) gives none
    (tmp_path / "profiles" / "attention_kernel_x.json").write_text(
        json.dumps({"dram_bytes_per_algorithmic_byte": 1.05, "stale": True}))
    assert bench._traffic_ratio_from_profiles("attention_kernel_x") is None


def test_untimed_steps_cover_warmup_and_one_pool_cycle():
    assert bench.untimed_steps(5, 16) == 17
    assert bench.untimed_steps(40, 16) == 40
    assert bench.untimed_steps(3, 1) == 3


def test_spin_is_bounded_and_covers_the_first_steps():
    for k in (1, 20, 2000, 10 ** 6):
        c = bench.spin_cycles(k)
        ms = c / 2.07e9 * 1e3
        assert 2.0 <= ms <= 50.0 + 1e-9


def test_both_arms_share_one_config():
    import argparse
    from workload import get_workload
    args = argparse.Namespace(compaction="tailfill")
    for name in ("qwen32b", "gpt2_b1"):
        w = get_workload(name)
        c = bench.bench_config(w, args, 1)
        assert c == bench.bench_config(w, args, 1)
        assert c["workload"] == name and c["vocab"] == w.V and c["heads"] == [w.Hq, w.Hkv]
    assert "larger than L2" in bench.bench_config(get_workload("qwen32b"), args, 1)["l2"]
    assert "fits the 129 MB L2" in bench.bench_config(get_workload("gpt2_b1"), args, 1)["l2"]


def test_blas_thread_count_is_reported():
    b = bench.blas_threads()
    assert set(b) == {"threads", "library", "how"}
    assert b["threads"] is None or b["threads"] >= 1


def test_clock_summary_uses_samples_under_load():
    rows = [["0", "1000", "2070", "100", "0x0", "Not Active", "Not Active", "Not Active", "Not Active", "0"],
            ["0", "2070", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Active", "100"],
            ["0", "2060", "2070", "950", "0x0", "Not Active", "Not Active", "Not Active", "Not Active", "97"]]
    c = bench.summarise_clocks(rows)
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3 and c["samples_under_load"] == 2
    assert bench.summarise_clocks([]) is None
