"""The multi-rank logic of bench.py on CPU with gloo, world size 2: each rank
runs an independent replica; the timing is the max over ranks and the value
is the whole-job rate.  The reference arm does its work on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _seed_worker(rank, port, results):
    # every rank draws its own replica: distinct seeds, distinct prefills
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    from workload import Workload, prefill_batch
    w = Workload(name="t_rank", B=1, L=1, Hq=2, Hkv=1, d=64, V=64, T0=32, steps=1,
                 n_high=(16,), n_low=(16,), P=4, W=8)
    seeds = [bench.replica_seed(4003, i, rank) for i in range(3)]
    k, _ = prefill_batch(w, seeds[0], "cpu")
    t = k.float().reshape(-1)
    got = [torch.zeros_like(t) for _ in range(2)]
    dist.all_gather(got, t)
    all_seeds = [None, None]
    dist.all_gather_object(all_seeds, seeds)
    results[rank] = (all_seeds, bool(torch.equal(got[0], got[1])))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_on_different_ranks_draw_different_inputs():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_seed_worker, args=(port, results), nprocs=2, start_method="spawn", join=True)
    seeds, same = results[0]
    assert not same
    assert len(set(seeds[0]) | set(seeds[1])) == 6     # three seeds per rank, none shared
    assert seeds[0] == [4003, 4004, 4005]


def _worker(rank, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    ms = 100.0 if rank == 0 else 250.0
    ms_max, value = bench.reduce_timing(ms, 50, 2, torch.device("cpu"))
    results[rank] = (ms_max, value)
    dist.barrier()
    dist.destroy_process_group()


def test_timing_is_max_over_ranks_and_value_is_whole_job():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(port, results), nprocs=2, start_method="spawn", join=True)
    for rank in (0, 1):
        ms_max, value = results[rank]
        assert ms_max == 250.0
        assert abs(value - 2 * 50 / 0.25) < 1e-9


def test_single_rank_needs_no_process_group():
    ms_max, value = bench.reduce_timing(40.0, 20, 1, torch.device("cpu"))
    assert ms_max == 40.0 and abs(value - 500.0) < 1e-9


def test_reference_arm_does_no_work_off_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    # the float64 oracle timed on the host: one JSON line with the same
    # metric and unit as the GPU arm, its own cpu_baseline and a host-only e2e
    import json
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--workload", "gpt2_b1", "--steps", "2",
                       "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "steps/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] >= 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "steps/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "gpt2_b1"
    # the GPU arm's config dict for the same arguments, the measured wall
    # time per timed step, and the extrapolation labelled with its sample
    import argparse
    from workload import get_workload
    assert line["config"] == bench.bench_config(get_workload("gpt2_b1"),
                                                argparse.Namespace(compaction="tailfill"), 1)
    assert line["ms_per_step"] > 0
    assert line["extrapolated"]["unit_steps_per_timed_step"] == 2
    assert line["extrapolated"]["unit_steps_per_whole_step"] == 12
    assert "threads" in line["cpu_baseline"]["blas"]
