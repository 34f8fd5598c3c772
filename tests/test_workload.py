"""The synthetic inputs follow the stated recipe: workload geometry and
hyper-parameters, the pyramidal budgets, N(0, 1) K/V with scaled heavy keys,
the planted needle key and the needle queries, and N(0, sigma) logits with one
spike.  Both generator back-ends (per-unit numpy streams and the torch
generator used by the benchmark) are checked; no GPU is needed."""
import numpy as np
import pytest
import torch

from workload import (WORKLOADS, heavy_positions, needle_position, prefill_batch_fast, prefill_unit,
                      step_logits, step_pool_fast, step_unit)
from workload.gen import _pyramid, q_direction

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


@pytest.mark.parametrize("name, geom", [
    # name: (B, L, Hq, Hkv, d, V, T0, steps, N_high, N_low, P, W, q dtype)
    ("gpt2_b1", (1, 12, 12, 12, 64, 50257, 600, 64, 256, 512, 32, 64, "f16")),
    ("qwen14b", (4, 48, 40, 8, 128, 152064, 8192, 256, 1024, 2048, 64, 256, "bf16")),
    ("qwen32b", (8, 64, 40, 8, 128, 152064, 4096, 4096, 1024, 2048, 64, 256, "bf16")),
    ("needle32k", (1, 64, 40, 8, 128, 152064, 32768, 128, 2048, 4096, 64, 256, "bf16")),
])
def test_workload_geometry(name, geom):
    w = WORKLOADS[name]
    B, L, Hq, Hkv, d, V, T0, steps, nh, nl, P, W, qd = geom
    assert (w.B, w.L, w.Hq, w.Hkv, w.d, w.V, w.T0, w.steps) == (B, L, Hq, Hkv, d, V, T0, steps)
    assert w.n_high == (nh,) * L and w.n_low == (nl,) * L
    assert (w.P, w.W, w.q_dtype) == (P, W, qd)
    assert (w.tau, w.alpha, w.lam, w.w_H, w.w_m, w.w_p) == (0.7, 0.65, 0.9, 0.4, 0.3, 0.3)


def test_gpt2_batch8_pyramidal_budgets():
    w = WORKLOADS["gpt2_b8_pyramid"]
    assert (w.B, w.L, w.T0, w.steps, w.P, w.W) == (8, 12, 128, 2048, 64, 128)
    # linear from the first to the last layer, rounded half to even
    assert w.n_low == (768, 721, 675, 628, 582, 535, 489, 442, 396, 349, 303, 256)
    assert w.n_high == (384, 361, 337, 314, 291, 268, 244, 221, 198, 175, 151, 128)
    assert _pyramid(3, 10, 5) == (10, 8, 5)   # 7.5 rounds to the even 8
    assert _pyramid(1, 10, 5) == (10,)


def test_heavy_keys_and_kv_distribution():
    w = WORKLOADS["gpt2_b1"]   # 8 heavy keys scaled by 4
    hp = heavy_positions(w, 5, 0)
    assert hp.size == w.heavy_count and len(set(hp.tolist())) == hp.size
    assert np.all((hp >= 0) & (hp < w.T0)) and np.all(np.diff(hp) > 0)
    k, v = prefill_unit(w, 5, 0, 3)
    assert k.shape == v.shape == (w.Hkv, w.T0, w.d) and k.dtype == np.float16
    light = np.setdiff1d(np.arange(w.T0), hp)
    kl = k[:, light, :].astype(np.float64)
    assert abs(kl.mean()) < 0.01 and abs(kl.std() - 1.0) < 0.01
    vv = v.astype(np.float64)
    assert abs(vv.mean()) < 0.01 and abs(vv.std() - 1.0) < 0.01
    # heavy keys: the same N(0, 1) draw scaled, so their RMS is ~4x; values stay N(0, 1)
    kh = k[:, hp, :].astype(np.float64)
    assert 3.6 < np.sqrt((kh ** 2).mean()) / np.sqrt((kl ** 2).mean()) < 4.4
    assert abs(np.sqrt((v[:, hp, :].astype(np.float64) ** 2).mean()) - 1.0) < 0.1
    # qwen32b: 0.5 % of a 4096-token prefill, scaled by 3
    w32 = WORKLOADS["qwen32b"]
    assert w32.heavy_count == round(0.005 * w32.T0) and w32.heavy_factor == 3.0


def test_needle_key_depth_and_queries():
    w = WORKLOADS["needle32k"].replace(T0=2048)
    depths = [needle_position(w, s, 0) / w.T0 for s in range(40)]
    assert min(depths) >= 0.1 and max(depths) < 0.9
    p = needle_position(w, 9, 0)
    for l in (0, 17):
        qd = q_direction(w, 9, l)
        np.testing.assert_allclose(np.linalg.norm(qd, axis=1), 1.0, rtol=1e-6)
        k, _ = prefill_unit(w, 9, 0, l)
        # the planted key is 6 * the unit query direction, in every KV head
        np.testing.assert_array_equal(k[:, p, :], (6.0 * qd).astype(np.float16))
        q, _, _ = step_unit(w, 9, 3, 0, l)
        dev = q.float().numpy() - np.repeat(qd, w.g, axis=0)   # q = q_dir + N(0, 0.3^2)
        assert abs(dev.mean()) < 0.03 and abs(dev.std() - 0.3) < 0.03
    assert w.spike_hi == 4.0   # low-confidence logits


@pytest.mark.parametrize("name", ["gpt2_b1", "qwen32b"])
def test_logits_are_gaussian_with_one_spike(name):
    w = WORKLOADS[name]
    z = step_logits(w, 11, 2, 0).astype(np.float64)
    assert z.shape == (w.V,)
    assert abs(z.mean()) < 0.02 * w.logit_sigma and abs(z.std() / w.logit_sigma - 1.0) < 0.02
    # at most one entry lies beyond the Gaussian's reach plus the spike
    assert z.max() < 6.5 * w.logit_sigma + w.spike_hi


def test_device_generators_follow_the_same_recipe():
    dev = torch.device("cpu")
    w = WORKLOADS["gpt2_b1"].replace(L=2, T0=256)
    k, v = prefill_batch_fast(w, 4, dev)
    assert k.shape == (2, 1, w.Hkv, 256, w.d) and k.dtype == torch.float16
    hp = torch.from_numpy(heavy_positions(w, 4, 0))
    light = torch.tensor(np.setdiff1d(np.arange(256), hp.numpy()))
    kl = k[:, 0][:, :, light].double()
    assert abs(kl.std().item() - 1.0) < 0.02
    ratio = k[:, 0][:, :, hp].double().pow(2).mean().sqrt() / kl.pow(2).mean().sqrt()
    assert 3.5 < ratio.item() < 4.5
    q, kn, vn, lg = step_pool_fast(w, 4, 3, dev)
    assert q.shape == (3, 2, 1, w.Hq, w.d) and q.dtype == torch.float16
    assert kn.shape == vn.shape == (3, 2, 1, w.Hkv, w.d) and lg.shape == (3, 1, w.V)
    assert abs(lg.double().std().item() / w.logit_sigma - 1.0) < 0.02
    wn = WORKLOADS["needle32k"].replace(L=2, T0=512)
    k, _ = prefill_batch_fast(wn, 4, dev)
    p = needle_position(wn, 4, 0)
    for l in range(2):
        qd = torch.from_numpy(q_direction(wn, 4, l))
        assert torch.equal(k[l, 0, :, p, :], (6.0 * qd).to(torch.float16))
    q, _, _, _ = step_pool_fast(wn, 4, 2, dev)
    qd = torch.stack([torch.from_numpy(q_direction(wn, 4, l)) for l in range(2)]).repeat_interleave(wn.g, 1)
    dev_q = q.float() - qd[None, :, None]
    assert abs(dev_q.std().item() - 0.3) < 0.03
