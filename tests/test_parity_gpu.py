"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that span several
16-token blocks, ragged tails, empty prefills, budget flips, the split-K
cluster path and both head dims."""
import numpy as np
import pytest
import torch

import confidence_gated_kv_gb300 as ck
from workload import Workload, get_workload, prefill_batch

from _parity import Pair, confident_logits, step_inputs

pytestmark = pytest.mark.gpu


# confkv_step modes: one fused launch per step where the shape allows it
# (the default), and the three separate kernels
MODES = [ck.binding.STEP_AUTO, ck.binding.STEP_SEPARATE]
MODE_IDS = ["fused", "separate"]


def _run(w, seed, steps, prefill_len=None, confident_every=0, cap=None, check_state=True, mode=0):
    p = Pair(w, seed, prefill_len=prefill_len, cap=cap, mode=mode)
    p.compare_states()
    for s in range(steps):
        q, kn, vn, lg = step_inputs(w, seed, s)
        if confident_every and s % confident_every == confident_every - 1:
            lg = confident_logits(w.V, w.B, seed * 1000 + s)
        p.step(q, kn, vn, lg, check_state=check_state)
    return p


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_gqa5_d128_ragged_prefills_and_flips(mode):
    w = Workload(name="t_gqa", B=3, L=2, Hq=10, Hkv=2, d=128, V=3000, T0=300, steps=40,
                 n_high=(40, 30), n_low=(120, 90), P=8, W=32, q_dtype="bf16",
                 heavy_count=5, heavy_factor=3.0, logit_sigma=1.5, spike_hi=14.0)
    p = _run(w, 11, 40, prefill_len=[300, 17, 0], confident_every=5, mode=mode)
    assert p.flags.evictions > 0
    assert p.flags.max_out_err <= 2e-3
    assert p.cache.stats()["launches"] == p.launches == (40 if mode == ck.binding.STEP_AUTO else 120)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_mha_d64_fp16_queries(mode):
    w = Workload(name="t_mha", B=2, L=3, Hq=4, Hkv=4, d=64, V=5000, T0=200, steps=30,
                 n_high=(64,) * 3, n_low=(128,) * 3, P=16, W=64, q_dtype="f16",
                 heavy_count=3, heavy_factor=4.0)
    p = _run(w, 12, 30, prefill_len=[200, 150], confident_every=4, mode=mode)
    assert p.flags.evictions > 0


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_gqa8_pyramidal_budgets(mode):
    w = Workload(name="t_g8", B=2, L=3, Hq=16, Hkv=2, d=128, V=2000, T0=160, steps=20,
                 n_high=(48, 40, 32), n_low=(96, 80, 64), P=12, W=24, q_dtype="f16")
    p = _run(w, 13, 20, confident_every=3, mode=mode)
    assert p.flags.evictions > 0


def test_persistent_kernel_several_units_per_cta_under_a_cta_cap():
    # 12 units (3 sequences x 2 layers x 2 KV heads).  A cap of 5 CTAs runs
    # the persistent kernel with 2 or 3 units per CTA (the double-buffered
    # header, partials and score slots turn over; rounds end ragged), a cap of
    # 4 with 3 units on every CTA.  Without a cap the 12 short units run one
    # per CTA.  The empty prefill gives one sequence units of ring blocks
    # only.
    w = Workload(name="t_cap", B=3, L=2, Hq=10, Hkv=2, d=128, V=3000, T0=300, steps=36,
                 n_high=(40, 30), n_low=(120, 90), P=8, W=32, q_dtype="bf16",
                 heavy_count=5, heavy_factor=3.0, logit_sigma=1.5, spike_hi=14.0)
    p = Pair(w, 31, prefill_len=[300, 17, 0])
    s = 0
    for cap, grid in [(5, (5, 1)), (4, (4, 1)), (0, (12, 1))]:
        p.cache.set_attention_ctas(cap)
        assert p.cache.attention_plan()[0] == 1
        assert p.cache.attention_grid() == grid
        for _ in range(12):
            q, kn, vn, lg = step_inputs(w, 31, s)
            if s % 5 == 4:
                lg = confident_logits(w.V, w.B, 31000 + s)
            p.step(q, kn, vn, lg)
            s += 1
    assert p.flags.evictions > 0
    assert p.flags.max_out_err <= 2e-3


@pytest.mark.parametrize("d, Hq, Hkv", [(128, 8, 2), (64, 4, 4)])
def test_split_k_cluster_path_and_large_first_eviction(d, Hq, Hkv):
    # units of 4000 tokens on 2-CTA clusters (at least 1024 tokens per CTA);
    # the launch shape follows the host's bound on the cache length (the
    # loose budget), so the confident step's cut to 1500 keeps it
    w = Workload(name="t_split", B=1, L=1, Hq=Hq, Hkv=Hkv, d=d, V=4000, T0=4000, steps=6,
                 n_high=(1500,), n_low=(3000,), P=16, W=64, q_dtype="bf16", heavy_count=10,
                 heavy_factor=3.0)
    p = Pair(w, 14)
    splits, smem = p.cache.attention_plan()
    assert splits > 1
    for s in range(6):
        assert p.cache.attention_plan()[0] == splits
        q, kn, vn, lg = step_inputs(w, 14, s)
        if s == 3:
            lg = confident_logits(w.V, w.B, 99)
        p.step(q, kn, vn, lg)
    assert p.flags.evictions >= 4000 - 1500


def test_long_int8_units_on_the_persistent_kernel():
    # One unit per sequence with a 32K-token INT8 region on the persistent
    # kernel (a cap of 2 CTAs keeps these two units off the split-K path):
    # every consumer warp runs ~500 INT8 blocks, so the kernel instance that
    # removes the INT8 V bias as it goes is launched.  Needle queries keep the
    # softmax flat.  With the bias left to the end of the INT8 blocks the
    # output was off by 2.7e-3 on such units.
    w = Workload(name="t_long", B=2, L=1, Hq=5, Hkv=1, d=128, V=2000, T0=32768, steps=3,
                 n_high=(40000,), n_low=(40000,), P=8, W=64, q_dtype="bf16", needle=True)
    p = Pair(w, 23)
    p.cache.set_attention_ctas(2)
    assert p.cache.attention_plan()[0] == 1
    assert p.cache.attention_grid() == (2, 1)
    for s in range(3):
        q, kn, vn, lg = step_inputs(w, 23, s)
        p.step(q, kn, vn, lg)
    assert p.flags.max_out_err <= 2e-3


def test_full_kv_long_ring_on_the_persistent_kernel():
    # full KV: no eviction and an FP16 window longer than every cache, so the
    # ring (1120 slots) is too long for the unit header and the persistent
    # kernel reads its positions from global memory; 608 units keep the
    # persistent launch shape
    L, B, Hkv = 19, 4, 8
    w = Workload(name="t_full", B=B, L=L, Hq=16, Hkv=Hkv, d=128, V=1000, T0=40, steps=6,
                 n_high=(1 << 30,) * L, n_low=(1 << 30,) * L, P=8, W=1100, q_dtype="bf16", cap=16)
    p = Pair(w, 17, prefill_len=[40, 7, 0, 33])
    splits, _ = p.cache.attention_plan()
    assert splits == 1
    for s in range(6):
        q, kn, vn, lg = step_inputs(w, 17, s)
        p.step(q, kn, vn, lg)
    st = p.cache.stats()
    assert st["evicted"] == 0 and st["requantised"] == 0
    assert p.flags.max_out_err <= 2e-3


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_sliding_window_policy_alpha_zero(mode):
    # recency only: alpha = 0 ranks by position, so every eviction takes the
    # oldest candidates
    w = Workload(name="t_slide", B=2, L=2, Hq=8, Hkv=2, d=64, V=800, T0=150, steps=12,
                 n_high=(64,) * 2, n_low=(64,) * 2, alpha=0.0, P=8, W=64, q_dtype="f16")
    p = _run(w, 18, 12, mode=mode)
    assert p.flags.evictions > 0


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_captured_step_replays_match_the_oracle(mode):
    # one step captured into a CUDA graph, replayed with new inputs copied
    # into the captured buffers: the device-side step index advances, the
    # host accounts for each replay inside a reservation
    w = Workload(name="t_graph", B=2, L=2, Hq=10, Hkv=2, d=128, V=3000, T0=260, steps=12,
                 n_high=(40, 30), n_low=(100, 90), P=8, W=32, q_dtype="bf16",
                 heavy_count=5, heavy_factor=3.0)
    p = Pair(w, 19, mode=mode)
    q0, kn0, vn0, lg0 = step_inputs(w, 19, 0)
    p.step(q0, kn0, vn0, lg0)                       # plain step first
    sq, skn, svn, slg = q0.cuda(), kn0.cuda(), vn0.cuda(), lg0.cuda()
    outs = p.cache.new_outputs()
    state = {}

    def capture():
        p.cache.graph_reserve(w.steps)
        state["g"] = p.cache.capture_step(sq, skn, svn, slg, outs)

    def replay(q, kn, vn, lg):
        if p.cache._h is not None and "g" not in state:
            capture()
        sq.copy_(q); skn.copy_(kn); svn.copy_(vn); slg.copy_(lg)
        state["g"].replay()
        p.cache.graph_advance(1)
        return outs

    capture()
    for s in range(1, w.steps):
        q, kn, vn, lg = step_inputs(w, 19, s)
        if s % 4 == 3:
            lg = confident_logits(w.V, w.B, 19000 + s)
        before = p.flags.ties + p.flags.budget
        p.step(q, kn, vn, lg, gpu_step=replay)
        if p.flags.ties + p.flags.budget != before:
            state.pop("g")                          # a resync drops the reservation
    assert p.flags.evictions > 0
    assert p.flags.max_out_err <= 2e-3


def test_capture_without_reservation_is_refused():
    w = Workload(name="t_graph2", B=1, L=1, Hq=4, Hkv=2, d=64, V=500, T0=40, steps=2,
                 n_high=(32,), n_low=(48,), P=4, W=16, q_dtype="f16")
    p = Pair(w, 20)
    q, kn, vn, lg = (x.cuda() for x in step_inputs(w, 20, 0))
    outs = p.cache.new_outputs()
    with pytest.raises(ck.ConfkvError):
        p.cache.capture_step(q, kn, vn, lg, outs)
    st = p.cache.stats()
    assert st["steps"] == 0 and st["device_status"] == 0


def test_order_preserving_compaction_ablation():
    # the ablation layout: survivors keep position order in the INT8 region
    # (every survivor above the first hole moves); same results as tail fill
    w = Workload(name="t_ord", B=3, L=2, Hq=10, Hkv=2, d=128, V=3000, T0=300, steps=24,
                 n_high=(40, 30), n_low=(120, 90), P=8, W=32, q_dtype="bf16",
                 heavy_count=5, heavy_factor=3.0)
    p = Pair(w, 21, prefill_len=[300, 17, 150], compaction=ck.binding.COMPACT_ORDERED)
    for s in range(w.steps):
        q, kn, vn, lg = step_inputs(w, 21, s)
        if s % 5 == 4:
            lg = confident_logits(w.V, w.B, 21000 + s)
        p.step(q, kn, vn, lg)
        for b in range(w.B):
            for l in range(w.L):
                pos8 = p.cache.export_unit(b, l)["pos8"]
                assert np.all(np.diff(pos8) > 0), "INT8 slots out of position order (b%d l%d)" % (b, l)
    assert p.flags.evictions > 0
    assert p.cache.stats()["moved"] > 0


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_bounded_wait_reports_a_timeout_and_the_context_survives(mode):
    # failure detection without a fault: a wait that nothing satisfies runs
    # out, the status word says so, and the context keeps working
    w = Workload(name="t_to", B=1, L=1, Hq=4, Hkv=2, d=64, V=500, T0=40, steps=2,
                 n_high=(32,), n_low=(48,), P=4, W=16, q_dtype="f16")
    p = Pair(w, 24, mode=mode)
    p.cache.selftest_timeout()
    st = p.cache.stats(check=False)
    assert st["device_status"] & ck.binding.STATUS_TIMEOUT
    with pytest.raises(ck.ConfkvError):
        p.cache.stats()
    # prefill clears the word; the context still steps correctly
    from workload import prefill_batch
    k, v = prefill_batch(w, 24, "cpu")
    p.cache.prefill(k.cuda(), v.cuda(), [w.T0])
    assert p.cache.stats()["device_status"] == 0
    q, kn, vn, lg = step_inputs(w, 24, 0)
    p.step(q, kn, vn, lg)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_no_eviction_limit_is_plain_attention(mode):
    # budgets above every cache length: nothing is evicted, nothing moves
    w = Workload(name="t_noop", B=2, L=2, Hq=6, Hkv=3, d=64, V=1000, T0=40, steps=12,
                 n_high=(10 ** 5,) * 2, n_low=(10 ** 5,) * 2, P=4, W=16, q_dtype="f16", cap=80)
    p = _run(w, 15, 12, mode=mode)
    assert p.flags.evictions == 0
    st = p.cache.stats()
    assert st["evicted"] == 0 and st["moved"] == 0
    assert st["requantised"] == 2 * 2 * 12


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_gpt2_small_batch1_full_trajectory(mode):
    # GPT-2-small geometry, 600-token prefill, all 64 decode steps free-running
    w = get_workload("gpt2_b1")
    p = _run(w, 1001, w.steps, check_state=False, mode=mode)
    assert p.cache.step_launches() == (1 if mode == ck.binding.STEP_AUTO else 3)
    p.compare_states()
    assert p.flags.steps == 64
    assert p.flags.max_out_err <= 2e-3


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_fused_step_with_no_sm_to_spare(mode):
    # As many units as SMs: no CTA is left for the vocabulary, so the units'
    # epilogue warps reduce the chunks (one each) in the fused step.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv = 8 if sms % 8 == 0 else 4 if sms % 4 == 0 else 0
    if Hkv == 0 or sms // Hkv > 64:
        pytest.skip("needs an SM count with a small divisor")
    L = sms // Hkv
    w = Workload(name="t_nospare", B=1, L=L, Hq=2 * Hkv, Hkv=Hkv, d=64, V=5000, T0=90, steps=12,
                 n_high=(32,) * L, n_low=(64,) * L, P=8, W=32, q_dtype="f16")
    p = _run(w, 17, 12, confident_every=4, mode=mode)
    assert p.cache.step_launches() == (1 if mode == ck.binding.STEP_AUTO else 3)
    assert p.flags.evictions > 0


def test_prepared_steps_match_step_calls():
    # Cache.prepared_steps makes the same confkv_step calls with arguments
    # prepared once: identical outputs and state to Cache.step
    w = Workload(name="t_prep", B=2, L=2, Hq=8, Hkv=2, d=64, V=3000, T0=80, steps=6,
                 n_high=(32, 32), n_low=(48, 48), P=8, W=16, q_dtype="bf16")
    k, v = prefill_batch(w, 23, "cpu")
    caches = []
    for _ in range(2):
        c = ck.Cache(ck.config_from_workload(w))
        c.prefill(k.cuda(), v.cuda(), [w.T0] * w.B)
        caches.append(c)
    inputs = [tuple(x.cuda() for x in step_inputs(w, 23, s)) for s in range(6)]
    outs = [caches[0].new_outputs(), caches[1].new_outputs()]
    run = caches[1].prepared_steps(inputs, outs[1])
    for s in range(6):
        caches[0].step(*inputs[s], outs[0])
        run(s)
        torch.cuda.synchronize()
        for key in ("out", "budget", "confidence", "n_evicted"):
            assert torch.equal(outs[0][key], outs[1][key]), (s, key)
        ne = outs[0]["n_evicted"].cpu()
        ev0, ev1 = outs[0]["evicted"].cpu(), outs[1]["evicted"].cpu()
        for l in range(w.L):
            for b in range(w.B):
                n = int(ne[l, b])   # only the first n_evicted entries of a row are written
                assert torch.equal(ev0[l, b, :n], ev1[l, b, :n]), (s, l, b)
    assert caches[0].stats()["evicted"] == caches[1].stats()["evicted"]


def test_gpt2_small_batch8_pyramid_prefix():
    w = get_workload("gpt2_b8_pyramid")
    p = _run(w, 1002, 24, confident_every=6, check_state=False)
    p.compare_states()


@pytest.mark.parametrize("kernel", ["split", "persistent"])
@pytest.mark.parametrize("pinned", [True, False, "mixed"])
def test_host_buffer_step_matches_device_step(pinned, kernel):
    # pinned buffers take the mapped mode (kernels read and write host memory
    # in place); pageable ones, or a mix, the staged copies.  The 8 units of
    # ~4100 tokens take the split-K kernel; units of 100 tokens under a cap of
    # 3 CTAs the persistent kernel, which then reads q and reduces the logits
    # from host memory.
    split = kernel == "split"
    w = Workload(name="t_host", B=2, L=2, Hq=8, Hkv=2, d=128, V=3000, T0=4200 if split else 100,
                 steps=5, n_high=(3000, 3000) if split else (40, 40),
                 n_low=(4100, 4100) if split else (64, 64), P=8, W=16, q_dtype="bf16")
    ctas = 0 if split else 3
    k, v = prefill_batch(w, 16, "cpu")
    a = ck.Cache(ck.config_from_workload(w))
    b = ck.Cache(ck.config_from_workload(w))
    a.prefill(k.cuda(), v.cuda(), [w.T0] * w.B)
    b.prefill(k.cuda(), v.cuda(), [w.T0] * w.B)
    a.set_attention_ctas(ctas)
    b.set_attention_ctas(ctas)
    assert (b.attention_plan()[0] > 1) == split
    hout = b.host_outputs(pin=pinned is not False)
    pin_in = pinned is True
    for s in range(5):
        q, kn, vn, lg = step_inputs(w, 16, s)
        o = a.step(q.cuda(), kn.cuda(), vn.cuda(), lg.cuda())
        ins = [x.pin_memory() if pin_in else x.clone() for x in (q, kn, vn, lg)]
        b.step_host(*ins, hout)
        torch.cuda.synchronize()
        assert b.stats()["host_h2d_bytes"] == sum(x.numel() * x.element_size() for x in (q, kn, vn, lg))
        assert torch.equal(o["out"].cpu(), hout["out"])
        assert torch.equal(o["budget"].cpu(), hout["budget"])
        # mapped steps on the persistent kernel reduce the logits in the
        # attention kernel (another summation order): c agrees to fp32 rounding
        assert torch.allclose(o["confidence"].cpu(), hout["confidence"], rtol=0, atol=1e-6)
        assert torch.equal(o["n_evicted"].cpu(), hout["n_evicted"])
        n = o["n_evicted"].cpu()
        for l in range(w.L):
            for bb in range(w.B):
                kk = int(n[l, bb])
                assert torch.equal(o["evicted"][l, bb, :kk].cpu(), hout["evicted"][l, bb, :kk])


def test_export_import_round_trip_resumes_identically():
    w = Workload(name="t_ckpt", B=2, L=2, Hq=8, Hkv=4, d=64, V=2000, T0=90, steps=8,
                 n_high=(30, 30), n_low=(60, 60), P=6, W=16, q_dtype="f16")
    k, v = prefill_batch(w, 17, "cpu")
    a = ck.Cache(ck.config_from_workload(w))
    a.prefill(k.cuda(), v.cuda(), [w.T0] * w.B)
    for s in range(4):
        a.step(*(t.cuda() for t in step_inputs(w, 17, s)))
    b = ck.Cache(ck.config_from_workload(w))
    for l in range(w.L):
        for bb in range(w.B):
            b.import_unit(bb, l, a.export_unit(bb, l))
    pl, steps = a.get_clock()
    b.set_clock(pl, steps)
    for s in range(4, 8):
        ins = [t.cuda() for t in step_inputs(w, 17, s)]
        oa = a.step(*ins)
        ob = b.step(*ins)
        torch.cuda.synchronize()
        assert torch.equal(oa["out"], ob["out"])
        assert torch.equal(oa["n_evicted"], ob["n_evicted"])


def test_capacity_is_checked_before_launch():
    w = Workload(name="t_cap", B=1, L=1, Hq=4, Hkv=4, d=64, V=1000, T0=40, steps=4,
                 n_high=(10 ** 5,), n_low=(10 ** 5,), P=4, W=8, q_dtype="f16", cap=48)
    k, v = prefill_batch(w, 18, "cpu")
    c = ck.Cache(ck.config_from_workload(w))
    c.prefill(k.cuda(), v.cuda(), [40])
    # 32 INT8 entries after prefill, one more per step: the 17th step would
    # need slot 48 of a 48-slot region
    for s in range(40):
        try:
            c.step(*(t.cuda() for t in step_inputs(w, 18, s)))
        except ck.ConfkvError as e:
            assert e.status == -2
            break
    else:
        pytest.fail("capacity overflow not reported")
    assert c.stats()["device_status"] == 0
    # a prefill longer than cap + W is rejected too
    k2 = torch.zeros((1, 1, 4, 80, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(ck.ConfkvError):
        c.prefill(k2, k2, [80])


def test_step_before_prefill_is_an_order_error():
    w = Workload(name="t_ord", B=1, L=1, Hq=4, Hkv=4, d=64, V=1000, T0=10, steps=1,
                 n_high=(16,), n_low=(16,), P=4, W=8)
    c = ck.Cache(ck.config_from_workload(w))
    with pytest.raises(ck.ConfkvError) as e:
        c.step(*(t.cuda() for t in step_inputs(w, 19, 0)))
    assert e.value.status == -7


def test_misaligned_buffers_are_refused_before_any_launch():
    # q is read with bulk copies (16-byte aligned sources), k_new / v_new as
    # 32-bit words: a view at an odd offset must come back as EINVAL with
    # nothing launched, and the context must still step correctly after
    import ctypes
    w = Workload(name="t_align", B=2, L=2, Hq=8, Hkv=2, d=64, V=700, T0=60, steps=2,
                 n_high=(24, 24), n_low=(40, 40), P=4, W=16, q_dtype="f16")
    p = Pair(w, 25)
    p.compare_states()
    q, kn, vn, lg = (t.cuda() for t in step_inputs(w, 25, 0))
    outs = p.cache.new_outputs()

    def shifted(t, elems):
        buf = torch.empty(t.numel() + 16, dtype=t.dtype, device="cuda")
        v = buf[elems:elems + t.numel()].view(t.shape)
        v.copy_(t)
        return v

    st0 = p.cache.stats()
    L = ck.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    cases = {"q +2 bytes": (shifted(q, 1), kn, vn, lg), "q +8 bytes": (shifted(q, 4), kn, vn, lg),
             "k_new +2 bytes": (q, shifted(kn, 1), vn, lg), "v_new +2 bytes": (q, kn, shifted(vn, 1), lg)}
    for name, (qq, kk, vv, ll) in cases.items():
        r = L.confkv_step(p.cache.handle, ptr(qq), ptr(kk), ptr(vv), ptr(ll), ptr(outs["out"]),
                          ptr(outs["budget"]), ptr(outs["confidence"]), ptr(outs["evicted"]),
                          ptr(outs["n_evicted"]), stream)
        assert r == ck.binding.EINVAL, "%s: status %d" % (name, r)
    torch.cuda.synchronize()
    st1 = p.cache.stats()
    assert st1["launches"] == st0["launches"] and st1["steps"] == st0["steps"]
    # a 16-byte-aligned view at an offset is fine
    q8 = shifted(q, 8)
    p.step(q.cpu(), kn.cpu(), vn.cpu(), lg.cpu(), gpu_step=lambda *a: p.cache.step(q8, kn, vn, lg))
    assert p.cache.stats()["launches"] == st0["launches"] + p.cache.step_launches()
    # the allocation-free confidence call checks its pointers the same way
    c = torch.empty(w.B + 1, dtype=torch.float32, device="cuda")
    lgs = shifted(lg, 1)
    assert L.confkv_confidence_noalloc(ctypes.c_void_p(lgs.data_ptr() + 2), w.B, w.V, 0.4, 0.3, 0.3, ptr(c),
                                       stream) == ck.binding.EINVAL
    assert L.confkv_confidence_noalloc(ptr(lgs), w.B, w.V, 0.4, 0.3, 0.3,
                                       ctypes.c_void_p(c.data_ptr() + 2), stream) == ck.binding.EINVAL


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_footprint_counters_follow_the_oracle(mode):
    # resident entries and K/V bytes at stored widths, and their exact peak
    # over the steps, against the oracle's state (Pair checks every step);
    # the workspace (allocator) bytes are the context's fixed footprint
    w = Workload(name="t_foot", B=3, L=2, Hq=10, Hkv=2, d=128, V=3000, T0=300, steps=20,
                 n_high=(40, 30), n_low=(120, 90), P=8, W=32, q_dtype="bf16")
    p = _run(w, 26, 20, prefill_len=[300, 17, 0], confident_every=4, mode=mode)
    st = p.cache.stats()
    assert st["peak_resident"] == p.peak_entries > 0
    assert st["peak_resident_bytes"] == p.peak_bytes > 0
    assert st["workspace_bytes"] == ck.workspace_bytes(p.cache.cfg) == p.cache.workspace.numel()
    assert st["steps"] == 20 and st["launches"] == p.launches == (20 if mode == ck.binding.STEP_AUTO else 60)
