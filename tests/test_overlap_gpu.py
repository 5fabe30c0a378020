"""Bucketed steps for overlap with backward (zr_step_bucket): launched bucket by bucket, as each bucket's
gradients become ready, they compute exactly what one zr_step computes, including a skip decided by a
non-finite value in any bucket (page "DP / DDP / DeepSpeed ZeRO-1/2/3", section 二; page "第 7 讲", Overlap)."""
import numpy as np
import pytest
import torch

import oracle
import zero_gradient_reduction_gb300 as zr
import zrgen
from zrgen.layout import Layout
from _harness import oracle_layout
from test_parity_gpu import HYPER, OHYPER, assert_state_close, u16

pytestmark = pytest.mark.gpu
F32 = np.float32
NUMELS = [30_000, 777, 61_000, 8, 12_345, 40_000]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _setup(W=3, dtype=zr.F16, S=1024.0, dynamic=False):
    plans = [zr.Plan(NUMELS, W=W, dtype=dtype, stage=2, cap=35_000, scaler=zr.Scaler(S, dynamic)) for _ in range(2)]
    _, ooff = oracle_layout(plans[0], NUMELS, 35_000, W)
    lay = Layout(NUMELS, ooff, np.full(len(NUMELS), 1e-2, F32), 3, dtype)
    table = torch.from_numpy(zrgen.normal_table().copy()).cuda()
    states = []
    for p in plans:
        st = p.new_state()
        st.master[0].zero_()
        lay.master_dev(st.master[0], table, torch.cuda.current_stream().cuda_stream)
        states.append(st)
    return plans, lay, table, states


def _live_bytes(st, k):
    return [t.cpu().contiguous().view(torch.int8).numpy().tobytes() for t in st.live(k).values()]


def test_bucketed_equals_single_launch():
    plans, lay, table, (sa, sb) = _setup()
    assert len(plans[0].buckets) >= 4
    n = plans[0].numel
    grads = [torch.zeros(n, dtype=torch.float16, device="cuda") for _ in range(3)]
    cs = torch.cuda.current_stream().cuda_stream
    for step in (1, 2, 3):
        for r in range(3):
            lay.grads_dev(grads[r], step, r, 1024.0, table, cs)
        ra = plans[0].step(grads, sa, HYPER, report=True)
        for b in range(len(plans[1].buckets)):
            plans[1].step_bucket(b, grads, sb, HYPER)
        rb = plans[1].report()
        assert (ra.current, ra.t, ra.overflow, ra.steps) == (rb.current, rb.t, rb.overflow, rb.steps)
        assert _live_bytes(sa, ra.current) == _live_bytes(sb, rb.current)


@pytest.mark.parametrize("cap", [1, 3, 16])
def test_bucket_block_cap_gives_the_same_bytes(cap):
    """zr_plan_set_bucket_blocks only changes the launch shape: every bucket launch capped at `cap` blocks
    (striding over its tiles) computes what one zr_step computes."""
    plans, lay, table, (sa, sb) = _setup()
    plans[1].set_bucket_blocks(cap)
    n = plans[0].numel
    grads = [torch.zeros(n, dtype=torch.float16, device="cuda") for _ in range(3)]
    cs = torch.cuda.current_stream().cuda_stream
    for step in (1, 2):
        for r in range(3):
            lay.grads_dev(grads[r], step, r, 1024.0, table, cs)
        ra = plans[0].step(grads, sa, HYPER, report=True)
        for b in range(len(plans[1].buckets)):
            plans[1].step_bucket(b, grads, sb, HYPER)
        rb = plans[1].report()
        assert (ra.current, ra.t, ra.overflow, ra.steps) == (rb.current, rb.t, rb.overflow, rb.steps)
        assert _live_bytes(sa, ra.current) == _live_bytes(sb, rb.current)
    plans[1].set_bucket_blocks(0)  # back to one block per tile, between steps
    ra = plans[0].step(grads, sa, HYPER, report=True)
    for b in range(len(plans[1].buckets)):
        plans[1].step_bucket(b, grads, sb, HYPER)
    rb = plans[1].report()
    assert ra.steps == rb.steps == 3 and _live_bytes(sa, ra.current) == _live_bytes(sb, rb.current)
    with pytest.raises(zr.ZrError):
        plans[1].set_bucket_blocks(-1)


def test_bucketed_skip_is_global():
    plans, lay, table, (sa, _) = _setup(W=2, S=65536.0, dynamic=True)
    p = plans[0]
    n = p.numel
    grads = [torch.zeros(n, dtype=torch.float16, device="cuda") for _ in range(2)]
    cs = torch.cuda.current_stream().cuda_stream
    for r in range(2):
        lay.grads_dev(grads[r], 1, r, 65536.0, table, cs)
    for b in range(len(p.buckets)):
        p.step_bucket(b, grads, sa, HYPER)
    r1 = p.report()
    before = _live_bytes(sa, r1.current)
    mid = len(p.buckets) // 2
    s0 = int(p.buckets[mid, 0])
    grads[1].view(torch.int16)[s0 + 5] = 0x7C00  # +inf inside a middle bucket
    for b in range(len(p.buckets)):
        p.step_bucket(b, grads, sa, HYPER)
    r2 = p.report()
    assert r2.overflow == 1 and r2.current == r1.current and r2.t == 1 and r2.scale == 32768.0
    assert _live_bytes(sa, r2.current) == before


def test_overlapped_schedule_matches_oracle():
    """A compute stream produces each bucket's gradients in bucket order and records an event; the step of
    bucket b waits for that event on a side stream. The result is the oracle's."""
    plans, lay, table, (sa, _) = _setup(W=4, dtype=zr.BF16, S=1.0)
    p = plans[0]
    n = p.numel
    W = 4
    grads = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    compute, side = torch.cuda.Stream(), torch.cuda.Stream()
    compute.wait_stream(torch.cuda.current_stream())  # zeroed buffers and the master init come first
    side.wait_stream(torch.cuda.current_stream())
    om = lay.master_host(0, n)
    o = [om, np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)]
    osc = oracle.new_scaler(1.0)
    ob, ooff = oracle_layout(p, NUMELS, 35_000, W)
    by_off = sorted(range(len(NUMELS)), key=lambda t: ooff[t])
    for step in (1, 2):
        events = []
        for b, (s0, ln, _) in enumerate(ob):
            with torch.cuda.stream(compute):
                for t in by_off:  # "backward" writes this bucket's tensors
                    off = int(ooff[t])
                    if s0 <= off < s0 + ln:
                        for r in range(W):
                            zrgen.fill_dev(grads[r].data_ptr() + 2 * off, NUMELS[t], zrgen.BF16, 3,
                                           zrgen.stream_id(zrgen.TAG_GRAD, step, r, t), 0, np.float32(1e-2),
                                           table.data_ptr(), compute.cuda_stream)
                ev = torch.cuda.Event()
                ev.record(compute)
                events.append(ev)
        p.step_overlapped(grads, sa, HYPER, events, side)
        torch.cuda.synchronize()
        rep = p.report()
        og = [lay.grads_host(0, n, step, r, 1.0) for r in range(W)]
        oracle.step(W, 1, zr.BF16, ob, og, *o, OHYPER, osc)
        L = sa.live(rep.current)
        assert_state_close(L["master"].cpu().numpy(), L["m"].cpu().numpy(), L["v"].cpu().numpy(),
                           u16(L["param"]), *o, exact=True, where=f"overlapped step {step}: ")


@pytest.mark.parametrize("staging", [zr.STAGING_REGISTERS, zr.STAGING_BULK])
def test_graph_replay_steps_like_direct_calls(staging):
    """A CUDA graph of one zr_step, replayed (the launch the benchmark times), keeps stepping (live set, scale
    and t come from device memory) and gives the same bytes as calling zr_step each time, with either load
    staging in the graph."""
    plans, lay, table, (sa, sb) = _setup(W=2, dtype=zr.BF16, S=1.0)
    plans[1].set_staging(staging)
    n = plans[0].numel
    grads = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for r in range(2):
        lay.grads_dev(grads[r], 1, r, 1.0, table, torch.cuda.current_stream().cuda_stream)
    g = plans[1].capture(grads, sb, HYPER)
    for _ in range(3):
        plans[0].step(grads, sa, HYPER)
        g.replay()
    torch.cuda.synchronize()
    ra, rb = plans[0].report(), plans[1].report()
    assert ra.t == rb.t == 3 and ra.current == rb.current
    assert _live_bytes(sa, ra.current) == _live_bytes(sb, rb.current)
