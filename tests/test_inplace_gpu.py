"""The in-place step (zr_step_inplace): one state set, a flag pass before the update.

It must give the oracle's bits, the same bits as the ping-pong step on the same inputs, and on an
overflow step it must leave the single set bit-unchanged (the skip of page "并行训练框架DeepSpeed介绍",
核心技术 (3), taken before anything is overwritten)."""
import numpy as np
import pytest
import torch

import zero_gradient_reduction_gb300 as zr
from test_parity_gpu import HYPER, FusedRun

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


class InPlaceRun(FusedRun):
    """FusedRun on a single state set, stepped with zr_step_inplace."""

    def __init__(self, *args, **kw):
        super().__init__(*args, **kw)
        s1 = self.plan.new_state1()
        s1.master.copy_(self.state.master[0])
        s1.param.copy_(self.state.param[0])
        self.state1 = s1
        self.state = None  # the ping-pong sets are not used

    def _launch(self, stage):
        rep = self.plan.step_inplace(self.grads, self.state1, HYPER, stage=stage, report=True)
        assert rep.current == 0
        return rep

    def live(self):
        s = self.state1
        return (s.master.cpu().numpy(), s.m.cpu().numpy(), s.v.cpu().numpy(),
                s.param.cpu().view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("W,A,dtype", [(1, 1, zr.BF16), (2, 1, zr.F16), (3, 1, zr.BF16), (5, 1, zr.F16),
                                       (6, 1, zr.BF16), (7, 1, zr.F16), (8, 1, zr.BF16), (2, 4, zr.BF16),
                                       (4, 4, zr.F16), (3, 3, zr.BF16), (16, 1, zr.F16), (17, 1, zr.BF16)])
def test_inplace_ragged_buckets_bit_exact(W, A, dtype):
    rng = np.random.default_rng(W * 100 + A + 7)
    numels = [1000, 37, 5000, 8, 123_457, 64, 9_999, 3, 40_000]
    order = list(rng.permutation(W))
    run = InPlaceRun(numels, W, A, dtype, cap=20_000, S=8.0, order=order, seed=4,
                     sigma=rng.uniform(1e-3, 1e-1, size=len(numels)))
    assert len(run.plan.buckets) >= 4
    for s in range(1, 4):
        rep, _ = run.step(s)
        assert rep.t == s
        run.check(f"in place W={W} A={A} step {s}: ")


def test_inplace_equals_pingpong_with_a_skip():
    """Same seeded inputs through both modes, an overflow at step 2: identical bytes after every step."""
    numels = [60_000, 333, 20_001]
    kw = dict(cap=30_000, S=65536.0, dynamic=True, seed=6, interval=2)
    pp = FusedRun(numels, 4, 1, zr.F16, **kw)
    ip = InPlaceRun(numels, 4, 1, zr.F16, **kw)
    inj = (2, int(pp.ooffsets[2]) + 5)
    for s in range(1, 6):
        rp, _ = pp.step(s, inject=inj if s == 2 else None)
        ri, _ = ip.step(s, inject=inj if s == 2 else None)
        for f in ("overflow", "skipped", "t", "steps", "skipped_total", "good"):
            assert getattr(rp, f) == getattr(ri, f), f
        assert rp.scale_used == ri.scale_used and rp.scale == ri.scale
        for x, y in zip(pp.live(), ip.live()):
            assert x.tobytes() == y.tobytes(), f"step {s}"


@pytest.mark.parametrize("dtype", [zr.F16, zr.BF16])
def test_inplace_skip_leaves_the_set_unchanged(dtype):
    numels = [20_000, 4_000, 30_000]
    run = InPlaceRun(numels, 2, 1, dtype, cap=25_000, S=65536.0, dynamic=True, seed=5)
    run.step(1)
    before = [x.copy() for x in run.live()]
    rep, _ = run.step(2, inject=(1, int(run.ooffsets[1]) + 99))
    assert rep.overflow == 1 and rep.skipped == 1 and rep.t == 1 and rep.scale == 32768.0
    for a, b in zip(run.live(), before):
        assert a.tobytes() == b.tobytes()
    for s in (3, 4):
        rep, _ = run.step(s)
        assert rep.overflow == 0
        run.check(f"resume step {s}: ")
    assert rep.t == 3 and rep.skipped_total == 1


def test_inplace_scale_growth():
    run = InPlaceRun([4096, 1000], 2, 1, zr.BF16, cap=10_000, S=4.0, dynamic=True, interval=2)
    scales = [run.step(s)[0].scale_used for s in range(1, 6)]
    assert scales == [4.0, 4.0, 8.0, 8.0, 16.0]
    run.check()


def test_inplace_graph_replay_equals_eager():
    """Both launches of an in-place step captured in a CUDA graph; replays keep stepping (the flag and the
    scaler live in device memory)."""
    numels = [50_000, 1234]
    a = InPlaceRun(numels, 3, 1, zr.BF16, cap=40_000, S=2.0, seed=8)
    b = InPlaceRun(numels, 3, 1, zr.BF16, cap=40_000, S=2.0, seed=8)
    st = torch.cuda.current_stream().cuda_stream
    for r in range(3):  # one fixed set of gradients, stepped three times
        a.layout.grads_dev(a.grads[r], 1, r, 2.0, a.table, st)
        b.layout.grads_dev(b.grads[r], 1, r, 2.0, b.table, st)
    for _ in range(3):
        a.plan.step_inplace(a.grads, a.state1, HYPER)
    g = b.plan.capture(b.grads, b.state1, HYPER, steps=1)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ra, rb = a.plan.report(), b.plan.report()
    assert ra.t == rb.t == 3 and ra.current == rb.current == 0
    for x, y in zip(a.live(), b.live()):
        assert x.tobytes() == y.tobytes()


def test_inplace_error_paths():
    plan = zr.Plan([1024], W=2, A=1, dtype=zr.BF16, stage=2, cap=2048)
    s1 = plan.new_state1()
    grads = [torch.zeros(plan.numel, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(zr.ZrError) as e:
        plan.step_inplace(grads, s1, HYPER, stage=4)
    assert e.value.status == 1
    with pytest.raises(zr.ZrError):
        plan.step_inplace([grads[0], grads[1][1:]], s1, HYPER)  # 2-byte offset: misaligned
    master = s1.master
    s1.master = master[1:]  # 4-byte offset: misaligned
    with pytest.raises(zr.ZrError):
        plan.step_inplace(grads, s1, HYPER)
    s1.master = master
    # nothing above launched, and the control block is untouched
    s1.master.zero_()
    r = plan.step_inplace(grads, s1, HYPER, report=True)
    assert r.t == 1 and r.steps == 1 and r.overflow == 0


def test_inplace_guard_bands_clean_and_skipped():
    """Both launches stay inside every buffer, on a clean step and on a skipped one."""
    from test_guards_gpu import Guarded
    numels = [12_345, 7, 40_000, 8, 999]
    for W, A in ((3, 1), (2, 4), (8, 1)):
        plan = zr.Plan(numels, W=W, A=A, dtype=zr.BF16, stage=2, cap=20_000, scaler=zr.Scaler(1.0))
        n = plan.numel
        grads = [Guarded(n, torch.bfloat16) for _ in range(W * A)]
        for g in grads:
            g.t.normal_()
        bufs = [Guarded(n, torch.float32) for _ in range(3)] + [Guarded(n, torch.bfloat16)]
        bufs[0].t.fill_(0.01)
        bufs[1].t.zero_()
        bufs[2].t.zero_()
        one = zr.State1.of(*(b.t for b in bufs))
        rep = plan.step_inplace([g.t for g in grads], one, HYPER, report=True)
        assert rep.overflow == 0
        grads[-1].t[n - 1] = float("nan")
        rep = plan.step_inplace([g.t for g in grads], one, HYPER, report=True)
        assert rep.overflow == 1 and rep.t == 1
        assert all(x.intact() for x in grads + bufs), (W, A)
        plan.close()


def test_inplace_max_workers_and_replicas_with_empty_tensors():
    """W = 64 and W*A = 256 (the limits), zero-size tensors in the list."""
    import oracle
    from test_parity_gpu import OHYPER, assert_state_close
    numels = [0, 5000, 0, 1, 20_000, 0]
    for W, A in ((64, 1), (64, 4)):
        plan = zr.Plan(numels, W=W, A=A, dtype=zr.BF16, stage=1, cap=8_000, scaler=zr.Scaler(1.0))
        n = plan.numel
        rng = np.random.default_rng(W * 3 + A)
        hg = [oracle.encode(zr.BF16, rng.normal(size=n).astype(np.float32)) for _ in range(W * A)]
        grads = [torch.from_numpy(g.view(np.int16).copy()).cuda().view(torch.bfloat16) for g in hg]
        one = plan.new_state1()
        master = (rng.normal(size=n) * 0.02).astype(np.float32)
        one.master.copy_(torch.from_numpy(master))
        rep = plan.step_inplace(grads, one, HYPER, report=True)
        o = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
        from _harness import oracle_layout
        ob, _ = oracle_layout(plan, numels, 8_000, W)
        orep, _ = oracle.step(W, A, zr.BF16, ob, hg, *o, OHYPER, oracle.new_scaler(1.0))
        assert rep.overflow == orep.overflow == 0 and rep.t == 1
        assert_state_close(one.master.cpu().numpy(), one.m.cpu().numpy(), one.v.cpu().numpy(),
                           one.param.cpu().view(torch.int16).numpy().view(np.uint16), *o, exact=True,
                           where=f"in place W={W} A={A}: ")
        plan.close()


def test_inplace_fp32_overflow_from_finite_bf16_skips():
    """Finite bf16 values whose fp32 ring sum is +inf: the flag pass must see the sum, not the inputs."""
    import oracle
    n = 64
    hg = [oracle.encode(zr.BF16, np.full(n, 3.0e38, np.float32)) for _ in range(2)]
    plan = zr.Plan([n], W=2, dtype=zr.BF16, stage=2, cap=n, scaler=zr.Scaler(1.0, dynamic=True))
    one = plan.new_state1()
    one.master.fill_(0.5)
    one.param.fill_(0.5)
    before = [t.clone() for t in (one.master, one.m, one.v, one.param)]
    grads = [torch.from_numpy(g.view(np.int16).copy()).cuda().view(torch.bfloat16) for g in hg]
    rep = plan.step_inplace(grads, one, HYPER, report=True)
    assert rep.overflow == 1 and rep.t == 0 and rep.skipped_total == 1
    for a, b in zip((one.master, one.m, one.v, one.param), before):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    plan.close()


@pytest.mark.parametrize("W,A", [(2, 4), (8, 2)])
def test_inplace_fp32_gradients_equal_pingpong(W, A):
    """A plan over fp32 micro-batch sums (zr_accumulate): in place and ping-pong give the same bytes."""
    numels = [40_000, 999, 77_777, 8]
    rng = np.random.default_rng(W + 5 * A)
    order = list(rng.permutation(W))
    kw = dict(W=W, A=1, dtype=zr.BF16, stage=2, cap=50_000, order=order, scaler=zr.Scaler(1.0), fp32_grads=True)
    pa, pb = zr.Plan(numels, **kw), zr.Plan(numels, **kw)
    n = pa.numel
    st = pa.new_state()
    st.master[0].copy_(torch.from_numpy((rng.normal(size=n) * 0.02).astype(np.float32)))
    one = pb.new_state1()
    one.master.copy_(st.master[0])
    accs = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(W)]
    for step in (1, 2, 3):
        for wk in range(W):
            for q in range(A):
                g = torch.from_numpy((rng.normal(size=n) * 1e-2).astype(np.float32)).cuda().to(torch.bfloat16)
                zr.accumulate(g, accs[wk], q == 0)
        ra = pa.step(accs, st, HYPER, report=True)
        rb = pb.step_inplace(accs, one, HYPER, report=True)
        assert ra.overflow == rb.overflow == 0 and ra.t == rb.t == step
        L = st.live(ra.current)
        for x, y in zip((L["master"], L["m"], L["v"], L["param"]), (one.master, one.m, one.v, one.param)):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), step
    pa.close()
    pb.close()


def test_inplace_checkpoint_resume_is_byte_identical():
    """Four in-place steps straight against two, a checkpoint (control block + the one set), a restore into
    a fresh plan and two more: the same bytes, with a skip in between."""
    import oracle
    numels = [30_000, 5_000, 17_000]
    kw = dict(cap=25_000, S=65536.0, dynamic=True, seed=9, interval=2)
    straight = InPlaceRun(numels, 2, 1, zr.F16, **kw)
    inj = (0, int(straight.ooffsets[1]) + 7)
    for s in range(1, 5):
        straight.step(s, inject=inj if s == 2 else None)
    first = InPlaceRun(numels, 2, 1, zr.F16, **kw)
    for s in (1, 2):
        first.step(s, inject=inj if s == 2 else None)
    ck = first.plan.checkpoint()
    assert ck.t == 1 and ck.skipped == 1 and ck.scale == 32768.0 and ck.current == 0
    second = InPlaceRun(numels, 2, 1, zr.F16, **kw)
    second.plan.restore(ck)
    for name in ("master", "m", "v", "param"):
        getattr(second.state1, name).copy_(getattr(first.state1, name))
    second.o = [x.copy() for x in first.o]
    second.osc = oracle.Scaler.from_buffer_copy(first.osc)
    second.S = ck.scale
    for s in (3, 4):
        second.step(s)
    for a, b in zip(straight.live(), second.live()):
        assert a.tobytes() == b.tobytes()
    second.check("resumed in place: ")


@pytest.mark.parametrize("pinned", [True, False])
def test_inplace_from_host_equals_inplace(pinned):
    """zr_step_inplace_from_host: the host gradients copied in, then the same in-place step."""
    numels = [50_000, 777, 12_345]
    a = InPlaceRun(numels, 3, 1, zr.F16, cap=40_000, S=1024.0, seed=2)
    b = InPlaceRun(numels, 3, 1, zr.F16, cap=40_000, S=1024.0, seed=2)
    for s in (1, 2):
        a.step(s)
        host = []
        for r in range(3):
            g = b.layout.grads_host(0, b.n, s, r, b.S)
            host.append(torch.from_numpy(g.view(np.int16).copy()).pin_memory() if pinned else g.copy())
        for d in b.grads:
            d.fill_(0)
        rep = b.plan.step_inplace_from_host(host, b.grads, b.state1, HYPER)
        assert rep.t == s and rep.overflow == 0 and rep.current == 0
        for x, y in zip(a.live(), b.live()):
            assert x.tobytes() == y.tobytes()
