"""Out-of-bounds checks without a sanitizer: every device buffer a call touches sits between guard bands of a
known pattern, which must be intact after the call. Plus the method's degenerate cases."""
import numpy as np
import pytest
import torch

import oracle
import zero_gradient_reduction_gb300 as zr
from _harness import oracle_layout
from test_parity_gpu import HYPER, OHYPER, assert_state_close, u16

pytestmark = pytest.mark.gpu
GUARD = 4096  # bytes on each side
PATTERN = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


class Guarded:
    """A device buffer of `n` elements of `dtype` with GUARD bytes of PATTERN before and after it."""

    def __init__(self, n, dtype):
        esz = torch.empty(0, dtype=dtype).element_size()
        self.raw = torch.full((GUARD * 2 + n * esz,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n * esz].view(dtype)

    def intact(self):
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[-GUARD:] == PATTERN).all())


def test_guards_fused_step_and_bucketed():
    numels = [12_345, 7, 40_000, 8, 999]
    for W, A in ((3, 1), (2, 4), (5, 2)):
        plan = zr.Plan(numels, W=W, A=A, dtype=zr.BF16, stage=2, cap=20_000, scaler=zr.Scaler(1.0))
        n = plan.numel
        grads = [Guarded(n, torch.bfloat16) for _ in range(W * A)]
        for g in grads:
            g.t.normal_()
        st = zr.State.__new__(zr.State)
        parts = {k: [Guarded(n, torch.float32) for _ in range(2)] for k in ("master", "m", "v")}
        prm = [Guarded(n, torch.bfloat16) for _ in range(2)]
        st.master = [p.t for p in parts["master"]]
        st.m = [p.t for p in parts["m"]]
        st.v = [p.t for p in parts["v"]]
        st.param = [p.t for p in prm]
        for k in range(2):
            st.m[k].zero_(); st.v[k].zero_(); st.master[k].fill_(0.01)
        plan.step([g.t for g in grads], st, HYPER)
        for b in range(len(plan.buckets)):
            plan.step_bucket(b, [g.t for g in grads], st, HYPER)
        torch.cuda.synchronize()
        everything = grads + prm + [p for v in parts.values() for p in v]
        assert all(x.intact() for x in everything), (W, A)
        plan.close()


def _guarded_state(n, tdt):
    st = zr.State.__new__(zr.State)
    parts = {k: [Guarded(n, torch.float32) for _ in range(2)] for k in ("master", "m", "v")}
    prm = [Guarded(n, tdt) for _ in range(2)]
    st.master = [p.t for p in parts["master"]]
    st.m = [p.t for p in parts["m"]]
    st.v = [p.t for p in parts["v"]]
    st.param = [p.t for p in prm]
    for k in range(2):
        st.m[k].zero_(); st.v[k].zero_(); st.master[k].fill_(0.01)
    return st, prm + [p for v in parts.values() for p in v]


@pytest.mark.parametrize("staging", [zr.STAGING_BULK, zr.STAGING_BULK_IO])
def test_guards_bulk_staging(staging):
    """Bulk-copy staging (loads, and loads + stores) writes nothing outside its buffers: ragged tensors, stages
    of 256 elements so that tiles end in partial stages, the specialised (W = 2, 8) and generic (W = 3, A = 2)
    kernels."""
    numels = [12_345, 7, 40_000, 8, 999]
    for W, A, dtype, shape in ((2, 1, zr.F16, (256, 2)), (8, 1, zr.BF16, (256, 3)), (3, 2, zr.BF16, (0, 0))):
        plan = zr.Plan(numels, W=W, A=A, dtype=dtype, stage=2, cap=20_000, scaler=zr.Scaler(1.0))
        plan.set_staging(staging, *shape)
        assert plan.staging == staging
        n = plan.numel
        tdt = plan.torch_dtype()
        grads = [Guarded(n, tdt) for _ in range(W * A)]
        for g in grads:
            g.t.normal_()
        st, bufs = _guarded_state(n, tdt)
        for _ in range(2):
            plan.step([g.t for g in grads], st, HYPER)
        torch.cuda.synchronize()
        assert all(x.intact() for x in grads + bufs), (staging, W, A)
        plan.close()


def test_guards_in_place_step():
    numels = [12_345, 7, 40_000, 8, 999]
    for W, A in ((2, 1), (3, 2)):
        plan = zr.Plan(numels, W=W, A=A, dtype=zr.F16, stage=1, cap=20_000, scaler=zr.Scaler(1.0))
        n = plan.numel
        grads = [Guarded(n, torch.float16) for _ in range(W * A)]
        for g in grads:
            g.t.normal_()
        bufs = [Guarded(n, torch.float32) for _ in range(3)] + [Guarded(n, torch.float16)]
        bufs[0].t.fill_(0.01); bufs[1].t.zero_(); bufs[2].t.zero_()
        one = zr.State1.of(bufs[0].t, bufs[1].t, bufs[2].t, bufs[3].t)
        plan.step_inplace([g.t for g in grads], one, HYPER)
        torch.cuda.synchronize()
        assert all(x.intact() for x in grads + bufs), (W, A)
        plan.close()


def test_guards_standalone_calls():
    rng_n = [1, 7, 9, 1000, 65_541]
    for n in rng_n:
        W = 3
        gs = [Guarded(n, torch.float16) for _ in range(W)]
        for g in gs:
            g.t.normal_()
        sums = Guarded(n, torch.float32)
        flag = Guarded(1, torch.int32)
        flag.t.zero_()
        zr.reduce_scatter([g.t for g in gs], sums.t, flag.t)
        ar = [Guarded(n, torch.float32) for _ in range(2)]
        zr.all_reduce([g.t for g in gs], [x.t for x in ar], flag.t)
        m, v, p = (Guarded(n, torch.float32) for _ in range(3))
        m.t.zero_(); v.t.zero_(); p.t.fill_(0.5)
        zr.adamw_shard_step(sums.t, m.t, v.t, p.t, HYPER, 1.0, W, 1, flag.t)
        reps = [Guarded(n, torch.float16) for _ in range(2)]
        zr.all_gather(p.t, [r.t for r in reps])
        acc = Guarded(n, torch.float32)
        zr.accumulate(gs[0].t, acc.t, True)
        zr.accumulate(gs[1].t, acc.t, False)
        torch.cuda.synchronize()
        assert all(x.intact() for x in gs + [sums, flag, m, v, p, acc] + reps + ar), n


def test_guards_zero3_and_noalloc():
    numels = [10_000, 333, 25_000]
    W = 4
    plan = zr.Plan(numels, W=W, dtype=zr.F16, stage=3, cap=15_000)
    n = plan.numel
    full = Guarded(n, torch.float16)
    full.t.normal_()
    shards = [Guarded(max(plan.shard_numel(w), 8), torch.float16) for w in range(W)]
    plan.shard_params(full.t, [s.t for s in shards])
    out = Guarded(n, torch.float16)
    plan.gather_params([s.t for s in shards], out.t, 0, len(plan.buckets))
    torch.cuda.synchronize()
    assert torch.equal(out.t.view(torch.int16), full.t.view(torch.int16))
    assert all(x.intact() for x in [full, out] + shards)
    # the no-allocation step on guarded state
    grads = [Guarded(n, torch.float16) for _ in range(W)]
    for g in grads:
        g.t.normal_()
    st = zr.State.__new__(zr.State)
    bufs = [Guarded(n, torch.float32) for _ in range(6)] + [Guarded(n, torch.float16) for _ in range(2)]
    st.master, st.m, st.v, st.param = [bufs[0].t, bufs[1].t], [bufs[2].t, bufs[3].t], [bufs[4].t, bufs[5].t], \
        [bufs[6].t, bufs[7].t]
    for b in bufs[:6]:
        b.t.zero_()
    of = torch.zeros(1, dtype=torch.int32, device="cuda")
    zr.step_noalloc(plan.buckets, W, 1, zr.F16, [g.t for g in grads], st, 0, HYPER, 1.0, 1, of)
    torch.cuda.synchronize()
    assert all(x.intact() for x in grads + bufs)
    plan.close()


def test_max_workers_and_replicas_with_empty_tensors():
    """W = 64 (the limit), W*A = 256 (the limit) and zero-size tensors in the list."""
    numels = [0, 5000, 0, 1, 20_000, 0]
    for W, A in ((64, 1), (64, 4)):
        plan = zr.Plan(numels, W=W, A=A, dtype=zr.BF16, stage=1, cap=8_000, scaler=zr.Scaler(1.0))
        n = plan.numel
        rng = np.random.default_rng(W + A)
        hg = [oracle.encode(zr.BF16, rng.normal(size=n).astype(np.float32)) for _ in range(W * A)]
        grads = [torch.from_numpy(g.view(np.int16).copy()).cuda().view(torch.bfloat16) for g in hg]
        st = plan.new_state()
        master = (rng.normal(size=n) * 0.02).astype(np.float32)
        st.master[0].copy_(torch.from_numpy(master))
        rep = plan.step(grads, st, HYPER, report=True)
        o = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
        ob, _ = oracle_layout(plan, numels, 8_000, W)
        orep, _ = oracle.step(W, A, zr.BF16, ob, hg, *o, OHYPER, oracle.new_scaler(1.0))
        assert rep.overflow == orep.overflow == 0
        L = st.live(rep.current)
        assert_state_close(L["master"].cpu().numpy(), L["m"].cpu().numpy(), L["v"].cpu().numpy(), u16(L["param"]),
                           *o, exact=True, where=f"W={W} A={A}: ")
        plan.close()


def test_fp32_overflow_from_finite_bf16_skips():
    """Two finite bf16 values near the top of the range sum to +inf in fp32: the step is skipped."""
    n = 64
    big = np.full(n, 3.0e38, np.float32)
    hg = [oracle.encode(zr.BF16, big) for _ in range(2)]
    assert np.all(np.isfinite(oracle.decode(zr.BF16, hg[0])))
    plan = zr.Plan([n], W=2, dtype=zr.BF16, stage=2, cap=n, scaler=zr.Scaler(1.0, dynamic=True))
    st = plan.new_state()
    st.master[0].fill_(0.5)
    grads = [torch.from_numpy(g.view(np.int16).copy()).cuda().view(torch.bfloat16) for g in hg]
    rep = plan.step(grads, st, HYPER, report=True)
    ob, _ = oracle_layout(plan, [n], n, 2)
    orep, _ = oracle.step(2, 1, zr.BF16, ob, hg, np.full(n, 0.5, np.float32), np.zeros(n, np.float32),
                          np.zeros(n, np.float32), np.zeros(n, np.uint16), OHYPER, oracle.new_scaler(1.0, dynamic=True))
    assert rep.overflow == orep.overflow == 1 and rep.current == 0 and rep.t == 0
    plan.close()


def test_signed_zero_gradients():
    """All-negative-zero gradients sum to -0 (the sum starts from the first worker's value, not +0)."""
    n = 32
    hg = [np.full(n, 0x8000, np.uint16) for _ in range(3)]  # -0.0 in fp16
    plan = zr.Plan([n], W=3, dtype=zr.F16, stage=2, cap=n, scaler=zr.Scaler(1.0))
    sums = torch.empty(n, dtype=torch.float32, device="cuda")
    of = torch.zeros(1, dtype=torch.int32, device="cuda")
    zr.reduce_scatter([torch.from_numpy(g.view(np.int16).copy()).cuda().view(torch.float16) for g in hg], sums, of)
    torch.cuda.synchronize()
    got = sums.cpu().numpy()
    assert np.all(got == 0) and np.all(np.signbit(got))
    z = np.zeros(n, np.float32)
    ob, _ = oracle_layout(plan, [n], n, 3)
    _, want = oracle.step(3, 1, zr.F16, ob, hg, z.copy(), z.copy(), z.copy(), np.zeros(n, np.uint16),
                          OHYPER, oracle.new_scaler(1.0), want_sums=True)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    plan.close()
