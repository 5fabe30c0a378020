"""GPU parity: every C-ABI call against the oracle, element by element, on seeded inputs.

Bar (the stated tolerances): reduced sums, overflow flag and skip decision bit-exact; fp32 master/m/v
within 2 ulp; 16-bit params within 1 ulp. The kernels follow the oracle's op order with IEEE
round-to-nearest ops and no contraction, so these tests also assert bit-exactness where it is expected.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import zero_gradient_reduction_gb300 as zr
import zrgen
from _harness import Layout, oracle_layout

pytestmark = pytest.mark.gpu

F32 = np.float32
HYPER = zr.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
OHYPER = oracle.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32bits(t) -> np.ndarray:
    a = t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else t
    return np.ascontiguousarray(a, dtype=F32).view(np.uint32)


def to_dev16(a: np.ndarray, dtype: int) -> torch.Tensor:
    tdt = torch.float16 if dtype == zr.F16 else torch.bfloat16
    return torch.from_numpy(a.view(np.int16).copy()).cuda().view(tdt)


def ulp_diff_f32(a: np.ndarray, b: np.ndarray) -> int:
    """Max distance in representable fp32 steps (sign-magnitude order)."""
    ia = np.asarray(a, F32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, F32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return int(np.max(np.abs(ia - ib))) if ia.size else 0


def ulp_diff_16(a: np.ndarray, b: np.ndarray) -> int:
    ia = np.asarray(a, np.uint16).astype(np.int64)
    ib = np.asarray(b, np.uint16).astype(np.int64)
    ia = np.where(ia & 0x8000, -(ia & 0x7FFF), ia)
    ib = np.where(ib & 0x8000, -(ib & 0x7FFF), ib)
    return int(np.max(np.abs(ia - ib))) if ia.size else 0


def assert_state_close(gm, gmm, gv, gp, om, omm, ov, op, exact=True, where=""):
    for name, g, o in (("master", gm, om), ("m", gmm, omm), ("v", gv, ov)):
        d = ulp_diff_f32(g, o)
        assert d <= 2, f"{where}{name}: {d} ulp"
        if exact:
            assert np.array_equal(np.asarray(g, F32).view(np.uint32), np.asarray(o, F32).view(np.uint32)), \
                f"{where}{name}: not bit-exact ({d} ulp)"
    d = ulp_diff_16(gp, op)
    assert d <= 1, f"{where}param: {d} ulp"
    if exact:
        assert np.array_equal(gp, op), f"{where}param: not bit-exact"


# ----------------------------------------------------------------------------- generator
@pytest.mark.parametrize("dt", [zrgen.F16, zrgen.BF16, zrgen.F32])
def test_generator_host_equals_device(dt):
    table = torch.from_numpy(zrgen.normal_table().copy()).cuda()
    for first, n, scale in ((0, 1, 1.0), (3, 1001, 0.5), (8, 65536, 655.36), (12345, 300_001, 1e-4)):
        host = zrgen.fill_host(n, dt, 7, 99, first, scale)
        tdt = {zrgen.F16: torch.float16, zrgen.BF16: torch.bfloat16, zrgen.F32: torch.float32}[dt]
        buf = torch.empty(n, dtype=tdt, device="cuda")
        zrgen.fill_dev(buf.data_ptr(), n, dt, 7, 99, first, scale, table.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        devb = u16(buf) if dt != zrgen.F32 else buf.cpu().numpy().view(np.uint32)
        hostb = host if dt != zrgen.F32 else host.view(np.uint32)
        assert np.array_equal(devb, hostb)


# ----------------------------------------------------------------------------- reduce-scatter
def _rand_grads(rng, W, n, dtype, scale=3.0):
    out = []
    for _ in range(W):
        out.append(oracle.encode(dtype, (rng.normal(size=n) * scale).astype(F32)))
    return out


def _oracle_sums(grads, W, n, dtype, order):
    C = oracle.chunk_size(n, W, 8)
    z = np.zeros(n, F32)
    rep, sums = oracle.step(W, 1, dtype, np.array([[0, n, C]]), grads, z.copy(), z.copy(), z.copy(),
                            np.zeros(n, np.uint16), OHYPER, oracle.new_scaler(), order=order, want_sums=True)
    return sums, rep.overflow


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("dtype", [zr.F16, zr.BF16])
def test_reduce_scatter_bit_exact(W, dtype):
    rng = np.random.default_rng(W * 10 + dtype)
    for n in (1, 7, 8, 100, 8 * W * 3 + 3, 65_541, 300_000):
        order = list(rng.permutation(W))
        grads = _rand_grads(rng, W, n, dtype)
        want, flag = _oracle_sums(grads, W, n, dtype, order)
        gd = [to_dev16(g, dtype) for g in grads]
        sums = torch.empty(n, dtype=torch.float32, device="cuda")
        of = torch.zeros(1, dtype=torch.int32, device="cuda")
        zr.reduce_scatter(gd, sums, of, order=order)
        torch.cuda.synchronize()
        assert np.array_equal(f32bits(sums), want.view(np.uint32)), (W, n)
        assert int(of.item()) == flag == 0


@pytest.mark.parametrize("W", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("dtype", [zr.F16, zr.BF16])
def test_all_reduce_bit_exact(W, dtype):
    """Every one of the R outputs equals what the oracle's hop-by-hop all-reduce leaves on every worker."""
    rng = np.random.default_rng(W * 17 + dtype)
    for n in (1, 9, 8 * W * 2 + 5, 70_003):
        order = list(rng.permutation(W))
        grads = _rand_grads(rng, W, n, dtype)
        xs = [oracle.decode(dtype, g) for g in grads]
        work = [xs[order[p]].copy() for p in range(W)]
        oracle.ring_all_reduce(work, oracle.chunk_size(n, W, 8))
        for p in range(1, W):
            assert np.array_equal(work[p].view(np.uint32), work[0].view(np.uint32))
        outs = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(W)]
        of = torch.zeros(1, dtype=torch.int32, device="cuda")
        zr.all_reduce([to_dev16(g, dtype) for g in grads], outs, of, order=order)
        torch.cuda.synchronize()
        for o in outs:
            assert np.array_equal(f32bits(o), work[0].view(np.uint32)), (W, n)
        assert int(of.item()) == 0
    # a non-finite input sets the flag; R = 1 is the reduce-scatter
    grads = _rand_grads(rng, W, 4096, dtype)
    grads[W - 1][100] = 0x7C00 if dtype == zr.F16 else 0x7F80
    gd = [to_dev16(g, dtype) for g in grads]
    one = torch.empty(4096, dtype=torch.float32, device="cuda")
    rs = torch.empty(4096, dtype=torch.float32, device="cuda")
    of1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    of2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    zr.all_reduce(gd, [one], of1)
    zr.reduce_scatter(gd, rs, of2)
    torch.cuda.synchronize()
    assert int(of1.item()) == int(of2.item()) == 1 and torch.equal(one.view(torch.int32), rs.view(torch.int32))


def test_reduce_scatter_overflow_flag_sticky():
    rng = np.random.default_rng(1)
    W, n = 4, 10_000
    grads = _rand_grads(rng, W, n, zr.F16)
    of = torch.zeros(1, dtype=torch.int32, device="cuda")
    sums = torch.empty(n, dtype=torch.float32, device="cuda")
    zr.reduce_scatter([to_dev16(g, zr.F16) for g in grads], sums, of)
    torch.cuda.synchronize()
    assert of.item() == 0
    for bad, pos in ((0x7C00, 9_999), (0x7E00, 5), (0xFC00, 4_321)):
        g2 = [g.copy() for g in grads]
        g2[2][pos] = bad
        want, flag = _oracle_sums(g2, W, n, zr.F16, None)
        of.zero_()
        zr.reduce_scatter([to_dev16(g, zr.F16) for g in g2], sums, of)
        torch.cuda.synchronize()
        assert of.item() == 1 == flag
        got = sums.cpu().numpy()
        assert np.array_equal(np.isnan(got), np.isnan(want))
        fin = np.isfinite(want)
        assert np.array_equal(got[fin].view(np.uint32), want[fin].view(np.uint32))
        # the flag is never cleared by a clean call
        zr.reduce_scatter([to_dev16(g, zr.F16) for g in grads], sums, of)
        torch.cuda.synchronize()
        assert of.item() == 1


# ----------------------------------------------------------------------------- AdamW shard step
@pytest.mark.parametrize("n", [1, 5, 4096, 100_003])
@pytest.mark.parametrize("t", [1, 7])
def test_adamw_shard_step_bit_exact(n, t):
    rng = np.random.default_rng(n + t)
    S, W = 1024.0, 3
    sums = (rng.normal(size=n) * 30.0).astype(F32)
    m = (rng.normal(size=n) * 1e-3).astype(F32)
    v = np.abs(rng.normal(size=n) * 1e-5).astype(F32)
    p = (rng.normal(size=n) * 0.02).astype(F32)
    dsums, dm, dv, dp = (torch.from_numpy(x.copy()).cuda() for x in (sums, m, v, p))
    of = torch.zeros(1, dtype=torch.int32, device="cuda")
    zr.adamw_shard_step(dsums, dm, dv, dp, HYPER, S, W, t, of)
    torch.cuda.synchronize()
    g = (sums * oracle.unscale_factor(S, W)).astype(F32)
    oracle.adamw(g, p, m, v, OHYPER, oracle.bias_correction(0.9, t), oracle.bias_correction(0.999, t))
    assert of.item() == 0
    for dev, host in ((dp, p), (dm, m), (dv, v)):
        assert np.array_equal(f32bits(dev), host.view(np.uint32))


def test_adamw_shard_step_skips_on_flag():
    rng = np.random.default_rng(3)
    n = 1000
    sums = (rng.normal(size=n)).astype(F32)
    arrs = [(rng.normal(size=n)).astype(F32) for _ in range(3)]
    arrs[1] = np.abs(arrs[1])
    dev = [torch.from_numpy(a.copy()).cuda() for a in arrs]
    # preset flag: no update
    of = torch.ones(1, dtype=torch.int32, device="cuda")
    zr.adamw_shard_step(torch.from_numpy(sums).cuda(), dev[0], dev[1], dev[2], HYPER, 1.0, 1, 1, of)
    torch.cuda.synchronize()
    for d, a in zip(dev, arrs):
        assert np.array_equal(f32bits(d), a.view(np.uint32))
    # non-finite shard value: the flag pass sets the flag and the update is skipped
    sums[777] = np.inf
    of.zero_()
    zr.adamw_shard_step(torch.from_numpy(sums).cuda(), dev[0], dev[1], dev[2], HYPER, 1.0, 1, 1, of)
    torch.cuda.synchronize()
    assert of.item() == 1
    for d, a in zip(dev, arrs):
        assert np.array_equal(f32bits(d), a.view(np.uint32))


# ----------------------------------------------------------------------------- all-gather
@pytest.mark.parametrize("dtype", [zr.F16, zr.BF16])
@pytest.mark.parametrize("R", [1, 3, 8])
def test_all_gather_bit_exact(dtype, R):
    rng = np.random.default_rng(R)
    n = 50_007
    x = (rng.normal(size=n) * rng.choice([1e-9, 1e-6, 1e-2, 1.0, 1e4, 7e4], size=n)).astype(F32)
    x[:6] = [0.0, -0.0, np.inf, -np.inf, 65519.0, 65520.0]
    want = oracle.encode(dtype, x)
    tdt = torch.float16 if dtype == zr.F16 else torch.bfloat16
    reps = [torch.empty(n, dtype=tdt, device="cuda") for _ in range(R)]
    zr.all_gather(torch.from_numpy(x).cuda(), reps)
    torch.cuda.synchronize()
    for r in reps:
        assert np.array_equal(u16(r), want)


# ----------------------------------------------------------------------------- fused step
class FusedRun:
    """A fused-step run on the GPU with the full oracle beside it (small sizes)."""

    def __init__(self, numels, W, A, dtype, cap, S, dynamic=False, order=None, seed=0, sigma=None, stage=2,
                 interval=1000, staging=None, backoff=0.5, growth=2.0, min_scale=1.0, hyper=None):
        self.hyper, self.ohyper = hyper or (HYPER, OHYPER)
        self.plan = zr.Plan(numels, W=W, A=A, dtype=dtype, stage=stage, cap=cap, order=order,
                            scaler=zr.Scaler(S, dynamic, backoff=backoff, growth=growth, min_scale=min_scale,
                                             growth_interval=interval))
        if staging is not None:  # (staging, stage_elems, stages) for zr_plan_set_staging
            self.plan.set_staging(*staging)
        self.W, self.A, self.dtype, self.order = W, A, dtype, order
        self.obuckets, self.ooffsets = oracle_layout(self.plan, numels, cap, W)
        sig = np.full(len(numels), 1e-2, F32) if sigma is None else np.asarray(sigma, F32)
        self.layout = Layout(numels, self.ooffsets, sig, seed, dtype)
        n = self.plan.numel
        self.n = n
        self.table = torch.from_numpy(zrgen.normal_table().copy()).cuda()
        self.state = self.plan.new_state()
        self.state.master[0].zero_()
        self.layout.master_dev(self.state.master[0], self.table, torch.cuda.current_stream().cuda_stream)
        zr.all_gather(self.state.master[0], [self.state.param[0]])
        self.grads = [torch.zeros(n, dtype=self.plan.torch_dtype(), device="cuda") for _ in range(W * A)]
        om = self.layout.master_host(0, n)
        self.o = [om, np.zeros(n, F32), np.zeros(n, F32), oracle.encode(dtype, om)]
        self.osc = oracle.new_scaler(S, dynamic, backoff=backoff, growth=growth, min_scale=min_scale,
                                     interval=interval)
        self.S = S
        self.current = 0

    def step(self, step, inject=None, stage=None):
        st = torch.cuda.current_stream().cuda_stream
        S = self.S
        ograds = []
        for r in range(self.W * self.A):
            self.layout.grads_dev(self.grads[r], step, r, S, self.table, st)
            ograds.append(self.layout.grads_host(0, self.n, step, r, S))
        if inject is not None:
            r, i = inject
            bits = 0x7C00 if self.dtype == zr.F16 else 0x7F80
            self.grads[r].view(torch.int16)[i] = np.int16(np.uint16(bits).view(np.int16))
            ograds[r][i] = bits
        rep = self._launch(stage)
        orep, _ = oracle.step(self.W, self.A, self.dtype, self.obuckets, ograds, *self.o, self.ohyper, self.osc,
                              order=self.order)
        assert rep.overflow == orep.overflow and rep.skipped == orep.skipped
        assert rep.scale_used == orep.scale_used and rep.scale == orep.scale_next
        assert rep.t == orep.t_after
        self.S = rep.scale
        self.current = rep.current
        return rep, orep

    def _launch(self, stage):
        return self.plan.step(self.grads, self.state, self.hyper, stage=stage, report=True)

    def live(self):
        L = self.state.live(self.current)
        return (L["master"].cpu().numpy(), L["m"].cpu().numpy(), L["v"].cpu().numpy(), u16(L["param"]))

    def check(self, where=""):
        assert_state_close(*self.live(), *self.o, exact=True, where=where)


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_fused_tiny_config_bit_exact(staging):
    """flat n = 786,432, W = 3, fp16, one bucket, S = 1024 static, 3 steps, seed 0; the plan's own staging
    (registers, for a plan this small) and bulk-copy staging."""
    w = zrgen.workload("tiny")
    run = FusedRun(list(w.tensors), w.W, w.A, w.dtype, w.cap, w.init_scale, w.dynamic, seed=w.seed,
                   sigma=zrgen.sigma_per_tensor(w), stage=w.stage,
                   staging=None if staging is None else (staging, 0, 0))
    # a plan this small (launch-bound, L2-resident) keeps register staging by default
    assert run.plan.staging == (zr.STAGING_REGISTERS if staging is None else staging)
    assert len(run.plan.buckets) == 1 and run.plan.numel == 786_432
    for s in range(1, w.steps + 1):
        rep, orep = run.step(s)
        assert rep.overflow == 0 and rep.current == s % 2 and rep.t == s
        run.check(f"step {s}: ")


@pytest.mark.parametrize("W,A,dtype", [(2, 1, zr.F16), (3, 1, zr.BF16), (5, 1, zr.F16), (6, 1, zr.BF16),
                                       (7, 1, zr.F16), (8, 1, zr.BF16), (2, 4, zr.BF16), (4, 4, zr.F16),
                                       (8, 4, zr.BF16), (3, 3, zr.BF16), (9, 1, zr.BF16), (16, 1, zr.F16),
                                       (17, 1, zr.BF16), (24, 1, zr.F16), (33, 1, zr.BF16)])
@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_fused_ragged_buckets(W, A, dtype, staging):
    rng = np.random.default_rng(W * 100 + A)
    numels = [1000, 37, 5000, 8, 123_457, 64, 9_999, 3, 40_000]
    order = list(rng.permutation(W))
    run = FusedRun(numels, W, A, dtype, cap=20_000, S=8.0, order=order, seed=3,
                   sigma=rng.uniform(1e-3, 1e-1, size=len(numels)),
                   staging=None if staging is None else (staging, 0, 0))
    # small plans keep register staging by default
    assert run.plan.staging == (zr.STAGING_REGISTERS if staging is None else staging)
    assert len(run.plan.buckets) >= 4
    for s in range(1, 4):
        run.step(s)
        run.check(f"W={W} A={A} step {s}: ")


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_fused_skip_then_resume(staging):
    numels = [20_000, 4_000, 30_000]
    run = FusedRun(numels, 2, 1, zr.F16, cap=25_000, S=65536.0, dynamic=True, seed=5,
                   staging=None if staging is None else (staging, 0, 0))
    run.step(1)
    before = [x.copy() for x in run.live()]
    cur = run.current
    rep, orep = run.step(2, inject=(1, int(run.ooffsets[2]) + 123))
    assert rep.overflow == 1 and rep.skipped == 1 and rep.current == cur and rep.t == 1
    assert rep.scale == 32768.0 and rep.skipped_total == 1
    after = run.live()
    for a, b in zip(after, before):
        assert a.tobytes() == b.tobytes()
    for s in (3, 4):
        run.step(s)
        run.check(f"resume step {s}: ")


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_non_finite_in_an_alignment_gap_skips(staging):
    """The gaps that align tensors to 8 elements are elements of the flat buffers: a +inf left in one is summed
    and flagged like any other, on both sides, and the step is skipped."""
    numels = [1, 7, 3000]
    run = FusedRun(numels, 2, 1, zr.BF16, cap=10_000, S=1.0, seed=31,
                   staging=None if staging is None else (staging, 0, 0))
    gaps = [i for i in range(run.n) if not any(o <= i < o + k for o, k in zip(run.ooffsets, numels))]
    assert gaps
    run.step(1)
    rep, orep = run.step(2, inject=(1, gaps[0]))
    assert rep.overflow == orep.overflow == 1
    run.grads[1].view(torch.int16)[gaps[0]] = 0  # the caller clears it again
    rep, _ = run.step(3)
    assert rep.overflow == 0
    run.check()


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_fused_scale_growth(staging):
    run = FusedRun([4096, 1000], 2, 1, zr.BF16, cap=10_000, S=4.0, dynamic=True, interval=2,
                   staging=None if staging is None else (staging, 0, 0))
    scales = []
    for s in range(1, 6):
        rep, _ = run.step(s)
        scales.append(rep.scale_used)
    assert scales == [4.0, 4.0, 8.0, 8.0, 16.0]
    run.check()


def _nan16(bits, dtype):
    return (bits & 0x7FFF) > (0x7C00 if dtype == zr.F16 else 0x7F80)


@pytest.mark.parametrize("dtype", [zr.F16, zr.BF16])
@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_non_finite_state_and_zero_over_zero(dtype, staging):
    """Degenerate states: a caller's master holding NaN and +-inf, and eps = 0 with a zero gradient (0/0 in the
    update). Results are NaN exactly where the oracle's are and bit-identical everywhere else. IEEE fixes neither
    the sign nor the payload of a NaN made by arithmetic or by a conversion (x86, Arm and the GPU each make their
    own), so NaN bits are the one thing not compared: the GPU's 16-bit cast writes one quiet NaN, the oracle's
    encoder the quiet NaN of the value's sign."""
    hyper = (zr.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=0.0, weight_decay=0.01),
             oracle.AdamW(1e-3, 0.9, 0.999, 0.0, 0.01))
    run = FusedRun([3000, 77, 5000], 2, 1, dtype, cap=6000, S=1.0, seed=29, hyper=hyper,
                   staging=None if staging is None else (staging, 0, 0))
    planted = {11: np.nan, 12: -np.nan, 13: np.inf, 14: -np.inf, 4000: np.nan}
    for i, x in planted.items():
        run.state.master[0][i] = float(x)
        run.o[0][i] = np.float32(x)
    zero_at = [100, 101, 5003]
    for s in (1, 2):
        st = torch.cuda.current_stream().cuda_stream
        for r in range(2):
            run.layout.grads_dev(run.grads[r], s, r, run.S, run.table, st)
        ograds = [run.layout.grads_host(0, run.n, s, r, run.S) for r in range(2)]
        for r in range(2):
            for i in zero_at:  # every worker's gradient exactly zero here: 0/0 once m and v are zero
                run.grads[r][i] = 0.0
                ograds[r][i] = 0
        rep = run._launch(None)
        orep, _ = oracle.step(2, 1, dtype, run.obuckets, ograds, *run.o, run.ohyper, run.osc)
        assert rep.overflow == orep.overflow == 0 and rep.t == orep.t_after
        run.current = rep.current
    gm, gmm, gv, gp = run.live()
    om, omm, ov, op = run.o
    for name, g, o in (("master", gm, om), ("m", gmm, omm), ("v", gv, ov)):
        gn, on = np.isnan(g), np.isnan(o)
        assert np.array_equal(gn, on), name
        assert np.array_equal(g[~gn].view(np.uint32), o[~on].view(np.uint32)), name
    # NaN at least where planted and where the gradient is zero (alignment padding, also zero, joins them)
    assert {11, 12, 4000, *zero_at} <= set(np.flatnonzero(np.isnan(gm)).tolist())
    assert np.isposinf(gm[13]) and np.isneginf(gm[14])
    gnan, onan = _nan16(gp, dtype), _nan16(op, dtype)
    assert np.array_equal(gnan, onan) and np.array_equal(gp[~gnan], op[~onan])


@pytest.mark.parametrize("S,dtype", [(2.0 ** 126, zr.BF16), (2.0 ** -20, zr.F16)])
@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_extreme_loss_scales(S, dtype, staging):
    """S = 2^126 at W = 3: r = fp32(1/(S*W)) is a subnormal fp32 factor (bf16 gradients near 1e36 still finite);
    S = 2^-20 in fp16: the scaled gradients fall into fp16's subnormal range. Both bit for bit the oracle's."""
    run = FusedRun([6000, 333, 9000], 3, 1, dtype, cap=10_000, S=S, seed=23,
                   staging=None if staging is None else (staging, 0, 0))
    for s in (1, 2):
        rep, _ = run.step(s)
        assert rep.overflow == 0
    run.check(f"S = {S}: ")


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_scaler_floor_and_custom_rule(staging):
    """A rule other than the default (backoff 0.25, growth 3, floor 2, interval 2): two skips in a row take the
    scale 8 -> 2 -> 2 (floored, not 0.5), two clean steps then grow it to 6; state bit for bit the oracle's."""
    run = FusedRun([4096, 1000], 2, 1, zr.F16, cap=10_000, S=8.0, dynamic=True, interval=2, backoff=0.25,
                   growth=3.0, min_scale=2.0, seed=21, staging=None if staging is None else (staging, 0, 0))
    want = [(8.0, 2.0, 1), (2.0, 2.0, 1), (2.0, 2.0, 0), (2.0, 6.0, 0), (6.0, 6.0, 0)]
    for s, (used, nxt, skipped) in enumerate(want, start=1):
        rep, _ = run.step(s, inject=(0, 17) if skipped else None)
        assert (rep.scale_used, rep.scale, rep.overflow) == (used, nxt, skipped), s
    assert rep.t == 3 and rep.skipped_total == 2
    run.check("after the floor: ")


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_default_growth_interval_over_a_thousand_steps(staging):
    """The default rule (growth after 1000 clean steps) run to its first growth: the scale doubles on step
    1001 exactly, a skip at step 1003 halves it and resets the count, and the state after 1005 steps is the
    oracle's, bit for bit (register staging, the plan's own for this size, and bulk-copy staging)."""
    run = FusedRun([2048, 1000], 2, 1, zr.F16, cap=4096, S=1024.0, dynamic=True, seed=13, interval=1000,
                   staging=None if staging is None else (staging, 0, 0))
    for s in range(1, 1006):
        rep, _ = run.step(s, inject=(1, 5) if s == 1003 else None)
        if s <= 1000:
            assert rep.scale_used == 1024.0
        if s == 1000:
            assert rep.scale == 2048.0 and rep.good == 0
        if s in (1001, 1002, 1003):
            assert rep.scale_used == 2048.0
        if s == 1003:
            assert rep.overflow == 1 and rep.scale == 1024.0 and rep.good == 0
    assert rep.t == 1004 and rep.steps == 1005 and rep.skipped_total == 1
    run.check("after 1005 steps: ")


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_stages_identical(staging):
    """DDP (stage 0) and ZeRO stages 1-3 give the same bytes."""
    outs = []
    for stage in (0, 1, 2, 3):
        run = FusedRun([70_000, 5000], 4, 1, zr.BF16, cap=50_000, S=1.0, seed=11, stage=stage,
                       staging=None if staging is None else (staging, 0, 0))
        for s in (1, 2):
            rep, _ = run.step(s, stage=stage)
            assert rep.stage == stage
        outs.append([x.tobytes() for x in run.live()])
    assert outs[0] == outs[1] == outs[2] == outs[3]


@pytest.mark.parametrize("pinned", [True, False])
def test_step_from_host_equals_step(pinned):
    """Pinned host gradients are read in place by the kernel; pageable ones are copied first."""
    numels = [50_000, 777, 12_345]
    a = FusedRun(numels, 3, 1, zr.F16, cap=40_000, S=1024.0, seed=2)
    b = FusedRun(numels, 3, 1, zr.F16, cap=40_000, S=1024.0, seed=2)
    for s in (1, 2):
        a.step(s)
        host = []
        for r in range(3):
            g = b.layout.grads_host(0, b.n, s, r, b.S)
            host.append(torch.from_numpy(g.view(np.int16).copy()).pin_memory() if pinned else g.copy())
        for d in b.grads:
            d.fill_(0)
        rep = b.plan.step_from_host(host, b.grads, b.state, HYPER)
        assert rep.t == s and rep.overflow == 0
        b.current = rep.current
        for x, y in zip(a.live(), b.live()):
            assert x.tobytes() == y.tobytes()
        # the copy path fills the device buffers; the in-place path leaves them alone
        assert (int(b.grads[0].view(torch.int16).abs().sum().item()) == 0) == pinned


def test_error_paths():
    plan = zr.Plan([1024], W=2, A=1, dtype=zr.BF16, stage=2, cap=2048)
    st = plan.new_state()
    grads = [torch.zeros(plan.numel, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(zr.ZrError) as e:
        plan.step(grads, st, HYPER, stage=4)
    assert e.value.status == 1
    with pytest.raises(zr.ZrError):
        plan.step(grads, st, HYPER, stage=-1)
    with pytest.raises(zr.ZrError):
        plan.step([grads[0], grads[1][1:]], st, HYPER)  # 2-byte offset: misaligned
    st.master[1] = st.master[0]
    with pytest.raises(zr.ZrError):
        plan.step(grads, st, HYPER)
    with pytest.raises(zr.ZrError):
        zr.Plan([8], W=65, A=1)
    with pytest.raises(zr.ZrError):
        zr.Plan([8], W=8, A=33)
    with pytest.raises(zr.ZrError):
        zr.reduce_scatter(grads, torch.empty(1024, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"),
                          order=[0, 0])
    # nothing above launched: the library still works
    plan.reset()
    st2 = plan.new_state()
    st2.master[0].zero_()
    r = plan.step(grads, st2, HYPER, report=True)
    assert r.t == 1 and r.overflow == 0


@pytest.mark.parametrize("staging", [None, zr.STAGING_BULK])
def test_checkpoint_resume_is_byte_identical(staging):
    """Run 4 steps straight; separately run 2, checkpoint (control block + live state), restore into a fresh
    plan and state, run steps 3-4: the live state matches byte for byte, with a skip in between."""
    numels = [30_000, 5_000, 17_000]
    stg = None if staging is None else (staging, 0, 0)
    straight = FusedRun(numels, 2, 1, zr.F16, cap=25_000, S=65536.0, dynamic=True, seed=9, interval=2,
                        staging=stg)
    inj = (0, int(straight.ooffsets[1]) + 7)
    for s in range(1, 5):
        straight.step(s, inject=inj if s == 2 else None)
    first = FusedRun(numels, 2, 1, zr.F16, cap=25_000, S=65536.0, dynamic=True, seed=9, interval=2, staging=stg)
    for s in (1, 2):
        first.step(s, inject=inj if s == 2 else None)
    ck = first.plan.checkpoint()
    saved = {k: v.clone() for k, v in first.state.live(ck.current).items()}
    assert ck.t == 1 and ck.skipped == 1 and ck.scale == 32768.0
    second = FusedRun(numels, 2, 1, zr.F16, cap=25_000, S=65536.0, dynamic=True, seed=9, interval=2, staging=stg)
    second.plan.restore(ck)
    live = second.state.live(ck.current)
    for k in saved:
        live[k].copy_(saved[k])
    second.o = [x.copy() for x in first.o]   # the oracle continues from the same point
    second.osc = oracle.Scaler.from_buffer_copy(first.osc)
    second.S = ck.scale
    second.current = ck.current
    for s in (3, 4):
        second.step(s)
    for a, b in zip(straight.live(), second.live()):
        assert a.tobytes() == b.tobytes()
    second.check("resumed: ")
    for bad in (zr.Checkpoint(2, 1.0, 0, 0, 0, 0, 1.0, 1.0), zr.Checkpoint(0, 0.0, 0, 0, 0, 0, 1.0, 1.0),
                zr.Checkpoint(0, 1.0, -1, 0, 0, 0, 1.0, 1.0), zr.Checkpoint(0, 1.0, 0, 0, 0, 0, 1.5, 1.0),
                zr.Checkpoint(0, 1.0, 0, 0, 0, 0, 0.5, float("nan")), zr.Checkpoint(0, 1.0, 0, 0, 0, 0, -0.1, 0.9)):
        with pytest.raises(zr.ZrError):
            second.plan.restore(bad)


@pytest.mark.parametrize("call", ["step", "step_inplace", "step_from_host"])
def test_plan_without_parameters_steps_clean(call):
    """Every tensor empty (the degenerate model): the reduce-scatter sums nothing, so each step is clean, as the
    oracle's step over no buckets is: t and the good-step count advance and the scale grows on the interval
    (the live set flips on the ping-pong paths). Zero-size tensors have null data pointers, which are accepted."""
    numels = [0, 0, 0]
    W = 2
    plan = zr.Plan(numels, W=W, dtype=zr.F16, stage=1, cap=100,
                   scaler=zr.Scaler(1024.0, dynamic=True, growth_interval=2))
    ob, _ = oracle.bucket_plan(numels, 100, W)
    assert plan.numel == 0 and len(plan.buckets) == 0 and ob.shape[0] == 0
    osc = oracle.new_scaler(1024.0, dynamic=True, interval=2)
    z, zu = np.zeros(0, np.float32), np.zeros(0, np.uint16)
    grads = [torch.empty(0, dtype=torch.float16, device="cuda") for _ in range(W)]
    st = plan.new_state1() if call == "step_inplace" else plan.new_state()
    host = [torch.empty(0, dtype=torch.float16) for _ in range(W)]
    for step in (1, 2, 3):
        if call == "step":
            rep = plan.step(grads, st, HYPER, report=True)
        elif call == "step_inplace":
            rep = plan.step_inplace(grads, st, HYPER, report=True)
        else:
            rep = plan.step_from_host(host, grads, st, HYPER)
        orep, _ = oracle.step(W, 1, zr.F16, ob, [zu, zu], z, z.copy(), z.copy(), zu.copy(), OHYPER, osc)
        assert rep.overflow == orep.overflow == 0
        assert (rep.t, rep.good, rep.scale, rep.steps) == (osc.t, osc.good, osc.scale, step)
        assert rep.current == (0 if call == "step_inplace" else step % 2)
    plan.close()


# ----------------------------------------------------------------------------- bulk-copy staging
@pytest.mark.parametrize("W,A,dtype,shape", [(1, 1, zr.BF16, (0, 0)), (2, 1, zr.F16, (0, 0)),
                                             (2, 1, zr.BF16, (256, 2)), (3, 1, zr.F16, (0, 0)),
                                             (5, 1, zr.BF16, (1024, 4)), (8, 1, zr.BF16, (0, 0)),
                                             (8, 1, zr.F16, (4096, 1)), (16, 1, zr.F16, (0, 0)),
                                             (64, 1, zr.BF16, (0, 0)), (2, 4, zr.BF16, (0, 0)), (4, 4, zr.F16, (0, 0)),
                                             (8, 4, zr.BF16, (0, 0)), (3, 3, zr.BF16, (512, 3)),
                                             (32, 8, zr.F16, (0, 0))])
@pytest.mark.parametrize("mode", [zr.STAGING_BULK, zr.STAGING_BULK_IO])
def test_bulk_staging_bit_exact(W, A, dtype, shape, mode):
    """zr_step with its loads (and with BULK_IO its results too) staged in shared memory by bulk copies gives
    the oracle's bytes: ragged buckets, a ring order, micro-batch accumulation (A > 1, up to W*A = 256 replica
    slices per stage), automatic and explicit stage shapes (down to stages of 256 elements and a single
    stage)."""
    rng = np.random.default_rng(W * 31 + A * 7 + dtype)
    numels = [1000, 37, 5000, 8, 123_457, 64, 9_999, 3, 40_000]
    order = [int(x) for x in rng.permutation(W)]
    run = FusedRun(numels, W, A, dtype, cap=20_000, S=8.0, order=order, seed=21,
                   sigma=rng.uniform(1e-3, 1e-1, size=len(numels)), staging=(mode,) + shape)
    assert run.plan.staging == mode
    for s in range(1, 4):
        run.step(s)
        run.check(f"bulk W={W} A={A} shape={shape} step {s}: ")


@pytest.mark.parametrize("mode", [zr.STAGING_BULK, zr.STAGING_BULK_IO])
def test_bulk_staging_skip_and_scale(mode):
    """A +inf in one bucket skips the whole bulk-staged step and halves the dynamic scale, like the register
    path; switching back to register staging between steps continues the same run."""
    numels = [30_000, 4_000, 70_000]
    run = FusedRun(numels, 2, 1, zr.F16, cap=25_000, S=65536.0, dynamic=True, seed=5, staging=(mode, 0, 0))
    rep, orep = run.step(1)
    assert rep.overflow == 0
    before = [x.copy() for x in run.live()]
    rep, orep = run.step(2, inject=(1, int(run.ooffsets[2]) + 123))
    assert rep.overflow == 1 and rep.scale == 32768.0 and rep.t == 1
    assert all(np.array_equal(a, b) for a, b in zip(before, run.live()))
    run.check("after skip: ")
    run.plan.set_staging(zr.STAGING_REGISTERS)
    run.step(3)
    run.check("register staging after bulk: ")
    run.plan.set_staging(mode)
    run.step(4)
    run.check("bulk staging again: ")


@pytest.mark.parametrize("mode", [zr.STAGING_BULK, zr.STAGING_BULK_IO])
def test_bulk_staging_large_plan_one_block_per_tile(mode):
    """A plan with more than four waves of 32K-element tiles: the bulk-staged step launches one block per
    tile (the launch shape the benchmark times)."""
    w = zrgen.workload("gpt2")
    run = FusedRun(list(w.tensors)[:25], 8, 1, zr.BF16, cap=w.cap, S=1.0, seed=w.seed, staging=(mode, 0, 0))
    assert run.plan.numel > 4 * 152 * 2 * 32768
    for s in (1, 2):
        run.step(s)
        run.check(f"large bulk step {s}: ")


@pytest.mark.parametrize("mode,W", [(zr.STAGING_BULK, 2), (zr.STAGING_BULK_IO, 2), (zr.STAGING_BULK, 16)])
def test_bulk_wait_timeout_reports_and_recovers(mode, W):
    """The bounded waits of bulk staging: with the test hook on, no stage's copies complete its barrier, so every
    wait runs out after its limit (2 s), the step is skipped with the live set unchanged, zr_plan_report returns
    ZR_ERR_TIMEOUT and the CUDA context stays usable; restoring the step state clears the error and the run
    continues, bit-exact against the oracle."""
    import time
    # W = 16 under ZR_STAGING_BULK runs the chunked kernel (stages of 8 replica slices)
    run = FusedRun([40_000, 3_000], W, 1, zr.F16, cap=50_000, S=1024.0, seed=31, staging=(mode, 0, 0))
    run.step(1)
    run.check("before the stalled step: ")
    ck = run.plan.checkpoint()
    before = [x.copy() for x in run.live()]
    cs = torch.cuda.current_stream().cuda_stream
    for r in range(W):
        run.layout.grads_dev(run.grads[r], 2, r, run.S, run.table, cs)
    assert zr.lib().zr_plan_stall_bulk_waits(run.plan._h, 1) == 0
    t0 = time.perf_counter()
    run.plan.step(run.grads, run.state, HYPER)  # no report: the call itself does not wait
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert zr.lib().zr_plan_stall_bulk_waits(run.plan._h, 0) == 0
    assert 1.5 < elapsed < 60.0, elapsed
    with pytest.raises(zr.ZrError) as err:
        run.plan.report()
    assert err.value.status == 5 and "gave up" in str(err.value)
    assert all(np.array_equal(a, b) for a, b in zip(before, run.live()))
    x = torch.arange(1024, device="cuda", dtype=torch.float32)  # the context still works
    assert float(x.sum()) == 1024 * 1023 / 2
    run.plan.restore(ck)  # a fresh control block with the step state before the stalled step
    run.step(2)
    run.check("after recovery: ")


def test_bulk_staging_rejects_unsupported():
    plan = zr.Plan([4096], W=2, A=1, dtype=zr.BF16, stage=2, cap=8192, fp32_grads=True)
    with pytest.raises(zr.ZrError):  # bulk staging needs 16-bit gradients
        plan.set_staging(zr.STAGING_BULK)
    plan.close()
    plan = zr.Plan([4096], W=2, A=1, dtype=zr.BF16, stage=2, cap=8192)
    for bad in ((3, 0, 0), (-1, 0, 0), (zr.STAGING_BULK, 12, 0), (zr.STAGING_BULK, 0, 5)):
        with pytest.raises(zr.ZrError):
            plan.set_staging(*bad)
    with pytest.raises(zr.ZrError):  # 4 stages of 65536 elements do not fit an SM
        plan.set_staging(zr.STAGING_BULK, 65536, 4)
    plan.close()
    plan = zr.Plan([4096], W=16, A=1, dtype=zr.BF16, stage=2, cap=8192)
    with pytest.raises(zr.ZrError):  # more than 8 replica slices: stages of 8 slices, at most 2048 elements
        plan.set_staging(zr.STAGING_BULK, 4096, 1)
    plan.set_staging(zr.STAGING_BULK, 2048, 1)
    plan.set_staging(zr.STAGING_BULK_IO, 4096, 1)  # the load + store variant keeps one stage for all slices
    plan.close()
    # a refused call leaves no CUDA error behind for the caller's next check
    x = torch.empty(1024, device="cuda")
    x.fill_(1.0)
    torch.cuda.synchronize()
    assert float(x.sum()) == 1024.0
