"""zr_step_noalloc, the fused step for callers that cannot allocate device memory.

Who needs it: a caller whose runtime hands out every byte of device memory from its own pool and
forbids allocations behind its back, a job whose memory budget was fixed before its first step, or a
path on which a cudaMalloc would synchronise the device. None of them can create a plan, because
zr_plan_create allocates a tile table and a control block. zr_step_noalloc keeps that scratch in a
static device array of the library instead; the caller passes every input and output and carries the
live set, the loss scale and t from call to call.

Every test here calls the entry point through the C ABI (ctypes on libzr.so) and checks each call bit
for bit against the oracle, which runs the ring hop by hop on the host, from the oracle's own bucket
table (the large plan against zr_step, itself bit-exact against the oracle in the other test files). The
cases cover both specialised kernel widths the workloads use (fp16 W = 2, bf16 W = 8), a width without
its own instantiation (W = 6), micro-batch accumulation (A = 2), a plan small enough that the call
halves its tile size, a layout of more than 64 buckets (several set-up launches), a skipped step, t far
beyond any training run, the empty plan, a plan large enough for bulk-copy staging (against zr_step),
and a warm call that must not change the device's free memory. The file's name sorts last, so a run that
stops at the first failure has run every other test before it; it also passes alone in a fresh process
(it builds the library and makes its own inputs).
"""
import ctypes
import os
import sys
import time

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

pytestmark = pytest.mark.gpu
F32 = np.float32


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    import zero_gradient_reduction_gb300 as zr
    import zrgen
    torch.cuda.set_device(0)
    fn = zr.lib().zr_step_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.POINTER(zr.StateC), ctypes.c_int, ctypes.POINTER(zr.Hyper),
                   ctypes.c_float, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    return dict(oracle=oracle, zr=zr, zrgen=zrgen, fn=fn,
                table=torch.from_numpy(zrgen.normal_table().copy()).cuda())


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.int32).numpy().view(np.uint32) if t.dtype == torch.float32 else \
        t.view(torch.int16).numpy().view(np.uint16)


def _running_product(beta: float, n: int) -> float:
    """beta^n as n double multiplications from 1.0, stopping once the product no longer changes."""
    p = 1.0
    b = float(np.float32(beta))
    for _ in range(n):
        q = p * b
        if q == p:
            break
        p = q
    return p


class Run:
    """One no-allocation run beside the oracle: state tensors made by the test, the bucket table from the
    oracle's builder, the live set, the scale and t carried here as a caller would carry them."""

    def __init__(self, env, numels, W, A, dtype, cap, S=1.0, order=None, seed=0):
        oracle, zr, zrgen = env["oracle"], env["zr"], env["zrgen"]
        from zrgen.layout import Layout
        self.env, self.W, self.A, self.dtype, self.S, self.order = env, W, A, dtype, float(S), order
        self.buckets, offsets = oracle.bucket_plan(list(numels), cap, W)
        self.n = int(max((s + ln for s, ln, _ in self.buckets), default=0))
        n = max(self.n, 8)
        self.tdt = torch.float16 if dtype == zr.F16 else torch.bfloat16
        self.layout = Layout(numels, offsets, np.full(len(numels), 1e-2, F32), seed, dtype)
        cs = torch.cuda.current_stream().cuda_stream
        self.state = zr.State(n, self.tdt)
        self.state.master[0].zero_()
        self.layout.master_dev(self.state.master[0], env["table"], cs)
        zr.all_gather(self.state.master[0], [self.state.param[0]])
        om = self.layout.master_host(0, n)
        self.o = [om, np.zeros(n, F32), np.zeros(n, F32), oracle.encode(dtype, om)]
        self.osc = oracle.new_scaler(S)
        self.ohyper = oracle.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)
        self.hyper = zr.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)
        self.grads = [torch.zeros(n, dtype=self.tdt, device="cuda") for _ in range(W * A)]
        self.btab = (zr.Bucket * max(len(self.buckets), 1))(
            *[zr.Bucket(int(s), int(ln), int(c)) for s, ln, c in self.buckets])
        self.ordc = (ctypes.c_int * W)(*order) if order is not None else None
        self.overflow = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        self.current = 0
        self.t = 0  # clean steps so far

    def fill(self, step, inject=None):
        """Step `step`'s gradients on the device and, for the oracle, on the host; inject = (replica, index)
        of a +inf."""
        cs = torch.cuda.current_stream().cuda_stream
        og = []
        for r in range(self.W * self.A):
            self.layout.grads_dev(self.grads[r], step, r, self.S, self.env["table"], cs)
            og.append(self.layout.grads_host(0, max(self.n, 8), step, r, self.S))
        if inject is not None:
            r, i = inject
            bits = 0x7C00 if self.dtype == self.env["zr"].F16 else 0x7F80
            self.grads[r].view(torch.int16)[i] = int(np.uint16(bits).view(np.int16))
            og[r][i] = bits
        return og

    def call(self, t=None):
        zr = self.env["zr"]
        gptr = (ctypes.c_void_p * (self.W * self.A))(*[g.data_ptr() for g in self.grads])
        stc = self.state.c()
        h = self.hyper.c()
        rc = self.env["fn"](ctypes.addressof(self.btab), len(self.buckets), self.W, self.A, self.dtype,
                            ctypes.addressof(self.ordc) if self.ordc is not None else None, ctypes.addressof(gptr),
                            ctypes.byref(stc), self.current, ctypes.byref(h), self.S,
                            self.t + 1 if t is None else t, self.overflow.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
        assert rc == 0, zr.lib().zr_last_error()

    def step(self, step, inject=None, t=None):
        """One call beside one oracle step; checks the flag and the live set bit for bit."""
        og = self.fill(step, inject)
        before = [_bits(x) for x in self.state.live(self.current).values()]
        self.call(t)
        torch.cuda.synchronize()
        flag = int(self.overflow.item())
        orep, _ = self.env["oracle"].step(self.W, self.A, self.dtype, self.buckets, og, *self.o, self.ohyper,
                                          self.osc, order=self.order)
        assert flag == orep.overflow, f"step {step}: overflow {flag}, oracle {orep.overflow}"
        if flag:
            # skipped: the caller keeps its live set, which the call has not touched
            after = [_bits(x) for x in self.state.live(self.current).values()]
            assert all(np.array_equal(a, b) for a, b in zip(before, after)), "a skipped step changed the live set"
        else:
            self.current = 1 - self.current
            self.t += 1
        self.check(f"step {step}: ")
        return flag

    def check(self, where=""):
        live = self.state.live(self.current)
        n = self.n
        for name, o in zip(("master", "m", "v"), self.o[:3]):
            assert np.array_equal(_bits(live[name])[:n], o[:n].view(np.uint32)), f"{where}{name} not bit-exact"
        assert np.array_equal(_bits(live["param"])[:n], self.o[3][:n]), f"{where}param not bit-exact"


def test_noalloc_bit_exact_with_skip_and_zr_step(env):
    """bf16, W = 4, A = 2, a ring order: three calls in a row (clean, skipped on an injected +inf, clean),
    each bit for bit against the oracle and against zr_step on a plan over the same inputs."""
    zr = env["zr"]
    numels = [50_000, 777, 123_457, 9_000, 64]
    run = Run(env, numels, 4, 2, zr.BF16, 60_000, order=[2, 0, 3, 1], seed=7)
    assert len(run.buckets) >= 3
    plan = zr.Plan(numels, W=4, A=2, dtype=zr.BF16, stage=2, cap=60_000, order=[2, 0, 3, 1])
    assert np.array_equal(plan.buckets, run.buckets)
    ref = plan.new_state()
    ref.master[0].copy_(run.state.master[0])
    ref.param[0].copy_(run.state.param[0])
    inj = (5, int(run.layout.offsets[2]) + 4321)
    for step, inject in ((1, None), (2, inj), (3, None)):
        flag = run.step(step, inject)
        rep = plan.step(run.grads, ref, run.hyper, report=True)
        assert rep.overflow == flag and rep.current == run.current and rep.t == run.t
        for name in ("master", "m", "v", "param"):
            assert torch.equal(ref.live(rep.current)[name].view(torch.int8),
                               run.state.live(run.current)[name].view(torch.int8)), f"step {step}: {name}"
    assert run.t == 2
    plan.close()


@pytest.mark.parametrize("case", ["f16_w2", "bf16_w8", "f16_w3_small", "bf16_w6_70_buckets"])
def test_noalloc_kernel_paths(env, case):
    """The kernel instantiations a no-allocation caller reaches: fp16 W = 2 (two groups per thread) and
    bf16 W = 8 (the specialised widths of the 7B and 1.3B workloads), W = 3 on a plan so small that the
    call halves its tile size, and W = 6 over 70 one-tensor buckets (more than one set-up launch)."""
    zr = env["zr"]
    rng = np.random.default_rng(11)
    if case == "f16_w2":
        run = Run(env, [300_000, 12_345, 50_001], 2, 1, zr.F16, 200_000, S=1024.0, order=[1, 0], seed=3)
    elif case == "bf16_w8":
        run = Run(env, [200_000, 3_000, 77_777, 8], 8, 1, zr.BF16, 150_000,
                  order=[int(x) for x in rng.permutation(8)], seed=4)
    elif case == "f16_w3_small":
        run = Run(env, [4_000, 1_000, 2_048], 3, 1, zr.F16, 5_000, S=1024.0, seed=5)
    else:
        numels = [int(x) for x in rng.integers(8, 3_000, size=70)]
        # a cap of one parameter: every tensor gets a bucket of its own
        run = Run(env, numels, 6, 1, zr.BF16, 1, order=[int(x) for x in rng.permutation(6)], seed=6)
        assert len(run.buckets) == 70
    site = int(run.layout.offsets[len(run.layout.offsets) // 2])
    assert run.step(1) == 0
    assert run.step(2, inject=(run.W * run.A - 1, site)) == 1
    assert run.step(3) == 0
    assert run.t == 2


def test_noalloc_large_t(env):
    """t = 10^6 and 10^6 + 1 (a resumed run), then t = 10^12: the bias corrections come from the running
    products of the betas, which settle long before such t; each call returns promptly and matches the
    oracle given the same products."""
    zr = env["zr"]
    run = Run(env, [40_000, 999], 2, 1, zr.F16, 50_000, S=1024.0, seed=8)
    for step, t in ((1, 10 ** 6), (2, 10 ** 6 + 1), (3, 10 ** 12)):
        run.osc.t = t - 1
        run.osc.prod1 = _running_product(0.9, t - 1)
        run.osc.prod2 = _running_product(0.999, t - 1)
        t0 = time.perf_counter()
        run.step(step, t=t)
        assert time.perf_counter() - t0 < 30.0


def test_noalloc_large_t_matches_restored_plan(env):
    """At t = 10^6 the call gives the bytes zr_step gives after zr_plan_restore to the same step state."""
    zr = env["zr"]
    numels = [40_000, 999]
    run = Run(env, numels, 2, 1, zr.F16, 50_000, S=1024.0, seed=9)
    plan = zr.Plan(numels, W=2, A=1, dtype=zr.F16, stage=1, cap=50_000, scaler=zr.Scaler(1024.0))
    ref = plan.new_state()
    ref.master[0].copy_(run.state.master[0])
    ref.param[0].copy_(run.state.param[0])
    t = 10 ** 6
    ck = plan.checkpoint()
    ck.t = t - 1
    ck.beta1_pow = _running_product(0.9, t - 1)
    ck.beta2_pow = _running_product(0.999, t - 1)
    plan.restore(ck)
    run.fill(1)
    run.call(t=t)
    rep = plan.step(run.grads, ref, run.hyper, report=True)
    torch.cuda.synchronize()
    assert int(run.overflow.item()) == 0 and rep.overflow == 0 and rep.t == t
    for name in ("master", "m", "v", "param"):
        assert torch.equal(ref.live(rep.current)[name].view(torch.int8),
                           run.state.live(1)[name].view(torch.int8)), name
    plan.close()


def test_noalloc_large_plan_matches_bulk_staged_zr_step(env):
    """A plan large enough to stream from HBM (about 48M params, more than four waves of tiles): the call stages its
    loads with bulk copies as zr_step does for such a plan, and two calls in a row give zr_step's bytes exactly."""
    zr = env["zr"]
    numels = [24_000_000, 3_000, 24_000_000]
    run = Run(env, numels, 2, 1, zr.F16, 30_000_000, S=1024.0, seed=12)
    plan = zr.Plan(numels, W=2, A=1, dtype=zr.F16, stage=1, cap=30_000_000, scaler=zr.Scaler(1024.0))
    assert np.array_equal(plan.buckets, run.buckets) and plan.staging == zr.STAGING_BULK
    ref = plan.new_state()
    ref.master[0].copy_(run.state.master[0])
    ref.param[0].copy_(run.state.param[0])
    for step in (1, 2):
        run.fill(step)
        run.call()
        rep = plan.step(run.grads, ref, run.hyper, report=True)
        torch.cuda.synchronize()
        assert int(run.overflow.item()) == 0 and rep.overflow == 0
        run.current, run.t = 1 - run.current, run.t + 1
        for name in ("master", "m", "v", "param"):
            assert torch.equal(ref.live(rep.current)[name].view(torch.int8),
                               run.state.live(run.current)[name].view(torch.int8)), f"step {step}: {name}"
    plan.close()


def test_noalloc_empty_and_warm_call_allocates_nothing(env):
    """An empty bucket table is a clean step (the flag reads 0, not a stale value); a warm call changes
    neither the device's free memory nor torch's allocation count; sizes beyond the static scratch are
    refused with a clear error."""
    zr = env["zr"]
    empty = Run(env, [], 2, 1, zr.BF16, 1_000)
    assert len(empty.buckets) == 0
    empty.call(t=1)
    torch.cuda.synchronize()
    assert int(empty.overflow.item()) == 0
    # with nothing to reduce the arrays may be zero-size tensors, whose data pointers are null
    of = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    zr.step_noalloc(np.zeros((0, 3), np.int64), 2, 1, zr.BF16, [torch.empty(0, dtype=torch.bfloat16, device="cuda")] * 2,
                    zr.State(0, torch.bfloat16), 0, zr.AdamW(), 1.0, 1, of)
    torch.cuda.synchronize()
    assert int(of.item()) == 0

    run = Run(env, [100_000, 5_000], 4, 1, zr.BF16, 60_000, seed=10)
    run.step(1)  # first call on this device in a fresh process resolves the scratch address
    run.fill(2)
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    run.call()
    torch.cuda.synchronize()
    free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    assert free1 == free0 and alloc1 == alloc0, (free0, free1, alloc0, alloc1)
    assert int(run.overflow.item()) == 0

    n = 8 * 8192 * 70_000  # needs more tiles than the static scratch holds
    huge = (zr.Bucket * 1)(zr.Bucket(0, n, zr.chunk_size(n, 8)))
    gptr = (ctypes.c_void_p * 8)(*[run.grads[0].data_ptr()] * 8)
    stc = run.state.c()
    h = run.hyper.c()
    rc = env["fn"](ctypes.addressof(huge), 1, 8, 1, zr.BF16, None, ctypes.addressof(gptr), ctypes.byref(stc), 0,
                   ctypes.byref(h), 1.0, 3, run.overflow.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 1 and b"static scratch limit" in zr.lib().zr_last_error()
