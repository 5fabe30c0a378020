"""ZeRO-Offload step: reduce-scatter on the GPU, AdamW on the host CPU over host-resident
master/m/v, parameters back to the device. Checked against the oracle bit for bit, including a skip."""
import numpy as np
import pytest
import torch

import oracle
import zero_gradient_reduction_gb300 as zr
import zrgen
from zrgen.layout import Layout
from _harness import oracle_layout
from test_parity_gpu import OHYPER, u16

pytestmark = pytest.mark.gpu
F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _pinned(n, np_dtype, tdt, kind, keep):
    """A page-locked host buffer: from cudaHostAlloc (torch's pin_memory), or pageable numpy memory registered
    with cudaHostRegister (kept in `keep` for unregistering)."""
    if kind == "alloc":
        return torch.empty(n, dtype=tdt, pin_memory=True)
    a = np.zeros(n, np_dtype)
    assert int(torch.cuda.cudart().cudaHostRegister(a.ctypes.data, a.nbytes, 0)) == 0
    keep.append(a)
    return torch.from_numpy(a).view(tdt)


@pytest.mark.parametrize("W,dtype,kind", [(2, zr.F16, "alloc"), (4, zr.BF16, "alloc"), (2, zr.BF16, "registered")])
def test_offload_step_matches_oracle(W, dtype, kind):
    numels = [300_000, 999, 120_000, 64]
    S = 1024.0 if dtype == zr.F16 else 1.0
    plan = zr.Plan(numels, W=W, dtype=dtype, stage=2, cap=200_000, order=list(range(W))[::-1])
    n = plan.numel
    ob, ooff = oracle_layout(plan, numels, 200_000, W)
    lay = Layout(numels, ooff, np.full(len(numels), 1e-2, F32), 6, dtype)
    table = torch.from_numpy(zrgen.normal_table().copy()).cuda()
    cs = torch.cuda.current_stream().cuda_stream
    tdt = plan.torch_dtype()
    grads = [torch.zeros(n, dtype=tdt, device="cuda") for _ in range(W)]
    sums_dev = torch.empty(n, dtype=torch.float32, device="cuda")
    keep = []
    sums_host = _pinned(n, F32, torch.float32, kind, keep)
    master = lay.master_host(0, n)
    m, v = np.zeros(n, F32), np.zeros(n, F32)
    param_host = _pinned(n, np.uint16, tdt, kind, keep)
    param_dev = torch.zeros(n, dtype=tdt, device="cuda")
    o = [master.copy(), m.copy(), v.copy(), np.zeros(n, np.uint16)]
    osc = oracle.new_scaler(S, dynamic=True)
    t = 0
    for step in (1, 2, 3):
        for r in range(W):
            lay.grads_dev(grads[r], step, r, S, table, cs)
        og = [lay.grads_host(0, n, step, r, S) for r in range(W)]
        if step == 2:  # a non-finite gradient: the whole step is skipped
            grads[1].view(torch.int16)[7] = 0x7C00 if dtype == zr.F16 else 0x7F80
            og[1][7] = 0x7C00 if dtype == zr.F16 else 0x7F80
        before = master.tobytes()
        of = plan.offload_step(grads, sums_dev, sums_host, master, m, v, param_host, param_dev, zr.AdamW(), S,
                               t + 1, nthreads=8)
        torch.cuda.synchronize()
        rep, _ = oracle.step(W, 1, dtype, ob, og, *o, OHYPER, osc, order=list(range(W))[::-1])
        assert of == rep.overflow == (1 if step == 2 else 0)
        if of:
            assert master.tobytes() == before
            S = osc.scale
            continue
        t += 1
        for a, b in zip((master, m, v), o[:3]):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(u16(param_dev), o[3])
    plan.close()
    torch.cuda.synchronize()
    for a in keep:
        assert int(torch.cuda.cudart().cudaHostUnregister(a.ctypes.data)) == 0


@pytest.mark.parametrize("case", range(8))
def test_offload_random_plans_and_thread_counts(case):
    """Random layouts, caps and host thread counts (1 to more threads than a bucket has elements per
    thread): the team's slices of every bucket cover it exactly once and the result is the oracle's."""
    rng = np.random.default_rng(500 + case)
    W = int(rng.choice([1, 2, 3, 5, 8]))
    dtype = int(rng.choice([zr.F16, zr.BF16]))
    numels = [int(x) for x in rng.choice([0, 1, 9, 1000, 33_333, 100_000], size=int(rng.integers(1, 8)))]
    if sum(numels) == 0:
        numels[0] = 500
    cap = int(rng.choice([8, 1000, 50_000, 1 << 20]))
    nthreads = int(rng.choice([1, 3, 16, 64]))
    order = [int(x) for x in rng.permutation(W)]
    plan = zr.Plan(numels, W=W, dtype=dtype, stage=2, cap=cap, order=order)
    n = plan.numel
    tdt = plan.torch_dtype()
    ob, ooff = oracle_layout(plan, numels, cap, W)
    lay = Layout(numels, ooff, np.full(len(numels), 1e-2, F32), 40 + case, dtype)
    table = torch.from_numpy(zrgen.normal_table().copy()).cuda()
    cs = torch.cuda.current_stream().cuda_stream
    grads = [torch.zeros(n, dtype=tdt, device="cuda") for _ in range(W)]
    for r in range(W):
        lay.grads_dev(grads[r], 1, r, 1.0, table, cs)
    og = [lay.grads_host(0, n, 1, r, 1.0) for r in range(W)]
    master = lay.master_host(0, n)
    m, v = np.zeros(n, F32), np.zeros(n, F32)
    o = [master.copy(), m.copy(), v.copy(), np.zeros(n, np.uint16)]
    sums_dev = torch.empty(max(n, 4), dtype=torch.float32, device="cuda")
    sums_host = torch.empty(max(n, 4), dtype=torch.float32, pin_memory=True)
    param_host = torch.empty(max(n, 8), dtype=tdt, pin_memory=True)
    param_dev = torch.zeros(max(n, 8), dtype=tdt, device="cuda")
    of = plan.offload_step(grads, sums_dev, sums_host, master, m, v, param_host, param_dev, zr.AdamW(), 1.0, 1,
                           nthreads=nthreads)
    torch.cuda.synchronize()
    rep, _ = oracle.step(W, 1, dtype, ob, og, *o, OHYPER, oracle.new_scaler(1.0), order=order)
    assert of == rep.overflow == 0
    for a, b in zip((master, m, v), o[:3]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (case, W, cap, nthreads)
    assert np.array_equal(u16(param_dev)[:n], o[3])
    plan.close()


def test_offload_step_plan_without_parameters():
    """Every tensor empty: nothing is reduced or copied, the step is clean, and the zero-size (null) arrays are
    accepted, as zr_step accepts them."""
    plan = zr.Plan([0, 0], W=2, dtype=zr.F16, stage=2, cap=100)
    assert plan.numel == 0
    e16 = torch.empty(0, dtype=torch.float16)
    of = plan.offload_step([torch.empty(0, dtype=torch.float16, device="cuda")] * 2,
                           torch.empty(0, device="cuda"), torch.empty(0), np.zeros(0, F32), np.zeros(0, F32),
                           np.zeros(0, F32), e16, torch.empty(0, dtype=torch.float16, device="cuda"), zr.AdamW(),
                           1.0, 1, nthreads=4)
    torch.cuda.synchronize()
    assert of == 0
    plan.close()

