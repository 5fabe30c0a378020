"""The standalone accumulate path (gradient accumulation with the synchronisation skipped, page
"第 7 讲：Parallelism（上）", Gradient Accumulation): zr_accumulate per micro-batch into fp32, then the ring over
fp32 inputs. It must give the same bits as the fused A-way step and as the oracle."""
import numpy as np
import pytest
import torch

import oracle
import zero_gradient_reduction_gb300 as zr
import zrgen
from zrgen.layout import Layout
from _harness import oracle_layout
from test_parity_gpu import HYPER, OHYPER, assert_state_close, f32bits, to_dev16, u16

pytestmark = pytest.mark.gpu
F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype", [zr.F16, zr.BF16])
def test_accumulate_bit_exact(dtype):
    rng = np.random.default_rng(4 + dtype)
    for n in (1, 9, 4096, 100_003):
        A = 4
        gs = [oracle.encode(dtype, (rng.normal(size=n) * 5).astype(F32)) for _ in range(A)]
        want = np.zeros(n, F32)
        acc = torch.empty(n, dtype=torch.float32, device="cuda")
        for a, g in enumerate(gs):
            oracle.accumulate(dtype, g, want, a == 0)
            zr.accumulate(to_dev16(g, dtype), acc, a == 0)
        torch.cuda.synchronize()
        assert np.array_equal(f32bits(acc), want.view(np.uint32))


def test_reduce_scatter_on_fp32_inputs():
    rng = np.random.default_rng(8)
    for W, n in ((2, 1000), (5, 4099), (8, 70_001)):
        xs = [(rng.normal(size=n) * 3).astype(F32) for _ in range(W)]
        order = list(rng.permutation(W))
        C = oracle.chunk_size(n, W, 8)
        work = [xs[order[p]].copy() for p in range(W)]
        oracle.ring_reduce_scatter(work, C)
        want = np.empty(n, F32)
        for p in range(W):
            c = (p + 1) % W
            lo, hi = min(c * C, n), min((c + 1) * C, n)
            want[lo:hi] = work[p][lo:hi]
        sums = torch.empty(n, dtype=torch.float32, device="cuda")
        of = torch.zeros(1, dtype=torch.int32, device="cuda")
        zr.reduce_scatter([torch.from_numpy(x).cuda() for x in xs], sums, of, order=order)
        torch.cuda.synchronize()
        assert np.array_equal(f32bits(sums), want.view(np.uint32)) and of.item() == 0


@pytest.mark.parametrize("W,A", [(2, 4), (4, 3), (8, 4)])
def test_accumulate_then_fp32_step_equals_fused_and_oracle(W, A):
    numels = [40_000, 999, 77_777, 8]
    rng = np.random.default_rng(W * 10 + A)
    order = list(rng.permutation(W))
    sig = rng.uniform(1e-3, 1e-1, size=len(numels)).astype(F32)
    fused = zr.Plan(numels, W=W, A=A, dtype=zr.BF16, stage=2, cap=50_000, order=order, scaler=zr.Scaler(1.0))
    acc_plan = zr.Plan(numels, W=W, A=1, dtype=zr.BF16, stage=2, cap=50_000, order=order, scaler=zr.Scaler(1.0),
                       fp32_grads=True)
    assert np.array_equal(fused.buckets, acc_plan.buckets)
    obuckets, ooffsets = oracle_layout(fused, numels, 50_000, W)
    lay = Layout(numels, ooffsets, sig, 5, zr.BF16)
    n = fused.numel
    table = torch.from_numpy(zrgen.normal_table().copy()).cuda()
    cs = torch.cuda.current_stream().cuda_stream
    st_f, st_a = fused.new_state(), acc_plan.new_state()
    for st in (st_f, st_a):
        st.master[0].zero_()
        lay.master_dev(st.master[0], table, cs)
    om = lay.master_host(0, n)
    o = [om, np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)]
    osc = oracle.new_scaler(1.0)
    grads = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(W * A)]
    accs = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(W)]
    for step in (1, 2):
        for r in range(W * A):
            lay.grads_dev(grads[r], step, r, 1.0, table, cs)
        rf = fused.step(grads, st_f, HYPER, report=True)
        for w in range(W):
            for a in range(A):
                zr.accumulate(grads[w * A + a], accs[w], a == 0)
        ra = acc_plan.step(accs, st_a, HYPER, report=True)
        assert rf.overflow == ra.overflow == 0 and rf.current == ra.current
        for x, y in zip(st_f.live(rf.current).values(), st_a.live(ra.current).values()):
            assert x.cpu().view(torch.int32 if x.element_size() == 4 else torch.int16).numpy().tobytes() == \
                y.cpu().view(torch.int32 if y.element_size() == 4 else torch.int16).numpy().tobytes()
        og = [lay.grads_host(0, n, step, r, 1.0) for r in range(W * A)]
        oracle.step(W, A, zr.BF16, obuckets, og, *o, OHYPER, osc, order=order)
        L = st_a.live(ra.current)
        assert_state_close(L["master"].cpu().numpy(), L["m"].cpu().numpy(), L["v"].cpu().numpy(), u16(L["param"]),
                           *o, exact=True, where=f"W={W} A={A} step {step}: ")
    fused.close()
    acc_plan.close()
