"""GPU parity of the ZeRO-3 parameter shards and the all-gather before forward/backward against the oracle
(bit-exact: these are copies), including after a fused step and on the 1.3B workload's layout."""
import numpy as np
import pytest
import torch

import oracle
import zero_gradient_reduction_gb300 as zr
from _harness import oracle_layout
import zrgen
from test_parity_gpu import HYPER, u16

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


def _bits(x: np.ndarray, dtype: int) -> torch.Tensor:
    tdt = torch.float16 if dtype == zr.F16 else torch.bfloat16
    return torch.from_numpy(x.view(np.int16).copy()).cuda().view(tdt)


@pytest.mark.parametrize("W,order_seed", [(1, 0), (2, 1), (3, 2), (5, 3), (8, 4)])
def test_shard_and_gather_match_oracle(W, order_seed):
    rng = np.random.default_rng(order_seed)
    numels = [int(x) for x in rng.integers(1, 40_000, size=9)]
    order = [int(x) for x in rng.permutation(W)]
    plan = zr.Plan(numels, W=W, A=1, dtype=zr.BF16, stage=3, cap=30_000, order=order)
    n = plan.numel
    ob, _ = oracle_layout(plan, numels, 30_000, W)
    assert [plan.shard_numel(w) for w in range(W)] == oracle.shard_sizes(ob, W, order)
    replica = rng.integers(0, 65536, size=n).astype(np.uint16)
    want = oracle.shard_params(W, ob, replica, order)
    shards = plan.new_shards()
    plan.shard_params(_bits(replica, zr.BF16), shards)
    torch.cuda.synchronize()
    for w in range(W):
        k = plan.shard_numel(w)
        assert np.array_equal(u16(shards[w])[:k], want[w][:k])
    for b in range(len(plan.buckets)):
        for wk in range(W):
            assert plan.shard_offset(b, wk) >= 0
    # gather bucket ranges into a transient replica that starts out filled with a marker
    nb = len(plan.buckets)
    for lo, hi in ((0, nb), (1, 2), (nb - 1, nb), (0, 0)):
        out = torch.full((n,), 0, dtype=torch.int16, device="cuda")
        out.fill_(7)
        ref = np.full(n, 7, np.uint16)
        oracle.param_all_gather(W, ob, want, ref, lo, hi, order)
        plan.gather_params(shards, out.view(torch.bfloat16), lo, hi)
        torch.cuda.synchronize()
        assert np.array_equal(u16(out), ref), (lo, hi)
    plan.close()


def test_zero3_step_shard_gather_roundtrip():
    """ZeRO-3 flow: fused step writes the full replica; each worker keeps its shard; the all-gather before the
    next forward rebuilds exactly that replica."""
    numels = [100_000, 3_000, 64_000]
    plan = zr.Plan(numels, W=4, A=1, dtype=zr.F16, stage=3, cap=80_000, scaler=zr.Scaler(1024.0))
    st = plan.new_state()
    st.master[0].normal_(0, 0.02)
    grads = [torch.randn(plan.numel, device="cuda").mul_(10).half() for _ in range(4)]
    rep = plan.step(grads, st, HYPER, stage=3, report=True)
    full = st.param[rep.current]
    shards = plan.new_shards()
    plan.shard_params(full, shards)
    transient = torch.empty_like(full)
    for b in range(len(plan.buckets)):  # layer by layer, as before each forward
        plan.gather_params(shards, transient, b, b + 1)
    torch.cuda.synchronize()
    assert torch.equal(transient.view(torch.int16), full.view(torch.int16))
    plan.close()


def test_1p3b_layout_gather_sampled():
    w = zrgen.workload("1p3b")
    plan = zr.Plan(list(w.tensors), W=w.W, A=1, dtype=w.dtype, stage=3, cap=w.cap)
    n = plan.numel
    g = torch.Generator(device="cuda").manual_seed(3)
    full = torch.randint(-32768, 32767, (n,), dtype=torch.int16, device="cuda", generator=g)
    shards = plan.new_shards()
    plan.shard_params(full.view(torch.bfloat16), shards)
    out = torch.zeros_like(full)
    plan.gather_params(shards, out.view(torch.bfloat16))
    torch.cuda.synchronize()
    assert torch.equal(out, full)
    # spot-check the layout against the oracle's definition on bucket 3's blocks
    ob, _ = oracle_layout(plan, w.tensors, w.cap, w.W)
    b = 3
    s0, ln, C = (int(x) for x in ob[b])
    for pos in range(w.W):
        blk = (pos + 1) % w.W
        lo, hi = min(blk * C, ln), min((blk + 1) * C, ln)
        off = plan.shard_offset(b, pos)
        assert torch.equal(shards[pos][off:off + (hi - lo)].view(torch.int16), full[s0 + lo:s0 + hi])
    plan.close()
