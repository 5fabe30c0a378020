"""Seeded random plans through the fused step, ping-pong and in place, against the oracle bit for bit.

Each case draws W (1-64), A, the dtype, the ring order, a tensor list with empty and tiny tensors, the
bucket cap, the loss scale and the step mode, so the tile schedule (small-plan tile search, ragged
blocks), the kernel instantiations (specialised widths and the batched path for any other W) and both
commit modes meet shapes no hand-written case lists."""
import numpy as np
import pytest
import torch

import zero_gradient_reduction_gb300 as zr
from test_inplace_gpu import InPlaceRun
from test_parity_gpu import FusedRun

pytestmark = pytest.mark.gpu

WIDTHS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 11, 12, 16, 24, 31, 32, 64]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("case", range(64))
def test_random_plan_matches_oracle(case):
    rng = np.random.default_rng(9000 + case)
    W = int(rng.choice(WIDTHS))
    A = int(rng.choice([1, 1, 1, 2, 4]))  # W * A <= 256 for every draw
    dtype = int(rng.choice([zr.F16, zr.BF16]))
    ntensors = int(rng.integers(1, 12))
    numels = [int(x) for x in rng.choice([0, 1, 7, 8, 100, 999, 4096, 12_345, 40_000, 65_537], size=ntensors)]
    if sum(numels) == 0:
        numels[0] = 1000
    cap = int(rng.choice([1, 64, 5_000, 30_000, 1 << 20]))
    order = [int(x) for x in rng.permutation(W)]
    S = float(rng.choice([1.0, 8.0, 1024.0]))
    dynamic = bool(rng.integers(0, 2))
    sigma = rng.uniform(1e-3, 1e-1, size=ntensors)
    cls = InPlaceRun if rng.integers(0, 2) else FusedRun
    # the plan's own staging, or one chosen; a bulk staging half of the time with a drawn stage shape (stages of
    # 256-4096 elements, 1-4 of them, as long as they fit a block's shared memory)
    pick = int(rng.integers(0, 4))
    staging = None if pick == 0 else ((zr.STAGING_REGISTERS, zr.STAGING_BULK, zr.STAGING_BULK_IO)[pick - 1], 0, 0)
    if pick >= 2 and rng.integers(0, 2):
        E = int(rng.choice([256, 512, 1024, 2048, 4096]))
        NS = int(rng.integers(1, 5))
        # bulk loads with more than 8 replica slices spread them over stages of 8 (stages of at most 2048)
        chunked = pick == 2 and W * A > 8
        E = min(E, 2048) if chunked else E
        stage_bytes = (lambda e: 2 * 8 * e + 12 * e) if chunked else (lambda e: 2 * W * A * e + 12 * e)
        while NS > 1 and NS * stage_bytes(E) > 200 * 1024:
            NS -= 1
        while E > 256 and NS * stage_bytes(E) > 200 * 1024:
            E //= 2
        staging = (staging[0], E, NS)
    run = cls(numels, W, A, dtype, cap=cap, S=S, dynamic=dynamic, order=order, seed=case, sigma=sigma,
              interval=2, staging=staging)
    where = f"case {case}: W={W} A={A} dtype={dtype} cap={cap} numels={numels} {cls.__name__}"
    for s in (1, 2, 3):
        run.step(s)
        run.check(f"{where} step {s}: ")


@pytest.mark.parametrize("case", range(32))
def test_random_plan_all_paths_agree(case):
    """For a random plan: the per-bucket launches (zr_step_bucket), the unfused chain (zr_reduce_scatter per
    bucket, zr_adamw_shard_step, zr_all_gather) and the fused step give the same bytes, and the ZeRO-3 shards
    of the result gather back into it."""
    rng = np.random.default_rng(7000 + case)
    W = int(rng.choice(WIDTHS))
    dtype = int(rng.choice([zr.F16, zr.BF16]))
    tdt = torch.float16 if dtype == zr.F16 else torch.bfloat16
    ntensors = int(rng.integers(1, 10))
    numels = [int(x) for x in rng.choice([0, 1, 9, 100, 4096, 12_345, 40_000], size=ntensors)]
    if sum(numels) == 0:
        numels[0] = 777
    cap = int(rng.choice([1, 64, 5_000, 1 << 20]))
    order = [int(x) for x in rng.permutation(W)]
    S = float(rng.choice([1.0, 1024.0]))
    mk = lambda: zr.Plan(numels, W=W, A=1, dtype=dtype, stage=3, cap=cap, order=order, scaler=zr.Scaler(S))
    fused, bucketed = mk(), mk()
    n = fused.numel
    grads = [(torch.randn(n, generator=torch.Generator().manual_seed(case * 100 + r)) * 0.01 * S).to(tdt).cuda()
             for r in range(W)]
    master0 = (torch.randn(n, generator=torch.Generator().manual_seed(case)) * 0.02).cuda()
    h = zr.AdamW(lr=1e-3, weight_decay=0.01)
    states = []
    for _ in range(3):
        st = fused.new_state()
        st.master[0].copy_(master0)
        zr.all_gather(st.master[0], [st.param[0]])
        states.append(st)
    rf = fused.step(grads, states[0], h, report=True)
    for b in range(len(bucketed.buckets)):
        bucketed.step_bucket(b, grads, states[1], h)
    rb = bucketed.report()
    assert rf.t == rb.t == 1 and rf.overflow == rb.overflow == 0 and rf.current == rb.current == 1
    # the unfused chain, in place on set 0 of the third state
    st = states[2]
    sums = torch.empty(n, dtype=torch.float32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    for (b0, blen, _c) in fused.buckets:
        zr.reduce_scatter([g[b0:b0 + blen] for g in grads], sums[b0:b0 + blen], flag, order=order)
    zr.adamw_shard_step(sums, st.m[0], st.v[0], st.master[0], h, S, W, 1, flag)
    zr.all_gather(st.master[0], [st.param[0]])
    torch.cuda.synchronize()
    chain = st.live(0)
    for name in ("master", "m", "v", "param"):
        a = states[0].live(1)[name]
        for other in (states[1].live(1)[name], chain[name]):
            assert torch.equal(a.view(torch.uint8), other.view(torch.uint8)), (case, name)
    # ZeRO-3: keep the owned blocks, gather them back
    shards = fused.new_shards()
    fused.shard_params(states[0].live(1)["param"], shards)
    back = torch.empty_like(states[0].param[0])
    fused.gather_params(shards, back)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), states[0].live(1)["param"].view(torch.int16))
