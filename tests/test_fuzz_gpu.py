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
    run = cls(numels, W, A, dtype, cap=cap, S=S, dynamic=dynamic, order=order, seed=case, sigma=sigma,
              interval=2)
    where = f"case {case}: W={W} A={A} dtype={dtype} cap={cap} numels={numels} {cls.__name__}"
    for s in (1, 2, 3):
        run.step(s)
        run.check(f"{where} step {s}: ")
