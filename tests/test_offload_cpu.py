"""ZeRO-Offload's host update (page "并行训练框架DeepSpeed介绍", (16) ZeRO-Offload: the optimizer update moves to
the CPU) against the oracle, without a GPU: same op order, so the same bits, for any thread count."""
import numpy as np
import pytest

import oracle

F32 = np.float32


@pytest.fixture(scope="module")
def zr():
    from zero_gradient_reduction_gb300 import build as zbuild
    zbuild.build()
    import zero_gradient_reduction_gb300 as z
    return z


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("nthreads", [1, 3, 16])
def test_offload_adamw_bit_exact(zr, dtype, nthreads):
    rng = np.random.default_rng(nthreads + 10 * dtype)
    for n, t, S, W in ((1, 1, 1.0, 1), (1000, 2, 1024.0, 3), (200_003, 7, 65536.0, 2)):
        sums = (rng.normal(size=n) * 40).astype(F32)
        p = (rng.normal(size=n) * 0.02).astype(F32)
        m = (rng.normal(size=n) * 1e-3).astype(F32)
        v = np.abs(rng.normal(size=n) * 1e-5).astype(F32)
        want = [p.copy(), m.copy(), v.copy()]
        g = (sums * oracle.unscale_factor(S, W)).astype(F32)
        oracle.adamw(g, *want, oracle.AdamW(), oracle.bias_correction(0.9, t), oracle.bias_correction(0.999, t))
        out = np.zeros(n, np.uint16)
        of = zr.offload_adamw(sums, p, m, v, out, dtype, zr.AdamW(), S, W, t, nthreads)
        assert of == 0
        for a, b in zip((p, m, v), want):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(out, oracle.encode(dtype, want[0]))


def test_offload_adamw_skips_on_nonfinite(zr):
    n = 300_000
    rng = np.random.default_rng(1)
    sums = rng.normal(size=n).astype(F32)
    sums[123_456] = np.nan
    arrs = [rng.normal(size=n).astype(F32) for _ in range(3)]
    arrs[2] = np.abs(arrs[2])
    before = [a.copy() for a in arrs]
    out = np.full(n, 7, np.uint16)
    assert zr.offload_adamw(sums, *arrs, out, 1, zr.AdamW(), 1.0, 1, 1, 8) == 1
    for a, b in zip(arrs, before):
        assert a.tobytes() == b.tobytes()
    assert np.all(out == 7)
