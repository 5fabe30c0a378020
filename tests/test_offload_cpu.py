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


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("n", [1, 7, 8, 4095, 4097, 100_003])
def test_offload_adamw_writes_nothing_outside(zr, dtype, n):
    """Guard bands around every host array: the vectorised update, its cast passes (fp16 per 4096-element chunk)
    and the thread split write only [0, n)."""
    G = 64
    rng = np.random.default_rng(n)

    def guarded(dt, fill):
        raw = np.empty(n + 2 * G, dt)
        raw.view(np.uint8)[:] = 0xA5
        raw[G:G + n] = fill
        return raw

    sums = guarded(F32, (rng.normal(size=n) * 10).astype(F32))
    p, m = guarded(F32, 0.5), guarded(F32, 0.0)
    v = guarded(F32, 0.0)
    out = guarded(np.uint16, 0)
    before = [a.copy() for a in (sums, p, m, v, out)]
    assert zr.offload_adamw(sums[G:G + n], p[G:G + n], m[G:G + n], v[G:G + n], out[G:G + n], dtype, zr.AdamW(),
                            1.0, 2, 1, 16) == 0
    for a, b in zip((sums, p, m, v, out), before):
        assert a[:G].tobytes() == b[:G].tobytes() and a[G + n:].tobytes() == b[G + n:].tobytes()
    assert not np.array_equal(p[G:G + n], before[1][G:G + n])  # the update did run


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
@pytest.mark.parametrize("where", [0, 37_499, 37_500, 123_456, 299_999])
def test_offload_adamw_skips_on_nonfinite(zr, bad, where):
    """One non-finite sum anywhere (the first and last element of a thread's slice of 37,500, the last element)
    skips the whole update: nothing is written."""
    n = 300_000
    rng = np.random.default_rng(1)
    sums = rng.normal(size=n).astype(F32)
    sums[where] = bad
    arrs = [rng.normal(size=n).astype(F32) for _ in range(3)]
    arrs[2] = np.abs(arrs[2])
    before = [a.copy() for a in arrs]
    out = np.full(n, 7, np.uint16)
    assert zr.offload_adamw(sums, *arrs, out, 1, zr.AdamW(), 1.0, 1, 1, 8) == 1
    for a, b in zip(arrs, before):
        assert a.tobytes() == b.tobytes()
    assert np.all(out == 7)


@pytest.mark.parametrize("dtype", [0, 1])
def test_offload_cast_every_boundary(zr, dtype):
    """The host cast to fp16 / bf16, exhaustively at its boundaries: with lr = weight decay = 0 the update leaves
    the master as it is (p * 1 - 0 * u), so the 16-bit output is the cast of the input, compared with the oracle's
    IEEE encoder on every 16-bit value's fp32 image, the midpoints between neighbours and one fp32 ulp on either
    side of each midpoint (the round-to-nearest-even ties and their neighbours), zeros, infinities, NaNs and the
    overflow threshold."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.decode(dtype, allbits)
    fin = vals[np.isfinite(vals)].astype(np.float64)
    fin = np.unique(fin)
    mids = ((fin[:-1] + fin[1:]) / 2).astype(F32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))])
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -np.nan, 65504.0, 65519.99, 65520.0, 3.4e38, -3.4e38,
                         1e-45, -1e-45, 2.0 ** -25, 2.0 ** -24, 2.0 ** -133, 2.0 ** -134], dtype=F32)
    p = np.concatenate([vals.astype(F32), near, specials]).astype(F32)
    n = p.size
    sums = np.zeros(n, F32)
    m = np.zeros(n, F32)
    v = np.zeros(n, F32)
    out = np.zeros(n, np.uint16)
    h = zr.AdamW(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    assert zr.offload_adamw(sums, p, m, v, out, dtype, h, 1.0, 1, 1, 4) == 0
    want = oracle.encode(dtype, p)
    nan = np.isnan(p)
    assert np.array_equal(out[~nan], want[~nan])
    # NaN: the canonical quiet NaN of its sign
    assert np.all((out[nan] & 0x7FFF) == (0x7E00 if dtype == 0 else 0x7FC0))
