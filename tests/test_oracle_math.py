"""Pins of the oracle's arithmetic: mean, AdamW, loss scaling, number formats and memory accounting.

Each check is tied to something the pages or mathematics fix, not to the oracle's own formulas:
- data-parallel mean == full-batch gradient of a tiny least-squares model (page "第 7 讲：Parallelism
  （上）", 数学等价性), exact in dyadic arithmetic;
- AdamW: the first step from m = v = 0, a constant-gradient closed form over many steps, the place of
  eps, and torch.optim.AdamW (the optimizer in that page's DDP loop) within 2 ulp;
- skipped steps leave the state byte-identical and halve the scale (page "并行训练框架DeepSpeed介绍",
  核心技术 (1)/(3): dynamic loss scaling);
- fp16/bf16 conversions equal torch's CPU casts on every 16-bit pattern and on a large float sample;
- model-state bytes equal the pages' printed numbers (tests/golden/memory_accounting.txt).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

F32 = np.float32


def f32ulp(x):
    return np.spacing(np.abs(np.asarray(x, dtype=np.float32))).astype(np.float64)


# ------------------------------------------------------------------ mean
def test_mean_equals_full_batch_gradient():
    """Least squares L = (1/B) sum (x_i . theta - y_i)^2 split over W workers (B/W samples each)."""
    rng = np.random.default_rng(0)
    B, W, d = 16, 4, 8
    X = rng.integers(-2, 3, size=(B, d)).astype(np.float64)
    theta = rng.integers(-2, 3, size=d).astype(np.float64)
    y = rng.integers(-4, 5, size=B).astype(np.float64)
    full = (2.0 / B) * X.T @ (X @ theta - y)
    per = []
    for k in range(W):
        Xk, yk = X[k * B // W:(k + 1) * B // W], y[k * B // W:(k + 1) * B // W]
        per.append((2.0 / (B / W)) * Xk.T @ (Xk @ theta - yk))
    for g in per:  # dyadic and small: exact in fp16
        assert np.array_equal(oracle.decode(oracle.F16, oracle.encode(oracle.F16, g.astype(F32))), g.astype(F32))
    grads = [oracle.encode(oracle.F16, g.astype(F32)) for g in per]
    n = d
    C = oracle.chunk_size(n, W, 2)
    zero = np.zeros(n, F32)
    for order in ([0, 1, 2, 3], [2, 0, 3, 1]):
        _, sums = oracle.step(W, 1, oracle.F16, np.array([[0, n, C]]), grads, zero.copy(), zero.copy(), zero.copy(),
                              np.zeros(n, np.uint16), oracle.AdamW(), oracle.new_scaler(1.0), order=order,
                              want_sums=True)
        mean = sums * oracle.unscale_factor(1.0, W)
        assert np.array_equal(mean.astype(np.float64), full)


def test_unscale_factor_removes_scale_and_count():
    for S, W in ((1024.0, 3), (65536.0, 2), (1.0, 8), (32768.0, 64)):
        r = oracle.unscale_factor(S, W)
        assert r == F32(1.0 / (S * W))
    # the mean of W identical scaled gradients is the unscaled gradient (powers of two: exact)
    assert F32(F32(8 * 3.0 * 1024) * oracle.unscale_factor(1024.0, 8)) == F32(3.0)


# ------------------------------------------------------------------ AdamW
H = oracle.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def test_first_step_moments_closed_form():
    rng = np.random.default_rng(1)
    g = rng.normal(size=4096).astype(F32) * F32(0.01)
    p = rng.normal(size=4096).astype(F32) * F32(0.02)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    bc1, bc2 = oracle.bias_correction(H.beta1, 1), oracle.bias_correction(H.beta2, 1)
    oracle.adamw(g, p.copy(), m, v, H, bc1, bc2)
    omb1 = F32(1.0) - F32(H.beta1)
    omb2 = F32(1.0) - F32(H.beta2)
    assert np.array_equal(m, (omb1 * g).astype(F32))
    assert np.array_equal(v, (omb2 * (g * g).astype(F32)).astype(F32))


def test_constant_gradient_closed_form():
    """With g constant, m_hat = g and v_hat = g^2 at every t, so each step is p <- p*d - lr*g/(|g|+eps)."""
    T = 25
    g = np.array([0.5, -0.25, 3.0, -7.0, 1e-3, -2e-4], dtype=F32)
    p0 = np.array([0.02, -0.01, 0.5, -0.3, 0.0, 1.0], dtype=F32)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    for t in range(1, T + 1):
        oracle.adamw(g, p, m, v, H, oracle.bias_correction(H.beta1, t), oracle.bias_correction(H.beta2, t))
        d = 1.0 - float(F32(H.lr)) * float(F32(H.weight_decay))
        u = g.astype(np.float64) / (np.abs(g.astype(np.float64)) + float(F32(H.eps)))
        want = p0.astype(np.float64) * d ** t - float(F32(H.lr)) * u * sum(d ** k for k in range(t))
        # fp32 recurrences: at most ~2 ulp of p and a 2e-6 relative error of the step per step taken
        tol = t * (2 * f32ulp(want) + float(F32(H.lr)) * 2e-6) + 1e-12
        assert np.all(np.abs(p - want) <= tol), (t, p, want)


def test_eps_outside_sqrt():
    """u = m_hat / (sqrt(v_hat) + eps): with |g| = eps the step is half of lr (eps inside sqrt gives ~1e-4)."""
    g = np.array([1e-8, -1e-8], dtype=F32)
    p = np.zeros(2, F32)
    m, v = np.zeros(2, F32), np.zeros(2, F32)
    h = oracle.AdamW(lr=1.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    oracle.adamw(g, p, m, v, h, oracle.bias_correction(0.9, 1), oracle.bias_correction(0.999, 1))
    assert np.allclose(p, [-0.5, 0.5], rtol=1e-5)


def test_bias_correction_is_one_minus_beta_power():
    for beta in (0.9, 0.999, 0.95):
        b = float(F32(beta))
        for t in (1, 2, 3, 10, 100, 1000):
            bc = oracle.bias_correction(beta, t)
            assert abs(float(bc) - (1.0 - b ** t)) <= float(f32ulp(1.0 - b ** t))


@pytest.mark.parametrize("steps", [1, 3])
def test_matches_torch_adamw(steps):
    """W=1, S=1: the update equals torch.optim.AdamW on the fp32 master within 4 ulp of the operands' scale
    (12 after 3 steps). torch folds lr into lr/bc1 and divides sqrt(v) by sqrt(bc2); those roundings differ by
    a few ulp of max(|p_before|, |p_after|, lr); a wrong term would be off by ~lr, i.e. ~10^7 such ulp."""
    rng = np.random.default_rng(2)
    n = 4096
    p0 = (rng.normal(size=n) * 0.02).astype(F32)
    gs = [(rng.normal(size=n) * 1e-2).astype(F32) for _ in range(steps)]
    # hyperparameters as the fp32 values the oracle holds, so that both sides start from the same numbers
    hp = dict(lr=float(F32(1e-3)), betas=(float(F32(0.9)), float(F32(0.999))), eps=float(F32(1e-8)),
              weight_decay=float(F32(0.01)))
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], foreach=False, **hp)
    p, m, v = p0.copy(), np.zeros(n, F32), np.zeros(n, F32)
    for t, g in enumerate(gs, start=1):
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
        oracle.adamw(g, p, m, v, H, oracle.bias_correction(0.9, t), oracle.bias_correction(0.999, t))
    want = tp.detach().numpy()
    tol = 4 if steps == 1 else 12
    scale = np.maximum(np.maximum(np.abs(want), np.abs(p0)), F32(1e-3))
    err = np.abs(p.astype(np.float64) - want) / f32ulp(scale)
    assert np.all(err <= tol), err.max()


# ------------------------------------------------------------------ step, skip, scaler
def _small_problem(W=2, n=64, dtype=oracle.F16, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    grads = [oracle.encode(dtype, (rng.normal(size=n) * scale).astype(F32)) for _ in range(W)]
    master = (rng.normal(size=n) * 0.02).astype(F32)
    return grads, master


def test_clean_step_params_are_cast_master():
    W, n = 3, 96
    grads, master = _small_problem(W, n, scale=10.0)
    m, v = np.zeros(n, F32), np.zeros(n, F32)
    param = np.zeros(n, np.uint16)
    rep, _ = oracle.step(W, 1, oracle.F16, np.array([[0, n, oracle.chunk_size(n, W, 8)]]), grads, master, m, v,
                         param, H, oracle.new_scaler(1024.0))
    assert rep.overflow == 0 and rep.t_after == 1
    assert np.array_equal(param, oracle.encode(oracle.F16, master))


def test_skip_leaves_state_identical_and_halves_scale():
    W, n = 2, 64
    grads, master = _small_problem(W, n, scale=100.0)
    grads[1][17] = 0x7C00  # +inf in fp16
    m = np.full(n, 0.5, F32)
    v = np.full(n, 0.25, F32)
    param = oracle.encode(oracle.F16, master)
    before = [a.copy() for a in (master, m, v, param)]
    sc = oracle.new_scaler(65536.0, dynamic=True)
    sc.t = 4
    rep, _ = oracle.step(W, 1, oracle.F16, np.array([[0, n, 32]]), grads, master, m, v, param, H, sc)
    assert rep.overflow == 1 and rep.skipped == 1
    for a, b in zip((master, m, v, param), before):
        assert a.tobytes() == b.tobytes()
    assert sc.scale == 32768.0 and sc.t == 4 and rep.t_after == 4


def test_nan_also_skips_and_scale_floor():
    W, n = 2, 16
    grads, master = _small_problem(W, n)
    grads[0][3] = 0x7E00  # NaN
    sc = oracle.new_scaler(1.0, dynamic=True)
    rep, _ = oracle.step(W, 1, oracle.F16, np.array([[0, n, 8]]), grads, master, np.zeros(n, F32),
                         np.zeros(n, F32), np.zeros(n, np.uint16), H, sc)
    assert rep.skipped == 1 and sc.scale == 1.0  # floored at min_scale


def test_static_scaler_skips_without_changing_scale():
    W, n = 2, 16
    grads, master = _small_problem(W, n)
    grads[0][0] = 0xFC00  # -inf
    sc = oracle.new_scaler(1024.0, dynamic=False)
    rep, _ = oracle.step(W, 1, oracle.F16, np.array([[0, n, 8]]), grads, master, np.zeros(n, F32),
                         np.zeros(n, F32), np.zeros(n, np.uint16), H, sc)
    assert rep.skipped == 1 and sc.scale == 1024.0 and sc.t == 0


def test_scale_growth_after_interval():
    W, n = 2, 16
    sc = oracle.new_scaler(4.0, dynamic=True, interval=3)
    m, v, param = np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)
    scales = []
    for s in range(7):
        grads, master0 = _small_problem(W, n, seed=s)
        if s == 0:
            master = master0
        rep, _ = oracle.step(W, 1, oracle.F16, np.array([[0, n, 8]]), grads, master, m, v, param, H, sc)
        scales.append(rep.scale_used)
    assert scales == [4.0, 4.0, 4.0, 8.0, 8.0, 8.0, 16.0]
    assert sc.t == 7


def test_overflow_flag_is_global_across_buckets():
    """One non-finite value in one bucket skips the update of every bucket."""
    W, n = 2, 64
    grads, master = _small_problem(W, n)
    grads[0][60] = 0x7C00  # in the second bucket
    buckets = np.array([[0, 32, 16], [32, 32, 16]])
    m, v = np.zeros(n, F32), np.zeros(n, F32)
    before = master.copy()
    rep, _ = oracle.step(W, 1, oracle.F16, buckets, grads, master, m, v, np.zeros(n, np.uint16), H,
                         oracle.new_scaler(8.0, dynamic=True))
    assert rep.skipped == 1 and np.array_equal(master, before)


def test_dynamic_scale_trace_with_injected_inf():
    """Six steps, +inf at step 3: S used 65536, 65536, 65536 (skip), 32768, 32768, 32768; t 1, 2, 2, 3, 4, 5."""
    W, n = 2, 64
    sc = oracle.new_scaler(65536.0, dynamic=True)
    rng = np.random.default_rng(5)
    master = (rng.normal(size=n) * 0.02).astype(F32)
    m, v, param = np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)
    used, ts = [], []
    for step in range(1, 7):
        S = sc.scale
        grads = [oracle.encode(oracle.F16, (rng.normal(size=n) * 1e-2 * S).astype(F32)) for _ in range(W)]
        if step == 3:
            grads[1][5] = 0x7C00
        rep, _ = oracle.step(W, 1, oracle.F16, np.array([[0, n, 32]]), grads, master, m, v, param, H, sc)
        used.append(rep.scale_used)
        ts.append(rep.t_after)
    assert used == [65536.0, 65536.0, 65536.0, 32768.0, 32768.0, 32768.0]
    assert ts == [1, 2, 2, 3, 4, 5]


def test_accumulation_sums_microbatches_first():
    """A micro-batches per worker: the reduced value is the ring sum of per-worker fp32 micro-batch sums."""
    W, A, n = 3, 4, 48
    rng = np.random.default_rng(9)
    ints = [rng.integers(-50, 50, size=n) for _ in range(W * A)]
    grads = [oracle.encode(oracle.BF16, x.astype(F32)) for x in ints]
    zero = np.zeros(n, F32)
    _, sums = oracle.step(W, A, oracle.BF16, np.array([[0, n, 16]]), grads, zero.copy(), zero.copy(), zero.copy(),
                          np.zeros(n, np.uint16), H, oracle.new_scaler(), want_sums=True)
    assert np.array_equal(sums, np.sum(np.stack(ints), axis=0).astype(F32))
    # effective batch: W * b * A samples contribute (page "第 7 讲", Gradient Accumulation)
    b = 2
    assert W * b * A == len(grads) * b


def test_standalone_accumulate_then_ring_equals_step():
    """zro_accumulate over A micro-batches, then the ring over the fp32 sums, equals the step's own S1 + S2."""
    W, A, n = 3, 4, 96
    rng = np.random.default_rng(12)
    grads = [oracle.encode(oracle.BF16, rng.normal(size=n).astype(F32)) for _ in range(W * A)]
    zero = np.zeros(n, F32)
    _, want = oracle.step(W, A, oracle.BF16, np.array([[0, n, 32]]), grads, zero.copy(), zero.copy(), zero.copy(),
                          np.zeros(n, np.uint16), H, oracle.new_scaler(), want_sums=True)
    work = []
    for w in range(W):
        acc = np.zeros(n, F32)
        for a in range(A):
            oracle.accumulate(oracle.BF16, grads[w * A + a], acc, a == 0)
        work.append(acc)
    # the accumulators are exactly the left fold of the decoded micro-batches
    for w in range(W):
        ref = oracle.decode(oracle.BF16, grads[w * A])
        for a in range(1, A):
            ref = (ref + oracle.decode(oracle.BF16, grads[w * A + a])).astype(F32)
        assert np.array_equal(work[w], ref)
    oracle.ring_reduce_scatter(work, 32)
    got = np.empty(n, F32)
    for p in range(W):
        c = (p + 1) % W
        got[c * 32:(c + 1) * 32] = work[p][c * 32:(c + 1) * 32]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_sampled_windows_match_full_run():
    """A bucket cut to the same window of every block, run as its own bucket, gives the same values."""
    W, n = 4, 4 * 64
    rng = np.random.default_rng(11)
    order = [2, 0, 3, 1]
    grads = [oracle.encode(oracle.BF16, rng.normal(size=n).astype(F32)) for _ in range(W)]
    master = (rng.normal(size=n) * 0.02).astype(F32)
    C = n // W
    full = [master.copy(), np.zeros(n, F32), np.zeros(n, F32), np.zeros(n, np.uint16)]
    oracle.step(W, 1, oracle.BF16, np.array([[0, n, C]]), grads, *full, H, oracle.new_scaler(), order=order)
    off, L = 16, 24
    idx = np.concatenate([np.arange(c * C + off, c * C + off + L) for c in range(W)])
    win = [master[idx].copy(), np.zeros(W * L, F32), np.zeros(W * L, F32), np.zeros(W * L, np.uint16)]
    oracle.step(W, 1, oracle.BF16, np.array([[0, W * L, L]]), [np.ascontiguousarray(g[idx]) for g in grads], *win,
                H, oracle.new_scaler(), order=order)
    for a, b in zip(win, full):
        assert a.tobytes() == b[idx].tobytes()


# ------------------------------------------------------------------ number formats
def _torch_bits(x: np.ndarray, dt) -> np.ndarray:
    return torch.from_numpy(x).to(dt).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype,tdt", [(oracle.F16, torch.float16), (oracle.BF16, torch.bfloat16)])
def test_decode_every_pattern(dtype, tdt):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(dtype, bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(tdt).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


@pytest.mark.parametrize("dtype,tdt", [(oracle.F16, torch.float16), (oracle.BF16, torch.bfloat16)])
def test_encode_matches_torch_rne(dtype, tdt):
    rng = np.random.default_rng(3)
    raw = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32).view(F32)
    normal = (rng.normal(size=200_000) * rng.choice([1e-6, 1e-3, 1.0, 1e3, 6e4], size=200_000)).astype(F32)
    # every value exactly halfway between two neighbours of the 16-bit grid, both parities
    halves = []
    for b in np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16):
        lo = oracle.decode(dtype, np.array([b], np.uint16))[0]
        hi = oracle.decode(dtype, np.array([b + 1], np.uint16))[0] if b != 0xFFFF else np.nan
        if np.isfinite(lo) and np.isfinite(hi) and np.sign(lo) == np.sign(hi) or lo == 0:
            halves.append(F32((np.float64(lo) + np.float64(hi)) / 2))
    edge = np.array([0.0, -0.0, np.inf, -np.inf, 65504, 65519.99, 65520, 65536, 6.1e-5, 5.96e-8, 2.98e-8,
                     2.9802322e-08, 3.0e-8, 1e-45, 3.4e38, -3.4e38, 3.3895314e38, 3.3961776e38], dtype=F32)
    x = np.concatenate([raw, normal, np.array(halves, F32), edge])
    x = x[~np.isnan(x)]
    assert np.array_equal(oracle.encode(dtype, x), _torch_bits(x, tdt))
    nan = np.array([np.nan, -np.nan], F32)
    assert np.all(np.isnan(oracle.decode(dtype, oracle.encode(dtype, nan))))


# ------------------------------------------------------------------ memory accounting
def test_model_state_bytes_golden():
    for stage, n, W, want, tol, src in read_golden("memory_accounting.txt"):
        got = oracle.model_state_bytes(int(stage), int(n), int(W))
        assert abs(got - int(want)) <= int(tol), (src, got, want)


def test_model_state_bytes_16_per_param_and_sharding():
    n = 123_456_789
    assert oracle.model_state_bytes(0, n, 8) == 16 * n
    for W in (1, 2, 4, 8, 64):
        # W = 1 shards nothing: every stage holds the full 16 bytes per parameter
        if W == 1:
            assert all(oracle.model_state_bytes(s, n, 1) == 16 * n for s in (0, 1, 2, 3))
        assert oracle.model_state_bytes(1, n, W) >= oracle.model_state_bytes(2, n, W) >= \
            oracle.model_state_bytes(3, n, W)
    # 7B states do not fit an 80 GB GPU unsharded but do at W = 8 with stage 3
    assert oracle.model_state_bytes(0, 7 * 10 ** 9, 8) > 80e9 > oracle.model_state_bytes(3, 7 * 10 ** 9, 8)
