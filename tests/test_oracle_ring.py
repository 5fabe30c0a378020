"""Pins of the oracle's ring collectives against what the pages and arithmetic fix.

- The three-GPU A/B/C walk-through (page "DP / DDP / DeepSpeed ZeRO-1/2/3", section 二 DDP):
  state after each scatter-reduce hop and each all-gather hop (tests/golden/ring_abc_3gpu.txt).
- Per-GPU traffic (same page, sections 二 and 三; page "第 7 讲：Parallelism（上）", 通信量分析):
  (W-1) * phi / W sent and received per phase, 2 (W-1) phi / W in total, tending to 2 phi.
- Brute force on tiny inputs: every reduced value equals the left fold in ring order starting at
  the block's origin; with integer-valued gradients it equals the exact integer sum; it is within
  W ulp of the double-precision sum.
"""
import numpy as np
import pytest

import oracle
from conftest import read_golden

BLOCK = {"A": 0, "B": 1, "C": 2}
GPU = {"GPU0": 0, "GPU1": 1, "GPU2": 2}


def _abc_value(term: str) -> float:
    # A_k = 2^k, B_k = 2^(k+3), C_k = 2^(k+6): every subset sum is distinct
    return float(2 ** (BLOCK[term[0]] * 3 + int(term[1])))


def _abc_work():
    return [np.array([_abc_value(f"{b}{k}") for b in "ABC"], dtype=np.float32) for k in range(3)]


def test_abc_scatter_reduce_hops():
    rows = read_golden("ring_abc_3gpu.txt")
    for hop in (1, 2):
        work = _abc_work()
        oracle.ring_reduce_scatter(work, 1, hops=range(0, hop))
        for phase, h, gpu, blk, contents in rows:
            if phase != "rs" or int(h) != hop:
                continue
            want = sum(_abc_value(t) for t in contents.split("+"))
            assert work[GPU[gpu]][BLOCK[blk]] == want, (hop, gpu, blk, contents)
    # after the full scatter reduce each GPU owns one total
    work = _abc_work()
    oracle.ring_reduce_scatter(work, 1)
    for phase, _, gpu, blk, contents in rows:
        if phase == "own":
            want = sum(_abc_value(t) for t in contents.split("+"))
            assert work[GPU[gpu]][BLOCK[blk]] == want
            # the owned block is (p + 1) mod W
            assert BLOCK[blk] == (GPU[gpu] + 1) % 3


def test_abc_first_hop_leaves_other_blocks():
    work = _abc_work()
    oracle.ring_reduce_scatter(work, 1, hops=range(0, 1))
    # after hop 1, GPU0 still holds its own A0 and B0; GPU1 its B1, C1; GPU2 its A2, C2
    assert work[0][0] == _abc_value("A0") and work[0][1] == _abc_value("B0")
    assert work[1][1] == _abc_value("B1") and work[1][2] == _abc_value("C1")
    assert work[2][0] == _abc_value("A2") and work[2][2] == _abc_value("C2")


def test_abc_all_gather_hops():
    rows = read_golden("ring_abc_3gpu.txt")
    marker = {0: 11, 1: 22, 2: 33}  # block -> 16-bit tag of its total
    for hop in (1, 2):
        reps = [np.zeros(3, dtype=np.uint16) for _ in range(3)]
        for p in range(3):
            own = (p + 1) % 3
            reps[p][own] = marker[own]
        oracle.ring_all_gather(reps, 1, hops=range(0, hop))
        for phase, h, gpu, blk, _ in rows:
            if phase == "ag" and int(h) == hop:
                assert reps[GPU[gpu]][BLOCK[blk]] == marker[BLOCK[blk]], (hop, gpu, blk)
        if hop == 1:
            # the second transfer has not happened yet: GPU1 does not have A
            assert reps[1][0] == 0
    reps = [np.zeros(3, dtype=np.uint16) for _ in range(3)]
    for p in range(3):
        reps[p][(p + 1) % 3] = marker[(p + 1) % 3]
    oracle.ring_all_gather(reps, 1)
    for p in range(3):
        assert list(reps[p]) == [11, 22, 33]


def test_abc_all_reduce_every_gpu_holds_every_total():
    """After the scatter reduce and the all-gather every GPU holds the totals of A, B and C (section 二:
    at the end of the all-gather phase all GPUs have all reduced gradients)."""
    rows = read_golden("ring_abc_3gpu.txt")
    totals = {}
    for phase, _, gpu, blk, contents in rows:
        if phase == "own":
            totals[BLOCK[blk]] = sum(_abc_value(t) for t in contents.split("+"))
    work = _abc_work()
    sent, recv = oracle.ring_all_reduce(work, 1)
    for p in range(3):
        assert [float(x) for x in work[p]] == [totals[0], totals[1], totals[2]]
    # two phases of W-1 = 2 one-element transfers per GPU
    assert list(sent) == [4, 4, 4] and list(recv) == [4, 4, 4]


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8, 9])
def test_all_reduce_is_the_reduce_scatter_on_every_worker(W):
    """Brute force: every position ends with every block's left fold in ring order (the reduce-scatter's
    owner values), bit for bit; traffic 2 (W-1) n / W per position when W divides n into 8-aligned blocks."""
    rng = np.random.default_rng(300 + W)
    for trial in range(5):
        n = 8 * W * int(rng.integers(1, 4)) if trial % 2 == 0 else int(rng.integers(1, 65))
        C = oracle.chunk_size(n, W, 8)
        xs = [rng.normal(scale=2.0, size=n).astype(np.float32) for _ in range(W)]
        order = list(rng.permutation(W))
        work = [xs[order[p]].copy() for p in range(W)]
        sent, recv = oracle.ring_all_reduce(work, C)
        want = _left_fold(xs, order, C, n)
        for p in range(W):
            assert np.array_equal(work[p].view(np.uint32), want.view(np.uint32)), (W, n, p)
        if n % (8 * W) == 0:
            assert all(int(x) == 2 * (W - 1) * n // W for x in sent)
            assert all(int(x) == 2 * (W - 1) * n // W for x in recv)


def test_all_reduce_integer_gradients_exact():
    rng = np.random.default_rng(11)
    W, n = 6, 96
    ints = [rng.integers(-50, 50, size=n) for _ in range(W)]
    work = [x.astype(np.float32) for x in ints]
    oracle.ring_all_reduce(work, oracle.chunk_size(n, W, 8))
    exact = np.sum(np.stack(ints), axis=0).astype(np.float32)
    for p in range(W):
        assert np.array_equal(work[p], exact)


@pytest.mark.parametrize("W", [2, 3, 4, 5, 7, 8, 9, 16])
def test_traffic_per_phase(W):
    rng = np.random.default_rng(W)
    k = int(rng.integers(1, 20))
    n = W * 8 * k
    sent, recv = oracle.ring_traffic(n, W, 8)
    assert all(s == (W - 1) * n // W for s in sent)
    assert all(r == (W - 1) * n // W for r in recv)
    # the hop-by-hop collectives count the same
    work = [np.zeros(n, dtype=np.float32) for _ in range(W)]
    s2, r2 = oracle.ring_reduce_scatter(work, n // W)
    assert list(s2) == list(sent) and list(r2) == list(recv)
    reps = [np.zeros(n, dtype=np.uint16) for _ in range(W)]
    s3, r3 = oracle.ring_all_gather(reps, n // W)
    assert list(s3) == list(sent) and list(r3) == list(recv)


def test_traffic_tends_to_2phi():
    n = 2 ** 20
    for W in (2, 4, 8, 16, 32, 64):
        sent, _ = oracle.ring_traffic(n, W, 8)
        total = 2 * int(sent[0])
        assert total == 2 * (W - 1) * n // W
        assert abs(total / n - 2.0) <= 2.0 / W + 1e-12


def test_step_traffic_zero1_equals_ddp():
    """ZeRO-1/2 move the same 2 (W-1) phi / W per worker as DDP's all-reduce."""
    W, n = 4, 4 * 8 * 5
    buckets = np.array([[0, n, n // W]])
    rng = np.random.default_rng(0)
    grads = [oracle.encode(oracle.F16, rng.normal(size=n).astype(np.float32)) for _ in range(W)]
    master = rng.normal(size=n).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    param = np.zeros(n, np.uint16)
    rep, _ = oracle.step(W, 1, oracle.F16, buckets, grads, master, m, v, param, oracle.AdamW(), oracle.new_scaler())
    for w in range(W):
        assert rep.rs_sent[w] == rep.rs_recv[w] == (W - 1) * n // W
        assert rep.ag_sent[w] == rep.ag_recv[w] == (W - 1) * n // W


def _left_fold(xs_by_worker, order, C, n):
    """Definition of a reduced value: start at the block's origin position, add positions in ring order."""
    W = len(order)
    out = np.empty(n, dtype=np.float32)
    for i in range(n):
        c = i // C
        s = np.float32(xs_by_worker[order[c]][i])
        for h in range(1, W):
            s = np.float32(s + np.float32(xs_by_worker[order[(c + h) % W]][i]))
        out[i] = s
    return out


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 7, 8, 9])
def test_brute_force_sums(W):
    rng = np.random.default_rng(100 + W)
    for trial in range(6):
        n = int(rng.integers(1, 65))
        n8 = ((n + 7) // 8) * 8  # tensors are aligned to 8 in the flat layout
        C = oracle.chunk_size(n8, W, 8)
        order = list(rng.permutation(W))
        dtype = oracle.F16 if trial % 2 == 0 else oracle.BF16
        grads = []
        for _ in range(W):
            x = np.zeros(n8, np.float32)
            x[:n] = rng.normal(scale=3.0, size=n)
            grads.append(oracle.encode(dtype, x))
        buckets = np.array([[0, n8, C]])
        zero = np.zeros(n8, np.float32)
        rep, sums = oracle.step(W, 1, dtype, buckets, grads, zero.copy(), zero.copy(), zero.copy(),
                                np.zeros(n8, np.uint16), oracle.AdamW(), oracle.new_scaler(), order=order,
                                want_sums=True)
        xs = [oracle.decode(dtype, g) for g in grads]
        want = _left_fold(xs, order, C, n8)
        assert np.array_equal(sums.view(np.uint32), want.view(np.uint32)), (W, n, order)
        # within W ulp of the double sum
        d = np.sum(np.stack([x.astype(np.float64) for x in xs]), axis=0)
        ulp = np.spacing(np.abs(d).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(sums.astype(np.float64) - d) <= W * ulp + 1e-30)


def test_integer_sums_exact_any_order():
    rng = np.random.default_rng(7)
    W, n = 9, 72
    C = oracle.chunk_size(n, W, 8)
    ints = [rng.integers(-100, 100, size=n) for _ in range(W)]
    grads = [oracle.encode(oracle.F16, x.astype(np.float32)) for x in ints]
    exact = np.sum(np.stack(ints), axis=0)
    for trial in range(4):
        order = list(rng.permutation(W))
        zero = np.zeros(n, np.float32)
        _, sums = oracle.step(W, 1, oracle.F16, np.array([[0, n, C]]), grads, zero.copy(), zero.copy(), zero.copy(),
                              np.zeros(n, np.uint16), oracle.AdamW(), oracle.new_scaler(), order=order,
                              want_sums=True)
        assert np.array_equal(sums, exact.astype(np.float32))


def test_ragged_chunks_cover_bucket_once():
    """Blocks of C = 8*ceil(n/(8W)) elements tile [0, n) exactly; short or empty blocks at the end."""
    for W in range(1, 12):
        for n in (8, 16, 24, 40, 64, 200, 1000, 1024):
            C = oracle.chunk_size(n, W, 8)
            assert C % 8 == 0 and C * W >= n and (C - 8) * W < n
            # a sum of ones counts each element exactly W times
            ones = [oracle.encode(oracle.F16, np.ones(n, np.float32)) for _ in range(W)]
            zero = np.zeros(n, np.float32)
            _, sums = oracle.step(W, 1, oracle.F16, np.array([[0, n, C]]), ones, zero.copy(), zero.copy(),
                                  zero.copy(), np.zeros(n, np.uint16), oracle.AdamW(), oracle.new_scaler(),
                                  want_sums=True)
            assert np.all(sums == W)
