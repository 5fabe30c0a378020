"""Pins of the oracle's reverse-order bucket builder.

The pages fix the order (page "DP / DDP / DeepSpeed ZeRO-1/2/3", section 二: parameters are laid out in the
reverse of their definition order, output layer first, and synchronised one full bucket at a time; page
"第 7 讲：Parallelism（上）", DDP 核心实现细节 3: buckets follow the reverse of the backward order). The
cap rule is the reading taken here: a non-empty bucket closes before a tensor that would take it past the cap.
The counts below follow from that reading and the shape lists by hand arithmetic (e.g. GPT-2: three layers
(21.24M) + norm_b + norm_a + fc2 = 23.60M; adding fc1 would pass 25M).
"""
import numpy as np
import pytest

import oracle
import zrgen


def test_gpt2_buckets():
    numels, names = zrgen.gpt2_small_tensors()
    assert len(numels) == 73 and sum(numels) == 123_586_560
    b, off = oracle.bucket_plan(numels, 25_000_000, 8)
    assert [int(x) for x in b[:, 1]] == [23_599_104, 24_187_392, 23_009_280, 14_157_312, 38_633_472]
    # output side first: the last-defined tensor (h11.norm_b) sits at flat offset 0, the embedding last
    assert off[-1] == 0 and names[-1] == "h11.norm_b"
    assert off[0] == sum(numels) - numels[0]
    assert b[-1, 0] == off[0] and b[-1, 1] == numels[0]


def test_1p3b_buckets():
    numels, _ = zrgen.gpt_1p3b_tensors()
    assert len(numels) == 145 and sum(numels) == 1_311_080_448
    b, off = oracle.bucket_plan(numels, 50_000_000, 8)
    assert len(b) == 33
    assert int(b[-1, 1]) == 50304 * 2048  # the embedding alone
    assert int(b[:, 1].sum()) == sum(numels)


@pytest.mark.parametrize("k,count", [(19, 121), (20, 121), (21, 121), (22, 121), (23, 121), (24, 97), (25, 49),
                                     (26, 25), (27, 11), (28, 6)])
def test_sweep_bucket_counts(k, count):
    numels, _ = zrgen.gpt_1p3b_tensors()
    b, _ = oracle.bucket_plan(numels, 1 << k, 8)
    assert len(b) == count


def test_flat_7b_in_200m_buckets():
    w = zrgen.workload("7b")
    b, _ = oracle.bucket_plan(list(w.tensors), w.cap, w.W)
    assert len(b) == 35 and all(int(x) == 200_000_000 for x in b[:, 1])
    assert all(int(c) == 100_000_000 for c in b[:, 2])


def test_flat_13b_in_200m_buckets_and_its_memory():
    """The 13B in-place workload: 65 full buckets; its two ping-pong sets would not fit one GB300 (288 GB)
    beside the gradients, one set does."""
    w = zrgen.workload("13b")
    b, _ = oracle.bucket_plan(list(w.tensors), w.cap, w.W)
    assert len(b) == 65 and int(b[:, 1].sum()) == 13_000_000_000 and w.state_sets == 1
    grads = 2 * w.W * w.A * w.n
    assert grads + 2 * 14 * w.n > 288e9 > grads + 14 * w.n


def test_contiguous_reverse_and_aligned():
    rng = np.random.default_rng(0)
    for trial in range(20):
        nt = int(rng.integers(1, 40))
        numels = [int(x) for x in rng.integers(1, 5000, size=nt)]
        cap = int(rng.integers(1, 20000))
        W = int(rng.integers(1, 10))
        b, off = oracle.bucket_plan(numels, cap, W, 8)
        # buckets tile the flat buffer in order
        assert b[0, 0] == 0
        for i in range(1, len(b)):
            assert b[i, 0] == b[i - 1, 0] + b[i - 1, 1]
        # tensors placed last-defined first, each at a multiple of 8, never overlapping
        order = sorted(range(nt), key=lambda t: off[t])
        assert order == list(range(nt - 1, -1, -1))
        for t in range(nt):
            assert off[t] % 8 == 0
            if t > 0:
                assert off[t - 1] == off[t] + ((numels[t] + 7) // 8) * 8
        # every tensor lies inside one bucket; a bucket over the cap holds one tensor
        for s, n, c in b:
            inside = [t for t in range(nt) if s <= off[t] < s + n]
            assert all(off[t] + numels[t] <= s + n for t in inside)
            if n > cap:
                assert len(inside) == 1
            assert c == oracle.chunk_size(int(n), W, 8)
        # closing rule: the first tensor of the next bucket would have overflowed this one
        for i in range(len(b) - 1):
            s, n, _ = b[i]
            nxt = [t for t in range(nt) if off[t] == b[i + 1, 0]][0]
            assert n + numels[nxt] > cap


def test_equal_to_cap_fits():
    b, _ = oracle.bucket_plan([8, 8, 8], 16, 2)
    assert [int(x) for x in b[:, 1]] == [16, 8]
    b, _ = oracle.bucket_plan([100, 8], 16, 2)  # 100 > cap sits alone
    assert [int(x) for x in b[:, 1]] == [8, 104]
