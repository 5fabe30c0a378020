"""Pins of the oracle's ZeRO-3 parameter shards and the all-gather before forward/backward.

Page "DP / DDP / DeepSpeed ZeRO-1/2/3", section 四: under ZeRO-3 the parameters are partitioned too; a GPU
missing a layer's parameters receives them before forward and again before backward, then drops them; the
extra all-gather makes the traffic 3 phi, 1.5x DDP. Page "第 7 讲：Parallelism（上）", ZeRO Stage 3: each GPU
stores 1/W of the parameters (2N/W bytes of the 16N/W total).
"""
import numpy as np
import pytest

import oracle


def test_abc_shards_are_the_owned_blocks():
    """Three GPUs, blocks A, B, C: after reduce-scatter GPU0 owns B, GPU1 C, GPU2 A, and keeps just that."""
    replica = np.array([11, 22, 33], np.uint16)  # A, B, C
    shards = oracle.shard_params(3, np.array([[0, 3, 1]]), replica)
    assert [list(s) for s in shards] == [[22], [33], [11]]
    out = np.zeros(3, np.uint16)
    oracle.param_all_gather(3, np.array([[0, 3, 1]]), shards, out, 0, 1)
    assert list(out) == [11, 22, 33]


@pytest.mark.parametrize("W", [1, 2, 3, 5, 8])
def test_gather_of_shards_restores_replica(W):
    rng = np.random.default_rng(W)
    for trial in range(5):
        numels = [int(x) for x in rng.integers(1, 3000, size=int(rng.integers(1, 12)))]
        buckets, _ = oracle.bucket_plan(numels, int(rng.integers(100, 6000)), W)
        n = int(buckets[-1, 0] + buckets[-1, 1])
        order = list(rng.permutation(W))
        replica = rng.integers(0, 65536, size=n).astype(np.uint16)
        shards = oracle.shard_params(W, buckets, replica, order)
        assert sum(oracle.shard_sizes(buckets, W, order)) == n
        out = np.zeros(n, np.uint16)
        oracle.param_all_gather(W, buckets, shards, out, 0, len(buckets), order)
        assert np.array_equal(out, replica)
        # a bucket range touches only those buckets
        lo = int(rng.integers(0, len(buckets)))
        hi = int(rng.integers(lo, len(buckets) + 1))
        part = np.full(n, 7, np.uint16)
        oracle.param_all_gather(W, buckets, shards, part, lo, hi, order)
        inside = np.zeros(n, bool)
        for s, ln, _ in buckets[lo:hi]:
            inside[s:s + ln] = True
        assert np.array_equal(part[inside], replica[inside]) and np.all(part[~inside] == 7)


def test_shard_is_one_wth_of_the_parameters():
    W, n = 8, 8 * 8 * 1000
    buckets, _ = oracle.bucket_plan([n], n, W)
    sizes = oracle.shard_sizes(buckets, W)
    assert sizes == [n // W] * W
    # parameter bytes per worker: 2N/W, the parameter term of stage 3's 16N/W
    assert 2 * sizes[0] == 2 * n // W and oracle.model_state_bytes(3, n, W) == 16 * n // W


def test_zero3_traffic_is_three_phi():
    """reduce-scatter + all-gather before forward + all-gather before backward: 3 (W-1) phi / W per worker."""
    W, n = 8, 8 * 8 * 512
    rs, _ = oracle.ring_traffic(n, W)
    reps = [np.zeros(n, np.uint16) for _ in range(W)]
    ag, _ = oracle.ring_all_gather(reps, n // W)
    per_worker = rs[0] + 2 * ag[0]
    assert per_worker == 3 * (W - 1) * n // W
    ddp = 2 * (W - 1) * n // W
    assert per_worker / ddp == 1.5
