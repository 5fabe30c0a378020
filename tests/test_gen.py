"""Pins of the synthetic input generator (inputs only; shared by the oracle tests and the CUDA path)."""
import numpy as np
import pytest
import torch

import zrgen
from conftest import read_golden


def test_philox_known_answers():
    for row in read_golden("philox4x32_10_kat.txt"):
        vals = [int(x, 16) for x in row]
        assert zrgen.philox(vals[0:4], vals[4:6]) == vals[6:10]


def test_normal_table():
    from scipy.special import ndtri
    t = zrgen.normal_table().astype(np.float64)
    assert np.all(np.diff(t) > 0)
    assert np.array_equal(t[::-1], -t)
    q = ndtri((np.arange(65536) + 0.5) / 65536.0)
    assert np.all(np.abs(t - q) <= np.spacing(np.abs(q).astype(np.float32)))
    assert abs(t.mean()) < 1e-12 and abs(t.std() - 1.0) < 1e-4


def test_fill_is_counter_based():
    seed, stream = 5, zrgen.stream_id(zrgen.TAG_GRAD, 2, 3, 4)
    full = zrgen.fill_host(1000, zrgen.BF16, seed, stream, 0, 0.5)
    for first, n in ((0, 1), (3, 17), (8, 8), (13, 987), (999, 1)):
        part = zrgen.fill_host(n, zrgen.BF16, seed, stream, first, 0.5)
        assert np.array_equal(part, full[first:first + n])
    for i in (0, 7, 8, 555):
        u = zrgen.host().zrgen_u16(seed, stream, i)
        want = zrgen.f32_to_bf16(np.float32(zrgen.normal_table()[u] * np.float32(0.5)))
        assert full[i] == want
    other = zrgen.fill_host(1000, zrgen.BF16, seed, stream + 1, 0, 0.5)
    assert not np.array_equal(other, full)


@pytest.mark.parametrize("dt,tdt,fn", [(zrgen.F16, torch.float16, zrgen.f32_to_f16),
                                       (zrgen.BF16, torch.bfloat16, zrgen.f32_to_bf16)])
def test_generator_rounding_matches_torch(dt, tdt, fn):
    x = (zrgen.fill_host(20000, zrgen.F32, 1, 9, 0, 1.0) *
         np.repeat(np.float32([1e-7, 1e-5, 1.0, 300.0, 65000.0]), 4000)).astype(np.float32)
    ours = zrgen.fill_host(20000, dt, 1, 9, 0, 1.0)
    base = zrgen.fill_host(20000, zrgen.F32, 1, 9, 0, 1.0)
    assert np.array_equal(ours, torch.from_numpy(base).to(tdt).view(torch.int16).numpy().view(np.uint16))
    bits = torch.from_numpy(x).to(tdt).view(torch.int16).numpy().view(np.uint16)
    assert all(fn(float(a)) == int(b) for a, b in zip(x[::37], bits[::37]))


def test_workload_shapes_and_sigmas():
    assert zrgen.workload("tiny").n == 786_432
    assert zrgen.workload("gpt2").n == 123_586_560
    assert zrgen.workload("1p3b").n == 1_311_080_448
    assert zrgen.workload("7b").n == 7_000_000_000
    assert len(zrgen.sweep_workloads()) == 30
    s = zrgen.sigma_per_tensor(zrgen.workload("1p3b"))
    assert s.dtype == np.float32 and np.all(s >= np.float32(1e-4)) and np.all(s <= np.float32(1e-1))
    assert np.array_equal(s, zrgen.sigma_per_tensor(zrgen.workload("1p3b")))
    w, t, i = zrgen.inject_site(zrgen.workload("7b"), 3)
    assert 0 <= w < 2 and 0 <= t < 35 and 0 <= i < 200_000_000
    assert zrgen.inject_site(zrgen.workload("7b"), 2) is None
