"""zr_step_noalloc, the fused step for callers that cannot allocate device memory, against zr_step.

Such callers (a runtime that hands out all device memory from its own pool, a fixed memory budget,
a path where an allocation would synchronise the device) cannot create a plan, which allocates a
tile table and a control block; zr_step_noalloc keeps that scratch in a static device array of the
library instead. This file runs last (its name sorts last) and stands alone: it builds the library,
creates its own inputs, and calls the entry point through the C ABI twice in a row, comparing each
call's output with what the plan-based zr_step produces from the same inputs.
"""
import ctypes
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


def _ulps_f32(a, b):
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return int(np.max(np.abs(ia - ib)))


def _ulps_16(a, b):
    ia = np.asarray(a, np.uint16).astype(np.int64)
    ib = np.asarray(b, np.uint16).astype(np.int64)
    ia = np.where(ia & 0x8000, -(ia & 0x7FFF), ia)
    ib = np.where(ib & 0x8000, -(ib & 0x7FFF), ib)
    return int(np.max(np.abs(ia - ib)))


def test_noalloc_matches_zr_step_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import zero_gradient_reduction_gb300 as zr
    import zrgen
    from zrgen.layout import Layout

    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    numels = [50_000, 777, 123_457, 9_000, 64]
    W, A, dtype, S = 4, 2, zr.BF16, 1.0
    order = [2, 0, 3, 1]
    hyper = zr.AdamW()
    plan = zr.Plan(numels, W=W, A=A, dtype=dtype, stage=2, cap=60_000, order=order, scaler=zr.Scaler(S))
    assert len(plan.buckets) >= 3
    layout = Layout(numels, plan.tensor_offsets, np.full(len(numels), 1e-2, np.float32), 7, dtype)
    table = torch.from_numpy(zrgen.normal_table().copy()).to(dev)
    cs = torch.cuda.current_stream().cuda_stream
    n = plan.numel

    ref = plan.new_state(dev)      # state driven by zr_step (plan)
    nal = plan.new_state(dev)      # state driven by zr_step_noalloc
    for st in (ref, nal):
        st.master[0].zero_()
        layout.master_dev(st.master[0], table, cs)
        st.param[0].copy_(st.master[0].to(torch.bfloat16))
    grads = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(W * A)]

    # the C-ABI entry point, called directly
    fn = zr.lib().zr_step_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.POINTER(zr.StateC), ctypes.c_int, ctypes.POINTER(zr.Hyper),
                   ctypes.c_float, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    btab = (zr.Bucket * len(plan.buckets))(*[zr.Bucket(int(s), int(l), int(c)) for s, l, c in plan.buckets])
    ordc = (ctypes.c_int * W)(*order)
    overflow = torch.full((1,), 7, dtype=torch.int32, device=dev)
    current = 0
    for step in (1, 2):
        for r in range(W * A):
            layout.grads_dev(grads[r], step, r, S, table, cs)
        rep = plan.step(grads, ref, hyper, report=True)
        assert rep.overflow == 0 and rep.t == step

        gptr = (ctypes.c_void_p * (W * A))(*[g.data_ptr() for g in grads])
        stc = nal.c()
        h = hyper.c()
        rc = fn(ctypes.addressof(btab), len(plan.buckets), W, A, dtype, ctypes.addressof(ordc),
                ctypes.addressof(gptr), ctypes.byref(stc), current, ctypes.byref(h), S, step,
                overflow.data_ptr(), cs)
        assert rc == 0, zr.lib().zr_last_error()
        torch.cuda.synchronize()
        assert int(overflow.item()) == 0
        current = 1 - current  # clean step: the written set becomes live

        want = ref.live(rep.current)
        got = nal.live(current)
        for name in ("master", "m", "v"):
            d = _ulps_f32(got[name].cpu().numpy(), want[name].cpu().numpy())
            assert d <= 2, f"call {step}: {name} differs by {d} ulp"
        d = _ulps_16(got["param"].cpu().view(torch.int16).numpy().view(np.uint16),
                     want["param"].cpu().view(torch.int16).numpy().view(np.uint16))
        assert d <= 1, f"call {step}: param differs by {d} ulp"

    # sizes beyond the static scratch are refused with a clear error, launching nothing
    huge = (zr.Bucket * 1)(zr.Bucket(0, 8 * 8192 * 70_000, zr.chunk_size(8 * 8192 * 70_000, 8)))
    gptr = (ctypes.c_void_p * 8)(*[grads[0].data_ptr()] * 8)
    stc = nal.c()
    rc = fn(ctypes.addressof(huge), 1, 8, 1, dtype, None, ctypes.addressof(gptr), ctypes.byref(stc), 0,
            ctypes.byref(h), S, 3, overflow.data_ptr(), cs)
    assert rc == 1 and b"static scratch limit" in zr.lib().zr_last_error()
    plan.close()
