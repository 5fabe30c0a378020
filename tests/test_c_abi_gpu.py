"""The C ABI used from plain C: tests/c_abi_step.c includes only zr.h and the CUDA runtime, allocates with
cudaMalloc and runs three fused steps through libzr.so (the plan's staging, bulk-copy staging, and
zr_step_noalloc), checking each result against its closed form."""
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "zero_gradient_reduction_gb300")


def test_plain_c_program_runs_a_step():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    out_dir = os.path.join(PKG, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "c_abi_step")
    cmd = ["nvcc", "-O2", "-cudart", "shared", os.path.join(ROOT, "tests", "c_abi_step.c"), "-o", exe,
           f"-I{os.path.join(ROOT, 'include')}", f"-L{PKG}", "-lzr", "-Xlinker", f"-rpath,{PKG}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
