"""zrgen: seeded, counter-based synthetic inputs shared by the oracle tests and the CUDA path.

Inputs only. Nothing here reduces, scales or updates anything: it draws gradient
replicas, fp32 masters and per-tensor sigmas, and describes the workloads (tensor
shape lists and step settings) of the ZeRO post-backward step. Values are defined
in ``zrgen.h``; the host fill (plain C) and the device fill (CUDA) give equal bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libzrgen_host.so")
DEV_LIB = os.path.join(_HERE, "libzrgen_dev.so")

F16, BF16, F32 = 0, 1, 2
NP_DTYPE = {F16: np.uint16, BF16: np.uint16, F32: np.float32}

# stream tags (top byte of the 64-bit Philox stream id)
TAG_GRAD, TAG_MASTER, TAG_SIGMA, TAG_INJECT = 1, 2, 3, 4

_lock = threading.Lock()
_host = None
_dev = None
_table = None


def _newer(target, sources):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(s) <= t for s in sources)


def build_host(force: bool = False) -> str:
    srcs = [os.path.join(_HERE, "zrgen_host.c"), os.path.join(_HERE, "zrgen.h")]
    if force or not _newer(HOST_LIB, srcs):
        tmp = HOST_LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                               srcs[0], "-lm", "-o", tmp])
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_dev(force: bool = False, arch: str = "103a") -> str:
    srcs = [os.path.join(_HERE, "zrgen_dev.cu"), os.path.join(_HERE, "zrgen.h")]
    if force or not _newer(DEV_LIB, srcs):
        tmp = DEV_LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["nvcc", f"-gencode=arch=compute_{arch},code=sm_{arch}", "-O3", "-lineinfo",
                               "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
                               srcs[0], "-o", tmp])
        os.replace(tmp, DEV_LIB)
    return DEV_LIB


def host():
    global _host
    with _lock:
        if _host is None:
            if not os.path.exists(HOST_LIB):
                build_host()
            lib = ctypes.CDLL(HOST_LIB)
            u32p = ctypes.POINTER(ctypes.c_uint32)
            lib.zrgen_philox4x32_10.argtypes = [u32p, u32p, u32p]
            lib.zrgen_philox4x32_10.restype = None
            lib.zrgen_normal_table.argtypes = [ctypes.c_void_p]
            lib.zrgen_normal_table.restype = None
            lib.zrgen_u16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.zrgen_u16.restype = ctypes.c_uint16
            lib.zrgen_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int]
            lib.zrgen_uniform.restype = ctypes.c_double
            lib.zrgen_fill_normal_host.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                                   ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p]
            lib.zrgen_fill_normal_host.restype = ctypes.c_int
            lib.zrgen_f32_to_f16.argtypes = [ctypes.c_float]
            lib.zrgen_f32_to_f16.restype = ctypes.c_uint16
            lib.zrgen_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.zrgen_f32_to_bf16.restype = ctypes.c_uint16
            _host = lib
    return _host


def dev():
    global _dev
    with _lock:
        if _dev is None:
            if not os.path.exists(DEV_LIB):
                raise RuntimeError(f"zrgen device library missing: {DEV_LIB} (run __graft_entry__.build())")
            lib = ctypes.CDLL(DEV_LIB)
            lib.zrgen_fill_normal_dev.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                                  ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p,
                                                  ctypes.c_void_p]
            lib.zrgen_fill_normal_dev.restype = ctypes.c_int
            _dev = lib
    return _dev


def philox(ctr, key):
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    host().zrgen_philox4x32_10(c, k, o)
    return [int(x) for x in o]


def normal_table() -> np.ndarray:
    global _table
    if _table is None:
        t = np.empty(65536, dtype=np.float32)
        host().zrgen_normal_table(t.ctypes.data)
        t.setflags(write=False)
        _table = t
    return _table


def stream_id(tag: int, step: int = 0, replica: int = 0, tensor: int = 0) -> int:
    assert 0 <= tag < 256 and 0 <= step < 65536 and 0 <= replica < 65536 and 0 <= tensor < (1 << 24)
    return (tag << 56) | (step << 40) | (replica << 24) | tensor


def fill_host(n: int, dtype: int, seed: int, stream: int, first: int, scale) -> np.ndarray:
    out = np.empty(int(n), dtype=NP_DTYPE[dtype])
    if n:
        rc = host().zrgen_fill_normal_host(out.ctypes.data, dtype, int(n), int(seed), int(stream), int(first),
                                           float(np.float32(scale)), normal_table().ctypes.data)
        assert rc == 0
    return out


def fill_dev(ptr: int, n: int, dtype: int, seed: int, stream: int, first: int, scale, table_dev_ptr: int,
             cuda_stream: int) -> None:
    rc = dev().zrgen_fill_normal_dev(ctypes.c_void_p(ptr), dtype, int(n), int(seed), int(stream), int(first),
                                     float(np.float32(scale)), ctypes.c_void_p(table_dev_ptr),
                                     ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"zrgen_fill_normal_dev failed rc={rc}")


def uniform(seed: int, stream: int, block: int = 0, word: int = 0) -> float:
    return float(host().zrgen_uniform(int(seed), int(stream), int(block), int(word)))


def u64(seed: int, stream: int, block: int = 0) -> int:
    o = philox([block & 0xFFFFFFFF, block >> 32, stream & 0xFFFFFFFF, stream >> 32],
               [seed & 0xFFFFFFFF, seed >> 32])
    return (o[0] << 32) | o[1]


def f32_to_f16(x) -> int:
    return int(host().zrgen_f32_to_f16(float(np.float32(x))))


def f32_to_bf16(x) -> int:
    return int(host().zrgen_f32_to_bf16(float(np.float32(x))))


from .workloads import *  # noqa: E402,F401,F403
