"""TEST INFRASTRUCTURE — Python access to the CPU oracle (zr_oracle.c) of the ZeRO post-backward step.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
may import this package. It shares no code with the CUDA path (the product never imports it).
The arithmetic lives in the C file; this module only builds it, marshals numpy arrays and
keeps the loss-scaler record between steps.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "liboracle.so")
SRC = [os.path.join(_HERE, "zr_oracle.c"), os.path.join(_HERE, "zr_oracle.h")]
MAX_W = 64
F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle: -O2 with FMA contraction off and no fast-math (every float op rounds once)."""
    fresh = os.path.exists(LIB) and all(os.path.getmtime(s) <= os.path.getmtime(LIB) for s in SRC)
    if force or not fresh:
        tmp = LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", SRC[0], "-lm", "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


class Bucket(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int64), ("len", ctypes.c_int64), ("chunk", ctypes.c_int64)]


class Hyper(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class Scaler(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("good", ctypes.c_int64), ("t", ctypes.c_int64),
                ("prod1", ctypes.c_double), ("prod2", ctypes.c_double), ("backoff", ctypes.c_float),
                ("growth", ctypes.c_float), ("min_scale", ctypes.c_float), ("interval", ctypes.c_int64),
                ("dynamic", ctypes.c_int)]


class Report(ctypes.Structure):
    _fields_ = [("overflow", ctypes.c_int), ("skipped", ctypes.c_int), ("scale_used", ctypes.c_float),
                ("scale_next", ctypes.c_float), ("t_after", ctypes.c_int64),
                ("rs_sent", ctypes.c_int64 * MAX_W), ("rs_recv", ctypes.c_int64 * MAX_W),
                ("ag_sent", ctypes.c_int64 * MAX_W), ("ag_recv", ctypes.c_int64 * MAX_W)]


_lock = threading.Lock()
_lib = None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            vp, i64 = ctypes.c_void_p, ctypes.c_int64
            L.zro_chunk_size.argtypes = [i64, ctypes.c_int, ctypes.c_int]
            L.zro_chunk_size.restype = i64
            L.zro_bucket_plan.argtypes = [vp, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int, vp,
                                          ctypes.POINTER(ctypes.c_int), vp]
            L.zro_bucket_plan.restype = ctypes.c_int
            for nm in ("zro_f16_to_f32", "zro_bf16_to_f32"):
                getattr(L, nm).argtypes = [ctypes.c_uint16]
                getattr(L, nm).restype = ctypes.c_float
            for nm in ("zro_f32_to_f16", "zro_f32_to_bf16"):
                getattr(L, nm).argtypes = [ctypes.c_float]
                getattr(L, nm).restype = ctypes.c_uint16
            L.zro_decode.argtypes = [ctypes.c_int, vp, vp, i64]
            L.zro_decode.restype = None
            L.zro_encode.argtypes = [ctypes.c_int, vp, vp, i64]
            L.zro_encode.restype = None
            L.zro_accumulate.argtypes = [ctypes.c_int, vp, vp, i64, ctypes.c_int]
            L.zro_accumulate.restype = None
            L.zro_shard_params.argtypes = [ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
            L.zro_shard_params.restype = None
            L.zro_param_all_gather.argtypes = [ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, vp,
                                               vp]
            L.zro_param_all_gather.restype = ctypes.c_int
            L.zro_ring_reduce_scatter.argtypes = [ctypes.c_int, i64, i64, vp, vp, vp, vp]
            L.zro_ring_reduce_scatter.restype = None
            L.zro_ring_all_gather.argtypes = [ctypes.c_int, i64, i64, vp, vp, vp, vp]
            L.zro_ring_all_gather.restype = None
            L.zro_ring_all_reduce.argtypes = [ctypes.c_int, i64, i64, vp, vp, vp, vp]
            L.zro_ring_all_reduce.restype = None
            L.zro_ring_reduce_scatter_hops.argtypes = [ctypes.c_int, i64, i64, vp, vp, vp, vp, ctypes.c_int,
                                                       ctypes.c_int]
            L.zro_ring_reduce_scatter_hops.restype = None
            L.zro_ring_all_gather_hops.argtypes = [ctypes.c_int, i64, i64, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int]
            L.zro_ring_all_gather_hops.restype = None
            L.zro_ring_traffic.argtypes = [i64, ctypes.c_int, ctypes.c_int, vp, vp]
            L.zro_ring_traffic.restype = None
            L.zro_unscale_factor.argtypes = [ctypes.c_float, ctypes.c_int]
            L.zro_unscale_factor.restype = ctypes.c_float
            L.zro_bias_correction.argtypes = [ctypes.c_float, i64]
            L.zro_bias_correction.restype = ctypes.c_float
            L.zro_adamw.argtypes = [i64, vp, vp, vp, vp, ctypes.POINTER(Hyper), ctypes.c_float, ctypes.c_float]
            L.zro_adamw.restype = None
            L.zro_step.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp, vp, vp,
                                   vp, ctypes.POINTER(Hyper), ctypes.POINTER(Scaler), ctypes.c_int, vp,
                                   ctypes.POINTER(Report)]
            L.zro_step.restype = ctypes.c_int
            L.zro_model_state_bytes.argtypes = [ctypes.c_int, i64, ctypes.c_int]
            L.zro_model_state_bytes.restype = i64
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- layout
def chunk_size(n: int, W: int, align: int = 8) -> int:
    return int(lib().zro_chunk_size(int(n), int(W), int(align)))


def bucket_plan(numels: Sequence[int], cap: int, W: int, align: int = 8):
    """Returns (buckets: int64 array [nb, 3] of (start, len, chunk), tensor_offset: int64 array)."""
    nt = len(numels)
    num = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    bk = (Bucket * max(nt, 1))()
    off = np.zeros(max(nt, 1), dtype=np.int64)
    nb = ctypes.c_int(0)
    rc = lib().zro_bucket_plan(_ptr(num) if nt else None, nt, int(cap), int(W), int(align), ctypes.addressof(bk),
                               ctypes.byref(nb), _ptr(off))
    if rc != 0:
        raise ValueError(f"zro_bucket_plan rc={rc}")
    out = np.array([[bk[i].start, bk[i].len, bk[i].chunk] for i in range(nb.value)], dtype=np.int64).reshape(-1, 3)
    return out, off[:nt]


def _buckets_struct(buckets: np.ndarray):
    b = np.asarray(buckets, dtype=np.int64).reshape(-1, 3)
    arr = (Bucket * max(len(b), 1))()
    for i, (s, n, c) in enumerate(b):
        arr[i].start, arr[i].len, arr[i].chunk = int(s), int(n), int(c)
    return arr, len(b)


# ---------------------------------------------------------------- formats
def decode(dtype: int, bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    lib().zro_decode(dtype, _ptr(bits), _ptr(out), bits.size)
    return out


def encode(dtype: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().zro_encode(dtype, _ptr(x), _ptr(out), x.size)
    return out


def accumulate(dtype: int, g: np.ndarray, acc: np.ndarray, first: bool) -> None:
    """In place: acc = fp32(g) if first else acc + fp32(g)."""
    g = np.ascontiguousarray(g, dtype=np.uint16)
    assert acc.dtype == np.float32 and acc.flags["C_CONTIGUOUS"] and acc.size == g.size
    lib().zro_accumulate(dtype, _ptr(g), _ptr(acc), g.size, 1 if first else 0)


# ---------------------------------------------------------------- ring
def ring_reduce_scatter(work: List[np.ndarray], C: int, hops: Optional[range] = None):
    """In place on the W fp32 position arrays; returns (sent, recv) element counts per position.

    hops: the hop range to run (default: all W-1 hops)."""
    W = len(work)
    n = work[0].size
    for w in work:
        assert w.dtype == np.float32 and w.size == n
    ptrs = (ctypes.c_void_p * W)(*[_ptr(w) for w in work])
    msg = np.empty(max(W * C, 1), dtype=np.float32)
    sent = np.zeros(W, dtype=np.int64)
    recv = np.zeros(W, dtype=np.int64)
    if hops is None:
        lib().zro_ring_reduce_scatter(W, n, int(C), ctypes.addressof(ptrs), _ptr(msg), _ptr(sent), _ptr(recv))
    else:
        lib().zro_ring_reduce_scatter_hops(W, n, int(C), ctypes.addressof(ptrs), _ptr(msg), _ptr(sent), _ptr(recv),
                                           hops.start, hops.stop)
    return sent, recv


def ring_all_gather(reps: List[np.ndarray], C: int, hops: Optional[range] = None):
    W = len(reps)
    n = reps[0].size
    for r in reps:
        assert r.dtype == np.uint16 and r.size == n
    ptrs = (ctypes.c_void_p * W)(*[_ptr(r) for r in reps])
    msg = np.empty(max(W * C, 1), dtype=np.uint16)
    sent = np.zeros(W, dtype=np.int64)
    recv = np.zeros(W, dtype=np.int64)
    if hops is None:
        lib().zro_ring_all_gather(W, n, int(C), ctypes.addressof(ptrs), _ptr(msg), _ptr(sent), _ptr(recv))
    else:
        lib().zro_ring_all_gather_hops(W, n, int(C), ctypes.addressof(ptrs), _ptr(msg), _ptr(sent), _ptr(recv),
                                       hops.start, hops.stop)
    return sent, recv


def ring_all_reduce(work: List[np.ndarray], C: int):
    """In place on the W fp32 position arrays (reduce-scatter hops, then all-gather hops of the reduced
    blocks); returns (sent, recv) element counts per position over both phases."""
    W = len(work)
    n = work[0].size
    for w in work:
        assert w.dtype == np.float32 and w.size == n
    ptrs = (ctypes.c_void_p * W)(*[_ptr(w) for w in work])
    msg = np.empty(max(W * C, 1), dtype=np.float32)
    sent = np.zeros(W, dtype=np.int64)
    recv = np.zeros(W, dtype=np.int64)
    lib().zro_ring_all_reduce(W, n, int(C), ctypes.addressof(ptrs), _ptr(msg), _ptr(sent), _ptr(recv))
    return sent, recv


def shard_sizes(buckets: np.ndarray, W: int, order: Optional[Sequence[int]] = None) -> List[int]:
    """Elements of each worker's ZeRO-3 shard: the sum of its owned block over the buckets."""
    order = list(order) if order is not None else list(range(W))
    sizes = [0] * W
    for _, n, C in np.asarray(buckets).reshape(-1, 3):
        for p in range(W):
            c = (p + 1) % W
            sizes[order[p]] += max(0, min(int(n), (c + 1) * int(C)) - min(int(n), c * int(C)))
    return sizes


def shard_params(W: int, buckets: np.ndarray, replica: np.ndarray, order: Optional[Sequence[int]] = None):
    """Per-worker ZeRO-3 shards of a full 16-bit replica (list indexed by worker id)."""
    shards = [np.zeros(max(s, 1), np.uint16) for s in shard_sizes(buckets, W, order)]
    bk, nb = _buckets_struct(buckets)
    ordc = (ctypes.c_int * W)(*(order if order is not None else range(W)))
    ptrs = (ctypes.c_void_p * W)(*[_ptr(s) for s in shards])
    rep = np.ascontiguousarray(replica, dtype=np.uint16)
    lib().zro_shard_params(W, ctypes.addressof(ordc), nb, ctypes.addressof(bk), _ptr(rep), ctypes.addressof(ptrs))
    return shards


def param_all_gather(W: int, buckets: np.ndarray, shards: List[np.ndarray], replica: np.ndarray, b_lo: int, b_hi: int,
                     order: Optional[Sequence[int]] = None) -> None:
    """In place on `replica`: the ring all-gather of buckets [b_lo, b_hi) from the shards."""
    bk, nb = _buckets_struct(buckets)
    ordc = (ctypes.c_int * W)(*(order if order is not None else range(W)))
    ptrs = (ctypes.c_void_p * W)(*[_ptr(s) for s in shards])
    assert replica.dtype == np.uint16 and replica.flags["C_CONTIGUOUS"]
    rc = lib().zro_param_all_gather(W, ctypes.addressof(ordc), nb, ctypes.addressof(bk), int(b_lo), int(b_hi),
                                    ctypes.addressof(ptrs), _ptr(replica))
    if rc != 0:
        raise RuntimeError(f"zro_param_all_gather rc={rc}")


def ring_traffic(n: int, W: int, align: int = 8):
    sent = np.zeros(W, dtype=np.int64)
    recv = np.zeros(W, dtype=np.int64)
    lib().zro_ring_traffic(int(n), int(W), int(align), _ptr(sent), _ptr(recv))
    return sent, recv


# ---------------------------------------------------------------- optimizer
@dataclasses.dataclass
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    def c(self) -> Hyper:
        return Hyper(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


def unscale_factor(scale: float, W: int) -> np.float32:
    return np.float32(lib().zro_unscale_factor(float(scale), int(W)))


def bias_correction(beta: float, t: int) -> np.float32:
    return np.float32(lib().zro_bias_correction(float(beta), int(t)))


def adamw(g, p, m, v, hyper: AdamW, bc1, bc2) -> None:
    """In-place AdamW on fp32 arrays p, m, v with unscaled fp32 gradient g."""
    for a in (g, p, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    h = hyper.c()
    lib().zro_adamw(g.size, _ptr(g), _ptr(p), _ptr(m), _ptr(v), ctypes.byref(h), float(bc1), float(bc2))


def model_state_bytes(stage: int, n: int, W: int) -> int:
    return int(lib().zro_model_state_bytes(int(stage), int(n), int(W)))


# ---------------------------------------------------------------- step
def new_scaler(init_scale: float = 1.0, dynamic: bool = False, backoff: float = 0.5, growth: float = 2.0,
               min_scale: float = 1.0, interval: int = 1000) -> Scaler:
    return Scaler(float(init_scale), 0, 0, 1.0, 1.0, float(backoff), float(growth), float(min_scale),
                  int(interval), 1 if dynamic else 0)


def step(W: int, A: int, dtype: int, buckets: np.ndarray, grads: Sequence[np.ndarray], master: np.ndarray,
         m: np.ndarray, v: np.ndarray, param: np.ndarray, hyper: AdamW, scaler: Scaler,
         order: Optional[Sequence[int]] = None, flag_override: int = -1, want_sums: bool = False):
    """One oracle step in place on master/m/v/param; returns (Report, sums or None)."""
    assert len(grads) == W * A
    for g in grads:
        assert g.dtype == np.uint16 and g.flags["C_CONTIGUOUS"]
    total = int(max((s + n for s, n, _ in np.asarray(buckets).reshape(-1, 3)), default=0))
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.size >= total
    assert param.dtype == np.uint16 and param.size >= total
    bk, nb = _buckets_struct(buckets)
    gp = (ctypes.c_void_p * (W * A))(*[_ptr(g) for g in grads])
    ordc = (ctypes.c_int * W)(*(order if order is not None else range(W)))
    sums = np.zeros(max(total, 1), dtype=np.float32) if want_sums else None
    rep = Report()
    h = hyper.c()
    rc = lib().zro_step(W, A, dtype, ctypes.addressof(ordc), nb, ctypes.addressof(bk), ctypes.addressof(gp),
                        _ptr(master), _ptr(m), _ptr(v), _ptr(param), ctypes.byref(h), ctypes.byref(scaler),
                        int(flag_override), _ptr(sums) if sums is not None else None, ctypes.byref(rep))
    if rc != 0:
        raise RuntimeError(f"zro_step rc={rc}")
    return rep, (sums[:total] if sums is not None else None)
