"""Python binding of libzr, the GB300-native post-backward ZeRO step (C ABI in include/zr.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.
PyTorch supplies device memory and streams. If libzr.so is missing this module raises
on import of the library (there is no fallback of any kind).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzr.so")

F16, BF16, F32 = 0, 1, 2
STAGING_REGISTERS, STAGING_BULK, STAGING_BULK_IO = 0, 1, 2  # zr_staging
MAX_W, MAX_REPLICAS, ALIGN = 64, 256, 8
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "out of memory", 5: "timeout"}


class ZrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Bucket(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int64), ("len", ctypes.c_int64), ("chunk", ctypes.c_int64)]


class Hyper(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class ScalerCfg(ctypes.Structure):
    _fields_ = [("init_scale", ctypes.c_float), ("backoff", ctypes.c_float), ("growth", ctypes.c_float),
                ("min_scale", ctypes.c_float), ("growth_interval", ctypes.c_int32), ("dynamic", ctypes.c_int32)]


class PlanDesc(ctypes.Structure):
    _fields_ = [("W", ctypes.c_int32), ("A", ctypes.c_int32), ("dtype", ctypes.c_int), ("stage", ctypes.c_int32),
                ("align", ctypes.c_int32), ("cap", ctypes.c_int64), ("ntensors", ctypes.c_int32),
                ("numels", ctypes.POINTER(ctypes.c_int64)), ("order", ctypes.POINTER(ctypes.c_int32)),
                ("scaler", ScalerCfg), ("fp32_grads", ctypes.c_int32)]


class StateC(ctypes.Structure):
    _fields_ = [("master", ctypes.c_void_p * 2), ("m", ctypes.c_void_p * 2), ("v", ctypes.c_void_p * 2),
                ("param", ctypes.c_void_p * 2)]


class StateC1(ctypes.Structure):
    _fields_ = [("master", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("param", ctypes.c_void_p)]


class Checkpoint(ctypes.Structure):
    _fields_ = [("current", ctypes.c_int32), ("scale", ctypes.c_float), ("good", ctypes.c_int64),
                ("t", ctypes.c_int64), ("steps", ctypes.c_int64), ("skipped", ctypes.c_int64),
                ("beta1_pow", ctypes.c_double), ("beta2_pow", ctypes.c_double)]


class StepReport(ctypes.Structure):
    _fields_ = [("overflow", ctypes.c_int32), ("skipped", ctypes.c_int32), ("current", ctypes.c_int32),
                ("stage", ctypes.c_int32), ("scale_used", ctypes.c_float), ("scale", ctypes.c_float),
                ("t", ctypes.c_int64), ("steps", ctypes.c_int64), ("skipped_total", ctypes.c_int64),
                ("good", ctypes.c_int64), ("n_real", ctypes.c_int64), ("bytes_alg", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded libzr (ctypes). Raises if the library has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libzr.so not found at {LIB_PATH}; build it with __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int
            sig = {
                "zr_chunk_size": (i64, [i64, i32, i32]),
                "zr_bucket_plan": (st, [vp, i32, i64, i32, i32, vp, ctypes.POINTER(ctypes.c_int), vp]),
                "zr_reduce_scatter": (st, [vp, i32, i64, i32, vp, vp, vp, vp]),
                "zr_adamw_shard_step": (st, [vp, vp, vp, vp, i64, ctypes.POINTER(Hyper), ctypes.c_float, i32, i64,
                                             vp, vp]),
                "zr_all_gather": (st, [vp, i64, i32, vp, i32, vp]),
                "zr_all_reduce": (st, [vp, i32, i64, i32, vp, vp, i32, vp, vp]),
                "zr_accumulate": (st, [vp, i32, vp, i64, i32, vp]),
                "zr_step_bucket": (st, [vp, i32, i32, vp, ctypes.POINTER(StateC), ctypes.POINTER(Hyper), vp]),
                "zr_plan_set_bucket_blocks": (st, [vp, i32]),
                "zr_plan_set_staging": (st, [vp, i32, i32, i32]),
                "zr_plan_staging": (i32, [vp]),
                "zr_plan_stall_bulk_waits": (st, [vp, i32]),
                "zr_offload_adamw": (st, [vp, vp, vp, vp, vp, i32, i64, ctypes.POINTER(Hyper), ctypes.c_float, i32,
                                          i64, i32, ctypes.POINTER(ctypes.c_int32)]),
                "zr_offload_step": (st, [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(Hyper),
                                         ctypes.c_float, i64, i32, vp, ctypes.POINTER(ctypes.c_int32)]),
                "zr_plan_shard_numel": (i64, [vp, i32]),
                "zr_plan_shard_offset": (st, [vp, i32, i32, ctypes.POINTER(ctypes.c_int64)]),
                "zr_shard_params": (st, [vp, vp, vp, vp]),
                "zr_gather_params": (st, [vp, i32, i32, vp, vp, vp]),
                "zr_plan_create": (st, [ctypes.POINTER(PlanDesc), ctypes.POINTER(vp)]),
                "zr_plan_destroy": (st, [vp]),
                "zr_plan_numel": (i64, [vp]),
                "zr_plan_nbuckets": (ctypes.c_int32, [vp]),
                "zr_plan_buckets": (st, [vp, vp, vp]),
                "zr_plan_reset": (st, [vp, vp]),
                "zr_step": (st, [vp, i32, vp, ctypes.POINTER(StateC), ctypes.POINTER(Hyper), vp,
                                 ctypes.POINTER(StepReport)]),
                "zr_step_inplace": (st, [vp, i32, vp, ctypes.POINTER(StateC1), ctypes.POINTER(Hyper), vp,
                                         ctypes.POINTER(StepReport)]),
                "zr_step_inplace_from_host": (st, [vp, i32, vp, vp, ctypes.POINTER(StateC1), ctypes.POINTER(Hyper),
                                                   vp, ctypes.POINTER(StepReport)]),
                "zr_step_from_host": (st, [vp, i32, vp, vp, ctypes.POINTER(StateC), ctypes.POINTER(Hyper), vp,
                                           ctypes.POINTER(StepReport)]),
                "zr_plan_report": (st, [vp, vp, ctypes.POINTER(StepReport)]),
                "zr_step_noalloc": (st, [vp, i32, i32, i32, i32, vp, vp, ctypes.POINTER(StateC), i32,
                                         ctypes.POINTER(Hyper), ctypes.c_float, i64, vp, vp]),
                "zr_plan_checkpoint": (st, [vp, vp, ctypes.POINTER(Checkpoint)]),
                "zr_plan_restore": (st, [vp, ctypes.POINTER(Checkpoint), vp]),
                "zr_model_state_bytes": (i64, [i32, i64, i32]),
                "zr_ring_traffic": (st, [i64, i32, i32, vp, vp, vp, vp]),
                "zr_status_str": (ctypes.c_char_p, [st]),
                "zr_last_error": (ctypes.c_char_p, []),
                "zr_version": (ctypes.c_char_p, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise ZrError(status, lib().zr_last_error().decode(errors="replace"))


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t) -> int:
    return int(t.data_ptr())


def _ptr_array(tensors) -> ctypes.Array:
    return (ctypes.c_void_p * len(tensors))(*[_ptr(t) for t in tensors])


def _host_ptr_array(arrays) -> ctypes.Array:
    ptrs = []
    for a in arrays:
        ptrs.append(a.ctypes.data if isinstance(a, np.ndarray) else int(a.data_ptr()))
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


# ----------------------------------------------------------------------------- layout and accounting
def chunk_size(n: int, W: int, align: int = ALIGN) -> int:
    return int(lib().zr_chunk_size(int(n), int(W), int(align)))


def bucket_plan(numels: Sequence[int], cap: int, W: int, align: int = ALIGN):
    """(buckets int64 [nb, 3] of (start, len, chunk), tensor_offsets int64 [ntensors])."""
    nt = len(numels)
    num = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    out = (Bucket * max(nt, 1))()
    offs = np.zeros(max(nt, 1), dtype=np.int64)
    nb = ctypes.c_int(0)
    _check(lib().zr_bucket_plan(num.ctypes.data if nt else None, nt, int(cap), int(W), int(align),
                                ctypes.addressof(out), ctypes.byref(nb), offs.ctypes.data))
    b = np.array([[out[i].start, out[i].len, out[i].chunk] for i in range(nb.value)], dtype=np.int64).reshape(-1, 3)
    return b, offs[:nt]


def model_state_bytes(stage: int, n: int, W: int) -> int:
    return int(lib().zr_model_state_bytes(int(stage), int(n), int(W)))


def ring_traffic(n: int, W: int, align: int = ALIGN):
    arrs = [np.zeros(W, dtype=np.int64) for _ in range(4)]
    _check(lib().zr_ring_traffic(int(n), int(W), int(align), *[a.ctypes.data for a in arrs]))
    return dict(zip(("rs_sent", "rs_recv", "ag_sent", "ag_recv"), arrs))


# ----------------------------------------------------------------------------- standalone collectives
@dataclasses.dataclass
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    def c(self) -> Hyper:
        return Hyper(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


def _dt_of(t) -> int:
    import torch
    return {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32}[t.dtype]


def reduce_scatter(grads: Sequence, sums, overflow, order: Optional[Sequence[int]] = None, n: Optional[int] = None,
                   stream=None) -> None:
    """Ring reduce-scatter of W device gradient tensors (fp16/bf16) into fp32 `sums` (see zr_reduce_scatter)."""
    W = len(grads)
    n = int(grads[0].numel()) if n is None else int(n)
    ordc = (ctypes.c_int * W)(*order) if order is not None else None
    arr = _ptr_array(grads)  # must outlive the call
    _check(lib().zr_reduce_scatter(ctypes.addressof(arr), _dt_of(grads[0]), n, W,
                                   ctypes.addressof(ordc) if ordc is not None else None, _ptr(sums), _ptr(overflow),
                                   _stream_handle(stream)))


def all_reduce(grads: Sequence, outs: Sequence, overflow, order: Optional[Sequence[int]] = None,
               n: Optional[int] = None, stream=None) -> None:
    """Ring all-reduce (zr_all_reduce): the ring sums of the W gradient replicas written to every fp32 output."""
    W = len(grads)
    n = int(grads[0].numel()) if n is None else int(n)
    arr = _ptr_array(grads)
    out = _ptr_array(outs)
    o = (ctypes.c_int * W)(*order) if order is not None else None
    _check(lib().zr_all_reduce(ctypes.addressof(arr), _dt_of(grads[0]), n, W,
                               ctypes.addressof(o) if o is not None else None, ctypes.addressof(out), len(outs),
                               _ptr(overflow), _stream_handle(stream)))


def adamw_shard_step(shard_sums, m, v, master, hyper: AdamW, loss_scale: float, W: int, t: int, overflow,
                     length: Optional[int] = None, stream=None) -> None:
    n = int(master.numel()) if length is None else int(length)
    h = hyper.c()
    _check(lib().zr_adamw_shard_step(_ptr(shard_sums), _ptr(m), _ptr(v), _ptr(master), n, ctypes.byref(h),
                                     float(loss_scale), int(W), int(t), _ptr(overflow), _stream_handle(stream)))


def accumulate(grad, acc, first: bool, n: Optional[int] = None, stream=None) -> None:
    """acc = fp32(grad) if first else acc + fp32(grad): one micro-batch of gradient accumulation (zr_accumulate)."""
    n = int(grad.numel()) if n is None else int(n)
    _check(lib().zr_accumulate(_ptr(grad), _dt_of(grad), _ptr(acc), n, 1 if first else 0, _stream_handle(stream)))


def _host_ptr(a) -> int:
    return a.ctypes.data if isinstance(a, np.ndarray) else int(a.data_ptr())


def offload_adamw(sums, master, m, v, param16, dtype: int, hyper: AdamW, loss_scale: float, W: int, t: int,
                  nthreads: int = 8) -> int:
    """ZeRO-Offload's host update (zr_offload_adamw) on host arrays (numpy or CPU tensors); returns the flag."""
    n = int(sums.size if isinstance(sums, np.ndarray) else sums.numel())
    h = hyper.c()
    of = ctypes.c_int32(0)
    _check(lib().zr_offload_adamw(_host_ptr(sums), _host_ptr(master), _host_ptr(m), _host_ptr(v),
                                  _host_ptr(param16) if param16 is not None else None, int(dtype), n, ctypes.byref(h),
                                  float(loss_scale), int(W), int(t), int(nthreads), ctypes.byref(of)))
    return int(of.value)


def all_gather(master, replicas: Sequence, n: Optional[int] = None, stream=None) -> None:
    n = int(master.numel()) if n is None else int(n)
    arr = _ptr_array(replicas)
    _check(lib().zr_all_gather(_ptr(master), n, _dt_of(replicas[0]), ctypes.addressof(arr), len(replicas),
                               _stream_handle(stream)))


# ----------------------------------------------------------------------------- fused step
@dataclasses.dataclass
class Scaler:
    init_scale: float = 1.0
    dynamic: bool = False
    backoff: float = 0.5
    growth: float = 2.0
    min_scale: float = 1.0
    growth_interval: int = 1000

    def c(self) -> ScalerCfg:
        return ScalerCfg(self.init_scale, self.backoff, self.growth, self.min_scale, self.growth_interval,
                         1 if self.dynamic else 0)


class State:
    """The two (ping-pong) sets of fp32 master/m/v and the 16-bit parameter replica, as torch tensors."""

    def __init__(self, numel: int, dtype, device="cuda"):
        import torch
        self.master = [torch.empty(numel, dtype=torch.float32, device=device) for _ in range(2)]
        self.m = [torch.zeros(numel, dtype=torch.float32, device=device) for _ in range(2)]
        self.v = [torch.zeros(numel, dtype=torch.float32, device=device) for _ in range(2)]
        self.param = [torch.empty(numel, dtype=dtype, device=device) for _ in range(2)]

    def c(self) -> StateC:
        s = StateC()
        for k in range(2):
            s.master[k] = _ptr(self.master[k])
            s.m[k] = _ptr(self.m[k])
            s.v[k] = _ptr(self.v[k])
            s.param[k] = _ptr(self.param[k])
        return s

    def live(self, k: int):
        return dict(master=self.master[k], m=self.m[k], v=self.v[k], param=self.param[k])


class State1:
    """ONE set of fp32 master/m/v and the 16-bit parameter replica (the in-place step), as torch tensors."""

    def __init__(self, numel: int, dtype, device="cuda"):
        import torch
        self.master = torch.empty(numel, dtype=torch.float32, device=device)
        self.m = torch.zeros(numel, dtype=torch.float32, device=device)
        self.v = torch.zeros(numel, dtype=torch.float32, device=device)
        self.param = torch.empty(numel, dtype=dtype, device=device)

    @classmethod
    def of(cls, master, m, v, param) -> "State1":
        """A State1 over existing tensors (e.g. one set of a State), with no allocation."""
        s = cls.__new__(cls)
        s.master, s.m, s.v, s.param = master, m, v, param
        return s

    def c(self) -> StateC1:
        return StateC1(_ptr(self.master), _ptr(self.m), _ptr(self.v), _ptr(self.param))

    def live(self, k: int = 0):
        return dict(master=self.master, m=self.m, v=self.v, param=self.param)


class Plan:
    """A bucketed ZeRO step over W emulated workers (zr_plan_create / zr_step); stage 0 is DDP, 1-3 ZeRO."""

    def __init__(self, numels: Sequence[int], W: int, A: int = 1, dtype: int = BF16, stage: int = 2,
                 cap: int = 25_000_000, order: Optional[Sequence[int]] = None, scaler: Scaler = Scaler(),
                 fp32_grads: bool = False):
        self._numels = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
        self._order = (ctypes.c_int32 * W)(*order) if order is not None else None
        d = PlanDesc()
        d.W, d.A, d.dtype, d.stage, d.align, d.cap = int(W), int(A), int(dtype), int(stage), ALIGN, int(cap)
        d.ntensors = len(self._numels)
        d.numels = self._numels.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        d.order = ctypes.cast(self._order, ctypes.POINTER(ctypes.c_int32)) if self._order is not None else None
        d.scaler = scaler.c()
        d.fp32_grads = 1 if fp32_grads else 0
        h = ctypes.c_void_p()
        _check(lib().zr_plan_create(ctypes.byref(d), ctypes.byref(h)))
        self._h = h
        self.W, self.A, self.dtype, self.stage = int(W), int(A), int(dtype), int(stage)
        self.fp32_grads = bool(fp32_grads)
        self.numel = int(lib().zr_plan_numel(h))
        nb = int(lib().zr_plan_nbuckets(h))
        b = (Bucket * max(nb, 1))()
        offs = np.zeros(len(self._numels), dtype=np.int64)
        _check(lib().zr_plan_buckets(h, ctypes.addressof(b), offs.ctypes.data))
        self.buckets = np.array([[b[i].start, b[i].len, b[i].chunk] for i in range(nb)], dtype=np.int64).reshape(-1, 3)
        self.tensor_offsets = offs
        self.n_real = int(self._numels.sum())

    @property
    def handle(self):
        return self._h

    def torch_dtype(self):
        """The parameter replica's torch dtype."""
        import torch
        return torch.float16 if self.dtype == F16 else torch.bfloat16

    def grad_torch_dtype(self):
        """The gradient replicas' torch dtype (fp32 for a plan over accumulated micro-batches)."""
        import torch
        return torch.float32 if self.fp32_grads else self.torch_dtype()

    def new_state(self, device="cuda") -> State:
        return State(self.numel, self.torch_dtype(), device)

    def step(self, grads: Sequence, state: State, hyper: AdamW, stage: Optional[int] = None, stream=None,
             report: bool = False):
        arr = _ptr_array(grads)
        st = state.c()
        h = hyper.c()
        rep = StepReport() if report else None
        _check(lib().zr_step(self._h, int(stage if stage is not None else self.stage), ctypes.addressof(arr),
                             ctypes.byref(st), ctypes.byref(h), _stream_handle(stream),
                             ctypes.byref(rep) if rep is not None else None))
        return rep

    def new_state1(self, device="cuda") -> State1:
        return State1(self.numel, self.torch_dtype(), device)

    def step_inplace(self, grads: Sequence, state: State1, hyper: AdamW, stage: Optional[int] = None, stream=None,
                     report: bool = False):
        """One step on a single state set, updated in place (zr_step_inplace): a flag pass, then the update."""
        arr = _ptr_array(grads)
        st = state.c()
        h = hyper.c()
        rep = StepReport() if report else None
        _check(lib().zr_step_inplace(self._h, int(stage if stage is not None else self.stage), ctypes.addressof(arr),
                                     ctypes.byref(st), ctypes.byref(h), _stream_handle(stream),
                                     ctypes.byref(rep) if rep is not None else None))
        return rep

    def step_inplace_from_host(self, host_grads: Sequence, dev_grads: Sequence, state: State1, hyper: AdamW,
                               stage: Optional[int] = None, stream=None) -> StepReport:
        """zr_step_inplace_from_host: host gradients copied into dev_grads, then the in-place step; report."""
        ha = _host_ptr_array(host_grads)
        da = _ptr_array(dev_grads)
        st = state.c()
        h = hyper.c()
        rep = StepReport()
        _check(lib().zr_step_inplace_from_host(self._h, int(stage if stage is not None else self.stage),
                                               ctypes.addressof(ha), ctypes.addressof(da), ctypes.byref(st),
                                               ctypes.byref(h), _stream_handle(stream), ctypes.byref(rep)))
        return rep

    def capture(self, grads: Sequence, state, hyper: AdamW, stage: Optional[int] = None, steps: int = 1):
        """A CUDA graph of `steps` fused steps on these buffers (torch.cuda.CUDAGraph; replay() runs them):
        ping-pong steps for a State, in-place steps for a State1. The step reads its live set, loss scale
        and t from device memory at run time, so replays keep stepping correctly; the graph keeps the buffer
        addresses it was captured with."""
        import torch
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=side):
            for _ in range(steps):
                if isinstance(state, State1):
                    self.step_inplace(grads, state, hyper, stage=stage, stream=side)
                else:
                    self.step(grads, state, hyper, stage=stage, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        return g

    def step_bucket(self, bucket: int, grads: Sequence, state: State, hyper: AdamW, stage: Optional[int] = None,
                    stream=None) -> None:
        """One bucket of a step (zr_step_bucket): call for buckets 0..nb-1 in order; the last commits."""
        arr = _ptr_array(grads)
        st = state.c()
        h = hyper.c()
        _check(lib().zr_step_bucket(self._h, int(stage if stage is not None else self.stage), int(bucket),
                                    ctypes.addressof(arr), ctypes.byref(st), ctypes.byref(h), _stream_handle(stream)))

    def set_staging(self, staging: int, stage_elems: int = 0, stages: int = 0) -> None:
        """zr_plan_set_staging: STAGING_BULK (the default where it applies) or STAGING_REGISTERS."""
        _check(lib().zr_plan_set_staging(self._h, int(staging), int(stage_elems), int(stages)))

    @property
    def staging(self) -> int:
        """The staging zr_step uses for this plan (zr_plan_staging)."""
        return int(lib().zr_plan_staging(self._h))

    def set_bucket_blocks(self, max_blocks: int) -> None:
        """Cap every zr_step_bucket launch at max_blocks thread blocks (0: no cap), between steps."""
        _check(lib().zr_plan_set_bucket_blocks(self._h, int(max_blocks)))

    def step_overlapped(self, grads: Sequence, state: State, hyper: AdamW, ready_events: Sequence, side_stream,
                        stage: Optional[int] = None) -> None:
        """Bucketed overlap with backward: ready_events[b] is recorded (on the compute stream) when bucket b's
        gradients exist; bucket b's step then runs on side_stream after that event, while backward continues."""
        assert len(ready_events) == len(self.buckets)
        for b, ev in enumerate(ready_events):
            side_stream.wait_event(ev)
            self.step_bucket(b, grads, state, hyper, stage=stage, stream=side_stream)

    def offload_step(self, grads: Sequence, sums_dev, sums_host, master, m, v, param_host, param_dev, hyper: AdamW,
                     loss_scale: float, t: int, nthreads: int = 8, stage: Optional[int] = None, stream=None) -> int:
        """ZeRO-Offload step (zr_offload_step): reduce-scatter on the GPU, AdamW on the host CPU over the host
        master/m/v, parameters copied back. Returns the overflow flag; the last copies are still queued."""
        arr = _ptr_array(grads)
        h = hyper.c()
        of = ctypes.c_int32(0)
        _check(lib().zr_offload_step(self._h, int(stage if stage is not None else self.stage), ctypes.addressof(arr),
                                     _ptr(sums_dev), _host_ptr(sums_host), _host_ptr(master), _host_ptr(m),
                                     _host_ptr(v), _host_ptr(param_host), _ptr(param_dev), ctypes.byref(h),
                                     float(loss_scale), int(t), int(nthreads), _stream_handle(stream),
                                     ctypes.byref(of)))
        return int(of.value)

    def step_from_host(self, host_grads: Sequence, dev_grads: Sequence, state: State, hyper: AdamW,
                       stage: Optional[int] = None, stream=None) -> StepReport:
        ha = _host_ptr_array(host_grads)
        da = _ptr_array(dev_grads)
        st = state.c()
        h = hyper.c()
        rep = StepReport()
        _check(lib().zr_step_from_host(self._h, int(stage if stage is not None else self.stage),
                                       ctypes.addressof(ha), ctypes.addressof(da), ctypes.byref(st), ctypes.byref(h),
                                       _stream_handle(stream), ctypes.byref(rep)))
        return rep

    def report(self, stream=None) -> StepReport:
        rep = StepReport()
        _check(lib().zr_plan_report(self._h, _stream_handle(stream), ctypes.byref(rep)))
        return rep

    # ---- ZeRO-3 parameter shards
    def shard_numel(self, worker: int) -> int:
        return int(lib().zr_plan_shard_numel(self._h, int(worker)))

    def shard_offset(self, bucket: int, worker: int) -> int:
        off = ctypes.c_int64()
        _check(lib().zr_plan_shard_offset(self._h, int(bucket), int(worker), ctypes.byref(off)))
        return int(off.value)

    def new_shards(self, device="cuda"):
        import torch
        return [torch.empty(max(self.shard_numel(w), 8), dtype=self.torch_dtype(), device=device)
                for w in range(self.W)]

    def shard_params(self, replica, shards: Sequence, stream=None) -> None:
        """Each worker keeps its owned blocks of the full replica (zr_shard_params)."""
        arr = _ptr_array(shards)
        _check(lib().zr_shard_params(self._h, _ptr(replica), ctypes.addressof(arr), _stream_handle(stream)))

    def gather_params(self, shards: Sequence, replica, bucket_lo: int = 0, bucket_hi: Optional[int] = None,
                      stream=None) -> None:
        """ZeRO-3 all-gather of buckets [bucket_lo, bucket_hi) into the transient replica (zr_gather_params)."""
        hi = len(self.buckets) if bucket_hi is None else int(bucket_hi)
        arr = _ptr_array(shards)
        _check(lib().zr_gather_params(self._h, int(bucket_lo), hi, ctypes.addressof(arr), _ptr(replica),
                                      _stream_handle(stream)))

    def checkpoint(self, stream=None) -> Checkpoint:
        """The control block's step state (live set, scale, t, ...); save the live state tensors with it."""
        c = Checkpoint()
        _check(lib().zr_plan_checkpoint(self._h, _stream_handle(stream), ctypes.byref(c)))
        return c

    def restore(self, ckpt: Checkpoint, stream=None) -> None:
        _check(lib().zr_plan_restore(self._h, ctypes.byref(ckpt), _stream_handle(stream)))

    def reset(self, stream=None) -> None:
        _check(lib().zr_plan_reset(self._h, _stream_handle(stream)))

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().zr_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def step_noalloc(buckets: np.ndarray, W: int, A: int, dtype: int, grads: Sequence, state: State, current: int,
                 hyper: AdamW, loss_scale: float, t: int, overflow, order: Optional[Sequence[int]] = None,
                 stream=None) -> None:
    """zr_step_noalloc: the fused step for callers that cannot allocate device memory (scratch lives in a
    static device array of the library; the caller carries the live set, the scale and t)."""
    fn = lib().zr_step_noalloc
    b = np.asarray(buckets, dtype=np.int64).reshape(-1, 3)
    table = (Bucket * max(len(b), 1))(*[Bucket(int(s), int(n), int(c)) for s, n, c in b])
    ordc = (ctypes.c_int * W)(*order) if order is not None else None
    arr = _ptr_array(grads)
    st = state.c()
    h = hyper.c()
    _check(fn(ctypes.addressof(table), len(b), int(W), int(A), int(dtype),
              ctypes.addressof(ordc) if ordc is not None else None, ctypes.addressof(arr), ctypes.byref(st),
              int(current), ctypes.byref(h), float(loss_scale), int(t), _ptr(overflow), _stream_handle(stream)))


__all__ = ["lib", "ZrError", "chunk_size", "bucket_plan", "model_state_bytes", "ring_traffic", "reduce_scatter",
           "all_reduce", "adamw_shard_step", "accumulate", "offload_adamw", "all_gather", "AdamW", "Scaler",
           "State", "State1", "Plan", "step_noalloc", "F16", "BF16", "F32", "STAGING_REGISTERS", "STAGING_BULK",
           "STAGING_BULK_IO"]
