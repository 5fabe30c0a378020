"""The five synthetic workloads of the post-backward ZeRO step, as data.

Each workload names its tensor shape list (in definition order), the number of
emulated data-parallel workers W, micro-batches A, gradient dtype, ZeRO stage,
bucket cap (in parameters), step count, seed, loss-scale settings and AdamW
hyperparameters. Gradients of tensor t are N(0, sigma_t) * loss_scale; masters are
N(0, 0.02) in fp32; m = v = 0 at the start. Nothing here computes the step.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np

__all__ = ["Workload", "WORKLOADS", "workload", "width_workload", "gpt2_small_tensors", "gpt_1p3b_tensors",
           "sweep_workloads",
           "sigma_per_tensor", "grad_scale", "inject_site"]


def gpt2_small_tensors() -> Tuple[List[int], List[str]]:
    """GPT-2-small shape list: 50304x768 embedding, then 12 layers of qkv, out, fc1, fc2, two norms."""
    d, v = 768, 50304
    numels, names = [v * d], ["wte"]
    for layer in range(12):
        for nm, n in (("qkv", d * 3 * d), ("out", d * d), ("fc1", d * 4 * d), ("fc2", 4 * d * d),
                      ("norm_a", d), ("norm_b", d)):
            numels.append(n)
            names.append(f"h{layer}.{nm}")
    return numels, names


def gpt_1p3b_tensors() -> Tuple[List[int], List[str]]:
    """1.3B transformer shape list: 50304x2048 embedding, then 24 layers of qkv, out, fc1, fc2, two norms."""
    d, v = 2048, 50304
    numels, names = [v * d], ["wte"]
    for layer in range(24):
        for nm, n in (("qkv", d * 3 * d), ("out", d * d), ("fc1", d * 4 * d), ("fc2", 4 * d * d),
                      ("norm_a", d), ("norm_b", d)):
            numels.append(n)
            names.append(f"h{layer}.{nm}")
    return numels, names


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tensors: Tuple[int, ...]          # numels, definition (registration) order
    W: int                            # emulated data-parallel workers
    A: int                            # micro-batches accumulated before the ring
    dtype: int                        # 0 = fp16, 1 = bf16 (grads and params)
    stage: int                        # ZeRO stage 1/2/3
    cap: int                          # bucket cap in parameters
    steps: int
    seed: int
    sigma: Optional[float]            # fixed grad sigma, or None = log-uniform per tensor in [1e-4, 1e-1]
    init_scale: float                 # loss scale S at step 1
    dynamic: bool                     # dynamic loss scaling
    inject_step: Optional[int] = None  # 1-based step whose grads get one +inf
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    master_sigma: float = 0.02
    align: int = 8
    description: str = ""
    state_sets: int = 2                # 2 = ping-pong sets (zr_step); 1 = one set updated in place only

    @property
    def n(self) -> int:
        return int(sum(self.tensors))

    def alg_bytes_per_param(self) -> int:
        """W*A 16-bit grad reads + 12 B master/m/v read + 12 B written + 2 B param written."""
        return 2 * self.W * self.A + 26


def _flat(n: int, parts: int = 1) -> Tuple[int, ...]:
    assert n % parts == 0
    return tuple([n // parts] * parts)


_g2, _ = gpt2_small_tensors()
_b13, _ = gpt_1p3b_tensors()

WORKLOADS = {
    "tiny": Workload("tiny", _flat(786_432), W=3, A=1, dtype=0, stage=2, cap=786_432, steps=3, seed=0,
                     sigma=1e-2, init_scale=1024.0, dynamic=False,
                     description="flat n=786,432 (3*2^18), W=3, fp16, one bucket, S=1024, 3 steps"),
    "gpt2": Workload("gpt2", tuple(_g2), W=8, A=1, dtype=1, stage=2, cap=25_000_000, steps=10, seed=0,
                     sigma=None, init_scale=1.0, dynamic=False,
                     description="GPT-2-small shapes, 73 tensors, 123,586,560 params, W=8, bf16, 25M-param buckets"),
    "1p3b": Workload("1p3b", tuple(_b13), W=8, A=1, dtype=1, stage=3, cap=50_000_000, steps=5, seed=0,
                     sigma=None, init_scale=1.0, dynamic=False,
                     description="1.3B shapes, 145 tensors, 1,311,080,448 params, W=8, bf16, ZeRO-3, 50M-param buckets"),
    "7b": Workload("7b", _flat(7_000_000_000, 35), W=2, A=1, dtype=0, stage=1, cap=200_000_000, steps=6, seed=0,
                   sigma=1e-2, init_scale=65536.0, dynamic=True, inject_step=3,
                   description="flat 7.0e9 params in 200M-param buckets, W=2, fp16, dynamic loss scale S0=65536, "
                               "+inf injected at step 3"),
    # the GPT-2 shapes with A = 4 micro-batches on W = 2 workers: a case small enough (about 6 GB on the
    # device) for full profiler captures of the accumulate path's kernels
    "gpt2_a4": Workload("gpt2_a4", tuple(_g2), W=2, A=4, dtype=1, stage=2, cap=25_000_000, steps=3, seed=0,
                        sigma=None, init_scale=1.0, dynamic=False,
                        description="GPT-2-small shapes, 123,586,560 params, W=2, A=4, bf16, 25M-param buckets"),
    # a model whose ping-pong state sets do not fit one GPU (1.3e10 x 32 B = 416 GB) but whose in-place step does
    # (1.3e10 x 18 B = 234 GB): the 13B size that ZeRO-Offload is said to train on a single GPU (page
    # "并行训练框架DeepSpeed介绍", (16) ZeRO-Offload), here with all of the optimizer state in HBM
    "13b": Workload("13b", _flat(13_000_000_000, 65), W=2, A=1, dtype=0, stage=1, cap=200_000_000, steps=6, seed=0,
                    sigma=1e-2, init_scale=65536.0, dynamic=True, inject_step=3, state_sets=1,
                    description="flat 1.3e10 params in 200M-param buckets, W=2, fp16, dynamic loss scale S0=65536, "
                                "+inf injected at step 3, one state set stepped in place"),
    # the 7B workload's kernel configuration (W=2, fp16, 200M-param buckets) at 1/35 of its size: a case small
    # enough for a full profiler capture
    "7b_slice": Workload("7b_slice", _flat(200_000_000, 1), W=2, A=1, dtype=0, stage=1, cap=200_000_000, steps=6,
                         seed=0, sigma=1e-2, init_scale=65536.0, dynamic=True,
                         description="one 200M-param bucket of the 7B workload (W=2, fp16, S0=65536)"),
}


def sweep_workloads() -> List[Workload]:
    """Bucket-size and accumulation sweep on the 1.3B shapes: W in {2,4,8}, caps 2^19..2^28 params, A=4."""
    out = []
    for W in (2, 4, 8):
        for k in range(19, 29):
            out.append(Workload(f"sweep_W{W}_cap2^{k}", tuple(_b13), W=W, A=4, dtype=1, stage=2, cap=1 << k,
                                steps=3, seed=0, sigma=None, init_scale=1.0, dynamic=False,
                                description=f"1.3B shapes, W={W}, A=4, cap {1 << k} params ({(1 << k) * 2 >> 20} MB bf16)"))
    return out


def width_workload(W: int) -> Workload:
    """The GPT-2 shapes (123,586,560 params, 25M-param buckets, bf16) on W workers: cases a few GB in size for
    widths with no workload of their own (W = 5, 6, 7, 16, 32, ...)."""
    return Workload(f"gpt2_W{W}", tuple(_g2), W=W, A=1, dtype=1, stage=2, cap=25_000_000, steps=10, seed=0,
                    sigma=None, init_scale=1.0, dynamic=False,
                    description=f"GPT-2-small shapes, 123,586,560 params, W={W}, bf16, 25M-param buckets")


def workload(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    for w in sweep_workloads():
        if w.name == name:
            return w
    if name.startswith("gpt2_W") and name[6:].isdigit() and 1 <= int(name[6:]) <= 64:
        return width_workload(int(name[6:]))
    raise KeyError(name)


def sigma_per_tensor(w: Workload) -> np.ndarray:
    """Per-tensor grad sigma (float32), fixed across steps: log-uniform in [1e-4, 1e-1] drawn once per tensor."""
    from . import uniform, stream_id, TAG_SIGMA
    if w.sigma is not None:
        return np.full(len(w.tensors), w.sigma, dtype=np.float32)
    out = np.empty(len(w.tensors), dtype=np.float32)
    for t in range(len(w.tensors)):
        u = uniform(w.seed, stream_id(TAG_SIGMA, 0, 0, t), 0, 0)
        out[t] = np.float32(10.0 ** (-4.0 + 3.0 * u))
    return out


def grad_scale(sigma_t: float, loss_scale: float) -> np.float32:
    """The single fp32 multiplier applied to the normal table for a gradient draw."""
    return np.float32(np.float32(sigma_t) * np.float32(loss_scale))


def inject_site(w: Workload, step: int) -> Optional[Tuple[int, int, int]]:
    """(worker, tensor, element within that tensor) of the +inf injected at `step` (1-based), else None.

    The element is drawn uniformly over the concatenation of the tensors in definition order."""
    from . import u64, stream_id, TAG_INJECT
    if w.inject_step is None or step != w.inject_step:
        return None
    r = u64(w.seed, stream_id(TAG_INJECT, step, 0, 0), 0)
    worker = int((r >> 48) % w.W)
    index = int((r & ((1 << 48) - 1)) % w.n)
    for t, n in enumerate(w.tensors):
        if index < n:
            return worker, t, index
        index -= n
    raise AssertionError("unreachable")
