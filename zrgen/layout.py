"""Seeded inputs in a plan's flat layout (tensors at their flat offsets, alignment gaps zero).

Tensor t of replica r at step s is the normal stream (GRAD, s, r, t), indexed from 0 within the
tensor, scaled by sigma_t * S; masters are stream (MASTER, 0, 0, t) scaled by 0.02. Inputs only.
"""
from __future__ import annotations

import numpy as np

from . import F32, fill_dev, fill_host, grad_scale, stream_id, TAG_GRAD, TAG_MASTER


def grad_stream(step: int, replica: int, tensor: int) -> int:
    return stream_id(TAG_GRAD, step, replica, tensor)


def master_stream(tensor: int) -> int:
    return stream_id(TAG_MASTER, 0, 0, tensor)


class Layout:
    """Tensor offsets of a plan plus the per-tensor sigmas of a workload."""

    def __init__(self, numels, offsets, sigma, seed, dtype, master_sigma=0.02):
        self.numels = [int(x) for x in numels]
        self.offsets = [int(x) for x in offsets]
        self.sigma = np.asarray(sigma, dtype=np.float32)
        self.seed = int(seed)
        self.dtype = int(dtype)
        self.master_sigma = float(master_sigma)
        # tensors sorted by flat offset for range queries
        self._by_off = sorted(range(len(self.numels)), key=lambda t: self.offsets[t])

    def _pieces(self, lo: int, hi: int):
        """(tensor, index in tensor, flat position, count) for the real elements in [lo, hi)."""
        out = []
        for t in self._by_off:
            a, b = self.offsets[t], self.offsets[t] + self.numels[t]
            if b <= lo:
                continue
            if a >= hi:
                break
            s, e = max(a, lo), min(b, hi)
            out.append((t, s - a, s, e - s))
        return out

    def grads_host(self, lo: int, hi: int, step: int, replica: int, S: float) -> np.ndarray:
        out = np.zeros(hi - lo, dtype=np.uint16)
        for t, i0, pos, cnt in self._pieces(lo, hi):
            out[pos - lo:pos - lo + cnt] = fill_host(cnt, self.dtype, self.seed, grad_stream(step, replica, t), i0,
                                                           grad_scale(self.sigma[t], S))
        return out

    def master_host(self, lo: int, hi: int) -> np.ndarray:
        out = np.zeros(hi - lo, dtype=np.float32)
        for t, i0, pos, cnt in self._pieces(lo, hi):
            out[pos - lo:pos - lo + cnt] = fill_host(cnt, F32, self.seed, master_stream(t), i0,
                                                           self.master_sigma)
        return out

    def grads_dev(self, buf, step: int, replica: int, S: float, table_dev, stream) -> None:
        """Fill a flat device buffer (torch, 16-bit) with replica `replica`'s step-`step` gradients."""
        for t, (cnt, off) in enumerate(zip(self.numels, self.offsets)):
            fill_dev(buf.data_ptr() + 2 * off, cnt, self.dtype, self.seed, grad_stream(step, replica, t), 0,
                           grad_scale(self.sigma[t], S), table_dev.data_ptr(), stream)

    def master_dev(self, buf, table_dev, stream) -> None:
        for t, (cnt, off) in enumerate(zip(self.numels, self.offsets)):
            fill_dev(buf.data_ptr() + 4 * off, cnt, F32, self.seed, master_stream(t), 0,
                           self.master_sigma, table_dev.data_ptr(), stream)
