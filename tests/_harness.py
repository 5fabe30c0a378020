"""Shared helpers for the GPU parity tests: seeded inputs in the plan's flat layout and the
oracle run on sampled windows of full-size workloads.

Inputs come from zrgen (host fill for the oracle, device fill for the GPU; a test checks that the
two give equal bytes). Tensor t of replica r at step s is stream (GRAD, s, r, t), element index
within the tensor, scale sigma_t * S. Masters are stream (MASTER, 0, 0, t), scale 0.02. The gap
elements that align each tensor to 8 are zero.
"""
from __future__ import annotations

import numpy as np

import oracle
from zrgen.layout import Layout, grad_stream, master_stream  # noqa: E402,F401


def oracle_layout(plan, numels, cap: int, W: int):
    """The oracle's own bucket table and tensor offsets for a layout (page "DP / DDP / DeepSpeed ZeRO-1/2/3",
    section 二, and page "第 7 讲", DDP 核心实现细节: buckets in reverse registration order). Asserts that the
    plan zr_plan_create built has the same, so that every oracle call and every oracle-side input uses a
    table the product did not make."""
    buckets, offsets = oracle.bucket_plan(list(numels), int(cap), int(W))
    assert np.array_equal(np.asarray(plan.buckets), buckets), "zr_plan_create's buckets differ from the oracle's"
    assert np.array_equal(np.asarray(plan.tensor_offsets), offsets), "zr_plan_create's offsets differ from the oracle's"
    return buckets, offsets


def sample_windows(buckets: np.ndarray, W: int, which, L: int = 256, rng=None, cover=()):
    """Index windows for the sampled buckets. Each window set is a mini-bucket: for every block c of
    the bucket, L consecutive flat indices inside block c (at its start, its end or a seeded point),
    so the oracle can run it as a bucket of block size L with the same ring assignment. `cover`: flat
    indices that must fall inside a window (their bucket gets one more window set placed on them).
    Returns a list of (flat index array, mini block size)."""
    rng = rng or np.random.default_rng(0)
    out = []
    which = list(which)
    for i in cover:
        b = int(np.searchsorted(buckets[:, 0], i, side="right") - 1)
        if b not in which:
            which.append(b)
    for b in which:
        start, n, C = (int(x) for x in buckets[b])
        lens = [max(0, min(C, n - c * C)) for c in range(W)]
        full = [c for c in range(W) if lens[c] > 0]
        if n <= 4096 or any(lens[c] < C for c in full[:-1]):
            out.append((np.arange(start, start + n, dtype=np.int64), C))
            continue
        Lw = min(L, min(lens[c] for c in full[:-1]) if len(full) > 1 else L)
        places = ["start", "end", "mid"] + [int(i) for i in cover if start <= int(i) < start + n]
        for where in places:
            idx = []
            for c in range(W):
                ln = lens[c]
                if ln == 0:
                    continue
                k = min(Lw, ln) if c == full[-1] else Lw
                if where == "start":
                    o = 0
                elif where == "end":
                    o = ln - k
                elif where == "mid":
                    o = int(rng.integers(0, ln - k + 1)) // 8 * 8
                else:  # a window of every block at the covered index's offset within its block
                    rel = (where - start) % C
                    o = min(rel // 8 * 8, ln - k)
                idx.append(np.arange(start + c * C + o, start + c * C + o + k, dtype=np.int64))
            out.append((np.concatenate(idx), Lw))
    return out


class OracleWindows:
    """Oracle state on sampled windows, advanced step by step alongside the GPU run."""

    def __init__(self, layout: Layout, windows, W: int, A: int, hyper, scaler, order=None):
        self.layout, self.windows, self.W, self.A = layout, windows, W, A
        self.hyper, self.scaler, self.order = hyper, scaler, order
        self.state = []
        for idx, _ in windows:
            master = self._gather_master(idx)
            n = len(idx)
            self.state.append([master, np.zeros(n, np.float32), np.zeros(n, np.float32),
                               oracle.encode(layout.dtype, master)])

    def _gather_master(self, idx):
        # windows are runs of consecutive indices: fill run by run
        out = np.empty(len(idx), np.float32)
        runs = np.flatnonzero(np.diff(idx) != 1) + 1
        for seg in np.split(np.arange(len(idx)), runs):
            lo, hi = int(idx[seg[0]]), int(idx[seg[-1]]) + 1
            out[seg] = self.layout.master_host(lo, hi)
        return out

    def _gather_grads(self, idx, step, replica, S, inject=None):
        out = np.empty(len(idx), np.uint16)
        runs = np.flatnonzero(np.diff(idx) != 1) + 1
        for seg in np.split(np.arange(len(idx)), runs):
            lo, hi = int(idx[seg[0]]), int(idx[seg[-1]]) + 1
            out[seg] = self.layout.grads_host(lo, hi, step, replica, S)
        if inject is not None and inject[0] == replica:
            hit = np.flatnonzero(idx == inject[1])
            out[hit] = 0x7C00 if self.layout.dtype == oracle.F16 else 0x7F80
        return out

    def step(self, step: int, S: float, global_flag: int, inject=None):
        """inject: (replica, flat index) of a +inf, or None. Returns the reports."""
        reps = []
        sc0 = oracle.Scaler.from_buffer_copy(self.scaler)
        sc = sc0
        for k, (idx, Lw) in enumerate(self.windows):
            grads = [self._gather_grads(idx, step, r, S, inject) for r in range(self.W * self.A)]
            sc = oracle.Scaler.from_buffer_copy(sc0)
            rep, _ = oracle.step(self.W, self.A, self.layout.dtype, np.array([[0, len(idx), Lw]]), grads,
                                 *self.state[k], self.hyper, sc, order=self.order, flag_override=global_flag)
            reps.append(rep)
        self.scaler = sc
        return reps
