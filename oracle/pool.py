"""Runs the float64 oracle's layer over a process pool, one task per expert.

TEST INFRASTRUCTURE ONLY, like the oracle itself: only tests, the smoke check
and the benchmark's CPU legs use it.  It adds no arithmetic of its own: the
routing, permutation and every expert FFN are the oracle's functions
(route, permute, expert_ffn), unchanged; this module only distributes the
per-expert calls and assembles the per-slot outputs.

The layer it computes is the oracle's definition,
    out[t] = sum_{j < k} w[t][j] * FFN_{ids[t][j]}(x[t])  (+ the shared expert),
summed in slot order j = 0..k-1 in float64 exactly as moe_forward does.  The
only difference from calling moe_forward in one process is that an expert's
rows may be multiplied in a different blocking by the BLAS library, which
changes float64 results at the level of 1e-16 relative.

Processes are started with "spawn" (never fork: the caller may hold a CUDA
context), each with a single BLAS thread, one per core visible to the caller
(os.sched_getaffinity) unless a count is given.
"""
from __future__ import annotations

import multiprocessing as _mp
import os

import numpy as np

from . import nvfp4_moe_oracle as _O

_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS")


class _OneExpert:
    """One expert's canonical NVFP4 bytes, shaped as the oracle's weights
    object with a single expert (index 0)."""

    def __init__(self, w13_q, w13_s, w2_q, w2_s, gscale):
        self.w13_q, self.w13_s = w13_q[None], w13_s[None]
        self.w2_q, self.w2_s = w2_q[None], w2_s[None]
        self.gscale = np.asarray(gscale, np.float32)[None]


def _ffn_task(args):
    """Worker: expert FFN of some rows, y = FFN_e(x) [m][H] float64."""
    tag, w13_q, w13_s, w2_q, w2_s, gscale, x_bits = args
    w = _OneExpert(w13_q, w13_s, w2_q, w2_s, gscale)
    return tag, _O.expert_ffn(w, 0, _O.bf16_bits_to_f64(x_bits))


def cores() -> int:
    """Cores visible to this process."""
    return len(os.sched_getaffinity(0))


def make_pool(procs: int | None = None):
    """A spawn pool whose workers each use one BLAS thread."""
    n = procs or cores()
    saved = {v: os.environ.get(v) for v in _BLAS_VARS}
    for v in _BLAS_VARS:
        os.environ[v] = "1"
    try:
        pool = _mp.get_context("spawn").Pool(n)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    return pool, n


def moe_forward_pool(logits, x_bits, weights, k: int, num_shared: int = 0, pool=None, procs=None,
                     return_y=False):
    """The oracle's layer (moe_forward) over a process pool.

    logits [T][E], x_bits [T][H] BF16 bit patterns, weights the oracle's
    weights object (w13_q/w13_s/w2_q/w2_s/gscale, the shared expert as index
    E when num_shared = 1).  Returns out [T][H] float64 and, with return_y,
    also y [T][k + num_shared][H] float64 (every slot's expert output).
    """
    logits = np.asarray(logits)
    x_bits = np.asarray(x_bits)
    T, E = logits.shape
    r = _O.route(logits, k)
    H = x_bits.shape[1]
    ks = k + num_shared
    tasks = []
    for e in np.unique(r.ids):
        rows, slots = np.nonzero(r.ids == e)
        tasks.append(((int(e), rows, slots), weights.w13_q[e], weights.w13_s[e], weights.w2_q[e],
                      weights.w2_s[e], weights.gscale[e], x_bits[rows]))
    if num_shared:
        rows = np.arange(T)
        tasks.append(((E, rows, np.full(T, k)), weights.w13_q[E], weights.w13_s[E], weights.w2_q[E],
                      weights.w2_s[E], weights.gscale[E], x_bits))
    own = pool is None
    if own:
        pool, _ = make_pool(procs)
    y = np.zeros((T, ks, H), dtype=np.float64)
    try:
        # largest tasks first, so the last ones to finish are small
        tasks.sort(key=lambda a: -len(a[0][1]))
        for (e, rows, slots), ye in pool.imap_unordered(_ffn_task, tasks):
            y[rows, slots] = ye
    finally:
        if own:
            pool.close()
            pool.join()
    out = np.zeros((T, H), dtype=np.float64)
    for j in range(k):
        out += r.weights[:, j:j + 1] * y[:, j]
    if num_shared:
        out += y[:, k]
    if return_y:
        return out, y
    return out
