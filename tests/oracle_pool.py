"""Float64 oracle over many heads at once, for the full-size GPU parity tests.

Each (b, h) head of attention is an independent problem, so the oracle runs
one head per task in a pool of worker processes.  The pool is started with
``spawn``: a process forked after the parent has touched CUDA can hang.  The
workers import only numpy and ``oracle`` (never torch or the CUDA library);
each is given a share of the host's BLAS threads.

A task gets one head's inputs (the bf16-rounded Q, K, V, dO as float32, which
upcast exactly) and the GPU's outputs for that head, runs the oracle and
returns, per tensor, max|x - ref|, max|ref| and whether x is finite.  The
parent combines them into the parity metric max|dX - ref| / max|ref|, per
head and over the whole tensor.  Imported only by tests.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from contextlib import contextmanager

import numpy as np

TENSORS = ("O", "L", "dQ", "dK", "dV")
_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def head_errors(task):
    """Oracle for one head; returns {tensor: (max|x - ref|, max|ref|, finite)}."""
    from oracle import attention_backward

    q, k, v, g, scale, causal, outs = task
    up = [np.asarray(t, dtype=np.float64) for t in (q, k, v, g)]
    ref = attention_backward(*up, scale, causal)
    res = {}
    for name in TENSORS:
        x = np.asarray(outs[name], dtype=np.float64)
        r = getattr(ref, name)[0, 0]
        fin = bool(np.all(np.isfinite(x)))
        res[name] = (float(np.abs(x - r).max()) if fin else float("inf"), float(np.abs(r).max()), fin)
    return res


@contextmanager
def _blas_threads(n):
    old = {k: os.environ.get(k) for k in _BLAS_VARS}
    for k in _BLAS_VARS:
        os.environ[k] = str(n)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def run_heads(tasks, workers=None):
    """head_errors over every task, in order, on a spawn pool."""
    cpus = os.cpu_count() or 1
    workers = workers or max(1, min(8, cpus, len(tasks)))
    if workers == 1:
        return [head_errors(t) for t in tasks]
    with _blas_threads(max(1, cpus // workers)):
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers) as pool:
            return pool.map(head_errors, tasks, chunksize=1)


def summarize(per_head):
    """Whole-tensor ratios and the worst per-head ratio for each tensor."""
    whole, worst = {}, {}
    for name in TENSORS:
        diff = max(h[name][0] for h in per_head)
        ref = max(h[name][1] for h in per_head)
        whole[name] = diff / max(ref, 1e-30)
        worst[name] = max(h[name][0] / max(h[name][1], 1e-30) for h in per_head)
    return whole, worst
