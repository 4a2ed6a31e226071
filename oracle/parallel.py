"""The plain oracle mapped over independent heads in worker processes.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see the package docstring).

Each (batch, head) pair is its own attention problem, so computing the heads in
separate processes changes nothing in the arithmetic of any of them: a worker
runs :func:`oracle.attention.attention_f64` on one head's Q, K, V, exactly as a
single-process call would.  The point is wall-clock time: the oracle's
exponentials run on one core per process, so whole full-size outputs (hundreds
of heads of 2048 to 8191 rows) take seconds instead of minutes.

Workers are started with the ``spawn`` method, never ``fork`` (a process forked
from one that holds a CUDA context can hang), and run with single-threaded BLAS
so that the processes, not BLAS threads, share the cores.  Inputs cross the
process boundary as float32 arrays, which hold bf16 values exactly; the worker
upcasts them to float64.
"""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from .attention import attention_f64

_ONE_THREAD = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _bwd_head_task(args):
    from .backward import attention_backward_f64

    index, q, k, v, do, scale, causal = args
    grads = attention_backward_f64(*(np.asarray(x, dtype=np.float64) for x in (q, k, v, do)), scale, causal)
    return (index,) + tuple(grads)


def _head_task(args):
    index, q, k, v, scale, causal = args
    o, lse = attention_f64(np.asarray(q, dtype=np.float64), np.asarray(k, dtype=np.float64),
                           np.asarray(v, dtype=np.float64), scale, causal)
    return index, o, lse


class HeadPool:
    """A pool of spawn-started worker processes that run the oracle per head.

    Use as a context manager.  ``workers`` defaults to the host's core count.
    """

    def __init__(self, workers: int | None = None):
        self.workers = max(1, int(workers or os.cpu_count() or 1))
        saved = {name: os.environ.get(name) for name in _ONE_THREAD}
        try:
            # Spawned children read their environment at start-up, before numpy
            # loads its BLAS; the parent's own BLAS is already loaded and keeps
            # its thread count.
            for name in _ONE_THREAD:
                os.environ[name] = "1"
            self._pool = mp.get_context("spawn").Pool(self.workers)
        finally:
            for name, value in saved.items():
                if value is None:
                    os.environ.pop(name, None)
                else:
                    os.environ[name] = value

    def heads(self, tasks):
        """``tasks`` yields ``(index, q [Nq, d], k [Nk, d], v [Nk, dv], scale,
        causal)``; yields ``(index, O [Nq, dv], LSE [Nq])`` in completion order."""
        yield from self._pool.imap_unordered(_head_task, tasks)

    def backward_heads(self, tasks):
        """``tasks`` yields ``(index, q, k, v, do, scale, causal)`` per head;
        yields ``(index, dQ, dK, dV)`` from
        :func:`oracle.backward.attention_backward_f64`, in completion order."""
        yield from self._pool.imap_unordered(_bwd_head_task, tasks)

    def close(self):
        self._pool.close()
        self._pool.join()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        if exc[0] is None:
            self.close()
        else:
            self._pool.terminate()
            self._pool.join()
        return False
