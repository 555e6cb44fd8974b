"""Run the float64 oracle over many (document, head) units in parallel on the
host cores, for the whole-workload parity tests.

Test infrastructure: it only splits a workload into independent units, hands
each to ``oracle.attention_single`` in a worker process and puts the results
back in place; it holds no attention arithmetic of its own.  The pool uses
the ``spawn`` start method (a process forked after the first CUDA call would
hang), and each worker runs single-threaded BLAS so that the workers do not
oversubscribe the cores.
"""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _unit(args):
    import oracle

    q, k, v, scale, causal = args
    return oracle.attention_single(q, k, v, scale, causal)


def _workers(peak_unit_bytes: int) -> int:
    n = min(16, os.cpu_count() or 1)
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
        n = max(1, min(n, int(0.5 * avail // max(1, peak_unit_bytes))))
    except (ValueError, OSError, AttributeError):
        pass
    return n


def run_units(units, peak_unit_bytes: int):
    """units: list of (q [Lq, Hq', D], k [Lk, Hkv', D], v, scale, causal)
    float32 numpy arrays (bf16 values, exact).  Returns the list of
    (out, lse) of oracle.attention_single, in order."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    saved = {n: os.environ.get(n) for n in _THREAD_VARS + ("PYTHONPATH",)}
    try:
        for n in _THREAD_VARS:
            os.environ[n] = "1"
        os.environ["PYTHONPATH"] = root + (os.pathsep + saved["PYTHONPATH"] if saved["PYTHONPATH"] else "")
        ctx = mp.get_context("spawn")
        pool = ctx.Pool(_workers(peak_unit_bytes))
    finally:
        for n, v in saved.items():
            if v is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = v
    try:
        return pool.map(_unit, units, chunksize=1)
    finally:
        pool.close()
        pool.join()


def f32(t) -> np.ndarray:
    """bf16 torch tensor -> float32 numpy (exact)."""
    return t.detach().cpu().float().numpy()


def score_bytes(lq: int, lk: int) -> int:
    """Rough peak memory of one oracle unit: a few float64 [Lq, Lk] arrays."""
    return 5 * 8 * lq * lk + (1 << 26)
