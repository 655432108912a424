"""The float64 oracle over many matrices at once, for the full-size parity
tests (test infrastructure only).

Jobs run in worker processes started with ``spawn`` (never ``fork``: the test
process has a CUDA context, and a forked child of it may hang), each worker
with single-threaded BLAS so that the host cores are shared by matrices
rather than by threads inside one product. A job carries the raw bits of one
bf16 input and of the GPU's result (bf16 or fp32); the worker rebuilds both in
float64, runs the oracle and returns the per-matrix relative Frobenius error.
No torch in the workers: bit patterns are widened with numpy alone.
"""

from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

from oracle import ns as ons

_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _decode(bits: np.ndarray) -> np.ndarray:
    if bits.dtype == np.uint16:
        return bf16_bits_to_f64(bits)
    return bits.view(np.float32).astype(np.float64)


def oracle_error(job) -> tuple:
    """job = (key, shape, input bits, output bits, steps, a, b, c, eps, ridge)
    -> (key, relative Frobenius error of the output against the oracle)."""
    key, shape, in_bits, out_bits, steps, a, b, c, eps, ridge = job
    x = _decode(in_bits).reshape(shape)
    y = _decode(out_bits).reshape(shape)
    ref = ons.newton_schulz(x, steps, a, b, c, eps, ridge=ridge)
    return key, ons.rel_fro_error(y, ref)


class OraclePool:
    """Context manager: ``errors(jobs)`` returns {key: error} for all jobs."""

    def __init__(self, workers: int | None = None):
        self.workers = workers or max(1, os.cpu_count() or 1)
        self._saved = {}
        self._ex = None

    def __enter__(self):
        # spawned workers read these at their own numpy import; the parent's
        # BLAS is already loaded and keeps its threads
        for k in _BLAS_ENV:
            self._saved[k] = os.environ.get(k)
            os.environ[k] = "1"
        self._ex = cf.ProcessPoolExecutor(max_workers=self.workers, mp_context=mp.get_context("spawn"))
        return self

    def errors(self, jobs) -> dict:
        # largest matrices first, so that no long job starts last
        jobs = sorted(jobs, key=lambda j: -int(np.prod(j[1])) * min(j[1][0], int(np.prod(j[1][1:]))))
        out = {}
        for key, err in self._ex.map(oracle_error, jobs, chunksize=1):
            out[key] = err
        return out

    def __exit__(self, *exc):
        self._ex.shutdown(wait=True, cancel_futures=True)
        for k, v in self._saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        return False
