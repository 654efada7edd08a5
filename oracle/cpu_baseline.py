"""Time the CPU oracle on bounded row samples, on the host's cores.

TEST/BENCH INFRASTRUCTURE ONLY: used by ``bench.py``'s CPU-baseline leg and
its ``--impl reference`` arm. The oracle runs as it stands, in a ``spawn``
process pool (one BLAS thread per worker), reading the problem from shared
memory; only the pool's map over the sampled rows is timed.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import time
from multiprocessing import shared_memory

import numpy as np

_W = {}
_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _attach(spec):
    for name, (shm_name, shape, dtype) in spec.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        _W.setdefault("_shm", []).append(shm)
        _W[name] = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)


def _work(args):
    rows, bs, scale = args
    from oracle.sel_attn import sel_attn_rows

    sel_attn_rows(_W["Q"], _W["K"], _W["V"], _W["idx"], rows, bs, scale)
    return len(rows)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class OracleTimer:
    """Spawn pool + shared problem, reused across timed samples.

    with OracleTimer(Q, K, V, idx, bs, scale) as t:
        seconds = t.time_rows([(b, m, g), ...])
    """

    def __init__(self, Q, K, V, idx, block_size, scale=None, workers=None, chunk=32):
        self.arrays = (("Q", Q), ("K", K), ("V", V), ("idx", idx))
        self.bs, self.scale = block_size, scale
        self.workers = workers or host_cores()
        self.chunk = chunk
        self.shms, self.pool = [], None

    def __enter__(self):
        spec = {}
        for name, a in self.arrays:
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            self.shms.append(shm)
            np.ndarray(a.shape, a.dtype, buffer=shm.buf)[...] = a
            spec[name] = (shm.name, a.shape, a.dtype.str)
        saved = {k: os.environ.get(k) for k in _BLAS_VARS}
        for k in _BLAS_VARS:
            os.environ[k] = "1"
        try:
            ctx = mp.get_context("spawn")
            self.pool = ctx.Pool(self.workers, initializer=_attach, initargs=(spec,))
            b, m, g = 0, 0, 0
            self.pool.map(_work, [([(b, m, g)], self.bs, self.scale)] * self.workers)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        return self

    def time_rows(self, rows) -> float:
        tasks = [(rows[i:i + self.chunk], self.bs, self.scale)
                 for i in range(0, len(rows), self.chunk)]
        t0 = time.perf_counter()
        done = sum(self.pool.map(_work, tasks, chunksize=1))
        secs = time.perf_counter() - t0
        assert done == len(rows)
        return secs

    def __exit__(self, *exc):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
        for shm in self.shms:
            shm.close()
            shm.unlink()
        return False
