"""Per-head fp64 oracle runs of the chunked prefill, spread over the host's cores.

The oracle's chunked prefill treats every head on its own, so a full-size workload
is checked head by head in worker processes.  Workers are spawned (never forked
from a process that holds a CUDA context); they import only the oracle.
"""
import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _one(job):
    from oracle import kda_oracle as O
    S0, q, k, v, g, beta, cu, stride, mode = job
    return O.prefill_chunked(S0, q, k, v, g, beta, cu_seqlens=cu, chunk=64, ckpt_stride=stride, mode=mode)


def prefill_chunked_per_head(S0, q, k, v, g, beta, cu, stride, heads, mode=0):
    """The oracle's prefill_chunked of each head in `heads`, one worker process per head.

    S0 (N, H, dk, dv) and q, k, g (T, H, dk), v (T, H, dv), beta (T, H) as numpy arrays
    (float32 holds bf16 inputs exactly; the oracle computes in float64).  Returns
    {h: (o (T, 1, dv), S_final (N, 1, dk, dv), ckpts)} as prefill_chunked does for one head.
    """
    heads = list(heads)
    jobs = [(np.ascontiguousarray(S0[:, h:h + 1]), np.ascontiguousarray(q[:, h:h + 1]),
             np.ascontiguousarray(k[:, h:h + 1]), np.ascontiguousarray(v[:, h:h + 1]),
             np.ascontiguousarray(g[:, h:h + 1]), np.ascontiguousarray(beta[:, h:h + 1]), cu, stride, mode)
            for h in heads]
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    # one BLAS thread per worker: the workers already fill the cores
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: "1" for k in keys})
    try:
        with ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
            return dict(zip(heads, ex.map(_one, jobs)))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
