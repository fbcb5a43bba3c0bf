"""Runs independent oracle calls in a pool of spawned CPU processes.

Test infrastructure.  Sequences and KV heads of a pack are independent in the
method (each query attends only to keys of its own sequence through its own
KV head), so the oracle called on the slice of one (sequence, KV head) gives
the same numbers as on the whole pack; slicing only keeps each task small.
The pool is created with the "spawn" start method (a process forked after
CUDA has started can hang), and its workers import numpy and the oracle only.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
               "NUMEXPR_NUM_THREADS", "BLIS_NUM_THREADS")


def _bwd_slice(task):
    from oracle import msa_oracle as O
    q, k, v, do, sel, blocks, scale = task
    L = q.shape[0]
    out = O.sparse_attn_bwd(q, k, v, do, sel, np.array([0, L]), scale,
                            dkv_blocks=[(0, 0, b) for b in blocks])
    return out["dkv"]


def dkv_blocks(q, k, v, do, sel, cu, scale, blocks, processes=None):
    """dk, dv of every (sequence s, KV head g, block b) in `blocks`, each a pair
    of arrays [keys of the block, D], from the oracle's sampled backward.
    q, do [T, Hq, D]; k, v [T, Hkv, D]; sel [T, Hkv, topk]; cu [S + 1]."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    groups = {}
    for i, (s, g, b) in enumerate(blocks):
        groups.setdefault((s, g), []).append((i, b))
    tasks, index = [], []
    for (s, g), items in groups.items():
        a, e = int(cu[s]), int(cu[s + 1])
        tasks.append((np.ascontiguousarray(q[a:e, g * G:(g + 1) * G], dtype=np.float32),
                      np.ascontiguousarray(k[a:e, g:g + 1], dtype=np.float32),
                      np.ascontiguousarray(v[a:e, g:g + 1], dtype=np.float32),
                      np.ascontiguousarray(do[a:e, g * G:(g + 1) * G], dtype=np.float32),
                      np.ascontiguousarray(sel[a:e, g:g + 1]), [b for _, b in items], scale))
        index.append([i for i, _ in items])
    n = processes or max(1, min(len(tasks), len(os.sched_getaffinity(0))))
    # one BLAS thread per worker: the workers already use every core
    saved = {var: os.environ.get(var) for var in THREAD_VARS}
    os.environ.update({var: "1" for var in THREAD_VARS})
    try:
        pool = mp.get_context("spawn").Pool(n)
    finally:
        for var, val in saved.items():
            if val is None:
                os.environ.pop(var, None)
            else:
                os.environ[var] = val
    with pool:
        results = pool.map(_bwd_slice, tasks, chunksize=1)
    out = [None] * len(blocks)
    for idx, res in zip(index, results):
        for i, r in zip(idx, res):
            out[i] = r
    return out
