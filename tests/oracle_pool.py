"""Runs the fp64 oracle on one KV head per query head in separate processes (test
harness only).

With grouped-query attention a KV head's dK and dV are, by definition, the sums over
its query heads of each head's gradient (the oracle pins GQA against multi-head
attention with repeated K/V), so the heads are independent oracle calls whose dK/dV
the harness adds up.  The oracle itself runs unchanged in each worker.  Workers are
started with the "spawn" method, never forked from a process that holds a CUDA
context.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _one_head(args):
    host, offsets, scale = args
    from oracle import attention as A
    return A.tree_attention_direct(host, offsets, scale)


def oracle_one_kv_head(host, offsets, scale, processes=None):
    """host: q_*/do_* [rows, r, D] (the KV head's r query heads), k_*/v_* [rows, 1, D].
    Returns the oracle's dict for that KV head: o/lse/dq per query head, dk/dv summed
    over the query heads."""
    r = host["q_p"].shape[1]
    jobs = []
    for h in range(r):
        sub = {n: (x[:, h:h + 1] if n[0] in "qd" else x) for n, x in host.items()}
        jobs.append((sub, offsets, scale))
    processes = processes or r
    threads = max(1, (os.cpu_count() or 1) // processes)
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = str(threads)
    try:
        with mp.get_context("spawn").Pool(processes) as pool:
            res = pool.map(_one_head, jobs)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    out = {}
    for n in ("o_p", "o_r", "dq_p", "dq_r"):
        out[n] = np.concatenate([x[n] for x in res], axis=1)
    for n in ("lse_p", "lse_r"):
        out[n] = np.concatenate([x[n] for x in res], axis=0)
    for n in ("dk_p", "dv_p", "dk_r", "dv_r"):
        out[n] = sum(x[n] for x in res)
    return out
