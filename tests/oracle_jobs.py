"""Per-head oracle jobs for the full-size parity tests.

The oracle itself is single-process; these helpers only split its work by
query head across spawned worker processes (each head's softmax rows are
independent), so the large workloads' sampled references finish in seconds.
Nothing here computes anything the oracle does not: each job is one call of
`oracle.attention_scores` on one query head and its KV head.
"""
from __future__ import annotations

import multiprocessing as mp
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _head_job(job):
    import oracle as O
    Qh, Kg, q_pos0, extra = job
    kw = {}
    if extra is not None:
        Vg, h, Wo_h = extra
        kw = {"V": Vg, "h": h, "W_O": Wo_h}
    out = O.attention_scores(Qh, Kg, q_pos0, row_chunk=256, **kw)
    return {k: v[0] for k, v in out.items()}


def per_head_scores(Q_heads, Kg, q_pos0, *, V=None, h=None, W_O_heads=None, workers=4):
    """Oracle scores of each query head in Q_heads [G', R, d] against one KV head
    Kg [N, d], rows at positions q_pos0 .. q_pos0+R-1.

    Returns a list (one dict per head) of lse [R], w_t [N], kvzip [N] and, with
    V/h/W_O_heads ([G', D, d] column slices of W_O), s_plus [N].
    """
    jobs = []
    for i in range(Q_heads.shape[0]):
        extra = None if V is None else (V[None], h, W_O_heads[i])
        jobs.append((Q_heads[i:i + 1], Kg[None], q_pos0, extra))
    ctx = mp.get_context("spawn")
    with ProcessPoolExecutor(max_workers=min(workers, len(jobs)), mp_context=ctx) as ex:
        return list(ex.map(_head_job, jobs))


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
