"""The float64 oracle's backward for one K/V-head group of a large workload, in parallel.

Only the oracle runs here (``oracle.attention.attention_bwd`` on contiguous chunks of query
rows, in spawned worker processes that never touch CUDA); the chunks' dk / dv
contributions are summed and their dq rows assembled. Used by the full-size GPU parity
tests to check every key row of one group, not only sampled rows.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_SHARED = {}


def _init(q, k, v, do, cu, causal):
    _SHARED.update(q=q, k=k, v=v, do=do, cu=cu, causal=causal)


def _chunk(rows):
    from oracle import attention as A

    s = _SHARED
    dq, dk, dv = A.attention_bwd(s["q"], s["k"], s["v"], s["do"], s["cu"], s["causal"], rows=rows)
    return rows, dq[rows], dk, dv


def _balanced_chunks(cu, causal, n_chunks):
    """Contiguous row ranges of about equal oracle cost (row i of a causal sequence costs
    i + 1 key visits)."""
    rows, cost = [], []
    for s0, s1 in zip(cu[:-1], cu[1:]):
        r = np.arange(int(s0), int(s1))
        rows.append(r)
        cost.append((r - s0 + 1.0) if causal else np.full(r.size, float(s1 - s0)))
    rows, cost = np.concatenate(rows), np.concatenate(cost)
    edges = np.searchsorted(np.cumsum(cost), np.linspace(0, cost.sum(), n_chunks + 1)[1:-1])
    return [c for c in np.split(rows, edges) if c.size]


def group_backward(q, k, v, do, cu, causal, hk, group, workers=None):
    """dq [T, group, Dh], dk and dv [T, 1, Dh] of K/V head ``hk`` (query heads
    hk*group .. hk*group+group-1), float64, from packed natural-order inputs."""
    qg = np.ascontiguousarray(q[:, hk * group:(hk + 1) * group], dtype=np.float64)
    kg = np.ascontiguousarray(k[:, hk:hk + 1], dtype=np.float64)
    vg = np.ascontiguousarray(v[:, hk:hk + 1], dtype=np.float64)
    dog = np.ascontiguousarray(do[:, hk * group:(hk + 1) * group], dtype=np.float64)
    workers = workers or max(1, min(8, (os.cpu_count() or 2) // 2))
    chunks = _balanced_chunks(np.asarray(cu), causal, 8 * workers)
    dq = np.full(qg.shape, np.nan)
    dk = np.zeros(kg.shape)
    dv = np.zeros(vg.shape)
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers, initializer=_init, initargs=(qg, kg, vg, dog, np.asarray(cu), causal)) as pool:
        for rows, dq_r, dk_c, dv_c in pool.imap_unordered(_chunk, chunks):
            dq[rows] = dq_r
            dk += dk_c
            dv += dv_c
    return dq, dk, dv
