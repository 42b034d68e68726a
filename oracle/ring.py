"""Explicit ring schedule in float64: block attention per step + log-sum-exp merge.

This follows the pages step by step, with D virtual ranks:

* Rank r keeps its query shard Q_r; K/V shards travel around the ring 0 -> 1 -> ... ->
  D-1 -> 0, so at step s rank r holds the K/V shard of rank (r - s) mod D (Ring Attention
  concept page, "Sequence sharding and the ring topology"; its two-device code has device
  0 see K0 then K1 and device 1 see K1 then K0).
* At every step the rank computes local attention of Q_r against the K/V it holds, giving a
  *normalised* block output and its log-sum-exp (nanotron how-to page, "Forward Pass
  Implementation", step 2), masked by *global* positions when causal (concept page,
  "Watch Out For": the mask must know the global position of each K/V block).
* ``update_out_and_lse`` folds each block into the running (out, lse) (how-to page, step 3
  and "Numerically-Stable Output Fusion"; interview question page: rescale the previous
  partial by exp(old - new) when the reference value changes).
* Backward ("Backward Pass and Gradient Accumulation"): the same steps again, each block's
  gradient taken against the *final* out and lse; dq accumulates on its own rank, dk and dv
  accumulate into the shard that owns the K/V block.

The merge is written in its log-sum-exp form:

    lse' = log(exp(lse) + exp(block_lse))
    out' = exp(lse - lse') * out + exp(block_lse - lse') * block_out

with lse = -inf (and out = 0) as the identity: an empty running state, or a block whose
rows see no key. The concept page's printed two-device combine weighs *unnormalised* block
outputs by sums taken against *different* per-block maxima; that combine is not exact (it
is off by about 0.2 on the page's own inputs), so the oracle uses the rule above, which the
same page's claim of exactness requires.
"""
from __future__ import annotations

import numpy as np

from .layouts import shard_positions

NEG_INF = -np.inf


def update_out_and_lse(out, lse, block_out, block_lse):
    """Merge a normalised block into (out, lse).

    ``out`` and ``block_out`` are [..., Dh]; ``lse`` and ``block_lse`` have the same shape
    without the last axis ([...]).
    """
    out = np.asarray(out, np.float64)
    lse = np.asarray(lse, np.float64)
    block_out = np.asarray(block_out, np.float64)
    block_lse = np.asarray(block_lse, np.float64)
    new_lse = np.logaddexp(lse, block_lse)
    finite = np.isfinite(new_lse)
    safe = np.where(finite, new_lse, 0.0)
    w_old = np.where(finite & np.isfinite(lse), np.exp(np.where(np.isfinite(lse), lse, 0.0) - safe), 0.0)
    w_new = np.where(finite & np.isfinite(block_lse),
                     np.exp(np.where(np.isfinite(block_lse), block_lse, 0.0) - safe), 0.0)
    new_out = w_old[..., None] * out + w_new[..., None] * block_out
    return new_out, new_lse


def block_attention(q, k, v, pos_q, pos_k, causal: bool, scale: float):
    """Normalised attention of one query shard against one K/V shard.

    q [L, Hq, Dh], k/v [L, Hkv, Dh]; pos_q/pos_k global positions (same sequence).
    Returns block_out [L, Hq, Dh] and block_lse [Hq, L]; a row with no allowed key gets
    block_lse = -inf and block_out = 0.
    """
    lq, hq, dh = q.shape
    g = hq // k.shape[1]
    out = np.zeros((lq, hq, dh))
    lse = np.full((hq, lq), NEG_INF)
    allowed = (pos_k[None, :] <= pos_q[:, None]) if causal else np.ones((lq, pos_k.size), bool)
    any_row = allowed.any(axis=1)
    for h in range(hq):
        kv = h // g
        s = scale * (q[:, h, :] @ k[:, kv, :].T)
        s = np.where(allowed, s, NEG_INF)
        m = np.where(any_row, s.max(axis=1), 0.0)
        e = np.where(allowed, np.exp(s - m[:, None]), 0.0)
        l = e.sum(axis=1)
        ok = l > 0
        out[ok, h, :] = (e[ok] / l[ok, None]) @ v[:, kv, :]
        lse[h, ok] = m[ok] + np.log(l[ok])
    return out, lse


def piece_rows(lengths, D: int, varlen: bool, seq: int, rank: int) -> np.ndarray:
    """Shard-major rows holding rank ``rank``'s local piece of sequence ``seq``."""
    starts = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    L = lengths[seq] // D
    if varlen:
        base = rank * (int(starts[-1]) // D) + int(starts[seq]) // D
    else:
        base = int(starts[seq]) + rank * L
    return base + np.arange(L, dtype=np.int64)


def ring_fwd(q, k, v, lengths, D: int, layout: str, causal: bool, varlen: bool,
             scale: float | None = None, steps=None):
    """Ring forward over shard-major packed tensors ([T, H, Dh], float64).

    Returns shard-major ``out`` [T, Hq, Dh] and ``lse`` [Hq, T]. ``steps`` (default all D)
    limits the ring to its first steps, leaving the partial state a resumed ring continues.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    t, hq, dh = q.shape
    scale = 1.0 / np.sqrt(dh) if scale is None else scale
    out = np.zeros((t, hq, dh))
    lse = np.full((hq, t), NEG_INF)
    n_steps = D if steps is None else steps
    for i, n in enumerate(lengths):
        pos = shard_positions(layout, D, n)
        for r in range(D):
            rq = piece_rows(lengths, D, varlen, i, r)
            o_r = np.zeros((rq.size, hq, dh))
            l_r = np.full((rq.size, hq), NEG_INF)
            for s in range(n_steps):
                j = (r - s) % D
                rk = piece_rows(lengths, D, varlen, i, j)
                bo, bl = block_attention(q[rq], k[rk], v[rk], pos[r], pos[j], causal, scale)
                o_r, l_r = update_out_and_lse(o_r, l_r, bo, bl.T)
            out[rq] = o_r
            lse[:, rq] = l_r.T
    return out, lse


def ring_bwd(q, k, v, out, lse, dout, lengths, D: int, layout: str, causal: bool,
             varlen: bool, scale: float | None = None, steps=None, ranks=None):
    """Ring backward over shard-major tensors, using the final ``out`` and ``lse``.

    Returns shard-major dq [T, Hq, Dh], dk and dv [T, Hkv, Dh]. ``steps`` and ``ranks``
    (default: all) keep only the terms of those ring steps and query ranks, i.e. the block
    gradients the unfused path adds one step at a time (how-to page, "Backward Pass and
    Gradient Accumulation": dq += block_dq per step; block_dk / block_dv travel back to the
    shard that owns the K/V).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    out = np.asarray(out, np.float64)
    lse = np.asarray(lse, np.float64)
    dout = np.asarray(dout, np.float64)
    t, hq, dh = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    scale = 1.0 / np.sqrt(dh) if scale is None else scale
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for i, n in enumerate(lengths):
        pos = shard_positions(layout, D, n)
        for r in range(D):
            if ranks is not None and r not in ranks:
                continue
            rq = piece_rows(lengths, D, varlen, i, r)
            delta = (dout[rq] * out[rq]).sum(axis=2)  # [L, Hq]: rowsum(dO * O), final O
            for s in range(D):
                if steps is not None and s not in steps:
                    continue
                j = (r - s) % D
                rk = piece_rows(lengths, D, varlen, i, j)
                allowed = ((pos[j][None, :] <= pos[r][:, None]) if causal
                           else np.ones((rq.size, rk.size), bool))
                for h in range(hq):
                    kv = h // g
                    sc = scale * (q[rq, h, :] @ k[rk, kv, :].T)
                    final_lse = lse[h, rq]
                    p = np.where(allowed, np.exp(np.where(allowed, sc, 0.0) - final_lse[:, None]), 0.0)
                    dv[rk, kv, :] += p.T @ dout[rq, h, :]
                    dp = dout[rq, h, :] @ v[rk, kv, :].T
                    ds = p * (dp - delta[:, h][:, None])
                    dq[rq, h, :] += scale * (ds @ k[rk, kv, :])
                    dk[rk, kv, :] += scale * (ds.T @ q[rq, h, :])
    return dq, dk, dv


def step_allowed(layout: str, D: int, n: int, rank: int, step: int, causal: bool):
    """Boolean [L, L] mask of (local query, local key) pairs rank ``rank`` computes at
    ``step`` for one sequence of length ``n`` (global-position rule)."""
    pos = shard_positions(layout, D, n)
    j = (rank - step) % D
    if not causal:
        return np.ones((n // D, n // D), bool)
    return pos[j][None, :] <= pos[rank][:, None]
