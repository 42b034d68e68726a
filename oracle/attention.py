"""Plain softmax attention in float64 — the result ring attention reaches exactly.

The Ring Attention concept page states that the ring's final output is exact ("Online
softmax across ring steps"; "Show Me the Code" checks a two-device ring against a
single-device pass) and the interview question page says it keeps "the same exact math".
So the oracle's definition of the hot path's result is single-pass attention:

    S   = scale * Q_h K_g^T            g = floor(h * Hkv / Hq)  (grouped-query heads)
    S  += mask                         -inf where the key is in another sequence, or,
                                       when causal, at a later global position
    lse = log sum_j exp(S_ij)          natural log, computed with the row max subtracted
    out = exp(S - lse) V_g

``scale`` defaults to 1/sqrt(Dh) (nanotron how-to page, "Calling the Ring Attention
Function Directly": ``scaling=None`` means 1/sqrt(head_dim); the concept page's code divides
the scores by d**0.5).

The backward is the textbook chain rule of that definition: dV = P^T dO, dP = dO V^T,
dS = P * (dP - rowsum(P * dP)), dQ = scale dS K, dK = scale dS^T Q, with dK and dV of a
KV head summed over its query heads. (rowsum(P * dP) equals rowsum(dO * O).)

All arrays are packed ``[T, H, Dh]`` float64 in natural order with ``cu_seqlens``; use
``to_packed`` / ``lse_from_packed`` for batch-mode ``[B, S, H, Dh]`` tensors. Query rows are
processed in independent blocks only to bound memory; for a causal block, keys after the
block's last row are left out, which drops exact zeros and nothing else.
"""
from __future__ import annotations

import numpy as np

ROW_BLOCK = 512


def default_scale(head_dim: int) -> float:
    return 1.0 / np.sqrt(head_dim)


def to_packed(x: np.ndarray) -> np.ndarray:
    """[B, S, H, Dh] -> [B*S, H, Dh] (varlen tensors pass through)."""
    if x.ndim == 4:
        return x.reshape(x.shape[0] * x.shape[1], x.shape[2], x.shape[3])
    return x


def lse_from_packed(lse: np.ndarray, batch: int) -> np.ndarray:
    """[Hq, B*S] -> [B, Hq, S] (batch mode); ``batch=0`` keeps the varlen [Hq, T] form."""
    if batch == 0:
        return lse
    hq, t = lse.shape
    return lse.reshape(hq, batch, t // batch).transpose(1, 0, 2).copy()


def _group(hq: int, hkv: int) -> int:
    if hq % hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    return hq // hkv


def attention_fwd(q, k, v, cu_seqlens, causal: bool, scale: float | None = None,
                  rows=None, heads=None):
    """Forward by definition. Returns ``out`` [T, Hq, Dh] and ``lse`` [Hq, T] (float64).

    ``rows`` (natural query rows) and ``heads`` restrict the evaluation; rows or heads that
    are not evaluated are left as NaN.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    t, hq, dh = q.shape
    g = _group(hq, k.shape[1])
    scale = default_scale(dh) if scale is None else scale
    out = np.full((t, hq, dh), np.nan)
    lse = np.full((hq, t), np.nan)
    heads = range(hq) if heads is None else heads
    want = None if rows is None else np.zeros(t, bool)
    if want is not None:
        want[np.asarray(rows)] = True
    for s0, s1 in zip(cu_seqlens[:-1], cu_seqlens[1:]):
        s0, s1 = int(s0), int(s1)
        seq_rows = np.arange(s0, s1)
        if want is not None:
            seq_rows = seq_rows[want[s0:s1]]
        for b0 in range(0, seq_rows.size, ROW_BLOCK):
            r = seq_rows[b0:b0 + ROW_BLOCK]
            kend = (int(r.max()) + 1) if causal else s1
            i_loc = r - s0
            j_loc = np.arange(kend - s0)
            allowed = (j_loc[None, :] <= i_loc[:, None]) if causal else None
            for h in heads:
                kv = h // g
                s = scale * (q[r, h, :] @ k[s0:kend, kv, :].T)
                if allowed is not None:
                    s = np.where(allowed, s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                l = e.sum(axis=1, keepdims=True)
                row_lse = m + np.log(l)
                out[r, h, :] = (e / l) @ v[s0:kend, kv, :]
                lse[h, r] = row_lse[:, 0]
    return out, lse


def attention_bwd(q, k, v, dout, cu_seqlens, causal: bool, scale: float | None = None,
                  rows=None, heads=None):
    """Backward by definition. Returns ``dq`` [T, Hq, Dh], ``dk``, ``dv`` [T, Hkv, Dh].

    ``rows`` restricts the query rows whose contributions are summed: dq is exact on those
    rows (NaN elsewhere); dk and dv hold the contributions of those rows only, which is the
    whole gradient for keys that only those rows can see. ``heads`` restricts query heads.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    t, hq, dh = q.shape
    hkv = k.shape[1]
    g = _group(hq, hkv)
    scale = default_scale(dh) if scale is None else scale
    dq = np.full((t, hq, dh), np.nan)
    dk = np.zeros((t, hkv, dh))
    dv = np.zeros((t, hkv, dh))
    heads = range(hq) if heads is None else heads
    want = None if rows is None else np.zeros(t, bool)
    if want is not None:
        want[np.asarray(rows)] = True
    for s0, s1 in zip(cu_seqlens[:-1], cu_seqlens[1:]):
        s0, s1 = int(s0), int(s1)
        seq_rows = np.arange(s0, s1)
        if want is not None:
            seq_rows = seq_rows[want[s0:s1]]
        for b0 in range(0, seq_rows.size, ROW_BLOCK):
            r = seq_rows[b0:b0 + ROW_BLOCK]
            kend = (int(r.max()) + 1) if causal else s1
            i_loc = r - s0
            j_loc = np.arange(kend - s0)
            allowed = (j_loc[None, :] <= i_loc[:, None]) if causal else None
            for h in heads:
                kv = h // g
                kk = k[s0:kend, kv, :]
                vv = v[s0:kend, kv, :]
                qq = q[r, h, :]
                do = dout[r, h, :]
                s = scale * (qq @ kk.T)
                if allowed is not None:
                    s = np.where(allowed, s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                p = e / e.sum(axis=1, keepdims=True)
                dv[s0:kend, kv, :] += p.T @ do
                dp = do @ vv.T
                ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
                dq[r, h, :] = scale * (ds @ kk)
                dk[s0:kend, kv, :] += scale * (ds.T @ qq)
    return dq, dk, dv
