"""Shard layouts of ring attention (oracle side, float64-free integer code).

A sequence of N tokens is split across D ranks, each holding N/D tokens ("Ring Attention"
concept page, section "Sequence sharding and the ring topology"). The ring-flash-attn
package card ("What it is and what it does") names three ways to split it:

* basic: rank r holds the contiguous block of tokens [r*N/D, (r+1)*N/D);
* zigzag ("more compute-balanced"): the sequence is cut into 2D equal chunks and rank r
  holds chunk r followed by chunk 2D-1-r;
* stripe (Striped Attention, interview question page): token t goes to rank t mod D, in
  increasing t.

Each function here builds the split literally (reshape and concatenate the list of global
token indices) rather than from a closed form, so that it checks the CUDA path's arithmetic.

Tensors handed to the ring are *shard-major*: the D local buffers concatenated. In batch
mode that is per batch element along S; in varlen (packed) mode each sequence is split
separately and rank r's buffer is the concatenation of its pieces of every sequence, so the
local ``cu_seqlens`` of every rank is ``cu_seqlens / D``.
"""
from __future__ import annotations

import numpy as np


def shard_positions(layout: str, D: int, n: int) -> np.ndarray:
    """Global position of every shard-major slot of one sequence of length ``n``.

    Returns ``pos`` of shape (D, n // D): ``pos[r, a]`` is the global index of local token
    ``a`` of rank ``r``.
    """
    if n % D:
        raise ValueError("sequence length must divide by D")
    tokens = np.arange(n, dtype=np.int64)
    if layout == "basic":
        return tokens.reshape(D, n // D).copy()
    if layout == "zigzag":
        if n % (2 * D):
            raise ValueError("zigzag needs the sequence length to divide by 2D")
        chunks = tokens.reshape(2 * D, n // (2 * D))
        return np.stack([np.concatenate([chunks[r], chunks[2 * D - 1 - r]])
                         for r in range(D)])
    if layout == "stripe":
        # token t lives on rank t mod D; listing tokens in rows of D puts rank r in column r
        return tokens.reshape(n // D, D).T.copy()
    raise ValueError(f"unknown layout {layout!r}")


def shard_major_rows(layout: str, D: int, lengths: list[int], varlen: bool) -> np.ndarray:
    """For the whole (flattened) token axis: natural row index of every shard-major row.

    Batch mode (``varlen=False``): the token axis is B*S, batch element b occupies rows
    [b*S, (b+1)*S) in both orders and is sharded on its own.
    Varlen mode: packed rows; rank r's buffer starts at r*T/D and holds, for every sequence
    i in order, that sequence's local piece of length len_i/D.
    """
    total = int(sum(lengths))
    out = np.empty(total, dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    if not varlen:
        for i, n in enumerate(lengths):
            pos = shard_positions(layout, D, n)  # (D, L)
            out[starts[i]:starts[i] + n] = starts[i] + pos.reshape(-1)
        return out
    if total % D:
        raise ValueError("total tokens must divide by D")
    per_rank = total // D
    for i, n in enumerate(lengths):
        pos = shard_positions(layout, D, n)
        L = n // D
        for r in range(D):
            base = r * per_rank + starts[i] // D
            out[base:base + L] = starts[i] + pos[r]
    return out


def shard(x: np.ndarray, rows: np.ndarray, axis: int) -> np.ndarray:
    """Natural order -> shard-major along ``axis`` (``rows`` from ``shard_major_rows``)."""
    return np.take(x, rows, axis=axis)


def unshard(x: np.ndarray, rows: np.ndarray, axis: int) -> np.ndarray:
    """Shard-major -> natural order along ``axis``."""
    inv = np.empty_like(rows)
    inv[rows] = np.arange(rows.size, dtype=rows.dtype)
    return np.take(x, inv, axis=axis)
