"""Autograd wrappers and a drop-in attention module over the ring-attention C ABI.

The ring-flash-attn package card ("quickstart") shows the adapter use of ring attention:
a model keeps its projections and swaps its attention call for the ring one, and the
nanotron how-to page ("Integrating with MultiHeadAttention") selects ring attention by
name in its attention registry. Here the same is done on one GPU: ``ring_attention`` is a
differentiable call (forward = ``ra_ring_attn_fwd``, backward = ``ra_ring_attn_bwd`` against
the saved out and lse), ``shard`` / ``unshard`` move token tensors between natural and
shard-major order with their inverse permutation as gradient, and ``RingSelfAttention``
is a multi-head (GQA) self-attention layer with random weights that uses them.
"""
from __future__ import annotations

import math

import torch

from . import ops


class _RingAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, prob):
        out, lse = ops.ring_attn_fwd(q, k, v, prob)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.prob = prob
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = ops.ring_attn_bwd(dout.contiguous(), q, k, v, out, lse, ctx.prob)
        return dq, dk, dv, None


class _Shard(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, prob, direction):
        ctx.prob = prob
        ctx.direction = direction
        x = x.contiguous()
        return ops.shard_tokens(x, prob) if direction == 0 else ops.unshard_tokens(x, prob)

    @staticmethod
    def backward(ctx, g):
        g = g.contiguous()
        back = ops.unshard_tokens(g, ctx.prob) if ctx.direction == 0 else ops.shard_tokens(g, ctx.prob)
        return back, None, None


def ring_attention(q, k, v, prob: ops.Problem):
    """Differentiable ring attention on shard-major q, k, v; returns (out, lse)."""
    return _RingAttention.apply(q, k, v, prob)


def shard(x, prob: ops.Problem):
    """Natural -> shard-major order (gradient: the inverse permutation)."""
    return _Shard.apply(x, prob, 0)


def unshard(x, prob: ops.Problem):
    """Shard-major -> natural order (gradient: the inverse permutation)."""
    return _Shard.apply(x, prob, 1)


class RingSelfAttention(torch.nn.Module):
    """Self-attention with ring attention as its attention call.

    x [B, S, hidden] (natural order) -> y [B, S, hidden]. Query / key / value / output
    projections are ordinary linear layers (random initialisation, no bias); the attention
    between them runs through the library with D virtual ring shards in the chosen layout.
    With ``shard_major=True`` x and y are already shard-major (a model that shards its
    tokens once at the input keeps them so through every token-wise layer).
    """

    def __init__(self, hidden: int, hq: int, hkv: int, head_dim: int, *, D: int,
                 layout: str = "zigzag", causal: bool = True, shard_major: bool = False,
                 device=None, dtype=torch.bfloat16, seed: int = 0):
        super().__init__()
        if hq % hkv:
            raise ValueError("hq must be a multiple of hkv")
        self.hq, self.hkv, self.head_dim = hq, hkv, head_dim
        self.D, self.layout, self.causal, self.shard_major = D, layout, causal, shard_major
        g = torch.Generator().manual_seed(seed)

        def lin(n_out, n_in):
            w = torch.randn(n_out, n_in, generator=g) / math.sqrt(n_in)
            return torch.nn.Parameter(w.to(device=device, dtype=dtype))

        self.wq = lin(hq * head_dim, hidden)
        self.wk = lin(hkv * head_dim, hidden)
        self.wv = lin(hkv * head_dim, hidden)
        self.wo = lin(hidden, hq * head_dim)

    def problem(self, batch: int, seqlen: int) -> ops.Problem:
        return ops.make_problem(dtype=self.wq.dtype, layout=self.layout, causal=self.causal,
                                D=self.D, hq=self.hq, hkv=self.hkv, head_dim=self.head_dim,
                                batch=batch, seqlen=seqlen)

    def forward(self, x):
        b, s, _ = x.shape
        prob = self.problem(b, s)
        q = (x @ self.wq.t()).view(b, s, self.hq, self.head_dim)
        k = (x @ self.wk.t()).view(b, s, self.hkv, self.head_dim)
        v = (x @ self.wv.t()).view(b, s, self.hkv, self.head_dim)
        if not self.shard_major:
            q, k, v = shard(q, prob), shard(k, prob), shard(v, prob)
        out, _ = ring_attention(q.contiguous(), k.contiguous(), v.contiguous(), prob)
        if not self.shard_major:
            out = unshard(out, prob)
        return out.reshape(b, s, self.hq * self.head_dim) @ self.wo.t()
