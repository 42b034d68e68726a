"""Seeded synthetic workloads for ring attention: shapes, seeds and input tensors only.

Both sides of the parity check draw their inputs from here: the CUDA path (tests, bench,
smoke) and the float64 oracle (tests, CPU baseline). This module therefore holds none of
the method's arithmetic. It draws normal random numbers, rounds them to the storage dtype
(round-to-nearest-even to bfloat16, or to float32) and describes the shapes.

The five named workloads follow the long-context training shapes the ring attention pages
describe (sequence split into D shards that each hold N/D tokens; "Ring Attention" concept
page, section "Sequence sharding and the ring topology"), plus the two-device NumPy check of
the same page (section "Show Me the Code": seed 5, n=8, d=16, inputs scaled by 0.1).

Tensors are returned in natural (global position) order. Batch mode is ``[B, S, H, Dh]``;
varlen mode is packed ``[T, H, Dh]`` with ``cu_seqlens`` (int32, n+1 entries).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

LAYOUTS = ("basic", "zigzag", "stripe")


@dataclass(frozen=True)
class Workload:
    """One ring-attention problem: shapes, ring size D, shard layout, seed."""

    name: str
    dtype: str  # "f32" or "bf16": storage dtype of q, k, v, out, dout
    layout: str  # "basic" | "zigzag" | "stripe"
    causal: bool
    D: int  # number of virtual ring shards
    hq: int
    hkv: int
    head_dim: int
    seed: int
    batch: int = 0  # batch mode: B (0 in varlen mode)
    seqlen: int = 0  # batch mode: S
    seqlens: tuple = field(default_factory=tuple)  # varlen mode: per-sequence lengths
    input_scale: float = 1.0
    backward: bool = True

    # ---- shape helpers -------------------------------------------------------------
    @property
    def varlen(self) -> bool:
        return len(self.seqlens) > 0

    @property
    def lengths(self) -> list[int]:
        """Per-sequence lengths (batch mode: B copies of S)."""
        return list(self.seqlens) if self.varlen else [self.seqlen] * self.batch

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    def token_shape(self, heads: int) -> tuple:
        if self.varlen:
            return (self.total_tokens, heads, self.head_dim)
        return (self.batch, self.seqlen, heads, self.head_dim)

    def lse_shape(self) -> tuple:
        if self.varlen:
            return (self.hq, self.total_tokens)
        return (self.batch, self.hq, self.seqlen)

    def with_layout(self, layout: str) -> "Workload":
        return replace(self, layout=layout, name=_rename(self.name, layout))

    def causal_pairs(self) -> int:
        """Number of (query, key) pairs the attention visits, summed over query heads."""
        n = 0
        for ln in self.lengths:
            n += ln * (ln + 1) // 2 if self.causal else ln * ln
        return n * self.hq

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOP: two GEMMs (QK^T and PV), 4*Dh per visited pair.

        The causal count uses S^2/2 pairs per sequence and head (the diagonal's extra S/2
        pairs are not counted), as is usual for attention FLOP accounting.
        """
        pairs = 0.0
        for ln in self.lengths:
            pairs += (ln * ln / 2.0) if self.causal else float(ln * ln)
        return 4.0 * self.head_dim * pairs * self.hq


def _rename(name: str, layout: str) -> str:
    for lay in LAYOUTS:
        if name.endswith("_" + lay):
            return name[: -len(lay)] + layout
    return name + "_" + layout


# ---- number generation ------------------------------------------------------------------

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return rounded.view(np.float32).reshape(x.shape)


def _draw(rng: np.random.Generator, shape: tuple, w: Workload) -> np.ndarray:
    if w.dtype == "f32":
        # float64 draws, as in the two-device NumPy check, stored as float32
        return (rng.standard_normal(shape) * w.input_scale).astype(np.float32)
    x = rng.standard_normal(shape, dtype=np.float32)
    if w.input_scale != 1.0:
        x *= np.float32(w.input_scale)
    return round_to_bf16(x)


def make_qkv(w: Workload) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Q, K, V in natural order, drawn in that order from ``default_rng(seed)``.

    Values are exactly representable in the storage dtype (float32 arrays whose values are
    bf16 numbers for bf16 workloads), so both sides read identical inputs.
    """
    rng = np.random.default_rng(w.seed)
    q = _draw(rng, w.token_shape(w.hq), w)
    k = _draw(rng, w.token_shape(w.hkv), w)
    v = _draw(rng, w.token_shape(w.hkv), w)
    return q, k, v


def make_dout(w: Workload) -> np.ndarray:
    """Upstream gradient dO ~ N(0,1) in the storage dtype, seed = workload seed + 1."""
    rng = np.random.default_rng(w.seed + 1)
    return _draw(rng, w.token_shape(w.hq), replace(w, input_scale=1.0))


def varlen_lengths(n: int = 16, total: int = 65536, lo: int = 256, hi: int = 16384,
                   multiple: int = 16, seed: int = 1003) -> tuple:
    """Log-uniform sequence lengths in [lo, hi] that sum to ``total``.

    Draw u_i ~ U(ln lo, ln hi); rescale e^{u_i} to the total and clip, a few times; round
    to multiples of ``multiple`` (2D, so every zigzag chunk is whole); then move the
    remainder in steps of ``multiple`` onto the lengths that stay in range.
    """
    rng = np.random.default_rng(seed)
    ln = np.exp(rng.uniform(np.log(lo), np.log(hi), n))
    for _ in range(8):
        ln = np.clip(ln * (total / ln.sum()), lo, hi)
    ln = np.clip(np.round(ln / multiple).astype(np.int64) * multiple, lo, hi)
    diff = total - int(ln.sum())
    guard = 0
    while diff != 0 and guard < 100000:
        guard += 1
        if diff > 0:
            order = np.argsort(ln, kind="stable")
            for i in order:
                if ln[i] + multiple <= hi:
                    ln[i] += multiple
                    diff -= multiple
                    break
        else:
            order = np.argsort(-ln, kind="stable")
            for i in order:
                if ln[i] - multiple >= lo:
                    ln[i] -= multiple
                    diff += multiple
                    break
    assert int(ln.sum()) == total
    return tuple(int(x) for x in ln)


# ---- the named workloads ----------------------------------------------------------------

TINY = Workload(
    name="tiny_f32_n8_dh16_D2_basic", dtype="f32", layout="basic", causal=False, D=2,
    hq=1, hkv=1, head_dim=16, seed=5, batch=1, seqlen=8, input_scale=0.1, backward=False)

BATCH = Workload(
    name="batch_b2_s4096_h8_dh64_D4_basic", dtype="bf16", layout="basic", causal=True, D=4,
    hq=8, hkv=8, head_dim=64, seed=1001, batch=2, seqlen=4096)

LONG32K = Workload(
    name="long_s32768_h16_dh128_D8_zigzag", dtype="bf16", layout="zigzag", causal=True,
    D=8, hq=16, hkv=16, head_dim=128, seed=1002, batch=1, seqlen=32768)

VARLEN = Workload(
    name="varlen_t65536_16seq_gqa32x8_dh128_D8_zigzag", dtype="bf16", layout="zigzag",
    causal=True, D=8, hq=32, hkv=8, head_dim=128, seed=1003,
    seqlens=varlen_lengths(seed=1003))

LONG128K = Workload(
    name="long_s131072_gqa32x8_dh128_D16_zigzag", dtype="bf16", layout="zigzag",
    causal=True, D=16, hq=32, hkv=8, head_dim=128, seed=1004, batch=1, seqlen=131072)

NAMED = {w.name: w for w in (TINY, BATCH, LONG32K, LONG32K.with_layout("stripe"), VARLEN,
                             VARLEN.with_layout("basic"), VARLEN.with_layout("stripe"),
                             LONG128K)}
