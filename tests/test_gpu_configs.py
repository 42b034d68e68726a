"""GPU parity on the named workloads, in the launch configuration the benchmark times.

The two-device page example and the 4096-token batch workload are checked against the full
oracle. The 32K, varlen 64K and 128K workloads are too large for a float64 CPU pass, so they
are checked on outputs the oracle computes one by one:

* out, lse and dq on sampled query rows of every head (rows at every shard / chunk boundary
  of the layout plus random rows): each is exact from its own row of scores;
* dk and dv on the K/V rows of the last 128 positions of every sequence: under the causal
  rule only the last 128 queries see them, so those queries' gradients give them exactly;
* at any size: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per K/V head and sequence;
* for the 32K (one head), varlen 64K and 128K (one group of four query heads) workloads,
  dq, dk and dv of one whole K/V-head group, every row, against the oracle's backward of
  that group (run over row chunks in spawned processes).
"""
import numpy as np
import pytest
import torch

import context_blockwise_attention_step_gb300 as ra
import workloads as W
from oracle import attention as A
from oracle import layouts as LY

from _gpu_path import assert_grad, assert_lse, assert_out, packed, run
from _oracle_pool import group_backward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ra.build()
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")


def test_two_device_page_example():
    w = W.TINY
    res, (q, k, v, _) = run(w)
    out, lse = A.attention_fwd(packed(q), packed(k), packed(v), w.cu_seqlens, False)
    assert_out(w, res["out"], out)
    assert_lse(w, res["lse"], lse)


def test_batch_4096_full_oracle():
    w = W.BATCH
    res, (q, k, v, do) = run(w)
    cu = w.cu_seqlens
    out, lse = A.attention_fwd(packed(q), packed(k), packed(v), cu, True)
    assert_out(w, res["out"], out)
    assert_lse(w, res["lse"], lse)
    grads = A.attention_bwd(packed(q), packed(k), packed(v), packed(do), cu, True)
    for name, ref in zip(("dq", "dk", "dv"), grads):
        assert_grad(w, name, res[name], ref)


def sample_rows(w: W.Workload, n_random=24, seed=99):
    """Natural-order query rows: boundaries of every shard piece and zigzag chunk, plus random."""
    rng = np.random.default_rng(seed)
    rows = []
    start = 0
    for n in w.lengths:
        L = n // w.D
        pos = LY.shard_positions(w.layout, w.D, n)
        edges = set()
        for r in range(w.D):
            for a in (0, 1, 127, 128, L // 2 - 1, L // 2, L - 2, L - 1):
                if 0 <= a < L:
                    edges.add(int(pos[r, a]))
        edges.update(int(x) for x in rng.integers(0, n, size=min(n, n_random)))
        rows.extend(start + p for p in sorted(edges))
        start += n
    return np.array(sorted(set(rows)), dtype=np.int64)


def tail_rows(w: W.Workload, width=128):
    rows, start = [], 0
    for n in w.lengths:
        rows.extend(range(start + max(0, n - width), start + n))
        start += n
    return np.array(rows, dtype=np.int64)


FULL_GROUP = {W.LONG32K.name, W.VARLEN.name, W.LONG128K.name}

LARGE = [W.LONG32K, W.LONG32K.with_layout("stripe"), W.VARLEN, W.VARLEN.with_layout("basic"),
         W.VARLEN.with_layout("stripe"), W.LONG128K]


@pytest.mark.slow
@pytest.mark.parametrize("w", LARGE, ids=lambda w: w.name)
def test_large_workload_sampled(w):
    res, (q, k, v, do) = run(w)
    cu = w.cu_seqlens
    qp, kp, vp, dop = (packed(x) for x in (q, k, v, do))
    rows = sample_rows(w)
    out, lse = A.attention_fwd(qp, kp, vp, cu, True, rows=rows)
    assert_out(w, res["out"], out, rows=rows)
    assert_lse(w, res["lse"], lse, rows=rows)
    dq, _, _ = A.attention_bwd(qp, kp, vp, dop, cu, True, rows=rows)
    assert_grad(w, "dq", res["dq"], dq, rows=rows)
    tail = tail_rows(w)
    _, dk, dv = A.attention_bwd(qp, kp, vp, dop, cu, True, rows=tail)
    assert_grad(w, "dk", res["dk"], dk, rows=tail)
    assert_grad(w, "dv", res["dv"], dv, rows=tail)
    # sum rules over every key of every sequence
    gdk, gdv = packed(res["dk"]).astype(np.float64), packed(res["dv"]).astype(np.float64)
    g = w.hq // w.hkv
    for s0, s1 in zip(cu[:-1], cu[1:]):
        sum_dk = gdk[s0:s1].sum(axis=0)
        scale_dk = np.abs(gdk[s0:s1]).sum(axis=0).max()
        assert np.abs(sum_dk).max() <= 2e-2 * scale_dk
        want = dop[s0:s1].astype(np.float64).reshape(s1 - s0, w.hkv, g, w.head_dim).sum(axis=(0, 2))
        got = gdv[s0:s1].sum(axis=0)
        assert np.linalg.norm(got - want) <= 2e-2 * np.linalg.norm(want) + 1e-3
    # every row of one whole K/V-head group
    if w.name in FULL_GROUP:
        hk = w.hkv - 1
        dq_g, dk_g, dv_g = group_backward(qp, kp, vp, dop, cu, True, hk, g)
        assert_grad(w, "dq (group)", packed(res["dq"])[:, hk * g:(hk + 1) * g], dq_g)
        assert_grad(w, "dk (group)", packed(res["dk"])[:, hk:hk + 1], dk_g)
        assert_grad(w, "dv (group)", packed(res["dv"])[:, hk:hk + 1], dv_g)
