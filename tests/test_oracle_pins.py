"""Pins of the float64 oracle to things other than itself (CPU only).

* the two-device worked example of the Ring Attention concept page ("Show Me the Code");
* brute force: pure-Python scalar loops over tiny inputs;
* closed forms: uniform weights when K = 0 or Q = 0 (lse = ln #keys, out = mean of V);
* invariants: softmax rows sum to 1, the merge is associative / commutative with -inf as
  identity, ring == single pass for every D, layout, mode;
* central finite differences for the backward;
* the layout and causal-rule fixtures under tests/golden.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import attention as A
from oracle import layouts as LY
from oracle import ring as R
import workloads as W


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------------------
# the concept page's two-device example
# ---------------------------------------------------------------------------------------

def _page_inputs(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "p3_two_device.json")))
    rng = np.random.default_rng(g["seed"])
    n, d = g["n"], g["d"]
    qkv = [rng.standard_normal((n, d)) * g["input_scale"] for _ in g["draw_order"]]
    return g, qkv


def test_two_device_example_ring_equals_single_pass(golden_dir):
    g, (q, k, v) = _page_inputs(golden_dir)
    n, d = g["n"], g["d"]
    qp, kp, vp = (x.reshape(n, 1, d) for x in (q, k, v))
    cu = np.array([0, n], np.int32)
    out_ref, lse_ref = A.attention_fwd(qp, kp, vp, cu, causal=False)
    out_ring, lse_ring = R.ring_fwd(qp, kp, vp, [n], g["devices"], "basic", False, False)
    # basic layout: shard-major order is the natural order
    assert np.abs(out_ring - out_ref).max() <= 10 * g["claimed_max_difference"]
    assert np.abs(lse_ring - lse_ref).max() <= 1e-14
    # tiny inputs: every score is near zero, so lse is near ln(n)
    assert np.abs(lse_ref - math.log(n)).max() < 0.02


def test_two_device_example_rotation(golden_dir):
    """Device 0 sees KV0 then KV1; device 1 sees KV1 then KV0."""
    g, _ = _page_inputs(golden_dir)
    D = g["devices"]
    seen = {f"device{r}": [f"KV{(r - s) % D}" for s in range(D)] for r in range(D)}
    assert seen == g["rotation"]


def test_two_device_example_printed_combine_is_not_exact(golden_dir):
    """The page's printed combine weighs unnormalised block outputs by sums taken against
    different per-block maxima. It misses the single pass by far more than rounding, which
    is why the oracle merges by log-sum-exp instead."""
    g, (q, k, v) = _page_inputs(golden_dir)
    n, d = g["n"], g["d"]
    h = n // 2

    def page_block(qq, kk, vv):
        s = qq @ kk.T / d ** 0.5
        s = s - s.max(-1, keepdims=True)
        w = np.exp(s)
        return w @ vv, w.sum(-1)

    halves = []
    for qq in (q[:h], q[h:]):
        oa, wa = page_block(qq, k[:h], v[:h])
        ob, wb = page_block(qq, k[h:], v[h:])
        halves.append((oa * wa[:, None] + ob * wb[:, None]) / (wa + wb)[:, None])
    printed = np.vstack(halves)
    ref, _ = A.attention_fwd(q.reshape(n, 1, d), k.reshape(n, 1, d), v.reshape(n, 1, d),
                             np.array([0, n]), causal=False)
    assert np.abs(printed - ref[:, 0, :]).max() > 1e-2


def test_tiny_workload_reproduces_page_inputs(golden_dir):
    _, (q, k, v) = _page_inputs(golden_dir)
    tq, tk, tv = W.make_qkv(W.TINY)
    assert tq.shape == (1, 8, 1, 16)
    for a, b in ((q, tq), (k, tk), (v, tv)):
        np.testing.assert_array_equal(a.astype(np.float32), b.reshape(8, 16))


# ---------------------------------------------------------------------------------------
# brute force on tiny inputs
# ---------------------------------------------------------------------------------------

def _brute_force(q, k, v, cu, causal, scale):
    t, hq, dh = q.shape
    g = hq // k.shape[1]
    out = np.zeros((t, hq, dh))
    lse = np.zeros((hq, t))
    for s0, s1 in zip(cu[:-1], cu[1:]):
        for i in range(s0, s1):
            for h in range(hq):
                keys = [j for j in range(s0, s1) if (not causal or j <= i)]
                sc = [scale * sum(float(q[i, h, c]) * float(k[j, h // g, c]) for c in range(dh))
                      for j in keys]
                mx = max(sc)
                ws = [math.exp(x - mx) for x in sc]
                tot = sum(ws)
                lse[h, i] = mx + math.log(tot)
                for c in range(dh):
                    out[i, h, c] = sum(w * float(v[j, h // g, c]) for w, j in zip(ws, keys)) / tot
    return out, lse


@pytest.mark.parametrize("causal", [False, True])
def test_plain_attention_matches_brute_force(causal):
    rng = _rng(11)
    cu = np.array([0, 5, 12], np.int32)
    q = rng.standard_normal((12, 4, 3))
    k = rng.standard_normal((12, 2, 3))
    v = rng.standard_normal((12, 2, 3))
    out, lse = A.attention_fwd(q, k, v, cu, causal, scale=0.7)
    bo, bl = _brute_force(q, k, v, cu, causal, 0.7)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def test_block_attention_matches_brute_force_with_global_positions():
    """A rank's block uses the global positions of its query and key tokens."""
    rng = _rng(12)
    q = rng.standard_normal((4, 2, 3))
    k = rng.standard_normal((4, 1, 3))
    v = rng.standard_normal((4, 1, 3))
    pos_q = np.array([2, 3, 12, 13])
    pos_k = np.array([0, 1, 14, 15])
    out, lse = R.block_attention(q, k, v, pos_q, pos_k, True, 0.5)
    for i in range(4):
        for h in range(2):
            keys = [j for j in range(4) if pos_k[j] <= pos_q[i]]
            sc = [0.5 * float(q[i, h] @ k[j, 0]) for j in keys]
            mx = max(sc)
            tot = sum(math.exp(x - mx) for x in sc)
            assert abs(lse[h, i] - (mx + math.log(tot))) < 1e-12
            ref = sum(math.exp(x - mx) * v[j, 0] for x, j in zip(sc, keys)) / tot
            np.testing.assert_allclose(out[i, h], ref, atol=1e-12)


def test_block_attention_fully_masked_rows():
    q = np.ones((2, 1, 2))
    k = np.ones((2, 1, 2))
    v = np.ones((2, 1, 2))
    out, lse = R.block_attention(q, k, v, np.array([0, 1]), np.array([5, 6]), True, 1.0)
    assert np.all(lse == -np.inf)
    assert np.all(out == 0)


# ---------------------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("zero", ["q", "k"])
@pytest.mark.parametrize("causal", [False, True])
def test_uniform_weights_closed_form(zero, causal):
    rng = _rng(13)
    cu = np.array([0, 7, 16], np.int32)
    q = rng.standard_normal((16, 2, 4))
    k = rng.standard_normal((16, 2, 4))
    v = rng.standard_normal((16, 2, 4))
    if zero == "q":
        q[:] = 0
    else:
        k[:] = 0
    out, lse = A.attention_fwd(q, k, v, cu, causal)
    for s0, s1 in zip(cu[:-1], cu[1:]):
        for i in range(s0, s1):
            n_keys = (i - s0 + 1) if causal else (s1 - s0)
            np.testing.assert_allclose(lse[:, i], math.log(n_keys), atol=1e-13)
            np.testing.assert_allclose(out[i], v[s0:s0 + n_keys].mean(axis=0), atol=1e-13)


def test_rows_sum_to_one_and_dominant_key():
    rng = _rng(14)
    cu = np.array([0, 9], np.int32)
    q = rng.standard_normal((9, 1, 4))
    k = rng.standard_normal((9, 1, 4))
    ones = np.ones((9, 1, 4))
    out, _ = A.attention_fwd(q, k, ones, cu, True)
    np.testing.assert_allclose(out, 1.0, atol=1e-14)
    # one key far above the rest takes all the weight
    k2 = np.zeros((9, 1, 4))
    k2[3, 0, 0] = 60.0
    q2 = np.zeros((9, 1, 4))
    q2[:, 0, 0] = 1.0
    v2 = rng.standard_normal((9, 1, 4))
    out2, _ = A.attention_fwd(q2, k2, v2, cu, False, scale=1.0)
    np.testing.assert_allclose(out2[:, 0], np.broadcast_to(v2[3, 0], (9, 4)), atol=1e-20)


# ---------------------------------------------------------------------------------------
# merge rule
# ---------------------------------------------------------------------------------------

def _blocks(rng, n=3):
    return [(rng.standard_normal((5, 2, 3)), rng.standard_normal((5, 2)) * 3) for _ in range(n)]  # out, lse


def test_merge_associative_commutative_identity():
    rng = _rng(15)
    (a, la), (b, lb), (c, lc) = _blocks(rng)
    ab = R.update_out_and_lse(a, la, b, lb)
    abc1 = R.update_out_and_lse(*ab, c, lc)
    bc = R.update_out_and_lse(b, lb, c, lc)
    abc2 = R.update_out_and_lse(a, la, *bc)
    np.testing.assert_allclose(abc1[0], abc2[0], atol=1e-14)
    np.testing.assert_allclose(abc1[1], abc2[1], atol=1e-14)
    ba = R.update_out_and_lse(b, lb, a, la)
    np.testing.assert_allclose(ab[0], ba[0], atol=1e-15)
    np.testing.assert_allclose(ab[1], ba[1], atol=1e-15)
    ninf = np.full_like(la, -np.inf)
    ident = R.update_out_and_lse(np.zeros_like(a), ninf, a, la)
    np.testing.assert_allclose(ident[0], a, atol=1e-15)
    np.testing.assert_array_equal(ident[1], la)
    both = R.update_out_and_lse(np.zeros_like(a), ninf, np.zeros_like(a), ninf)
    assert np.all(both[1] == -np.inf) and np.all(both[0] == 0) and not np.isnan(both[0]).any()


def test_merge_of_disjoint_key_sets_equals_attention_over_union():
    rng = _rng(16)
    q = rng.standard_normal((6, 1, 4))
    k = rng.standard_normal((10, 1, 4))
    v = rng.standard_normal((10, 1, 4))
    parts = [np.arange(0, 3), np.arange(3, 7), np.arange(7, 10)]
    out = np.zeros((6, 1, 4))
    lse = np.full((6, 1), -np.inf)
    posq = np.full(6, 100)
    for p in rng.permutation(3):
        bo, bl = R.block_attention(q, k[parts[p]], v[parts[p]], posq, parts[p], False, 0.5)
        out, lse = R.update_out_and_lse(out, lse, bo, bl.T)
    s = 0.5 * q[:, 0] @ k[:, 0].T
    ref_lse = np.log(np.exp(s).sum(1))
    ref = (np.exp(s - ref_lse[:, None])) @ v[:, 0]
    np.testing.assert_allclose(lse[:, 0], ref_lse, atol=1e-14)
    np.testing.assert_allclose(out[:, 0], ref, atol=1e-14)


# ---------------------------------------------------------------------------------------
# layouts and the per-step causal structure
# ---------------------------------------------------------------------------------------

def test_layout_fixture(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "layouts_D4_n16.json")))
    for lay in W.LAYOUTS:
        np.testing.assert_array_equal(LY.shard_positions(lay, g["D"], g["n"]), np.array(g[lay]))


@pytest.mark.parametrize("layout", W.LAYOUTS)
@pytest.mark.parametrize("D", [1, 2, 3, 4, 8])
def test_layout_is_a_bijection_and_monotone_per_shard(layout, D):
    n = 2 * D * 6
    pos = LY.shard_positions(layout, D, n)
    assert sorted(pos.reshape(-1).tolist()) == list(range(n))
    assert np.all(np.diff(pos, axis=1) > 0)


@pytest.mark.parametrize("varlen", [False, True])
def test_shard_unshard_roundtrip(varlen):
    lengths = [16, 48, 32] if varlen else [32, 32]
    rows = LY.shard_major_rows("zigzag", 4, lengths, varlen)
    x = np.arange(sum(lengths) * 2).reshape(-1, 2)
    np.testing.assert_array_equal(LY.unshard(LY.shard(x, rows, 0), rows, 0), x)


def test_causal_rule_basic_layout(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "causal_rule_basic.json")))
    for D in g["checked_D"]:
        n = 4 * D
        for r in range(D):
            for s in range(D):
                active = R.step_allowed("basic", D, n, r, s, True).any()
                assert active == (s <= r), (D, r, s)


@pytest.mark.parametrize("layout", W.LAYOUTS)
@pytest.mark.parametrize("D", [1, 2, 3, 4, 8])
def test_union_of_step_masks_is_the_causal_mask(layout, D):
    n = 2 * D * 4
    L = n // D
    pos = LY.shard_positions(layout, D, n)
    cover = np.zeros((n, n), int)
    for r in range(D):
        for s in range(D):
            j = (r - s) % D
            m = R.step_allowed(layout, D, n, r, s, True)
            for a in range(L):
                for b in range(L):
                    if m[a, b]:
                        cover[pos[r, a], pos[j, b]] += 1
    np.testing.assert_array_equal(cover, np.tril(np.ones((n, n), int)))


@pytest.mark.parametrize("D", [2, 4, 8])
def test_zigzag_and_stripe_balance(D):
    n = 2 * D * 8
    L = n // D
    for r in range(D):
        for s in range(1, D):
            assert R.step_allowed("zigzag", D, n, r, s, True).sum() == L * L // 2
            cnt = R.step_allowed("stripe", D, n, r, s, True).sum()
            assert cnt == (L * (L + 1) // 2 if s <= r else L * (L - 1) // 2)


# ---------------------------------------------------------------------------------------
# ring == single pass, forward and backward
# ---------------------------------------------------------------------------------------

def _case(rng, lengths, hq, hkv, dh, varlen):
    t = sum(lengths)
    q = rng.standard_normal((t, hq, dh))
    k = rng.standard_normal((t, hkv, dh))
    v = rng.standard_normal((t, hkv, dh))
    do = rng.standard_normal((t, hq, dh))
    return q, k, v, do


@pytest.mark.parametrize("layout", W.LAYOUTS)
@pytest.mark.parametrize("D", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("varlen", [False, True])
def test_ring_equals_single_pass(layout, D, causal, varlen):
    rng = _rng(100 + D)
    lengths = [2 * D * 2, 2 * D * 5, 2 * D] if varlen else [2 * D * 3, 2 * D * 3]
    q, k, v, do = _case(rng, lengths, 4, 2, 8, varlen)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    out, lse = A.attention_fwd(q, k, v, cu, causal)
    dq, dk, dv = A.attention_bwd(q, k, v, do, cu, causal)
    rows = LY.shard_major_rows(layout, D, lengths, varlen)
    sm = lambda x: LY.shard(x, rows, 0)
    o_r, l_r = R.ring_fwd(sm(q), sm(k), sm(v), lengths, D, layout, causal, varlen)
    np.testing.assert_allclose(LY.unshard(o_r, rows, 0), out, atol=1e-12)
    np.testing.assert_allclose(LY.unshard(l_r, rows, 1), lse, atol=1e-12)
    g = R.ring_bwd(sm(q), sm(k), sm(v), o_r, l_r, sm(do), lengths, D, layout, causal, varlen)
    for got, ref in zip(g, (dq, dk, dv)):
        np.testing.assert_allclose(LY.unshard(got, rows, 0), ref, atol=1e-11)


@pytest.mark.parametrize("layout", W.LAYOUTS)
def test_per_step_backward_blocks(layout):
    """The per-(rank, step) backward terms of the unfused path: the dk / dv a rank's step
    adds into K/V shard (r - s) mod D are the gradient that rank's query rows alone give
    those keys (plain definition restricted to the rank's rows), and summing the steps'
    dq, dk, dv gives the whole gradient."""
    rng = _rng(23)
    D, lengths = 4, [48, 16]
    q, k, v, do = _case(rng, lengths, 4, 2, 6, True)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    rows = LY.shard_major_rows(layout, D, lengths, True)
    sm = lambda x: LY.shard(x, rows, 0)
    un = lambda x: LY.unshard(x, rows, 0)
    out, lse = A.attention_fwd(q, k, v, cu, True)
    dq, dk, dv = A.attention_bwd(q, k, v, do, cu, True)
    o_s, l_s = sm(out), LY.shard(lse, rows, 1)
    tot = [np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv)]
    for r in range(D):
        # natural rows of rank r's query pieces
        nat_rows = np.sort(np.concatenate([rows[R.piece_rows(lengths, D, True, i, r)]
                                           for i in range(len(lengths))]))
        _, dk_r, dv_r = A.attention_bwd(q, k, v, do, cu, True, rows=nat_rows)
        for s in range(D):
            g = R.ring_bwd(sm(q), sm(k), sm(v), o_s, l_s, sm(do), lengths, D, layout, True, True,
                           steps=[s], ranks=[r])
            j = (r - s) % D
            kj = np.concatenate([R.piece_rows(lengths, D, True, i, j) for i in range(len(lengths))])
            np.testing.assert_allclose(g[1][kj], sm(dk_r)[kj], atol=1e-12)
            np.testing.assert_allclose(g[2][kj], sm(dv_r)[kj], atol=1e-12)
            others = np.setdiff1d(np.arange(sum(lengths)), kj)
            assert not g[1][others].any() and not g[2][others].any()
            for acc, x in zip(tot, g):
                acc += un(x)
    for got, ref in zip(tot, (dq, dk, dv)):
        np.testing.assert_allclose(got, ref, atol=1e-11)


def test_partial_ring_resumes():
    """(out, lse) after k steps is the ring's whole state: merging the remaining steps'
    blocks into it gives the full result."""
    rng = _rng(21)
    D, lengths = 4, [32]
    q, k, v, _ = _case(rng, lengths, 2, 2, 4, False)
    full_o, full_l = R.ring_fwd(q, k, v, lengths, D, "zigzag", True, False)
    part_o, part_l = R.ring_fwd(q, k, v, lengths, D, "zigzag", True, False, steps=2)
    pos = LY.shard_positions("zigzag", D, 32)
    for r in range(D):
        rq = R.piece_rows(lengths, D, False, 0, r)
        o, l = part_o[rq], part_l[:, rq].T
        for s in range(2, D):
            rk = R.piece_rows(lengths, D, False, 0, (r - s) % D)
            bo, bl = R.block_attention(q[rq], k[rk], v[rk], pos[r], pos[(r - s) % D], True, 0.5)
            o, l = R.update_out_and_lse(o, l, bo, bl.T)
        np.testing.assert_allclose(o, full_o[rq], atol=1e-13)
        np.testing.assert_allclose(l.T, full_l[:, rq], atol=1e-13)


# ---------------------------------------------------------------------------------------
# backward: central finite differences
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    rng = _rng(31)
    cu = np.array([0, 5, 11], np.int32)
    q, k, v, do = _case(rng, [5, 6], 2, 1, 3, True)

    def loss(q_, k_, v_):
        o, _ = A.attention_fwd(q_, k_, v_, cu, causal, scale=0.8)
        return float((o * do).sum())

    dq, dk, dv = A.attention_bwd(q, k, v, do, cu, causal, scale=0.8)
    eps = 1e-6
    for x, gx in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            up = loss(q, k, v)
            x[idx] = old - eps
            dn = loss(q, k, v)
            x[idx] = old
            num[idx] = (up - dn) / (2 * eps)
        err = np.linalg.norm(num - gx) / np.linalg.norm(num)
        assert err < 1e-6, err


def test_gradient_sum_invariants():
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (per KV head, over its query heads)."""
    rng = _rng(32)
    cu = np.array([0, 24], np.int32)
    q, k, v, do = _case(rng, [24], 4, 2, 5, False)
    dq, dk, dv = A.attention_bwd(q, k, v, do, cu, True)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=0), do.reshape(24, 2, 2, 5).sum(axis=(0, 2)), atol=1e-12)


def test_row_subset_evaluation():
    """Rows evaluated alone equal the same rows of the full evaluation; keys that only the
    evaluated rows can see get their whole gradient."""
    rng = _rng(33)
    cu = np.array([0, 40], np.int32)
    q, k, v, do = _case(rng, [40], 2, 1, 4, False)
    out, lse = A.attention_fwd(q, k, v, cu, True)
    rows = np.array([0, 7, 39])
    o2, l2 = A.attention_fwd(q, k, v, cu, True, rows=rows)
    np.testing.assert_allclose(o2[rows], out[rows], atol=1e-14)
    np.testing.assert_allclose(l2[:, rows], lse[:, rows], atol=1e-14)
    dq, dk, dv = A.attention_bwd(q, k, v, do, cu, True)
    tail = np.arange(30, 40)
    dq2, dk2, dv2 = A.attention_bwd(q, k, v, do, cu, True, rows=tail)
    np.testing.assert_allclose(dq2[tail], dq[tail], atol=1e-13)
    np.testing.assert_allclose(dk2[tail], dk[tail], atol=1e-13)
    np.testing.assert_allclose(dv2[tail], dv[tail], atol=1e-13)
