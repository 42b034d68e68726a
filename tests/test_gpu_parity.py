"""GPU parity of the CUDA path (through the C ABI) against the float64 oracle, on small
seeded problems that still span several tiles and ragged tails.

Tolerances: bf16 inputs with f32 accumulation: out |gpu-ref| <= 2e-2 + 1e-2 |ref|, lse within
1e-3, dq / dk / dv within 3e-2 relative L2; f32: out and lse within 1e-5, gradients within
1e-5 relative L2 (f32 arithmetic over at most a few thousand terms).
"""
import os

import numpy as np
import pytest
import torch

import context_blockwise_attention_step_gb300 as ra
import workloads as W
from oracle import attention as A
from oracle import layouts as LY
from oracle import ring as R

from _gpu_path import (assert_grad, assert_lse, assert_out, packed, problem, run, upload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ra.build()
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")


def wl(name, dtype="bf16", layout="basic", causal=True, D=4, hq=4, hkv=2, dh=128, batch=1,
       seqlen=0, seqlens=(), seed=0):
    return W.Workload(name=name, dtype=dtype, layout=layout, causal=causal, D=D, hq=hq, hkv=hkv,
                      head_dim=dh, seed=seed or 1, batch=batch if not seqlens else 0,
                      seqlen=seqlen, seqlens=tuple(seqlens))


SMALL = [
    wl("basic_ragged_b2", layout="basic", D=4, batch=2, seqlen=4 * 200, seed=11),
    wl("zigzag_ragged", layout="zigzag", D=4, seqlen=8 * 130, seed=12),
    wl("stripe_D3", layout="stripe", D=3, seqlen=3 * 300, seed=13),
    wl("basic_dh64_mha", layout="basic", D=2, hq=8, hkv=8, dh=64, batch=2, seqlen=2 * 384, seed=14),
    wl("zigzag_dh64_noncausal", layout="zigzag", causal=False, D=4, dh=64, seqlen=1024, seed=15),
    wl("stripe_noncausal_D8", layout="stripe", causal=False, D=8, seqlen=8 * 136, seed=16),
    wl("single_rank", layout="basic", D=1, seqlen=640, seed=17),
    wl("varlen_zigzag", layout="zigzag", D=4, hq=8, hkv=2, seqlens=(24, 1200, 8, 512), seed=18),
    wl("varlen_stripe_dh64", layout="stripe", D=8, dh=64, seqlens=(160, 1600, 528), seed=19),
    wl("varlen_basic_D2", layout="basic", D=2, hq=2, hkv=1, seqlens=(1400, 10, 514), seed=20),
    wl("gqa8_zigzag_D8", layout="zigzag", D=8, hq=8, hkv=1, seqlen=16 * 40, seed=21),
]

F32 = [
    W.TINY,
    wl("f32_zigzag_varlen", dtype="f32", layout="zigzag", D=4, hq=4, hkv=2, dh=32,
       seqlens=(40, 96, 8), seed=22),
    wl("f32_stripe_batch", dtype="f32", layout="stripe", D=2, hq=2, hkv=2, dh=16, batch=2,
       seqlen=64, seed=23),
]


def oracle(w, inputs, backward=True):
    q, k, v, do = inputs
    cu = w.cu_seqlens
    out, lse = A.attention_fwd(packed(q), packed(k), packed(v), cu, w.causal)
    grads = A.attention_bwd(packed(q), packed(k), packed(v), packed(do), cu, w.causal) if backward else None
    return out, lse, grads


@pytest.mark.parametrize("w", SMALL + F32, ids=lambda w: w.name)
def test_ring_fwd_bwd_matches_oracle(w):
    res, inputs = run(w)
    out, lse, grads = oracle(w, inputs, w.backward)
    assert_out(w, res["out"], out)
    assert_lse(w, res["lse"], lse)
    if w.backward:
        for name, ref in zip(("dq", "dk", "dv"), grads):
            assert_grad(w, name, res[name], ref)


@pytest.mark.parametrize("w", [SMALL[1], SMALL[7]], ids=lambda w: w.name)
def test_cuda_core_cross_check_path(w, monkeypatch):
    """The CUDA-core kernels (forced for bf16) agree with the oracle too."""
    monkeypatch.setenv("RA_IMPL", "simt")
    res, inputs = run(w)
    out, lse, grads = oracle(w, inputs)
    assert_out(w, res["out"], out)
    assert_lse(w, res["lse"], lse)
    for name, ref in zip(("dq", "dk", "dv"), grads):
        assert_grad(w, name, res[name], ref)


# f32 head dims whose rows do not fill a warp evenly (48 and 96: 12 and 24 four-element
# pieces; 18: not a multiple of 4, one element per lane) exercise the merge's row split.
MERGE_F32 = [
    wl("f32_merge_dh48", dtype="f32", layout="zigzag", D=4, hq=4, hkv=2, dh=48,
       seqlens=(40, 96, 8), seed=24),
    wl("f32_merge_dh96", dtype="f32", layout="basic", D=2, hq=2, hkv=1, dh=96, batch=2,
       seqlen=72, seed=25),
    wl("f32_merge_dh18", dtype="f32", layout="stripe", D=3, hq=3, hkv=3, dh=18, batch=1,
       seqlen=66, seed=26),
]


@pytest.mark.parametrize("w", [SMALL[0], SMALL[2], SMALL[7], F32[1]] + MERGE_F32,
                         ids=lambda w: w.name)
@pytest.mark.parametrize("block_dtype", [torch.float32, torch.bfloat16])
def test_unfused_steps_and_merge(w, block_dtype):
    """Per-step block_attn_fwd equals the oracle's block of every (rank, step); merging the
    D blocks with update_out_and_lse gives the single-pass result."""
    if w.dtype == "f32" and block_dtype == torch.bfloat16:
        pytest.skip("f32 problems produce f32 blocks")
    q, k, v = W.make_qkv(w)
    qd, kd, vd = (upload(x, w) for x in (q, k, v))
    prob = problem(w, qd, kd)
    qs, ks, vs = (ra.shard_tokens(x, prob) for x in (qd, kd, vd))
    rows = LY.shard_major_rows(w.layout, w.D, w.lengths, w.varlen)
    q_sm, k_sm, v_sm = (LY.shard(packed(x).astype(np.float64), rows, 0) for x in (q, k, v))
    out = torch.zeros(qs.shape, device="cuda", dtype=torch.float32)
    lse = torch.full(ra.ops._lse_shape(prob), float("-inf"), device="cuda")
    scale = 1.0 / np.sqrt(w.head_dim)
    for s in range(w.D):
        bo, bl = ra.block_attn_fwd(qs, ks, vs, prob, rank=-1, step=s, out_dtype=block_dtype)
        bo_np = packed(bo.float().cpu().numpy())
        bl_np = bl.cpu().numpy()
        bl_np = bl_np if w.varlen else bl_np.transpose(1, 0, 2).reshape(w.hq, -1)
        for i, n in enumerate(w.lengths):
            pos = LY.shard_positions(w.layout, w.D, n)
            for r in range(w.D):
                j = (r - s) % w.D
                rq = R.piece_rows(w.lengths, w.D, w.varlen, i, r)
                rk = R.piece_rows(w.lengths, w.D, w.varlen, i, j)
                ro, rl = R.block_attention(q_sm[rq], k_sm[rk], v_sm[rk], pos[r], pos[j], w.causal, scale)
                masked = ~np.isfinite(rl)
                np.testing.assert_array_equal(~np.isfinite(bl_np[:, rq]), masked)
                assert np.all(bo_np[rq][masked.T] == 0)
                tol = 1e-5 if w.dtype == "f32" else 1e-3
                np.testing.assert_allclose(bl_np[:, rq][~masked], rl[~masked], atol=tol)
                otol = 1e-5 if w.dtype == "f32" else (2e-2 if block_dtype == torch.bfloat16 else 1e-2)
                np.testing.assert_allclose(bo_np[rq], ro, atol=otol, rtol=1e-2)
        ra.update_out_and_lse(out, lse, bo, bl, prob)
    out_nat = ra.unshard_tokens(out, prob).cpu().numpy()
    lse_nat = ra.unshard_lse(lse, prob).cpu().numpy()
    ref_out, ref_lse = A.attention_fwd(packed(q), packed(k), packed(v), w.cu_seqlens, w.causal)
    assert_out(w, out_nat, ref_out)
    assert_lse(w, lse_nat, ref_lse)


def test_single_rank_block_writes_only_its_rows():
    w = SMALL[1]
    q, k, v = W.make_qkv(w)
    qd, kd, vd = (upload(x, w) for x in (q, k, v))
    prob = problem(w, qd, kd)
    qs, ks, vs = (ra.shard_tokens(x, prob) for x in (qd, kd, vd))
    sentinel = 7.0
    bo = torch.full(qs.shape, sentinel, device="cuda", dtype=torch.float32)
    bl = torch.full(ra.ops._lse_shape(prob), sentinel, device="cuda")
    ra.block_attn_fwd(qs, ks, vs, prob, rank=2, step=1, block_out=bo, block_lse=bl)
    L = w.seqlen // w.D
    bo_np = bo.cpu().numpy()[0]
    mine = np.zeros(w.seqlen, bool)
    mine[2 * L:3 * L] = True
    assert np.all(bo_np[~mine] == sentinel)
    assert not np.any(bo_np[mine] == sentinel)


def test_merge_identity_and_empty_blocks():
    """-inf is the merge's identity on the GPU too, and -inf with -inf stays 0 / -inf."""
    w = SMALL[0]
    prob = ra.make_problem(dtype=torch.bfloat16, layout="basic", causal=True, D=4, hq=4, hkv=2,
                           head_dim=128, batch=2, seqlen=w.seqlen)
    shape = (2, w.seqlen, 4, 128)
    g = torch.Generator(device="cuda").manual_seed(3)
    bo = torch.randn(shape, device="cuda", generator=g)
    bl = torch.randn((2, 4, w.seqlen), device="cuda", generator=g)
    out = torch.zeros(shape, device="cuda")
    lse = torch.full((2, 4, w.seqlen), float("-inf"), device="cuda")
    ra.update_out_and_lse(out, lse, bo, bl, prob)
    torch.testing.assert_close(out, bo, atol=1e-6, rtol=1e-6)
    torch.testing.assert_close(lse, bl, atol=1e-6, rtol=1e-6)
    out2 = torch.zeros(shape, device="cuda")
    lse2 = torch.full((2, 4, w.seqlen), float("-inf"), device="cuda")
    ra.update_out_and_lse(out2, lse2, torch.zeros(shape, device="cuda"), lse2.clone(), prob)
    assert torch.all(out2 == 0) and torch.all(torch.isneginf(lse2))


@pytest.mark.parametrize("w", [SMALL[0], SMALL[1], SMALL[2], SMALL[7], SMALL[8]], ids=lambda w: w.name)
def test_shard_unshard_bit_exact(w):
    q, _, _ = W.make_qkv(w)
    qd = upload(q, w)
    prob = problem(w, qd, qd)
    qs = ra.shard_tokens(qd, prob)
    rows = LY.shard_major_rows(w.layout, w.D, w.lengths, w.varlen)
    ref = LY.shard(packed(q), rows, 0)
    got = packed(qs.float().cpu().numpy())
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
    back = ra.unshard_tokens(qs, prob)
    assert torch.equal(back.view(torch.int16), qd.view(torch.int16))
    lse = torch.arange(np.prod(ra.ops._lse_shape(prob)), device="cuda", dtype=torch.float32)
    lse = lse.reshape(ra.ops._lse_shape(prob))
    assert torch.equal(ra.unshard_lse(ra.shard_lse(lse, prob), prob), lse)


def test_bounded_wait_reports_timeout_and_recovers():
    assert ra.check_device_status(reset=True) == 0
    ra.test_wait_timeout(2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert ra.check_device_status(reset=True) == ra._abi.RA_ERR_DEVICE_TIMEOUT
    assert ra.check_device_status(reset=True) == 0
    # the context is still usable
    res, inputs = run(SMALL[6], backward=False)
    out, lse, _ = oracle(SMALL[6], inputs, backward=False)
    assert_out(SMALL[6], res["out"], out)


def test_repeated_calls_are_stable():
    """Two forward calls give bit-identical outputs (no state carried between launches)."""
    w = SMALL[7]
    res1, inputs = run(w, backward=False)
    res2, _ = run(w, inputs=inputs, backward=False)
    np.testing.assert_array_equal(res1["out"], res2["out"])
    np.testing.assert_array_equal(res1["lse"], res2["lse"])


# ---------------------------------------------------------------------------------------
# unfused backward: one ring step at a time
# ---------------------------------------------------------------------------------------

def _shard_major_inputs(w):
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    qd, kd, vd, dod = (upload(x, w) for x in (q, k, v, do))
    prob = problem(w, qd, kd)
    qs, ks, vs, dos = (ra.shard_tokens(x, prob) for x in (qd, kd, vd, dod))
    rows = LY.shard_major_rows(w.layout, w.D, w.lengths, w.varlen)
    host = tuple(LY.shard(packed(x).astype(np.float64), rows, 0) for x in (q, k, v, do))
    return prob, (qs, ks, vs, dos), host, rows


@pytest.mark.parametrize("w", [SMALL[1], SMALL[2], SMALL[7], SMALL[8], F32[1]], ids=lambda w: w.name)
def test_block_backward_per_step_matches_oracle(w):
    """ra_block_attn_bwd of every step (all ranks), each added into zeroed float32
    accumulators, equals the oracle's per-step terms of the ring backward; the sum over the
    steps equals the fused backward. The block backward has no atomics: a repeated call
    gives the same bits."""
    prob, (qs, ks, vs, dos), (q_h, k_h, v_h, do_h), rows = _shard_major_inputs(w)
    out_s, lse_s = ra.ring_attn_fwd(qs, ks, vs, prob)
    o_h = packed(out_s.float().cpu().numpy()).astype(np.float64)
    l_h = lse_s.cpu().numpy().astype(np.float64)
    l_h = l_h if w.varlen else l_h.transpose(1, 0, 2).reshape(w.hq, -1)
    tot = [torch.zeros(t.shape, device="cuda") for t in (qs, ks, vs)]
    for s in range(w.D):
        acc = [torch.zeros(t.shape, device="cuda") for t in (qs, ks, vs)]
        ra.block_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob, -1, s, *acc)
        ref = R.ring_bwd(q_h, k_h, v_h, o_h, l_h, do_h, w.lengths, w.D, w.layout, w.causal,
                         w.varlen, steps=[s])
        for name, a, r_ in zip(("dq", "dk", "dv"), acc, ref):
            assert_grad(w, f"{name} step {s}", packed(a.cpu().numpy()), r_)
        if s == w.D - 1:
            again = [torch.zeros(t.shape, device="cuda") for t in (qs, ks, vs)]
            ra.block_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob, -1, s, *again)
            for name, a, b in zip(("dq", "dk", "dv"), acc, again):
                assert torch.equal(a, b), f"{name} step {s}: repeated call differs"
        for t, a in zip(tot, acc):
            t += a
    fused = ra.ring_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob)
    for name, t, f in zip(("dq", "dk", "dv"), tot, fused):
        assert_grad(w, f"{name} sum of steps", packed(t.cpu().numpy()), packed(f.float().cpu().numpy()))
    assert ra.check_device_status() == 0, ra.last_error()


@pytest.mark.parametrize("w", [SMALL[1], SMALL[7]], ids=lambda w: w.name)
def test_block_backward_single_rank(w):
    """One (rank, step) call touches only that rank's dq rows and shard (rank - step) mod
    D's dk / dv rows, and matches the oracle's term of that pair."""
    prob, (qs, ks, vs, dos), (q_h, k_h, v_h, do_h), rows = _shard_major_inputs(w)
    out_s, lse_s = ra.ring_attn_fwd(qs, ks, vs, prob)
    o_h = packed(out_s.float().cpu().numpy()).astype(np.float64)
    l_h = lse_s.cpu().numpy().astype(np.float64)
    l_h = l_h if w.varlen else l_h.transpose(1, 0, 2).reshape(w.hq, -1)
    sentinel = 0.5
    for r, s in ((1, 0), (2, 3), (3, 1)):
        acc = [torch.full(t.shape, sentinel, device="cuda") for t in (qs, ks, vs)]
        ra.block_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob, r, s, *acc)
        ref = R.ring_bwd(q_h, k_h, v_h, o_h, l_h, do_h, w.lengths, w.D, w.layout, w.causal,
                         w.varlen, steps=[s], ranks=[r])
        j = (r - s) % w.D
        mine_q = np.concatenate([R.piece_rows(w.lengths, w.D, w.varlen, i, r) for i in range(len(w.lengths))])
        mine_k = np.concatenate([R.piece_rows(w.lengths, w.D, w.varlen, i, j) for i in range(len(w.lengths))])
        for name, a, r_, mine in zip(("dq", "dk", "dv"), acc, ref, (mine_q, mine_k, mine_k)):
            a = packed(a.cpu().numpy()).astype(np.float64)
            others = np.setdiff1d(np.arange(a.shape[0]), mine)
            assert np.all(a[others] == sentinel), name
            assert_grad(w, name, a[mine] - sentinel, r_[mine])


# ---------------------------------------------------------------------------------------
# deterministic backward
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("w", [SMALL[0], SMALL[1], SMALL[3], SMALL[7], SMALL[10]], ids=lambda w: w.name)
def test_deterministic_backward_is_bitwise_repeatable(w):
    """deterministic = 1 (tensor-core K/V pass + query-tile dq pass, no atomics): parity
    with the oracle, two runs give bit-identical dq, dk, dv, and so does the default
    (deterministic = 0) problem, which takes the same atomic-free path."""
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    qd, kd, vd, dod = (upload(x, w) for x in (q, k, v, do))
    prob = ra.problem_for(qd, kd, D=w.D, layout=w.layout, causal=w.causal,
                          cu_seqlens=w.cu_seqlens if w.varlen else None, deterministic=True)
    qs, ks, vs, dos = (ra.shard_tokens(x, prob) for x in (qd, kd, vd, dod))
    out_s, lse_s = ra.ring_attn_fwd(qs, ks, vs, prob)
    g1 = [t.clone() for t in ra.ring_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob)]
    g2 = ra.ring_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob)
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    g3 = ra.ring_attn_bwd(dos, qs, ks, vs, out_s, lse_s, problem(w, qd, kd))
    for a, b in zip(g1, g3):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref = A.attention_bwd(packed(q), packed(k), packed(v), packed(do), w.cu_seqlens, w.causal)
    for name, g, r_ in zip(("dq", "dk", "dv"), g1, ref):
        assert_grad(w, name, ra.unshard_tokens(g, prob).float().cpu().numpy(), r_)
    assert ra.check_device_status() == 0, ra.last_error()


def test_fma_pipe_exp2_error_bound():
    """The forward's FMA-pipe 2^x (range split + fitted cubic) stays within its stated
    relative error bound against float64 2^x over the softmax's input range, and clamps
    below -125."""
    x = np.concatenate([np.linspace(-125.0, 8.0, 200001), np.linspace(-0.5, 0.5, 10001),
                        np.arange(-20, 9, dtype=np.float64)]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    ra._abi.check(ra._abi.lib().ra_test_exp2_poly(ra.ops._p(xd), ra.ops._p(yd), x.size,
                                                  ra.ops._stream()))
    y = yd.cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() < 8e-5, rel.max()
    low = torch.tensor([-126.0, -1000.0, float("-inf")], device="cuda")
    out = torch.empty_like(low)
    ra._abi.check(ra._abi.lib().ra_test_exp2_poly(ra.ops._p(low), ra.ops._p(out), 3, ra.ops._stream()))
    np.testing.assert_allclose(out.cpu().numpy(), np.exp2(-125.0) * np.ones(3), rtol=1e-4)


@pytest.mark.parametrize("w", [SMALL[0], SMALL[7], SMALL[10]], ids=lambda w: w.name)
def test_fused_backward_variant_matches_oracle(w, monkeypatch):
    """The single-pass backward with float reductions for dq (RA_BWD=fused) stays correct,
    for the whole ring and for the per-step block backward it then also runs."""
    monkeypatch.setenv("RA_BWD", "fused")
    res, inputs = run(w)
    out, lse, grads = oracle(w, inputs)
    for name, ref in zip(("dq", "dk", "dv"), grads):
        assert_grad(w, name, res[name], ref)
    prob, (qs, ks, vs, dos), (q_h, k_h, v_h, do_h), rows = _shard_major_inputs(w)
    out_s, lse_s = ra.ring_attn_fwd(qs, ks, vs, prob)
    o_h = packed(out_s.float().cpu().numpy()).astype(np.float64)
    l_h = lse_s.cpu().numpy().astype(np.float64)
    l_h = l_h if w.varlen else l_h.transpose(1, 0, 2).reshape(w.hq, -1)
    s = w.D - 1
    acc = [torch.zeros(t.shape, device="cuda") for t in (qs, ks, vs)]
    ra.block_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob, -1, s, *acc)
    ref = R.ring_bwd(q_h, k_h, v_h, o_h, l_h, do_h, w.lengths, w.D, w.layout, w.causal,
                     w.varlen, steps=[s])
    for name, a, r_ in zip(("dq", "dk", "dv"), acc, ref):
        assert_grad(w, f"block {name} step {s}", packed(a.cpu().numpy()), r_)
    assert ra.check_device_status() == 0, ra.last_error()
