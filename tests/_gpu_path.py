"""Run the CUDA path of one workload through the C ABI and return natural-order results.

Shared by the GPU tests; holds no attention arithmetic (inputs come from ``workloads``,
the computation from the library, the expected values from ``oracle`` in each test).
"""
from __future__ import annotations

import numpy as np
import torch

import context_blockwise_attention_step_gb300 as ra
import workloads as W

BF16_OUT_ABS, BF16_OUT_REL, BF16_LSE_ABS, GRAD_REL_L2 = 2e-2, 1e-2, 1e-3, 3e-2
F32_ABS = 1e-5
F32_GRAD_REL_L2 = 1e-5


def torch_dtype(w: W.Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def upload(x: np.ndarray, w: W.Workload) -> torch.Tensor:
    return torch.from_numpy(x).to("cuda").to(torch_dtype(w))


def problem(w: W.Workload, q: torch.Tensor, k: torch.Tensor):
    return ra.problem_for(q, k, D=w.D, layout=w.layout, causal=w.causal,
                          cu_seqlens=w.cu_seqlens if w.varlen else None)


def run(w: W.Workload, inputs=None, backward: bool | None = None):
    """Returns (results dict of natural-order float arrays, inputs tuple)."""
    if inputs is None:
        q, k, v = W.make_qkv(w)
        do = W.make_dout(w)
        inputs = (q, k, v, do)
    q, k, v, do = inputs
    backward = w.backward if backward is None else backward
    qd, kd, vd = (upload(x, w) for x in (q, k, v))
    prob = problem(w, qd, kd)
    qs, ks, vs = (ra.shard_tokens(x, prob) for x in (qd, kd, vd))
    out_s, lse_s = ra.ring_attn_fwd(qs, ks, vs, prob)
    res = {"out_sm": out_s, "lse_sm": lse_s, "prob": prob, "q_sm": qs, "k_sm": ks, "v_sm": vs}
    res["out"] = ra.unshard_tokens(out_s, prob).float().cpu().numpy()
    res["lse"] = ra.unshard_lse(lse_s, prob).cpu().numpy()
    if backward:
        dod = upload(do, w)
        dos = ra.shard_tokens(dod, prob)
        dq, dk, dv = ra.ring_attn_bwd(dos, qs, ks, vs, out_s, lse_s, prob)
        for name, g in (("dq", dq), ("dk", dk), ("dv", dv)):
            res[name] = ra.unshard_tokens(g, prob).float().cpu().numpy()
    torch.cuda.synchronize()
    assert ra.check_device_status() == 0, ra.last_error()
    return res, inputs


def packed(x: np.ndarray) -> np.ndarray:
    return x.reshape(-1, x.shape[-2], x.shape[-1])


def lse_packed(lse: np.ndarray, w: W.Workload) -> np.ndarray:
    """[B, Hq, S] -> [Hq, B*S] (varlen lse is already [Hq, T])."""
    if w.varlen:
        return lse
    return lse.transpose(1, 0, 2).reshape(lse.shape[1], -1)


def assert_out(w, got, ref, rows=None):
    got, ref = packed(got), packed(ref)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    ok = np.isfinite(ref).all()
    assert ok
    err = np.abs(got - ref)
    if w.dtype == "bf16":
        bad = err > BF16_OUT_ABS + BF16_OUT_REL * np.abs(ref)
        assert not bad.any(), f"out: {bad.sum()} elements out of tolerance, max err {err.max()}"
    else:
        assert err.max() <= F32_ABS, f"out max err {err.max()}"


def assert_lse(w, got, ref, rows=None):
    got = lse_packed(got, w)
    if rows is not None:
        got, ref = got[:, rows], ref[:, rows]
    err = np.abs(got - ref).max()
    assert err <= (BF16_LSE_ABS if w.dtype == "bf16" else F32_ABS), f"lse max err {err}"


def rel_l2(got, ref):
    got, ref = np.asarray(got, np.float64).reshape(-1), np.asarray(ref, np.float64).reshape(-1)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def assert_grad(w, name, got, ref, rows=None):
    got, ref = packed(got), packed(ref)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    e = rel_l2(got, ref)
    tol = GRAD_REL_L2 if w.dtype == "bf16" else F32_GRAD_REL_L2
    assert e <= tol, f"{name} rel-L2 {e:.3e} > {tol}"
