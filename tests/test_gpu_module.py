"""The autograd wrapper and the drop-in attention module on the GPU, against the oracle.

``RingSelfAttention`` projects with random bf16 weights, shards the tokens, runs ring
attention through the C ABI and unshards. The expected values come from the float64
oracle's plain attention and its gradient, with the linear layers around it differentiated
by the chain rule (dW = g^T x, dx = g W) on the same bf16 weights and inputs. Tolerance:
relative L2 3e-2 on the output and on every gradient (bf16 storage of the projected
q, k, v, out and of every gradient, float32 accumulation).
"""
import numpy as np
import pytest
import torch

import context_blockwise_attention_step_gb300 as ra
from oracle import attention as A

from _gpu_path import GRAD_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ra.build()
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")


@pytest.mark.parametrize("layout,D,hq,hkv", [("zigzag", 4, 4, 2), ("stripe", 2, 2, 2)])
def test_module_forward_backward_matches_oracle(layout, D, hq, hkv):
    hidden, dh, B, S = 192, 128, 1, 768
    m = ra.RingSelfAttention(hidden, hq, hkv, dh, D=D, layout=layout, device="cuda", seed=3)
    g = torch.Generator().manual_seed(4)
    x = torch.randn(B, S, hidden, generator=g).to("cuda", torch.bfloat16).requires_grad_(True)
    gy = torch.randn(B, S, hidden, generator=g).to("cuda", torch.bfloat16)
    y = m(x)
    (y.float() * gy.float()).sum().backward()
    assert ra.check_device_status() == 0, ra.last_error()

    f64 = lambda t: t.detach().double().cpu().numpy()
    X, GY = f64(x)[0], f64(gy)[0]
    Wq, Wk, Wv, Wo = (f64(p) for p in (m.wq, m.wk, m.wv, m.wo))
    q = (X @ Wq.T).reshape(S, hq, dh)
    k = (X @ Wk.T).reshape(S, hkv, dh)
    v = (X @ Wv.T).reshape(S, hkv, dh)
    cu = np.array([0, S])
    out, _ = A.attention_fwd(q, k, v, cu, True)
    o2 = out.reshape(S, hq * dh)
    y_ref = o2 @ Wo.T
    d_o2 = GY @ Wo
    dq, dk, dv = A.attention_bwd(q, k, v, d_o2.reshape(S, hq, dh), cu, True)
    dq2, dk2, dv2 = dq.reshape(S, -1), dk.reshape(S, -1), dv.reshape(S, -1)
    want = {
        "y": y_ref,
        "x": dq2 @ Wq + dk2 @ Wk + dv2 @ Wv,
        "wq": dq2.T @ X, "wk": dk2.T @ X, "wv": dv2.T @ X, "wo": GY.T @ o2,
    }
    got = {"y": f64(y)[0], "x": f64(x.grad)[0], "wq": f64(m.wq.grad), "wk": f64(m.wk.grad),
           "wv": f64(m.wv.grad), "wo": f64(m.wo.grad)}
    for name in want:
        e = rel_l2(got[name], want[name])
        assert e <= GRAD_REL_L2, f"{name}: rel-L2 {e:.3e}"


def test_ring_attention_function_gradcheck_against_fused_call():
    """The Function's backward is ra_ring_attn_bwd on the saved out / lse: its gradients
    equal a direct call of the C ABI on the same tensors, bit for bit."""
    import workloads as W

    w = W.Workload(name="fn_b1_s512_gqa4x1_dh64_D2_basic", dtype="bf16", layout="basic",
                   causal=True, D=2, hq=4, hkv=1, head_dim=64, seed=41, batch=1, seqlen=512)
    q, k, v = (torch.from_numpy(t).to("cuda", torch.bfloat16) for t in W.make_qkv(w))
    do = torch.from_numpy(W.make_dout(w)).to("cuda", torch.bfloat16)
    prob = ra.problem_for(q, k, D=w.D, layout=w.layout, causal=w.causal, deterministic=True)
    qs, ks, vs, dos = (ra.shard_tokens(t, prob) for t in (q, k, v, do))
    leaves = [t.clone().requires_grad_(True) for t in (qs, ks, vs)]
    out, lse = ra.ring_attention(*leaves, prob)
    out.backward(dos)
    o2, l2 = ra.ring_attn_fwd(qs, ks, vs, prob)
    assert torch.equal(out.detach(), o2) and torch.equal(lse, l2)
    direct = ra.ring_attn_bwd(dos, qs, ks, vs, o2, l2, prob)
    for leaf, d in zip(leaves, direct):
        assert torch.equal(leaf.grad, d)
