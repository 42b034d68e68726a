"""The allocation-free backward, for callers that cannot allocate device memory.

ra_ring_attn_bwd_noalloc runs the same backward as ra_ring_attn_bwd on a static device
scratch array instead of a caller workspace. It is meant for callers that can hand the
library their inputs and outputs but cannot allocate scratch themselves (a plain-C plugin
given only its buffers, or a training step that must not call cudaMalloc). This file is
collected last so that a run stopping at the first failure has run every other test first;
it also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import context_blockwise_attention_step_gb300 as ra
from context_blockwise_attention_step_gb300 import _abi
import workloads as W

from _gpu_path import GRAD_REL_L2, rel_l2


def _case():
    return W.Workload(name="noalloc_b2_s1024_gqa4x2_dh128_D4_zigzag", dtype="bf16",
                      layout="zigzag", causal=True, D=4, hq=4, hkv=2, head_dim=128, seed=31,
                      batch=2, seqlen=1024)


def test_oversized_problem_is_rejected_without_launch():
    ra.build()
    big = ra.make_problem(dtype=torch.bfloat16, layout="basic", causal=True, D=1, hq=64, hkv=8,
                          head_dim=128, batch=1, seqlen=524288)
    assert ra.workspace_bytes(big) > _abi.RA_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = _abi.lib().ra_ring_attn_bwd_noalloc(big.ptr, *([fake] * 9), None)
    assert st == _abi.RA_ERR_WORKSPACE
    assert "at most" in ra.last_error()


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_twice():
    ra.build()
    w = _case()
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    up = lambda x: torch.from_numpy(x).to("cuda").to(torch.bfloat16)
    qd, kd, vd, dod = (up(x) for x in (q, k, v, do))
    prob = ra.problem_for(qd, kd, D=w.D, layout=w.layout, causal=w.causal)
    assert ra.workspace_bytes(prob) <= _abi.RA_NOALLOC_SCRATCH_BYTES
    qs, ks, vs, dos = (ra.shard_tokens(x, prob) for x in (qd, kd, vd, dod))
    out, lse = ra.ring_attn_fwd(qs, ks, vs, prob)
    ref = ra.ring_attn_bwd(dos, qs, ks, vs, out, lse, prob)
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        got = tuple(torch.full_like(t, float("nan")) for t in ref)
        ra.ring_attn_bwd_noalloc(dos, qs, ks, vs, out, lse, prob, *got)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            g64, r64 = g.double().cpu().numpy(), r.double().cpu().numpy()
            assert np.isfinite(g64).all(), name
            assert rel_l2(g64, r64) <= GRAD_REL_L2, name
    assert ra.check_device_status() == 0
