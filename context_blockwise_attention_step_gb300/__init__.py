"""Ring attention (the context-parallel blockwise attention step) on one GB300 GPU.

The D ring ranks are virtual shards of one sequence resident in HBM; the ring is a step
schedule over K/V shards, fused into hand-written sm_103a kernels behind the C ABI in
include/ringattn.h. This package is the thin Python binding over that ABI.
"""
from ._build import build  # noqa: F401
from ._abi import RingAttnError, EXPORTS  # noqa: F401
from .ops import (  # noqa: F401
    Problem, make_problem, problem_for, ring_attn_fwd, ring_attn_bwd, ring_attn_bwd_noalloc,
    block_attn_fwd, block_attn_bwd,
    update_out_and_lse, workspace_bytes, shard_tokens, unshard_tokens, shard_lse, unshard_lse,
    validate, layout_positions, step_counts, work_items, check_device_status,
    test_wait_timeout, profile_events, profile_split_event, last_error, version,
)
from .autograd import RingSelfAttention, ring_attention, shard, unshard  # noqa: F401,E402
