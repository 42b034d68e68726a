"""Python binding of the ring-attention C ABI: the same entry points, torch tensors in.

PyTorch provides device memory and the current CUDA stream; every step of the path runs in
the library's kernels. Tensors are shard-major (see include/ringattn.h): use
``shard_tokens`` / ``unshard_tokens`` to convert from natural order.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import _abi
from ._abi import RA_BF16, RA_F32, LAYOUTS, RaProblem, check, lib


@dataclass
class Problem:
    """A ring-attention problem; ``raw`` is the C struct handed to the library."""

    raw: RaProblem
    cu_host: np.ndarray | None  # keeps the host cu_seqlens alive
    token_dtype: torch.dtype
    rows: int

    @property
    def ptr(self):
        return ctypes.byref(self.raw)


def make_problem(*, dtype: torch.dtype, layout: str, causal: bool, D: int, hq: int, hkv: int,
                 head_dim: int, batch: int = 0, seqlen: int = 0, cu_seqlens=None,
                 scale: float | None = None, deterministic: bool = False) -> Problem:
    """Describe a problem. Batch mode: ``batch``, ``seqlen``. Varlen mode: ``cu_seqlens``
    (natural-order offsets; a host copy is kept)."""
    if dtype == torch.bfloat16:
        dt = RA_BF16
    elif dtype == torch.float32:
        dt = RA_F32
    else:
        raise ValueError(f"unsupported dtype {dtype}")
    raw = RaProblem()
    raw.dtype = dt
    raw.layout = LAYOUTS[layout]
    raw.causal = 1 if causal else 0
    raw.D = D
    raw.hq = hq
    raw.hkv = hkv
    raw.head_dim = head_dim
    raw.scale = 0.0 if scale is None else float(scale)
    raw.deterministic = 1 if deterministic else 0
    cu_host = None
    if cu_seqlens is None:
        raw.batch = batch
        raw.seqlen = seqlen
        rows = batch * seqlen
    else:
        if isinstance(cu_seqlens, torch.Tensor):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu_host = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        raw.batch = 0
        raw.n_seqs = cu_host.size - 1
        raw.cu_seqlens = cu_host.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        rows = int(cu_host[-1])
    return Problem(raw=raw, cu_host=cu_host, token_dtype=dtype, rows=rows)


def problem_for(q: torch.Tensor, k: torch.Tensor, *, D: int, layout: str = "basic",
                causal: bool = True, cu_seqlens=None, scale: float | None = None,
                deterministic: bool = False) -> Problem:
    """Problem from tensor shapes: [B, S, Hq, Dh] (batch) or [T, Hq, Dh] + cu_seqlens."""
    if q.dim() == 4:
        return make_problem(dtype=q.dtype, layout=layout, causal=causal, D=D, hq=q.shape[2],
                            hkv=k.shape[2], head_dim=q.shape[3], batch=q.shape[0],
                            seqlen=q.shape[1], scale=scale, deterministic=deterministic)
    if cu_seqlens is None:
        raise ValueError("varlen tensors need cu_seqlens")
    return make_problem(dtype=q.dtype, layout=layout, causal=causal, D=D, hq=q.shape[1],
                        hkv=k.shape[1], head_dim=q.shape[2], cu_seqlens=cu_seqlens, scale=scale,
                        deterministic=deterministic)


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _p(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _lse_shape(prob: Problem) -> tuple:
    r = prob.raw
    if r.batch > 0:
        return (r.batch, r.hq, r.seqlen)
    return (r.hq, prob.rows)


def _check_tensor(t: torch.Tensor, dtype, numel: int, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def ring_attn_fwd(q, k, v, prob: Problem, out=None, lse=None, stream=None, workspace=None):
    """Fused ring forward -> (out, lse), shard-major. lse is float32, natural log. The
    workspace (``workspace_bytes(prob, 0)`` bytes; allocated when not given) holds the
    counter the CTAs take their work items from."""
    r = prob.raw
    nq, nk = prob.rows * r.hq * r.head_dim, prob.rows * r.hkv * r.head_dim
    _check_tensor(q, prob.token_dtype, nq, "q")
    _check_tensor(k, prob.token_dtype, nk, "k")
    _check_tensor(v, prob.token_dtype, nk, "v")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(_lse_shape(prob), device=q.device, dtype=torch.float32) if lse is None else lse
    _check_tensor(out, prob.token_dtype, nq, "out")
    _check_tensor(lse, torch.float32, prob.rows * r.hq, "lse")
    need = workspace_bytes(prob, 0)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(lib().ra_ring_attn_fwd(prob.ptr, _p(q), _p(k), _p(v), _p(out), _p(lse),
                                 None if workspace is None else _p(workspace), wsz, _stream(stream)))
    return out, lse


def block_attn_fwd(q, k, v, prob: Problem, rank: int, step: int, out_dtype=torch.float32,
                   block_out=None, block_lse=None, stream=None):
    """One ring step of the unfused path for ``rank`` (all ranks if -1)."""
    r = prob.raw
    block_out = (torch.empty(q.shape, device=q.device, dtype=out_dtype)
                 if block_out is None else block_out)
    block_lse = (torch.empty(_lse_shape(prob), device=q.device, dtype=torch.float32)
                 if block_lse is None else block_lse)
    _check_tensor(block_out, out_dtype, prob.rows * r.hq * r.head_dim, "block_out")
    odt = RA_F32 if out_dtype == torch.float32 else RA_BF16
    check(lib().ra_block_attn_fwd(prob.ptr, rank, step, _p(q), _p(k), _p(v), _p(block_out), odt,
                                  _p(block_lse), _stream(stream)))
    return block_out, block_lse


def update_out_and_lse(out, lse, block_out, block_lse, prob: Problem, rank: int = -1, stream=None):
    """In-place log-sum-exp merge of (block_out, block_lse) into float32 (out, lse)."""
    r = prob.raw
    _check_tensor(out, torch.float32, prob.rows * r.hq * r.head_dim, "out")
    _check_tensor(lse, torch.float32, prob.rows * r.hq, "lse")
    odt = RA_F32 if block_out.dtype == torch.float32 else RA_BF16
    check(lib().ra_update_out_and_lse(prob.ptr, rank, _p(out), _p(lse), _p(block_out), odt,
                                      _p(block_lse), _stream(stream)))
    return out, lse


def workspace_bytes(prob: Problem, which: int = 1) -> int:
    return int(lib().ra_workspace_bytes(prob.ptr, which))


def ring_attn_bwd(dout, q, k, v, out, lse, prob: Problem, dq=None, dk=None, dv=None,
                  workspace=None, stream=None):
    """Ring backward -> (dq, dk, dv), shard-major, in the problem dtype."""
    r = prob.raw
    nq, nk = prob.rows * r.hq * r.head_dim, prob.rows * r.hkv * r.head_dim
    for t, n, name in ((dout, nq, "dout"), (q, nq, "q"), (k, nk, "k"), (v, nk, "v"), (out, nq, "out")):
        _check_tensor(t, prob.token_dtype, n, name)
    _check_tensor(lse, torch.float32, prob.rows * r.hq, "lse")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = workspace_bytes(prob)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    check(lib().ra_ring_attn_bwd(prob.ptr, _p(q), _p(k), _p(v), _p(out), _p(lse), _p(dout),
                                 _p(dq), _p(dk), _p(dv), _p(workspace), workspace.numel(),
                                 _stream(stream)))
    return dq, dk, dv


def block_attn_bwd(dout, q, k, v, out, lse, prob: Problem, rank: int, step: int, dq_acc, dk_acc,
                   dv_acc, workspace=None, stream=None):
    """One ring step of the unfused backward: adds the float32 block gradients of ``rank``
    (every rank if -1) at ``step`` into ``dq_acc`` (rank's rows) and ``dk_acc`` / ``dv_acc``
    (rows of shard (rank - step) mod D)."""
    r = prob.raw
    nq, nk = prob.rows * r.hq * r.head_dim, prob.rows * r.hkv * r.head_dim
    for t, n, name in ((dout, nq, "dout"), (q, nq, "q"), (k, nk, "k"), (v, nk, "v"), (out, nq, "out")):
        _check_tensor(t, prob.token_dtype, n, name)
    _check_tensor(lse, torch.float32, prob.rows * r.hq, "lse")
    for t, n, name in ((dq_acc, nq, "dq_acc"), (dk_acc, nk, "dk_acc"), (dv_acc, nk, "dv_acc")):
        _check_tensor(t, torch.float32, n, name)
    if workspace is None:
        workspace = torch.empty(max(workspace_bytes(prob, 2), 1), device=q.device, dtype=torch.uint8)
    check(lib().ra_block_attn_bwd(prob.ptr, rank, step, _p(q), _p(k), _p(v), _p(out), _p(lse),
                                  _p(dout), _p(dq_acc), _p(dk_acc), _p(dv_acc), _p(workspace),
                                  workspace.numel(), _stream(stream)))
    return dq_acc, dk_acc, dv_acc


def ring_attn_bwd_noalloc(dout, q, k, v, out, lse, prob: Problem, dq, dk, dv, stream=None):
    """ring_attn_bwd without a caller workspace, for callers that cannot allocate device
    memory: the library's static scratch array is used (problems up to
    RA_NOALLOC_SCRATCH_BYTES of scratch; calls overlapping on the GPU race on it). The
    outputs dq, dk, dv must be passed in."""
    r = prob.raw
    nq, nk = prob.rows * r.hq * r.head_dim, prob.rows * r.hkv * r.head_dim
    for t, n, name in ((dout, nq, "dout"), (q, nq, "q"), (k, nk, "k"), (v, nk, "v"),
                       (out, nq, "out"), (dq, nq, "dq"), (dk, nk, "dk"), (dv, nk, "dv")):
        _check_tensor(t, prob.token_dtype, n, name)
    _check_tensor(lse, torch.float32, prob.rows * r.hq, "lse")
    check(lib().ra_ring_attn_bwd_noalloc(prob.ptr, _p(q), _p(k), _p(v), _p(out), _p(lse),
                                         _p(dout), _p(dq), _p(dk), _p(dv), _stream(stream)))
    return dq, dk, dv


def shard_tokens(x: torch.Tensor, prob: Problem, out=None, stream=None):
    """Natural order -> shard-major (bit-exact copy)."""
    out = torch.empty_like(x) if out is None else out
    row_bytes = x.numel() * x.element_size() // prob.rows
    check(lib().ra_shard_tokens(prob.ptr, 0, _p(x), _p(out), row_bytes, _stream(stream)))
    return out


def unshard_tokens(x: torch.Tensor, prob: Problem, out=None, stream=None):
    """Shard-major -> natural order (bit-exact copy)."""
    out = torch.empty_like(x) if out is None else out
    row_bytes = x.numel() * x.element_size() // prob.rows
    check(lib().ra_shard_tokens(prob.ptr, 1, _p(x), _p(out), row_bytes, _stream(stream)))
    return out


def shard_lse(x: torch.Tensor, prob: Problem, out=None, stream=None):
    out = torch.empty_like(x) if out is None else out
    check(lib().ra_shard_lse(prob.ptr, 0, _p(x), _p(out), _stream(stream)))
    return out


def unshard_lse(x: torch.Tensor, prob: Problem, out=None, stream=None):
    out = torch.empty_like(x) if out is None else out
    check(lib().ra_shard_lse(prob.ptr, 1, _p(x), _p(out), _stream(stream)))
    return out


# ---- host-side integer helpers (no GPU) -------------------------------------------------

def validate(prob: Problem) -> int:
    return int(lib().ra_validate(prob.ptr))


def layout_positions(prob: Problem, seq: int) -> np.ndarray:
    r = prob.raw
    n = (r.seqlen if r.batch > 0 else int(prob.cu_host[seq + 1] - prob.cu_host[seq]))
    out = np.zeros(n, dtype=np.int64)
    check(lib().ra_layout_positions(prob.ptr, seq, out.ctypes.data_as(ctypes.c_void_p)))
    return out.reshape(r.D, n // r.D)


def step_counts(prob: Problem, seq: int, rank: int, step: int):
    r = prob.raw
    n = (r.seqlen if r.batch > 0 else int(prob.cu_host[seq + 1] - prob.cu_host[seq]))
    out = np.zeros(n // r.D, dtype=np.int32)
    active = np.zeros(1, dtype=np.int32)
    check(lib().ra_step_counts(prob.ptr, seq, rank, step, out.ctypes.data_as(ctypes.c_void_p),
                               active.ctypes.data_as(ctypes.c_void_p)))
    return out, bool(active[0])


def work_items(prob: Problem, which: int) -> np.ndarray:
    n = check(lib().ra_work_items(prob.ptr, which, None, 0))
    out = np.zeros((max(n, 1), 4), dtype=np.int32)
    check(lib().ra_work_items(prob.ptr, which, out.ctypes.data_as(ctypes.c_void_p), n))
    return out[:n]


def check_device_status(reset: bool = True) -> int:
    return int(lib().ra_check_device_status(1 if reset else 0))


def test_wait_timeout(timeout_ns: int, stream=None) -> int:
    return check(lib().ra_test_wait_timeout(timeout_ns, _stream(stream)))


def profile_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event ``start`` / ``stop`` around the main kernel of the next
    ring_attn_fwd / ring_attn_bwd calls (None, None switches the hook off)."""
    if start is None:
        check(lib().ra_profile_events(None, None))
        return
    for e in (start, stop):
        if e.cuda_event == 0:  # torch creates events lazily
            e.record()
    check(lib().ra_profile_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event)))


def profile_split_event(mid=None) -> None:
    """Record torch.cuda.Event ``mid`` between the two passes of the next ring_attn_bwd
    calls (None switches it off)."""
    if mid is None:
        check(lib().ra_profile_split_event(None))
        return
    if mid.cuda_event == 0:
        mid.record()
    check(lib().ra_profile_split_event(ctypes.c_void_p(mid.cuda_event)))


def last_error() -> str:
    return lib().ra_last_error().decode()


def version() -> int:
    return int(lib().ra_version())
