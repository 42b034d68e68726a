"""ctypes declarations of the C ABI in include/ringattn.h (one function per export).

Loading fails loudly when the library has not been built: there is no other code path.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH

RA_OK = 0
RA_ERR_INVALID_ARG = -1
RA_ERR_UNSUPPORTED = -2
RA_ERR_SHAPE = -3
RA_ERR_WORKSPACE = -4
RA_ERR_CUDA = -5
RA_ERR_DEVICE_TIMEOUT = -6
RA_F32 = 0
RA_BF16 = 1
LAYOUTS = {"basic": 0, "zigzag": 1, "stripe": 2}
RA_MAX_SEQS = 1024
RA_NOALLOC_SCRATCH_BYTES = 64 << 20

# every symbol include/ringattn.h declares
EXPORTS = (
    "ra_ring_attn_fwd", "ra_block_attn_fwd", "ra_update_out_and_lse", "ra_workspace_bytes",
    "ra_ring_attn_bwd", "ra_block_attn_bwd", "ra_ring_attn_bwd_noalloc", "ra_shard_tokens", "ra_shard_lse", "ra_validate",
    "ra_layout_positions", "ra_step_counts", "ra_work_items", "ra_check_device_status",
    "ra_test_wait_timeout", "ra_test_exp2_poly", "ra_profile_events", "ra_profile_split_event",
    "ra_last_error",
    "ra_version",
)


class RaProblem(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("seqlen", ctypes.c_int32),
        ("n_seqs", ctypes.c_int32),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("deterministic", ctypes.c_int32),
    ]


class RingAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"ringattn status {status}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(RaProblem)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    sig = {
        "ra_ring_attn_fwd": (i32, [P, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]),
        "ra_block_attn_fwd": (i32, [P, i32, i32, vp, vp, vp, vp, i32, vp, vp]),
        "ra_update_out_and_lse": (i32, [P, i32, vp, vp, vp, i32, vp, vp]),
        "ra_workspace_bytes": (ctypes.c_size_t, [P, i32]),
        "ra_ring_attn_bwd": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]),
        "ra_ring_attn_bwd_noalloc": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "ra_block_attn_bwd": (i32, [P, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    ctypes.c_size_t, vp]),
        "ra_shard_tokens": (i32, [P, i32, vp, vp, i64, vp]),
        "ra_shard_lse": (i32, [P, i32, vp, vp, vp]),
        "ra_validate": (i32, [P]),
        "ra_layout_positions": (i32, [P, i32, vp]),
        "ra_step_counts": (i32, [P, i32, i32, i32, vp, vp]),
        "ra_work_items": (i32, [P, i32, vp, i32]),
        "ra_check_device_status": (i32, [i32]),
        "ra_test_wait_timeout": (i32, [ctypes.c_uint64, vp]),
        "ra_test_exp2_poly": (i32, [vp, vp, i32, vp]),
        "ra_profile_events": (i32, [vp, vp]),
        "ra_profile_split_event": (i32, [vp]),
        "ra_last_error": (ctypes.c_char_p, []),
        "ra_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def check(status: int) -> int:
    if status < 0:
        raise RingAttnError(status, lib().ra_last_error().decode())
    return status
