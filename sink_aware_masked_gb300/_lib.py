"""ctypes view of libsinkattn.so (the C ABI declared in include/sinkattn.h)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libsinkattn.so")

STATUS = {
    0: "SINKATTN_OK",
    1: "SINKATTN_ERR_INVALID_ARG",
    2: "SINKATTN_ERR_UNSUPPORTED",
    3: "SINKATTN_ERR_ALIGNMENT",
    4: "SINKATTN_ERR_WORKSPACE",
    5: "SINKATTN_ERR_CUDA",
    6: "SINKATTN_ERR_TIMEOUT",
}

# Every entry point include/sinkattn.h declares: name -> (restype, argtypes).
_vp, _sz, _i32, _i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64


class Problem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("seqlen", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("cu_seqlens_host", ctypes.c_void_p),
        ("total_tokens", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32),
        ("num_heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("window", ctypes.c_int64),
        ("prefix", ctypes.c_int64),
        ("causal", ctypes.c_int32),
        ("scale", ctypes.c_float),
    ]


class GrpoProblem(ctypes.Structure):
    _fields_ = [
        ("num_rollouts", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("cu_tokens", ctypes.c_void_p),
        ("cu_tokens_host", ctypes.c_void_p),
        ("total_tokens", ctypes.c_int32),
        ("clip_eps", ctypes.c_float),
        ("adv_eps", ctypes.c_float),
        ("kl_beta", ctypes.c_float),
    ]


_PP = ctypes.POINTER(Problem)
_GP = ctypes.POINTER(GrpoProblem)
SIGNATURES = {
    "sinkattn_fwd_workspace_size": (_sz, [_PP]),
    "sinkattn_bwd_workspace_size": (_sz, [_PP]),
    "sinkattn_kernel_launches": (_i32, [_PP, _i32]),
    "sinkattn_fwd": (ctypes.c_int, [_PP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sinkattn_bwd": (ctypes.c_int, [_PP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sinkattn_bwd_noalloc": (ctypes.c_int, [_PP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "sinkattn_decode_workspace_size": (_sz, [_PP, _i32]),
    "sinkattn_decode_fwd": (ctypes.c_int, [_PP, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sinkattn_grpo_workspace_size": (_sz, [_GP]),
    "sinkattn_grpo_loss": (ctypes.c_int, [_GP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sinkattn_varlen_plan": (ctypes.c_int, [_vp, _i32, _vp, _vp]),
    "sinkattn_pack": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "sinkattn_unpack": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "sinkattn_get_device_status": (ctypes.c_int, [_vp]),
    "sinkattn_set_profile_events": (ctypes.c_int, [_i32, _vp, _vp]),
    "sinkattn_selftest_wait_timeout": (ctypes.c_int, [_i64, _vp]),
    "sinkattn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sinkattn_version": (_i32, []),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once; raises if it is missing (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libsinkattn.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class SinkAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


def check(fn: str, status: int) -> None:
    if status != 0:
        raise SinkAttnError(fn, status)
