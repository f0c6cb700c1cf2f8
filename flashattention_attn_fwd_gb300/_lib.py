"""ctypes view of the C ABI declared in include/flattn.h.

This module only loads ``libflattn.so`` and mirrors its types; it performs no
computation.  The library must have been built (``__graft_entry__.build()``
or ``python -m flashattention_attn_fwd_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflattn.so")

FL_OK = 0
FL_ERR_INVALID_ARG = 1
FL_ERR_UNSUPPORTED = 2
FL_ERR_ALIGNMENT = 3
FL_ERR_CUDA = 4
FL_ERR_TIMEOUT = 5
FL_ERR_DEVICE_BOUNDS = 6

MASKS = {"none": 0, "causal": 1, "window": 2, "prefix_lm": 3, "document": 4}
SCORE_MODS = {"none": 0, "alibi": 1, "softcap": 2}
FL_DEBUG_SKIP_KV_LOAD = 0x1
FL_DEBUG_KEY_SPLIT = 0x2

# Every symbol include/flattn.h declares.
EXPORTS = (
    "fl_attn_desc_init",
    "fl_attn_fwd",
    "fl_diffattn_fwd",
    "fl_evoformer_gated_attn_fwd",
    "fl_evoformer_col_gated_attn_fwd",
    "fl_sync_status",
    "fl_status_string",
    "fl_abi_version",
    "fl_attn_desc_size",
    "fl_attn_fwd_noalloc",
    "fl_attn_decode_fwd",
    "fl_attn_decode_workspace_size",
    "fl_attn_bwd",
    "fl_attn_bwd_workspace_size",
    "fl_diffattn_bwd",
    "fl_diffattn_bwd_workspace_size",
    "fl_last_error_detail",
    "fl_attn_schedule",
)


class AttnDesc(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("Lq", ctypes.c_int32), ("Lk", ctypes.c_int32), ("d", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("mask_kind", ctypes.c_int32), ("doc_causal", ctypes.c_int32),
        ("window", ctypes.c_int32), ("prefix_len", ctypes.c_int32),
        ("score_mod", ctypes.c_int32), ("softcap", ctypes.c_float),
        ("alibi_slopes", ctypes.c_void_p), ("doc_offsets", ctypes.c_void_p),
        ("num_docs", ctypes.c_int32),
        ("q_strides", ctypes.c_int64 * 4), ("k_strides", ctypes.c_int64 * 4),
        ("v_strides", ctypes.c_int64 * 4), ("o_strides", ctypes.c_int64 * 4),
        ("stream", ctypes.c_void_p),
        ("debug_flags", ctypes.c_uint32), ("debug_arg", ctypes.c_int32),
        ("wait_limit_ms", ctypes.c_uint32),
        ("reserved", ctypes.c_int32 * 7),
    ]


class FlattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == FL_ERR_CUDA:
            detail = lib().fl_last_error_detail().decode()
        super().__init__(f"{what}: {status_string(status)} (status {status})" + (f" [{detail}]" if detail else ""))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(the CUDA library is required; there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        L.fl_attn_desc_init.argtypes = [ctypes.POINTER(AttnDesc)]
        L.fl_attn_desc_init.restype = None
        L.fl_attn_fwd.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(AttnDesc)]
        L.fl_attn_fwd.restype = i32
        L.fl_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(AttnDesc)]
        L.fl_attn_fwd_noalloc.restype = i32
        L.fl_diffattn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, ctypes.POINTER(AttnDesc)]
        L.fl_diffattn_fwd.restype = i32
        L.fl_evoformer_gated_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
        L.fl_evoformer_gated_attn_fwd.restype = i32
        L.fl_evoformer_col_gated_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
        L.fl_evoformer_col_gated_attn_fwd.restype = i32
        L.fl_attn_decode_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(AttnDesc)]
        L.fl_attn_decode_fwd.restype = i32
        L.fl_attn_decode_workspace_size.argtypes = [ctypes.POINTER(AttnDesc)]
        L.fl_attn_decode_workspace_size.restype = ctypes.c_size_t
        L.fl_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(AttnDesc)]
        L.fl_attn_bwd.restype = i32
        L.fl_attn_bwd_workspace_size.argtypes = [ctypes.POINTER(AttnDesc)]
        L.fl_attn_bwd_workspace_size.restype = ctypes.c_size_t
        L.fl_diffattn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_size_t, ctypes.POINTER(AttnDesc)]
        L.fl_diffattn_bwd.restype = i32
        L.fl_diffattn_bwd_workspace_size.argtypes = [ctypes.POINTER(AttnDesc)]
        L.fl_diffattn_bwd_workspace_size.restype = ctypes.c_size_t
        L.fl_sync_status.argtypes = [vp]
        L.fl_sync_status.restype = i32
        L.fl_attn_schedule.argtypes = [ctypes.POINTER(AttnDesc), vp, ctypes.POINTER(ctypes.c_int64)]
        L.fl_attn_schedule.restype = i32
        L.fl_last_error_detail.argtypes = []
        L.fl_last_error_detail.restype = ctypes.c_char_p
        L.fl_status_string.argtypes = [i32]
        L.fl_status_string.restype = ctypes.c_char_p
        L.fl_abi_version.argtypes = []
        L.fl_abi_version.restype = i32
        L.fl_attn_desc_size.argtypes = []
        L.fl_attn_desc_size.restype = i32
        if L.fl_attn_desc_size() != ctypes.sizeof(AttnDesc):
            raise RuntimeError("fl_attn_desc layout mismatch between flattn.h and the binding")
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fl_status_string(int(status)).decode()


def new_desc() -> AttnDesc:
    d = AttnDesc()
    lib().fl_attn_desc_init(ctypes.byref(d))
    return d


def check(status: int, what: str) -> None:
    if status != FL_OK:
        raise FlattnError(status, what)
