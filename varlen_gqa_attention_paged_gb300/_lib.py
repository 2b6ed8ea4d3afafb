"""ctypes declarations of the C ABI in include/ua.h (libua.so next to this file)."""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libua.so")

# ua_status_t
UA_OK, UA_ERR_INVALID_ARG, UA_ERR_UNSUPPORTED, UA_ERR_CUDA = 0, 1, 2, 3
UA_ERR_WORKSPACE, UA_ERR_DEVICE_CHECK, UA_ERR_TIMEOUT, UA_ERR_SCRATCH_LIMIT = 4, 5, 6, 7
UA_NOALLOC_SCRATCH_BYTES = 16 << 20
# ua_dtype_t
UA_DT_F16, UA_DT_BF16, UA_DT_F8E4M3, UA_DT_F32 = 0, 1, 2, 3
# ua_backend_t
UA_BACKEND_AUTO, UA_BACKEND_2D, UA_BACKEND_SPLIT = 0, 1, 2
# ua_path_t
UA_PATH_2D, UA_PATH_SPLIT = 1, 2

# every symbol include/ua.h declares
EXPORTS = ("ua_unified_attention", "ua_unified_attention_noalloc", "ua_plan", "ua_workspace_bytes", "ua_device_status",
           "ua_device_status_reset", "ua_status_string", "ua_version")


class UaShape(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_q", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32),
        ("max_seqlen_k", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("qq_bias_stride", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("events", ctypes.c_void_p),
        ("k_scale_tok", ctypes.c_void_p),
        ("v_scale_tok", ctypes.c_void_p),
        ("k_scale_stride", ctypes.c_int64 * 3),
        ("v_scale_stride", ctypes.c_int64 * 3),
    ]


class UaPlan(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("block_m", ctypes.c_int32),
        ("n_part", ctypes.c_int32),
        ("grid_x", ctypes.c_int32),
        ("grid_y", ctypes.c_int32),
        ("grid_z", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("cluster_y", ctypes.c_int32),
        ("cluster_z", ctypes.c_int32),
        ("slot_per_seq", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_LOCK = threading.Lock()
_LIB = None


def load():
    """The loaded libua.so.  Raises if the CUDA library has not been built."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(varlen_gqa_attention_paged_gb300.build.build()); there is no CPU fallback")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.ua_unified_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                                             f32, i32, vp, vp, vp, i32, vp, i32, vp,
                                             ctypes.POINTER(UaShape)]
        lib.ua_unified_attention.restype = ctypes.c_int
        lib.ua_unified_attention_noalloc.argtypes = lib.ua_unified_attention.argtypes
        lib.ua_unified_attention_noalloc.restype = ctypes.c_int
        lib.ua_plan.argtypes = [ctypes.POINTER(UaShape), i32, i32, i32, i32, i32, i32, i32, i32,
                                ctypes.POINTER(UaPlan)]
        lib.ua_plan.restype = ctypes.c_int
        lib.ua_workspace_bytes.argtypes = [ctypes.POINTER(UaShape), i32, i32, i32, i32, i32, i32,
                                           i32]
        lib.ua_workspace_bytes.restype = ctypes.c_size_t
        lib.ua_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        lib.ua_device_status.restype = ctypes.c_int
        lib.ua_device_status_reset.argtypes = [vp]
        lib.ua_device_status_reset.restype = ctypes.c_int
        lib.ua_status_string.argtypes = [ctypes.c_int]
        lib.ua_status_string.restype = ctypes.c_char_p
        lib.ua_version.argtypes = []
        lib.ua_version.restype = ctypes.c_int
        _LIB = lib
        return lib
