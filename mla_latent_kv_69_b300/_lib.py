"""ctypes view of libmla_b300.so (the C ABI declared in include/mla.h).

The shared object is loaded on first use; if it is missing every call raises
ImportError. There is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("MLA_B300_LIB", os.path.join(_HERE, "lib", "libmla_b300.so"))

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_TIMEOUT = 5
MLA_ERR_DEVICE_BOUNDS = 6
MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_MAX_SPLITS = 256
MLA_STATIC_SCRATCH_BYTES = 64 << 20

EXPORTS = [
    "mla_absorb_q", "mla_decode_fwd", "mla_combine", "mla_up_v", "mla_quantize_fp8",
    "mla_num_splits", "mla_split_range", "mla_status_string", "mla_abi_version", "mla_decode_kernel",
    "mla_decode_combine_static", "mla_test_decode_stalled", "mla_cache_append", "mla_absorb_q_ex",
    "mla_cache_append_ex", "mla_multi_token_view", "mla_combine_up_v", "mla_quantize_fp6",
]


class MlaCache(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("data", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("max_pages", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("seq_stride_tokens", ctypes.c_int64),
        ("num_rows", ctypes.c_int64),
    ]


class MlaRope(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_float),
        ("yarn_scale", ctypes.c_float),
        ("yarn_alpha", ctypes.c_float),
        ("yarn_beta", ctypes.c_float),
        ("original_max_pos", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libmla_b300.so not found at {LIB_PATH}; build it with "
            "`python -m mla_latent_kv_69_b300.build` (there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.mla_absorb_q.argtypes = [vp, vp, vp, i32, i32, f32, vp, vp]
    lib.mla_decode_fwd.argtypes = [vp, ctypes.POINTER(MlaCache), vp, i32, i32, i32, f32, i32, vp, vp, vp, vp]
    lib.mla_combine.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    lib.mla_decode_combine_static.argtypes = [vp, ctypes.POINTER(MlaCache), vp, i32, i32, i32, f32, i32, vp, vp, vp,
                                              vp]
    lib.mla_test_decode_stalled.argtypes = [vp, ctypes.POINTER(MlaCache), vp, i32, i32, i32, f32, i32, vp, vp, vp,
                                            ctypes.c_uint64, vp]
    lib.mla_up_v.argtypes = [vp, vp, i32, i32, vp, vp]
    lib.mla_combine_up_v.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.mla_cache_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, f32, ctypes.POINTER(MlaCache), i32, vp, vp, vp]
    lib.mla_cache_append_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, ctypes.POINTER(MlaRope),
                                        ctypes.POINTER(MlaCache), i32, vp, vp, vp]
    lib.mla_absorb_q_ex.argtypes = [vp, vp, vp, i32, i32, ctypes.POINTER(MlaRope), vp, vp]
    lib.mla_multi_token_view.argtypes = [ctypes.POINTER(MlaCache), vp, i32, i32, i32, vp, vp, vp, i32,
                                         ctypes.POINTER(MlaCache), vp]
    lib.mla_quantize_fp8.argtypes = [vp, i64, vp, vp, vp]
    lib.mla_quantize_fp6.argtypes = [vp, i64, vp, vp, vp]
    lib.mla_num_splits.argtypes = [i32, i32, i32]
    lib.mla_decode_kernel.argtypes = [i32, i32]
    lib.mla_split_range.argtypes = [i32, i32, i32, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.mla_status_string.argtypes = [i32]
    lib.mla_status_string.restype = ctypes.c_char_p
    for fn in ("mla_absorb_q", "mla_decode_fwd", "mla_combine", "mla_up_v", "mla_quantize_fp8",
               "mla_num_splits", "mla_split_range", "mla_abi_version", "mla_decode_kernel",
               "mla_decode_combine_static", "mla_test_decode_stalled", "mla_cache_append", "mla_absorb_q_ex",
               "mla_cache_append_ex", "mla_multi_token_view", "mla_combine_up_v", "mla_quantize_fp6"):
        getattr(lib, fn).restype = ctypes.c_int
    return lib


_LIB = None


def get():
    """The loaded library (loads it on first call; raises ImportError if absent)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def status_string(status: int) -> str:
    return get().mla_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != MLA_OK:
        raise MlaError(fn, status)
