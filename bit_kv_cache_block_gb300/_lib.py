"""ctypes mirror of include/kvq.h: the structs, the status codes and every entry point.

Argument marshalling only. The library is loaded from this package directory and nothing
falls back to Python or the CPU: a missing or unloadable libkvq.so raises.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")

KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CAPACITY, KVQ_ERR_ALIGNMENT, KVQ_ERR_CUDA, \
    KVQ_ERR_TIMEOUT, KVQ_ERR_PAGE = range(8)
KVQ_RTN, KVQ_NUQ, KVQ_VARN, KVQ_INT4 = range(4)
KVQ_F16, KVQ_BF16 = 0, 1
KVQ_LAYOUT_ROWS, KVQ_LAYOUT_MMA = 0, 1
LAYOUTS = {"rows": KVQ_LAYOUT_ROWS, "mma": KVQ_LAYOUT_MMA}
KVQ_FORMAT_VERSION = 2
KVQ_STATIC_WORKSPACE_BYTES = 8 << 20
METHODS = {"rtn": KVQ_RTN, "nuq": KVQ_NUQ, "varn": KVQ_VARN, "int4": KVQ_INT4}

# every entry point declared in include/kvq.h
EXPORTS = ["kvq_status_str", "kvq_dense_kv_bytes", "kvq_layout", "kvq_cache_init", "kvq_append_block",
           "kvq_truncate", "kvq_reset", "kvq_debug_stall_decode", "kvq_decode_splits", "kvq_decode_workspace_bytes", "kvq_decode_bytes",
           "kvq_decode_attn", "kvq_decode_attn_ex", "kvq_decode_attn_static", "kvq_dequant", "kvq_calibrate_keys", "kvq_error_stats",
           "kvq_error_topk_workspace_bytes", "kvq_error_topk", "kvq_fit_codebook_workspace_bytes",
           "kvq_fit_codebook"]


class kvq_config(C.Structure):
    _fields_ = [("method", C.c_int32), ("bits", C.c_int32), ("batch", C.c_int32), ("n_kv_heads", C.c_int32),
                ("n_q_heads", C.c_int32), ("head_dim", C.c_int32), ("block", C.c_int32),
                ("max_blocks", C.c_int32), ("in_dtype", C.c_int32), ("pre_rope", C.c_int32),
                ("rope_theta", C.c_double), ("outlier_frac", C.c_float), ("varn_iters", C.c_int32),
                ("hadamard", C.c_int32), ("layout", C.c_int32), ("n_pages", C.c_int32),
                ("key_calib", C.c_int32), ("sink", C.c_int32), ("scale_group", C.c_int32),
                ("v_csc", C.c_int32)]


class kvq_layout_t(C.Structure):
    _fields_ = [("record_bytes", C.c_uint64), ("codes_off", C.c_uint64 * 2), ("codes_bytes", C.c_uint64 * 2),
                ("meta_off", C.c_uint64 * 2), ("meta_bytes", C.c_uint64 * 2), ("csr_off", C.c_uint64 * 2),
                ("csr_bytes", C.c_uint64 * 2), ("records_bytes", C.c_uint64), ("rope_off", C.c_uint64),
                ("rope_bytes", C.c_uint64), ("total_bytes", C.c_uint64), ("words_per_row", C.c_int32),
                ("n_outliers", C.c_int32), ("format_version", C.c_uint32), ("reserved", C.c_int32),
                ("calib_off", C.c_uint64), ("calib_bytes", C.c_uint64), ("sink_off", C.c_uint64),
                ("sink_bytes", C.c_uint64)]


class kvq_cache(C.Structure):
    _fields_ = [("cfg", kvq_config), ("lay", kvq_layout_t), ("base", C.c_void_p), ("codebook", C.c_void_p),
                ("dev_status", C.c_void_p), ("n_blocks", C.c_int32), ("device", C.c_int32),
                ("block_table", C.c_void_p), ("calibrated", C.c_int32)]


_lib = None


def lib() -> C.CDLL:
    """The loaded libkvq.so (loads it on first use; raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libkvq.so not found at {LIB_PATH}: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'` (the CUDA path has no fallback)")
    L = C.CDLL(LIB_PATH)
    vp, i32, u64, sz = C.c_void_p, C.c_int32, C.c_uint64, C.c_size_t
    P = C.POINTER
    L.kvq_status_str.restype = C.c_char_p
    L.kvq_status_str.argtypes = [C.c_int]
    L.kvq_dense_kv_bytes.restype = u64
    L.kvq_dense_kv_bytes.argtypes = [C.c_int64] * 6
    L.kvq_layout.restype = C.c_int
    L.kvq_layout.argtypes = [P(kvq_config), P(kvq_layout_t)]
    L.kvq_cache_init.restype = C.c_int
    L.kvq_cache_init.argtypes = [P(kvq_cache), P(kvq_config), vp, sz, vp, vp, vp]
    L.kvq_append_block.restype = C.c_int
    L.kvq_append_block.argtypes = [P(kvq_cache), vp, vp, i32, vp, vp]
    L.kvq_truncate.restype = C.c_int
    L.kvq_truncate.argtypes = [P(kvq_cache), i32]
    L.kvq_reset.restype = C.c_int
    L.kvq_reset.argtypes = [P(kvq_cache)]
    L.kvq_debug_stall_decode.restype = C.c_int
    L.kvq_debug_stall_decode.argtypes = [i32]
    L.kvq_decode_splits.restype = i32
    L.kvq_decode_splits.argtypes = [P(kvq_config), i32]
    L.kvq_decode_workspace_bytes.restype = C.c_int
    L.kvq_decode_workspace_bytes.argtypes = [P(kvq_config), i32, P(sz)]
    L.kvq_decode_bytes.restype = u64
    L.kvq_decode_bytes.argtypes = [P(kvq_config), i32]
    L.kvq_decode_attn.restype = C.c_int
    L.kvq_decode_attn.argtypes = [P(kvq_cache), vp, vp, vp, i32, vp, vp, sz, vp]
    L.kvq_decode_attn_ex.restype = C.c_int
    L.kvq_decode_attn_ex.argtypes = [P(kvq_cache), vp, vp, vp, i32, C.c_int64, C.c_int64, vp, vp, sz, vp]
    L.kvq_decode_attn_static.restype = C.c_int
    L.kvq_decode_attn_static.argtypes = [P(kvq_cache), vp, vp, vp, i32, vp, vp]
    L.kvq_dequant.restype = C.c_int
    L.kvq_dequant.argtypes = [P(kvq_cache), i32, i32, i32, vp, vp, vp]
    L.kvq_calibrate_keys.restype = C.c_int
    L.kvq_calibrate_keys.argtypes = [P(kvq_cache), vp, i32, vp]
    L.kvq_error_stats.restype = C.c_int
    L.kvq_error_stats.argtypes = [P(kvq_cache), vp, vp, i32, i32, vp, vp, vp]
    L.kvq_error_topk_workspace_bytes.restype = sz
    L.kvq_error_topk_workspace_bytes.argtypes = []
    L.kvq_fit_codebook_workspace_bytes.restype = sz
    L.kvq_fit_codebook_workspace_bytes.argtypes = [i32, C.c_int64]
    L.kvq_fit_codebook.restype = C.c_int
    L.kvq_fit_codebook.argtypes = [vp, vp, i32, C.c_int64, i32, i32, vp, vp, sz, vp]
    L.kvq_error_topk.restype = C.c_int
    L.kvq_error_topk.argtypes = [vp, C.c_int64, P(C.c_double), i32, vp, vp, sz, vp]
    _lib = L
    return L


class KVQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


def status_str(s: int) -> str:
    return lib().kvq_status_str(int(s)).decode()


def check(status: int, where: str) -> None:
    if status != KVQ_OK:
        raise KVQError(status, where)
