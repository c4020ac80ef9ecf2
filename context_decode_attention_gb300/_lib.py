"""Loading libdcp.so and declaring its C signatures (include/dcp.h)."""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libdcp.so")

DCP_F32, DCP_BF16, DCP_FP8_E4M3 = 0, 1, 2
DCP_LAYOUT_GQA, DCP_LAYOUT_MLA = 0, 1

# every symbol include/dcp.h declares
EXPORTS = [
    "dcp_version", "dcp_error_string", "dcp_launch_count", "dcp_attention_kernel", "dcp_workspace_size", "dcp_workspace_init", "dcp_get_error",
    "dcp_slot_mapping", "dcp_transfer_blocks", "dcp_pcp_partition", "dcp_prefill_attention",
    "dcp_sparse_workspace_size", "dcp_sparse_localize", "dcp_sparse_decode_attention", "dcp_partial_attention", "dcp_lse_merge", "dcp_decode_attention", "dcp_decode_plan", "dcp_decode_attention_planned",
    "dcp_decode_attention_noalloc", "dcp_noalloc_get_error",
]


class DcpError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(msg)
        self.code = code


class DcpParams(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int32), ("I", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("layout", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32), ("Tq", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("kv_scale", ctypes.c_float), ("softmax_scale", ctypes.c_float),
    ]


_lib = None


def lib_path():
    return _LIB_PATH


def lib():
    """The loaded libdcp (raises if it was never built or cannot load)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"libdcp.so is missing at {_LIB_PATH}: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (there is no CPU fallback)")
    L = ctypes.CDLL(_LIB_PATH)
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER(DcpParams)
    sig = {
        "dcp_version": (ctypes.c_int, []),
        "dcp_error_string": (ctypes.c_char_p, [ctypes.c_int]),
        "dcp_launch_count": (ctypes.c_uint64, []),
        "dcp_attention_kernel": (ctypes.c_char_p, [P]),
        "dcp_workspace_size": (ctypes.c_int, [P, i32, i64, ctypes.POINTER(sz)]),
        "dcp_workspace_init": (ctypes.c_int, [p, sz, p]),
        "dcp_get_error": (ctypes.c_int, [p, p, ctypes.POINTER(ctypes.c_uint32)]),
        "dcp_slot_mapping": (ctypes.c_int, [P, i32, p, i64, p, p, p, i32, i64, p, p, p, p, p, p, p, p, p, p, sz, p]),
        "dcp_transfer_blocks": (ctypes.c_int, [P, i32, p, p, i32, i64, p, p, p, p, p, sz, p]),
        "dcp_pcp_partition": (ctypes.c_int, [i32, i32, p, p, i32, p, p, p, sz, p]),
        "dcp_sparse_workspace_size": (ctypes.c_int, [P, i32, i32, ctypes.POINTER(sz)]),
        "dcp_sparse_localize": (ctypes.c_int, [P, i32, i32, p, p, p, p, p, sz, p]),
        "dcp_sparse_decode_attention": (ctypes.c_int, [P, i32, i32, p, p, p, i64, p, i32, p, p, p, p, sz, p]),
        "dcp_prefill_attention": (ctypes.c_int, [P, i32, i32, p, p, p, p, i64, p, i32, p, p, p, p, p, p, p, sz, p]),
        "dcp_partial_attention": (ctypes.c_int, [P, i32, p, p, p, i64, p, i32, p, p, p, p, p, sz, p]),
        "dcp_lse_merge": (ctypes.c_int, [i32, i64, i32, p, p, p, i32, p, p]),
        "dcp_decode_attention": (ctypes.c_int, [P, i32, p, p, p, i64, p, i32, p, p, p, p, p, sz, p]),
        "dcp_decode_plan": (ctypes.c_int, [P, i32, p, p, i32, p, sz, p]),
        "dcp_decode_attention_planned": (ctypes.c_int, [P, i32, p, p, p, i64, p, i32, p, p, p, p, p, sz, p]),
        "dcp_decode_attention_noalloc": (ctypes.c_int, [P, i32, p, p, p, i64, p, i32, p, p, p, p, p]),
        "dcp_noalloc_get_error": (ctypes.c_int, [p, ctypes.POINTER(ctypes.c_uint32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L
