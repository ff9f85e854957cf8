"""ctypes declarations of libtxl.so (the C ABI in include/txl.h).

Argument marshalling only.  There is no fallback: if the library is missing the import of the
binding raises, and every non-OK status of a call raises ``TxlError``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# TXL_CHECKED=1 selects the range-checked build of the same library (built on request by
# _build.py --checked)
LIB_PATH = os.path.join(_HERE, "libtxl_checked.so" if os.environ.get("TXL_CHECKED") == "1" else "libtxl.so")

TXL_OK, TXL_ERR_INVALID_ARG, TXL_ERR_UNSUPPORTED, TXL_ERR_ALIGNMENT = 0, 1, 2, 3
TXL_ERR_CUDA, TXL_ERR_TIMEOUT, TXL_ERR_WORKSPACE = 4, 5, 6
TXL_F32, TXL_BF16 = 0, 1

# every function include/txl.h declares
EXPORTS = (
    "txl_status_str", "txl_version", "txl_rel_pos_gen", "txl_rel_attn_fwd",
    "txl_rel_attn_workspace_size", "txl_rel_attn_path", "txl_rel_attn_decode",
    "txl_rel_attn_decode_workspace_size", "txl_rel_attn_decode_noalloc", "txl_mem_push",
    "txl_selftest_wait_timeout", "txl_linear", "txl_rel_attn_layer", "txl_rel_attn_layer_workspace_size",
    "txl_rel_attn_layer_fused", "txl_rel_attn_layer_fused_workspace_size",
    "txl_checked_build", "txl_range_errors", "txl_range_errors_clear", "txl_selftest_range_check",
    "txl_rel_attn_bwd", "txl_rel_attn_bwd_workspace_size", "txl_rel_pos_bwd", "txl_rel_attn_table_fwd",
    "txl_rel_attn_table_path", "txl_rel_attn_decode_path", "txl_rel_attn_fwd_lse", "txl_rel_attn_bwd_lse",
    "txl_rel_attn_bwd_path",
)


class TxlView(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_t", ctypes.c_int64), ("stride_h", ctypes.c_int64)]


class TxlMem(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("stride_b", ctypes.c_int64), ("stride_t", ctypes.c_int64),
                ("stride_h", ctypes.c_int64),
                ("B", ctypes.c_int), ("M", ctypes.c_int), ("H", ctypes.c_int), ("D", ctypes.c_int),
                ("dtype", ctypes.c_int), ("wp", ctypes.c_int), ("valid", ctypes.c_int)]


class TxlError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_str(status), status))


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtxl.so once.  Raises ImportError when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libtxl.so is not built (expected at %s); run "
                          "`python -c \"import __graft_entry__ as g; g.build()\"`" % path)
    lib = ctypes.CDLL(path)
    V = ctypes.POINTER(TxlView)
    Mp = ctypes.POINTER(TxlMem)
    i, i64, vp, fp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
    lib.txl_status_str.argtypes = [i]
    lib.txl_status_str.restype = ctypes.c_char_p
    lib.txl_version.argtypes = []
    lib.txl_version.restype = i
    lib.txl_rel_pos_gen.argtypes = [i, i, i, i, vp, i64, vp, i64, i, vp]
    lib.txl_rel_pos_gen.restype = i
    lib.txl_rel_attn_fwd.argtypes = [i, i, i, i, i, V, Mp, V, V, vp, vp, vp, i64, i, fp, V, i,
                                     vp, ctypes.c_size_t, vp, vp]
    lib.txl_rel_attn_fwd.restype = i
    lib.txl_rel_attn_workspace_size.argtypes = [i, i, i, i, Mp, i]
    lib.txl_rel_attn_workspace_size.restype = ctypes.c_size_t
    lib.txl_rel_attn_path.argtypes = [i, i, i, i, V, Mp, V, V, vp, i64, V, i]
    lib.txl_rel_attn_path.restype = i
    lib.txl_rel_attn_decode.argtypes = [i, i, i, i, i, V, Mp, V, V, vp, vp, vp, i64, i, fp, V, i,
                                        vp, ctypes.c_size_t, vp]
    lib.txl_rel_attn_decode.restype = i
    lib.txl_rel_attn_decode_workspace_size.argtypes = [i, i, i, i, Mp]
    lib.txl_rel_attn_decode_workspace_size.restype = ctypes.c_size_t
    lib.txl_rel_attn_decode_noalloc.argtypes = [i, i, i, i, i, V, Mp, V, V, vp, vp, vp, i64, i, fp, V,
                                                i, vp]
    lib.txl_rel_attn_decode_noalloc.restype = i
    lib.txl_mem_push.argtypes = [Mp, V, V, i, vp]
    lib.txl_mem_push.restype = i
    lib.txl_checked_build.argtypes = []
    lib.txl_checked_build.restype = i
    lib.txl_range_errors.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.txl_range_errors.restype = i
    lib.txl_range_errors_clear.argtypes = []
    lib.txl_range_errors_clear.restype = i
    lib.txl_selftest_range_check.argtypes = [vp]
    lib.txl_selftest_range_check.restype = i
    lib.txl_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint, vp]
    lib.txl_selftest_wait_timeout.restype = i
    lib.txl_linear.argtypes = [i, i, i, vp, i64, vp, i64, vp, i64, i, vp, vp]
    lib.txl_linear.restype = i
    lib.txl_rel_attn_layer.argtypes = [i, i, i, i, i, i, vp, i64, Mp, vp, vp, vp, vp, vp, i64, i, fp,
                                       vp, i64, vp, ctypes.c_size_t, vp, vp]
    lib.txl_rel_attn_layer.restype = i
    lib.txl_rel_attn_layer_workspace_size.argtypes = [i, i, i, i]
    lib.txl_rel_attn_layer_workspace_size.restype = ctypes.c_size_t
    lib.txl_rel_attn_layer_fused.argtypes = [i, i, i, i, i, i, vp, i64, Mp, i, vp, vp, vp, vp, vp, i64, i, fp,
                                             vp, i64, vp, ctypes.c_size_t, vp, vp]
    lib.txl_rel_attn_layer_fused.restype = i
    lib.txl_rel_attn_layer_fused_workspace_size.argtypes = [i, i, i, i]
    lib.txl_rel_attn_layer_fused_workspace_size.restype = ctypes.c_size_t
    lib.txl_rel_attn_bwd.argtypes = [i, i, i, i, i, V, Mp, V, V, vp, vp, vp, i64, i, fp, V, V,
                                     vp, vp, vp, vp, vp, vp, i, vp, ctypes.c_size_t, vp]
    lib.txl_rel_attn_bwd.restype = i
    lib.txl_rel_attn_fwd_lse.argtypes = [i, i, i, i, i, V, Mp, V, V, vp, vp, vp, i64, i, fp, V, vp, i,
                                         vp, ctypes.c_size_t, vp, vp]
    lib.txl_rel_attn_fwd_lse.restype = i
    lib.txl_rel_attn_bwd_lse.argtypes = [i, i, i, i, i, V, Mp, V, V, vp, vp, vp, i64, i, fp, V, V, vp,
                                         vp, vp, vp, vp, vp, vp, i, vp, ctypes.c_size_t, vp]
    lib.txl_rel_attn_bwd_lse.restype = i
    lib.txl_rel_attn_bwd_path.argtypes = [i, i, i, i, V, Mp, V, V, vp, i64, V, V, vp, vp, vp, vp, i]
    lib.txl_rel_attn_bwd_path.restype = i
    lib.txl_rel_attn_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.txl_rel_attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.txl_rel_pos_bwd.argtypes = [i, i, i, i, vp, vp, i64, vp]
    lib.txl_rel_pos_bwd.restype = i
    lib.txl_rel_attn_table_fwd.argtypes = [i, i, i, i, i, V, V, V, vp, vp, vp, i64, vp, fp, V, i, vp]
    lib.txl_rel_attn_table_fwd.restype = i
    lib.txl_rel_attn_table_path.argtypes = [i, i, i, i, i, V, V, V, vp, i64, vp, V, i]
    lib.txl_rel_attn_table_path.restype = i
    lib.txl_rel_attn_decode_path.argtypes = [i, i, i, i, V, Mp, V, V, vp, i64, V, i]
    lib.txl_rel_attn_decode_path.restype = i
    _lib = lib
    return lib


def status_str(status: int) -> str:
    try:
        return load().txl_status_str(int(status)).decode()
    except ImportError:
        return "status %d" % status


def check(status: int, what: str) -> None:
    if status != TXL_OK:
        raise TxlError(status, what)
