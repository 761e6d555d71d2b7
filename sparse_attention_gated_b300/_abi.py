"""ctypes mirror of include/hyb.h (argument marshalling only).

Loads the in-tree ``libhyb.so``.  There is no fallback: if the library is
missing or cannot be loaded, importing the ops raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhyb.so")

HYB_F32, HYB_BF16, HYB_E4M3, HYB_MXFP4 = 0, 1, 2, 3
HYB_DEV_BAD_INDEX, HYB_DEV_TIMEOUT = 0x1, 0x2
HYB_NOALLOC_SCRATCH_BYTES = 32 << 20  # include/hyb.h

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f = ctypes.c_float


class CompressArgs(ctypes.Structure):
    _fields_ = [("ca", _p), ("cb", _p), ("za", _p), ("zb", _p), ("bias", _p), ("out", _p), ("out_scale", _p),
                ("batch", _i64), ("n_rows", _i64), ("c", _i64), ("m", _i64), ("first_block", _i64),
                ("out_batch_stride", _i64), ("in_batch_stride", _i64), ("overlap", _i32), ("in_dtype", _i32),
                ("out_dtype", _i32),
                ("dev_status", _p)]


class IndexArgs(ctypes.Structure):
    _fields_ = [("qI", _p), ("qI_scale", _p), ("w", _p), ("kI", _p), ("kI_scale", _p), ("idx", _p), ("scores", _p),
                ("batch", _i64), ("n_q", _i64), ("n_entries", _i64), ("kv_stride", _i64), ("n_ih", _i64),
                ("c_I", _i64), ("m", _i64), ("k", _i64), ("q_pos0", _i64), ("dtype", _i32), ("dev_status", _p),
                ("ev_scores_begin", _p), ("ev_scores_end", _p), ("q_pos", _p)]


class Window(ctypes.Structure):
    _fields_ = [("kw", _p), ("n_kv", _i64), ("kv_pos0", _i64), ("q_pos0", _i64), ("n_win", _i64), ("out", _p),
                ("out_dtype", _i32), ("q_pos", _p), ("kv_pos0s", _p)]


class CsaAttendArgs(ctypes.Structure):
    _fields_ = [("q", _p), ("kc", _p), ("vc", _p), ("idx", _p), ("o", _p), ("lse", _p), ("batch", _i64),
                ("n_q", _i64), ("n_h", _i64), ("c", _i64), ("n_entries", _i64), ("kv_stride", _i64), ("k", _i64),
                ("scale", _f), ("dtype", _i32), ("dev_status", _p), ("window", _p), ("sink", _p)]


class HcaAttendArgs(ctypes.Structure):
    _fields_ = [("q", _p), ("kc", _p), ("vc", _p), ("o", _p), ("lse", _p), ("batch", _i64), ("n_q", _i64),
                ("n_h", _i64), ("c", _i64), ("n_entries", _i64), ("kv_stride", _i64), ("m", _i64), ("q_pos0", _i64),
                ("scale", _f), ("dtype", _i32), ("dev_status", _p), ("window", _p), ("sink", _p), ("q_pos", _p)]


class NormRopeArgs(ctypes.Structure):
    _fields_ = [("x", _p), ("rows", _i64), ("c", _i64), ("gamma", _p), ("eps", _f), ("dtype", _i32), ("pos", _p),
                ("rows_per_pos", _i64), ("rope_dims", _i64), ("theta", ctypes.c_double), ("row_stride", _i64)]


class GprojArgs(ctypes.Structure):
    _fields_ = [("o", _p), ("w", _p), ("out", _p), ("rows", _i64), ("n_h", _i64), ("c", _i64), ("g", _i64),
                ("d_g", _i64), ("dtype", _i32), ("out_dtype", _i32), ("dev_status", _p), ("out_row_stride", _i64)]


class SwaArgs(ctypes.Structure):
    _fields_ = [("q", _p), ("kw", _p), ("vw", _p), ("o_in", _p), ("lse_in", _p), ("out", _p), ("lse_out", _p),
                ("batch", _i64), ("n_q", _i64), ("n_h", _i64), ("c", _i64), ("n_kv", _i64), ("kv_pos0", _i64),
                ("q_pos0", _i64), ("n_win", _i64), ("scale", _f), ("dtype", _i32), ("out_dtype", _i32),
                ("dev_status", _p), ("q_pos", _p), ("kv_pos0s", _p)]


# every symbol include/hyb.h declares, with (restype, argtypes)
SIGNATURES = {
    "hyb_compress_out_count": (_i64, [_i64, _i64, _i32, _i64]),
    "hyb_compress_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(CompressArgs)]),
    "hyb_compress": (ctypes.c_int, [ctypes.POINTER(CompressArgs), _p, ctypes.c_size_t, _p]),
    "hyb_compress_batch": (ctypes.c_int, [ctypes.POINTER(CompressArgs), ctypes.c_int32, _p]),
    "csa_index_topk_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(IndexArgs)]),
    "csa_index_topk_counter_bytes": (ctypes.c_size_t, []),
    "csa_index_topk": (ctypes.c_int, [ctypes.POINTER(IndexArgs), _p, ctypes.c_size_t, _p]),
    "csa_index_topk_noalloc": (ctypes.c_int, [ctypes.POINTER(IndexArgs), _p]),
    "csa_index_topk_noalloc_reset": (ctypes.c_int, [_p]),
    "hyb_set_grid_wait_limit": (_i64, [_i64]),
    "csa_attend_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(CsaAttendArgs)]),
    "csa_attend": (ctypes.c_int, [ctypes.POINTER(CsaAttendArgs), _p, ctypes.c_size_t, _p]),
    "hca_attend_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(HcaAttendArgs)]),
    "hca_attend": (ctypes.c_int, [ctypes.POINTER(HcaAttendArgs), _p, ctypes.c_size_t, _p]),
    "swa_merge_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(SwaArgs)]),
    "swa_merge": (ctypes.c_int, [ctypes.POINTER(SwaArgs), _p, ctypes.c_size_t, _p]),
    "hyb_rmsnorm_rope": (ctypes.c_int, [ctypes.POINTER(NormRopeArgs), _p]),
    "hyb_rmsnorm_rope_batch": (ctypes.c_int, [ctypes.POINTER(NormRopeArgs), ctypes.c_int32, _p]),
    "hyb_grouped_out_proj": (ctypes.c_int, [ctypes.POINTER(GprojArgs), _p]),
    "hyb_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "hyb_last_error": (ctypes.c_char_p, []),
    "hyb_version": (_i32, []),
    "hyb_built_arch": (_i32, []),
}

_lib = None


class HybError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        self.status = status
        msg = lib.hyb_status_string(status).decode()
        detail = lib.hyb_last_error().decode()
        super().__init__(f"{where}: {msg}: {detail}")


def load(path: str = LIB_PATH):
    """Load libhyb.so (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"the CUDA library {path} is missing; build it with "
                               "`python -m sparse_attention_gated_b300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(status: int, where: str) -> None:
    if status != 0:
        raise HybError(status, where)
