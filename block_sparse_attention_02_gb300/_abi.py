"""ctypes mirror of include/msa.h and the loader of libmsa.so.

Nothing here computes: it declares the C structs and function signatures and
loads the in-tree library built by ``build.py``.  There is no fallback; if the
library is missing the import of the binding raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmsa.so")

MSA_OK = 0
MSA_ERR_INVALID_ARG = 1
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_CUDA = 3
MSA_ERR_DEVICE_CHECK = 4
MSA_ERR_WORKSPACE = 5

MSA_DEVERR_TIMEOUT = 0x1
MSA_DEVERR_BAD_PAGE = 0x2
MSA_DEVERR_BAD_SEL = 0x4
MSA_DEVERR_BAD_LEN = 0x8

MSA_MODE_PREFILL = 0
MSA_MODE_DECODE = 1
MSA_MODE_CHUNK = 2

_p = C.c_void_p
_i64x2 = C.c_int64 * 2
_i64x3 = C.c_int64 * 3
_i64x4 = C.c_int64 * 4


class IndexArgs(C.Structure):
    _fields_ = [
        ("mode", C.c_int), ("B", C.c_int), ("S", C.c_int), ("Hkv", C.c_int), ("HI", C.c_int),
        ("dI", C.c_int), ("Bk", C.c_int),
        ("q_idx", _p), ("q_idx_stride", _i64x4),
        ("w", _p), ("w_stride", _i64x3),
        ("k_idx", _p), ("k_idx_stride", _i64x3),
        ("num_pages", C.c_int64), ("seq_pt", _p), ("max_pages", C.c_int64), ("seq_len", _p),
        ("C", _p), ("C_stride", _i64x3), ("nb_stride", C.c_int),
        ("dev_err", _p),
        ("k", C.c_int), ("sel", _p), ("count", _p), ("pt", _p), ("n", _p), ("last_len", _p),
        ("row_scratch", _p), ("scratch_zeroed", C.c_int),
        ("q_pos", _p),
    ]


class TopkArgs(C.Structure):
    _fields_ = [
        ("mode", C.c_int), ("B", C.c_int), ("S", C.c_int), ("Hkv", C.c_int), ("Bk", C.c_int), ("k", C.c_int),
        ("C", _p), ("C_stride", _i64x3), ("nb_stride", C.c_int),
        ("seq_len", _p), ("sel", _p), ("count", _p), ("dev_err", _p),
        ("q_pos", _p),
    ]


class PrefillArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("S", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("D", C.c_int), ("Bk", C.c_int),
        ("k", C.c_int), ("softmax_scale", C.c_float),
        ("Q", _p), ("Q_stride", _i64x3), ("K", _p), ("K_stride", _i64x3), ("V", _p), ("V_stride", _i64x3),
        ("sel", _p), ("count", _p), ("O", _p), ("LSE", _p), ("dev_err", _p),
        ("mode", C.c_int), ("seq_pt", _p), ("max_pages", C.c_int64), ("num_pages", C.c_int64), ("q_pos", _p),
    ]


class DecodeArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("D", C.c_int), ("Bk", C.c_int), ("k", C.c_int),
        ("softmax_scale", C.c_float),
        ("Q", _p), ("Q_stride", _i64x2), ("K_pool", _p), ("V_pool", _p), ("kv_stride", _i64x3),
        ("num_pages", C.c_int64), ("pt", _p), ("n", _p), ("last_len", _p),
        ("O", _p), ("LSE", _p), ("dev_err", _p), ("scratch_zeroed", C.c_int),
    ]


class AppendArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("Hkv", C.c_int), ("D", C.c_int), ("dI", C.c_int), ("Bk", C.c_int),
        ("K_new", _p), ("K_new_stride", _i64x2), ("V_new", _p), ("V_new_stride", _i64x2),
        ("kidx_new", _p), ("kidx_new_stride", _i64x2),
        ("K_pool", _p), ("V_pool", _p), ("kv_stride", _i64x3), ("kidx_pool", _p), ("kidx_stride", _i64x3),
        ("num_pages", C.c_int64), ("seq_pt", _p), ("max_pages", C.c_int64), ("seq_len", _p), ("dev_err", _p),
        ("T", C.c_int), ("new_t_stride", _i64x3),
    ]


class DenseDecodeArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("D", C.c_int), ("Bk", C.c_int),
        ("softmax_scale", C.c_float),
        ("Q", _p), ("Q_stride", _i64x2), ("K_pool", _p), ("V_pool", _p), ("kv_stride", _i64x3),
        ("num_pages", C.c_int64), ("seq_pt", _p), ("max_pages", C.c_int64), ("seq_len", _p),
        ("O", _p), ("LSE", _p), ("dev_err", _p), ("scratch_zeroed", C.c_int),
    ]


class DensePrefillArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("S", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("D", C.c_int),
        ("softmax_scale", C.c_float),
        ("Q", _p), ("Q_stride", _i64x3), ("K", _p), ("K_stride", _i64x3), ("V", _p), ("V_stride", _i64x3),
        ("O", _p), ("LSE", _p), ("dev_err", _p),
    ]


# exported function name -> (restype, argtypes)
SIGNATURES = {
    "msa_version": (C.c_int, []),
    "msa_last_error_string": (C.c_char_p, []),
    "msa_status_string": (C.c_char_p, [C.c_int]),
    "msa_index_score": (C.c_int, [C.POINTER(IndexArgs), _p]),
    "msa_topk_blocks": (C.c_int, [C.POINTER(TopkArgs), _p]),
    "msa_build_page_table": (C.c_int, [_p, _p, _p, C.c_int64, _p, C.c_int, C.c_int, C.c_int, C.c_int,
                                       _p, _p, _p, _p, _p]),
    "msa_sparse_attn_prefill_workspace_size": (C.c_size_t, [C.POINTER(PrefillArgs), C.c_int64]),
    "msa_sparse_attn_prefill": (C.c_int, [C.POINTER(PrefillArgs), _p, C.c_size_t, _p]),
    "msa_sparse_attn_decode_workspace_size": (C.c_size_t, [C.POINTER(DecodeArgs)]),
    "msa_sparse_attn_decode": (C.c_int, [C.POINTER(DecodeArgs), _p, C.c_size_t, _p]),
    "msa_sparse_attn_decode_noalloc": (C.c_int, [C.POINTER(DecodeArgs), _p]),
    "msa_lse_merge": (C.c_int, [_p, _p, C.c_int64, C.c_int, C.c_int, _p, _p, _p, _p]),
    "msa_cache_append": (C.c_int, [C.POINTER(AppendArgs), _p]),
    "msa_dense_attn_decode_workspace_size": (C.c_size_t, [C.POINTER(DenseDecodeArgs)]),
    "msa_dense_attn_decode": (C.c_int, [C.POINTER(DenseDecodeArgs), _p, C.c_size_t, _p]),
    "msa_dense_attn_prefill": (C.c_int, [C.POINTER(DensePrefillArgs), _p]),
}

_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libmsa.so (built in-tree); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
            lib = C.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


class MSAError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        name = load().msa_status_string(status).decode()
        super().__init__(f"{func}: {name}: {detail}")


def check(status: int, func: str) -> None:
    if status != MSA_OK:
        raise MSAError(status, func, load().msa_last_error_string().decode())
