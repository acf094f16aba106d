"""ctypes declarations of the C ABI in include/emb.h (libemb.so, built in-tree).

Importing this module loads the CUDA library; if it has not been built the
import fails loudly -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libemb.so")

# emb_status
EMB_OK = 0
EMB_ERR_INVALID_ARG = -1
EMB_ERR_OOM = -2
EMB_ERR_CUDA = -3
EMB_ERR_KEY_RANGE = -4
EMB_ERR_CAPACITY = -5
EMB_ERR_TIMEOUT = -6
EMB_ERR_STATE = -7

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
POOLINGS = {"sum": 0, "mean": 1}
OPTS = {"sgd": 0, "adagrad": 1, "rowwise_adagrad": 2}
VARIANTS = {"reduction": 0, "unique_sort": 1, "unique_hash": 2}

# every symbol the header declares
EXPORTS = (
    "emb_create", "emb_destroy", "emb_init_uniform", "emb_forward", "emb_backward_update",
    "emb_set_keep_dedup", "emb_dedup_result", "emb_unique_workspace", "emb_unique",
    "emb_get_rows", "emb_set_rows", "emb_gather_rows", "emb_sync_status", "emb_launch_count",
    "emb_set_timing", "emb_phase_times", "emb_unique_noalloc", "emb_set_early_dedup",
    "emb_get_master_rows", "emb_set_master_rows", "emb_gather_master_rows", "emb_find_keys",
    "emb_cache_build", "emb_forward_infer", "emb_status_string",
)
UNIQUE_NOALLOC_MAX_KEYS = 262144
PHASES = ("forward", "dedup", "reduce_update")


class EmbTableSpec(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("pooling", ctypes.c_int32), ("opt", ctypes.c_int32), ("lr", ctypes.c_float),
                ("eps", ctypes.c_float), ("init_acc", ctypes.c_float), ("master_fp32", ctypes.c_int32),
                ("dynamic", ctypes.c_int32)]


class EmbError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = lib.emb_status_string(status).decode()
        super().__init__("%s%s (status %d)" % (what + ": " if what else "", msg, status))


def check(status: int, what: str = "") -> None:
    if status != EMB_OK:
        raise EmbError(status, what)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libemb.so is not built; run `python dlrm_sparse_embedding_gb300/build.py` "
                          "(needs nvcc).  There is no CPU fallback.")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    c_int = ctypes.c_int
    L.emb_create.argtypes = [ctypes.POINTER(EmbTableSpec), i32, i32, i64, ctypes.POINTER(vp)]
    L.emb_destroy.argtypes = [vp]
    L.emb_init_uniform.argtypes = [vp, ctypes.c_uint64, f32, f32, vp]
    L.emb_forward.argtypes = [vp, vp, vp, vp, i64, i32, vp, vp]
    L.emb_backward_update.argtypes = [vp, vp, i32, vp]
    L.emb_set_keep_dedup.argtypes = [vp, i32]
    L.emb_set_early_dedup.argtypes = [vp, i32]
    L.emb_dedup_result.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.POINTER(i64), vp]
    L.emb_unique_workspace.argtypes = [i64, ctypes.POINTER(ctypes.c_size_t)]
    L.emb_unique.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.emb_unique_noalloc.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp]
    L.emb_get_rows.argtypes = [vp, i32, i64, i64, vp, vp, vp]
    L.emb_set_rows.argtypes = [vp, i32, i64, i64, vp, vp, vp]
    L.emb_gather_rows.argtypes = [vp, i32, vp, i64, vp, vp, vp]
    L.emb_get_master_rows.argtypes = [vp, i32, i64, i64, vp, vp]
    L.emb_set_master_rows.argtypes = [vp, i32, i64, i64, vp, vp]
    L.emb_gather_master_rows.argtypes = [vp, i32, vp, i64, vp, vp]
    L.emb_find_keys.argtypes = [vp, i32, vp, i64, vp, vp]
    L.emb_cache_build.argtypes = [vp, i32, vp, i64, vp]
    L.emb_forward_infer.argtypes = [vp, vp, vp, vp, i64, i32, vp, vp]
    L.emb_sync_status.argtypes = [vp, vp]
    L.emb_launch_count.argtypes = [vp, ctypes.POINTER(i64), i32]
    L.emb_set_timing.argtypes = [vp, i32]
    L.emb_phase_times.argtypes = [vp, ctypes.POINTER(f32), i32, ctypes.POINTER(i64), i32]
    L.emb_status_string.argtypes = [c_int]
    L.emb_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name != "emb_status_string":
            getattr(L, name).restype = c_int
    return L


lib = _load()
