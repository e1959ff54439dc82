"""ctypes declarations of the C ABI in include/dbspmspv.h (marshalling only).

Loading fails loudly when libdbspmspv.so has not been built: there is no
fallback implementation of any step.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

I32, I64, F64, P = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p

DBS_OK = 0
STATUS_NAMES = {0: "DBS_OK", 1: "DBS_ERR_INVALID_ARG", 2: "DBS_ERR_OOM", 3: "DBS_ERR_CUDA",
                4: "DBS_ERR_TIMEOUT", 5: "DBS_ERR_UNSUPPORTED", 6: "DBS_ERR_INTERNAL"}
NUM_FORMATS = 5


class dbs_build_opts(ctypes.Structure):
    _fields_ = [("th0", I32), ("th1", I32), ("th2", F64), ("force_format", I32),
                ("tile_weight", I32), ("tile_max_row_blocks", I32), ("keep_host", I32),
                ("host_only", I32), ("num_threads", I32), ("device_convert", I32), ("dense_spmv", I32)]


class dbs_exec_opts(ctypes.Structure):
    _fields_ = [("th3", F64), ("local_pull_min", I32), ("collect_stats", I32),
                ("wait_timeout_ns", I64), ("push_work_frac", F64), ("spmv_x_frac", F64)]


class dbs_matrix_info(ctypes.Structure):
    _fields_ = [("m", I64), ("n", I64), ("nnz", I64), ("nbr", I64), ("nbc", I64),
                ("nblocks", I64), ("blocks_by_format", I64 * NUM_FORMATS),
                ("nnz_by_format", I64 * NUM_FORMATS), ("ntiles", I64), ("payload_bytes", I64),
                ("view_bytes", I64), ("total_bytes", I64), ("csr_bytes", I64),
                ("csr_csc_bytes", I64), ("valued", I32), ("on_device", I32),
                ("build_seconds", F64), ("spmv_bytes", I64), ("build_peak_bytes", I64)]


class dbs_stats(ctypes.Structure):
    _fields_ = [("path", I32), ("status", I32), ("n_nzblk", I64), ("n_blk", I64),
                ("x_active", I64), ("visited_blocks", I64), ("hit_blocks", I64),
                ("touched_nnz", I64), ("bytes_alg", I64), ("y_nnz", I64),
                ("bfs_levels", I32), ("bfs_push_levels", I32), ("phase_ns", I64 * 3)]


# name -> (restype, argtypes)
PROTOTYPES = {
    "dbs_build_opts_default": (None, [P]),
    "dbs_exec_opts_default": (None, [P]),
    "dbs_matrix_build_csr": (I32, [I64, I64, I64, P, P, P, ctypes.c_int, P, P, P]),
    "dbs_matrix_destroy": (I32, [P]),
    "dbs_matrix_info_get": (I32, [P, P]),
    "dbs_matrix_export_views": (I32, [P, P, P, P, P, P, P, P]),
    "dbs_matrix_export_csr": (I32, [P, P, P, P]),
    "dbs_workspace_create": (I32, [P, P]),
    "dbs_workspace_destroy": (I32, [P]),
    "dbs_workspace_set_opts": (I32, [P, P]),
    "dbs_workspace_check": (I32, [P, P]),
    "dbs_spmspv": (I32, [P, ctypes.c_int, P, P, I64, P, P, P, P, ctypes.c_int, P, P]),
    "dbs_spmspv_dense": (I32, [P, P, P, ctypes.c_int, P, P]),
    "dbs_spmspv_dense_noalloc": (I32, [P, P, P, P]),
    "dbs_spmspv_dense_noalloc_check": (I32, [P]),
    "dbs_debug_fail_alloc": (I32, [I64, P]),
    "dbs_decode_layer": (I32, [P, P, ctypes.c_float, P, P, P]),
    "dbs_matrix_export_raw": (I32, [P, I32, P, I64, P]),
    "dbs_spmv_plan_create": (I32, [I64, I64, I64, P, P, P, P, P]),
    "dbs_spmv": (I32, [P, P, P, P]),
    "dbs_spmv_plan_info": (I32, [P, P, P]),
    "dbs_spmv_plan_destroy": (I32, [P]),
    "dbs_bfs": (I32, [P, I64, P, P, ctypes.c_int, P, P]),
    "dbs_last_stats": (I32, [P, P, P]),
    "dbs_selftest_wait_timeout": (I32, [P, P]),
    "dbs_bfs_level_stats": (I32, [P, P, I32, P, P, P, P, P]),
    "dbs_status_string": (ctypes.c_char_p, [I32]),
    "dbs_version": (ctypes.c_char_p, []),
}

_lib = None


class DbsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libdbspmspv.so (built by __graft_entry__.build()); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def check(fn: str, status: int):
    if status != DBS_OK:
        raise DbsError(fn, status)
