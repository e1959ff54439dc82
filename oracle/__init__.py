"""CPU oracle for DB-SpMSpV -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
product path (``dynamic_sparsity_spmspv_gb300``) never does: it runs on the
CUDA library or fails.

The arithmetic lives in ``oracle.c`` (plain C, fp64); this module compiles it
with gcc and marshals numpy arrays through ctypes.  Every function cites the
part of the DB-SpMSpV paper (Cong et al., ICPP '26) that it restates; see the
header of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_lib = None

COO, DENSE, FORCE_CSR, FORCE_CSC, PATCHED_CSR = 0, 1, 2, 3, 4
PLUS_TIMES, OR_AND = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (plain gcc, -O2)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        # OpenMP only splits the rows of the all-cores baseline; without it
        # those functions run on one thread
        if subprocess.call(base + ["-fopenmp"], stderr=subprocess.DEVNULL) != 0:
            subprocess.check_call(base)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load(path: Optional[str] = None):
    global _lib
    if _lib is not None and path is None:
        return _lib
    lib = ctypes.CDLL(path or build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_csc_build.restype = P
    lib.oracle_csc_build.argtypes = [I64, I64, P, P, P]
    lib.oracle_csc_free.restype = None
    lib.oracle_csc_free.argtypes = [P]
    lib.oracle_spmspv_push.restype = I64
    lib.oracle_spmspv_push.argtypes = [P, ctypes.c_int, I64, P, P, P, P, P, P]
    lib.oracle_spmspv_pull.restype = I64
    lib.oracle_spmspv_pull.argtypes = [I64, I64, P, P, P, ctypes.c_int, I64, P, P, P, P, P, P]
    lib.oracle_bfs_queue.restype = I64
    lib.oracle_bfs_queue.argtypes = [P, I64, P]
    lib.oracle_bfs_spmspv.restype = I64
    lib.oracle_bfs_spmspv.argtypes = [P, I64, P]
    lib.oracle_activation_mask.restype = I64
    lib.oracle_activation_mask.argtypes = [I64, P, ctypes.c_float, P]
    lib.oracle_spmv_csr.restype = None
    lib.oracle_spmv_csr.argtypes = [I64, I64, P, P, P, P, P, P]
    lib.oracle_spmspv_pull_par.restype = I64
    lib.oracle_spmspv_pull_par.argtypes = [I64, I64, P, P, P, ctypes.c_int, I64, P, P, P, P, P, P]
    lib.oracle_bfs_pull_par.restype = I64
    lib.oracle_bfs_pull_par.argtypes = [I64, P, P, I64, P]
    lib.oracle_par_threads.restype = ctypes.c_int
    lib.oracle_par_threads.argtypes = []
    lib.oracle_block_views.restype = I64
    lib.oracle_block_views.argtypes = [I64, I64, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, P, P, P, P, P, P, P]
    if path is None:
        _lib = lib
    return lib


class use_library:
    """Swap in another build of oracle.c (tests plant mistakes in a mutated
    copy to check that the pins catch them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = _lib
        _lib = _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _csr_arrays(A):
    rp = np.ascontiguousarray(A.row_ptr, dtype=np.int64)
    ci = np.ascontiguousarray(A.col_idx, dtype=np.int32)
    va = None if A.vals is None else np.ascontiguousarray(A.vals, dtype=np.float32)
    return rp, ci, va


class Oracle:
    """Holds the oracle's own column-major copy of A (built once)."""

    def __init__(self, A):
        self.A = A
        self._rp, self._ci, self._va = _csr_arrays(A)
        lib = _load()
        self._h = lib.oracle_csc_build(A.m, A.n, _ptr(self._rp), _ptr(self._ci), _ptr(self._va))
        if not self._h:
            raise MemoryError("oracle_csc_build failed")

    def close(self):
        if getattr(self, "_h", None):
            _load().oracle_csc_free(self._h)
            self._h = None

    def __del__(self):
        self.close()

    # Algorithm 1, push (the oracle proper)
    def spmspv(self, x, semiring: int = PLUS_TIMES, visited: Optional[np.ndarray] = None):
        """Returns (idx int32[k], val float64[k] or None, abs_sum float64[k] or None)."""
        m = self.A.m
        idx = np.ascontiguousarray(x.idx, dtype=np.int32)
        val = None if x.val is None else np.ascontiguousarray(x.val, dtype=np.float32)
        vis = None if visited is None else np.ascontiguousarray(visited, dtype=np.uint8)
        y_idx = np.empty(max(m, 1), dtype=np.int32)
        y_val = np.empty(max(m, 1), dtype=np.float64) if semiring == PLUS_TIMES else None
        y_abs = np.empty(max(m, 1), dtype=np.float64) if semiring == PLUS_TIMES else None
        k = _load().oracle_spmspv_push(self._h, semiring, idx.shape[0], _ptr(idx), _ptr(val),
                                       _ptr(vis), _ptr(y_idx), _ptr(y_val), _ptr(y_abs))
        if k < 0:
            raise MemoryError("oracle_spmspv_push failed")
        if semiring == PLUS_TIMES:
            return y_idx[:k].copy(), y_val[:k].copy(), y_abs[:k].copy()
        return y_idx[:k].copy(), None, None

    # Section 4.3 (DB-Decoding): y = A x' for x' = x thresholded by magnitude
    def decode_layer(self, x: np.ndarray, tau: float):
        """Dense results of one decoding layer: (y float64[m], abs_sum
        float64[m], touched bool[m]); rows nothing reaches are 0."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        keep = activation_mask(x, tau)
        ri, rv, rs = self.spmspv(_SparseX(self.A.n, keep, x[keep]))
        m = self.A.m
        y, s, t = np.zeros(m), np.zeros(m), np.zeros(m, bool)
        y[ri], s[ri], t[ri] = rv, rs, True
        return y, s, t

    def bfs_queue(self, src: int) -> np.ndarray:
        lev = np.empty(self.A.n, dtype=np.int32)
        r = _load().oracle_bfs_queue(self._h, int(src), _ptr(lev))
        if r < 0:
            raise MemoryError("oracle_bfs_queue failed")
        return lev

    def bfs_spmspv(self, src: int) -> np.ndarray:
        lev = np.empty(self.A.n, dtype=np.int32)
        r = _load().oracle_bfs_spmspv(self._h, int(src), _ptr(lev))
        if r == -2:
            raise RuntimeError("oracle_bfs_spmspv: more than n levels")
        if r < 0:
            raise MemoryError("oracle_bfs_spmspv failed")
        return lev


class _SparseX:
    def __init__(self, n, idx, val):
        self.n, self.idx, self.val = n, idx, val


def spmv_csr(A, x: np.ndarray):
    """Dense-input regime: y = A x over every stored entry (x used as
    given).  Returns (y float64[m], abs_sum float64[m])."""
    if A.vals is None:
        raise ValueError("spmv_csr needs a valued matrix")
    rp, ci, va = _csr_arrays(A)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(max(A.m, 1), dtype=np.float64)
    s = np.empty(max(A.m, 1), dtype=np.float64)
    _load().oracle_spmv_csr(A.m, A.n, _ptr(rp), _ptr(ci), _ptr(va), _ptr(x), _ptr(y), _ptr(s))
    return y[:A.m].copy(), s[:A.m].copy()


def activation_mask(x: np.ndarray, tau: float) -> np.ndarray:
    """Section 4.3 / 5 (DB-Decoding, magnitude thresholding): ascending
    int32 indices j with |x_j| > tau (NaN entries kept)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(max(x.shape[0], 1), dtype=np.int32)
    k = _load().oracle_activation_mask(x.shape[0], _ptr(x), float(tau), _ptr(out))
    return out[:k].copy()


def spmspv_pull(A, x, semiring: int = PLUS_TIMES, visited: Optional[np.ndarray] = None):
    """Algorithm 1, pull (row-wise cross-check).  Same return shape as
    ``Oracle.spmspv``."""
    rp, ci, va = _csr_arrays(A)
    idx = np.ascontiguousarray(x.idx, dtype=np.int32)
    val = None if x.val is None else np.ascontiguousarray(x.val, dtype=np.float32)
    vis = None if visited is None else np.ascontiguousarray(visited, dtype=np.uint8)
    y_idx = np.empty(max(A.m, 1), dtype=np.int32)
    y_val = np.empty(max(A.m, 1), dtype=np.float64) if semiring == PLUS_TIMES else None
    y_abs = np.empty(max(A.m, 1), dtype=np.float64) if semiring == PLUS_TIMES else None
    k = _load().oracle_spmspv_pull(A.m, A.n, _ptr(rp), _ptr(ci), _ptr(va), semiring,
                                   idx.shape[0], _ptr(idx), _ptr(val), _ptr(vis),
                                   _ptr(y_idx), _ptr(y_val), _ptr(y_abs))
    if k < 0:
        raise MemoryError("oracle_spmspv_pull failed")
    if semiring == PLUS_TIMES:
        return y_idx[:k].copy(), y_val[:k].copy(), y_abs[:k].copy()
    return y_idx[:k].copy(), None, None


def par_threads() -> int:
    """Threads the all-cores baseline functions use (1 without OpenMP)."""
    return int(_load().oracle_par_threads())


def spmspv_pull_par(A, x, semiring: int = PLUS_TIMES, visited: Optional[np.ndarray] = None):
    """The all-cores CPU baseline: Algorithm 1 (bottom) with the rows split
    among OpenMP threads.  Same return shape as ``Oracle.spmspv``."""
    rp, ci, va = _csr_arrays(A)
    idx = np.ascontiguousarray(x.idx, dtype=np.int32)
    val = None if x.val is None else np.ascontiguousarray(x.val, dtype=np.float32)
    vis = None if visited is None else np.ascontiguousarray(visited, dtype=np.uint8)
    y_idx = np.empty(max(A.m, 1), dtype=np.int32)
    y_val = np.empty(max(A.m, 1), dtype=np.float64) if semiring == PLUS_TIMES else None
    y_abs = np.empty(max(A.m, 1), dtype=np.float64) if semiring == PLUS_TIMES else None
    k = _load().oracle_spmspv_pull_par(A.m, A.n, _ptr(rp), _ptr(ci), _ptr(va), semiring,
                                       idx.shape[0], _ptr(idx), _ptr(val), _ptr(vis),
                                       _ptr(y_idx), _ptr(y_val), _ptr(y_abs))
    if k < 0:
        raise MemoryError("oracle_spmspv_pull_par failed")
    if semiring == PLUS_TIMES:
        return y_idx[:k].copy(), y_val[:k].copy(), y_abs[:k].copy()
    return y_idx[:k].copy(), None, None


def bfs_pull_par(A, src: int) -> np.ndarray:
    """The all-cores CPU baseline's BFS: level-synchronous, each level one
    row-parallel pull.  Levels as ``Oracle.bfs_queue``."""
    rp, ci, _ = _csr_arrays(A)
    lev = np.empty(max(A.n, 1), dtype=np.int32)
    r = _load().oracle_bfs_pull_par(A.n, _ptr(rp), _ptr(ci), int(src), _ptr(lev))
    if r < 0:
        raise MemoryError("oracle_bfs_pull_par failed")
    return lev[:A.n].copy()


def block_views(A, bs: int = 16, th0: int = 32, th1: int = 128, th2: float = 2.0) -> dict:
    """Section 3.2.1 / Figure 5(b): dual block views, csc2csr, nnz and class
    of every nonzero block."""
    rp, ci, _ = _csr_arrays(A)
    nbr = (A.m + bs - 1) // bs
    nbc = (A.n + bs - 1) // bs
    cap = max(A.nnz, 1)
    out = dict(
        blk_row_ptr=np.empty(nbr + 1, np.int64), blk_col_idx=np.empty(cap, np.int64),
        blk_col_ptr=np.empty(nbc + 1, np.int64), blk_row_idx=np.empty(cap, np.int64),
        blk_csc2csr=np.empty(cap, np.int64), blk_nnz=np.empty(cap, np.int32),
        blk_class=np.empty(cap, np.int32))
    B = _load().oracle_block_views(A.m, A.n, _ptr(rp), _ptr(ci), bs, th0, th1, float(th2),
                                   *[_ptr(out[k]) for k in ("blk_row_ptr", "blk_col_idx",
                                                            "blk_col_ptr", "blk_row_idx",
                                                            "blk_csc2csr", "blk_nnz",
                                                            "blk_class")])
    if B < 0:
        raise MemoryError("oracle_block_views failed")
    for k in ("blk_col_idx", "blk_row_idx", "blk_csc2csr", "blk_nnz", "blk_class"):
        out[k] = out[k][:B].copy()
    out["B"] = int(B)
    return out


def tolerance_ok(y_gpu: np.ndarray, y_ref: np.ndarray, abs_sum: np.ndarray) -> np.ndarray:
    """Per-entry acceptance for fp32 plus-times: |y_gpu - y_ref| <= 1e-5 * S_i + 1e-30,
    with S_i = sum_j |a_ij x_j| from the oracle."""
    diff = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    return diff <= 1e-5 * abs_sum + 1e-30
