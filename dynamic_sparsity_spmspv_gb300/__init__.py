"""GB300 DB-SpMSpV: dual-view blocked sparse-matrix x sparse-vector products.

A thin binding over the C ABI of libdbspmspv.so (include/dbspmspv.h): every
step of the computation runs in the library's CUDA kernels (or, for the
one-time format conversion, its native host builder).  This module only
marshals arguments; PyTorch provides device memory and streams.

Method: Cong et al., "DB-SpMSpV: Dual-View Blocked Sparse Matrix-Sparse Vector
Multiplication for Dynamic GPU Workloads", ICPP '26.

    A = DBMatrix(m, n, row_ptr, col_idx, vals)      # build once (Section 3.2)
    ws = Workspace(A)
    y_idx, y_val, y_nnz = spmspv(A, x_idx, x_val, ws=ws)   # per x (3.3, 4.1)
    y = spmspv_dense(A, x_dense, ws=ws)                  # decoding form (4.3)
    levels, nlev = bfs(A, src, ws=ws)                    # DB-BFS (4.2)
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import _lib
from ._lib import DbsError, dbs_build_opts, dbs_exec_opts, dbs_matrix_info, dbs_stats  # noqa: F401

PLUS_TIMES, OR_AND = 0, 1
PATH_AUTO, PATH_PUSH, PATH_PULL, PATH_SPMV = 0, 1, 2, 3
FMT_AUTO, FMT_COO, FMT_DENSE, FMT_FORCE_CSR, FMT_FORCE_CSC, FMT_PATCHED_CSR = -1, 0, 1, 2, 3, 4
FORMAT_NAMES = ("coo", "dense", "force_csr", "force_csc", "patched_csr")

_PATHS = {"auto": PATH_AUTO, "push": PATH_PUSH, "pull": PATH_PULL, "spmv": PATH_SPMV}
_SEMIRINGS = {"plus_times": PLUS_TIMES, "or_and": OR_AND}


def _torch():
    import torch
    return torch


def _stream_handle(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _path(p) -> int:
    return _PATHS[p] if isinstance(p, str) else int(p)


def _semiring(s) -> int:
    return _SEMIRINGS[s] if isinstance(s, str) else int(s)


def _set_fields(o, kw):
    names = {f for f, _ in type(o)._fields_}
    for k, v in kw.items():
        if k not in names:
            raise TypeError(f"{type(o).__name__} has no field {k!r}")
        setattr(o, k, v)
    return o


def build_opts(**kw) -> dbs_build_opts:
    o = dbs_build_opts()
    _lib.load().dbs_build_opts_default(ctypes.byref(o))
    return _set_fields(o, kw)


def exec_opts(**kw) -> dbs_exec_opts:
    o = dbs_exec_opts()
    _lib.load().dbs_exec_opts_default(ctypes.byref(o))
    return _set_fields(o, kw)


class DBMatrix:
    """dbs_matrix_build_csr: the blocked dual-view matrix (library-owned HBM).

    row_ptr int64[m+1], col_idx int32[nnz], vals float32[nnz] or None, as
    numpy arrays (host) or torch CUDA tensors (device)."""

    def __init__(self, m: int, n: int, row_ptr, col_idx, vals=None, *, opts: Optional[dbs_build_opts] = None,
                 stream=None, **opt_kw):
        lib = _lib.load()
        if opts is None:
            opts = build_opts(**opt_kw)
        on_dev = not isinstance(row_ptr, np.ndarray)
        if on_dev:
            torch = _torch()
            row_ptr = row_ptr.to(torch.int64).contiguous()
            col_idx = col_idx.to(torch.int32).contiguous()
            vals = None if vals is None else vals.to(torch.float32).contiguous()
        else:
            row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
            col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
            vals = None if vals is None else np.ascontiguousarray(vals, dtype=np.float32)
        nnz = int(row_ptr[-1])
        handle = P = ctypes.c_void_p()
        s = None if opts.host_only else _stream_handle(stream)
        st = lib.dbs_matrix_build_csr(int(m), int(n), nnz, _ptr(row_ptr), _ptr(col_idx), _ptr(vals),
                                      1 if on_dev else 0, ctypes.byref(opts), s, ctypes.byref(handle))
        _lib.check("dbs_matrix_build_csr", st)
        self._h = P
        self.m, self.n, self.nnz = int(m), int(n), nnz
        self.valued = vals is not None

    @classmethod
    def from_csr(cls, A, **kw) -> "DBMatrix":
        """From any object with m, n, row_ptr, col_idx, vals (e.g. synth.CSR)."""
        return cls(A.m, A.n, A.row_ptr, A.col_idx, A.vals, **kw)

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        inf = dbs_matrix_info()
        _lib.check("dbs_matrix_info_get", _lib.load().dbs_matrix_info_get(self._h, ctypes.byref(inf)))
        d = {f: getattr(inf, f) for f, _ in inf._fields_}
        d["blocks_by_format"] = list(inf.blocks_by_format)
        d["nnz_by_format"] = list(inf.nnz_by_format)
        return d

    def export_views(self) -> dict:
        inf = self.info()
        B, nbr, nbc = inf["nblocks"], inf["nbr"], inf["nbc"]
        out = dict(blk_row_ptr=np.empty(nbr + 1, np.int64), blk_col_idx=np.empty(B, np.int64),
                   blk_col_ptr=np.empty(nbc + 1, np.int64), blk_row_idx=np.empty(B, np.int64),
                   blk_csc2csr=np.empty(B, np.int64), blk_nnz=np.empty(B, np.int32),
                   blk_format=np.empty(B, np.int32))
        st = _lib.load().dbs_matrix_export_views(self._h, *[_ptr(out[k]) for k in (
            "blk_row_ptr", "blk_col_idx", "blk_col_ptr", "blk_row_idx", "blk_csc2csr", "blk_nnz",
            "blk_format")])
        _lib.check("dbs_matrix_export_views", st)
        out["B"] = B
        return out

    RAW_ARRAYS = ("rb_ptr", "blk_desc", "blk_ref", "cb_ptr", "csc_desc", "csc_ref", "payload", "tiles",
                  "rb_rows")

    def export_raw(self, name: str) -> np.ndarray:
        """dbs_matrix_export_raw: one internal array as raw bytes (uint8)."""
        which = self.RAW_ARRAYS.index(name)
        lib = _lib.load()
        nb = ctypes.c_int64(0)
        _lib.check("dbs_matrix_export_raw", lib.dbs_matrix_export_raw(self._h, which, None, 0, ctypes.byref(nb)))
        out = np.zeros(max(nb.value, 1), dtype=np.uint8)
        _lib.check("dbs_matrix_export_raw",
                   lib.dbs_matrix_export_raw(self._h, which, out.ctypes.data, out.nbytes, ctypes.byref(nb)))
        return out[:nb.value]

    def export_csr(self):
        rp = np.empty(self.m + 1, np.int64)
        ci = np.empty(max(self.nnz, 1), np.int32)
        va = np.empty(max(self.nnz, 1), np.float32) if self.valued else None
        _lib.check("dbs_matrix_export_csr", _lib.load().dbs_matrix_export_csr(self._h, _ptr(rp), _ptr(ci), _ptr(va)))
        return rp, ci[:self.nnz], None if va is None else va[:self.nnz]

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.load().dbs_matrix_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Workspace:
    """dbs_workspace_create: per-stream scratch for calls on one matrix."""

    def __init__(self, A: DBMatrix, opts: Optional[dbs_exec_opts] = None, **opt_kw):
        self.A = A
        h = ctypes.c_void_p()
        _lib.check("dbs_workspace_create", _lib.load().dbs_workspace_create(A.handle, ctypes.byref(h)))
        self._h = h
        if opts is not None or opt_kw:
            self.set_opts(opts or exec_opts(**opt_kw))

    @property
    def handle(self):
        return self._h

    def set_opts(self, opts: dbs_exec_opts):
        _lib.check("dbs_workspace_set_opts", _lib.load().dbs_workspace_set_opts(self._h, ctypes.byref(opts)))

    def check(self, stream=None) -> int:
        """dbs_workspace_check: returns the latched device status (and clears it)."""
        return _lib.load().dbs_workspace_check(self._h, _stream_handle(stream))

    def stats(self, stream=None) -> dict:
        s = dbs_stats()
        _lib.check("dbs_last_stats", _lib.load().dbs_last_stats(self._h, _stream_handle(stream), ctypes.byref(s)))
        d = {f: getattr(s, f) for f, _ in s._fields_}
        d["phase_ns"] = list(s.phase_ns)
        return d

    def bfs_levels(self, max_levels: int = 64, stream=None) -> dict:
        """dbs_bfs_level_stats: per-level frontier blocks, push work (matrix
        blocks in the frontier's column blocks), path and device time."""
        fb = np.zeros(max_levels, np.int64)
        pw = np.zeros(max_levels, np.int64)
        pa = np.zeros(max_levels, np.int32)
        ns = np.zeros(max_levels, np.int64)
        tr = np.zeros(max_levels, np.int64)
        _lib.check("dbs_bfs_level_stats", _lib.load().dbs_bfs_level_stats(
            self._h, _stream_handle(stream), max_levels, _ptr(fb), _ptr(pw), _ptr(pa), _ptr(ns), _ptr(tr)))
        n = int((pa > 0).sum())
        return {"frontier_blocks": fb[:n].tolist(), "push_work": pw[:n].tolist(),
                "path": ["push" if p == 1 else "pull" for p in pa[:n]],
                "level_us": (ns[:n] / 1e3).round(2).tolist(), "traversal_us": (tr[:n] / 1e3).round(2).tolist()}

    def selftest_wait_timeout(self, stream=None):
        _lib.check("dbs_selftest_wait_timeout",
                   _lib.load().dbs_selftest_wait_timeout(self._h, _stream_handle(stream)))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.load().dbs_workspace_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dbs_spmspv(A: DBMatrix, x_idx, x_val=None, *, semiring="plus_times", visited=None, path="auto",
               ws: Workspace, y_idx=None, y_val=None, y_nnz=None, stream=None):
    """dbs_spmspv: y = A x for a sparse x given as CUDA tensors (x_idx int32,
    x_val float32 or None).  Returns CUDA tensors (y_idx[:cap], y_val or None,
    y_nnz int64[1]); the first y_nnz entries are valid once the stream gets
    there.  Asynchronous."""
    torch = _torch()
    sr = _semiring(semiring)
    dev = x_idx.device
    if y_idx is None:
        y_idx = torch.empty(max(A.m, 1), dtype=torch.int32, device=dev)
    if sr == PLUS_TIMES and y_val is None:
        y_val = torch.empty(max(A.m, 1), dtype=torch.float32, device=dev)
    if y_nnz is None:
        y_nnz = torch.empty(1, dtype=torch.int64, device=dev)
    st = _lib.load().dbs_spmspv(A.handle, sr, _ptr(x_idx), _ptr(x_val), int(x_idx.numel()), _ptr(visited),
                                _ptr(y_idx), _ptr(y_val) if sr == PLUS_TIMES else None, _ptr(y_nnz),
                                _path(path), ws.handle, _stream_handle(stream))
    _lib.check("dbs_spmspv", st)
    return y_idx, (y_val if sr == PLUS_TIMES else None), y_nnz


def dbs_spmspv_dense(A: DBMatrix, x, *, y=None, path="auto", ws: Workspace, stream=None):
    """dbs_spmspv_dense: dense CUDA float32 x (zeros inactive) -> dense y."""
    torch = _torch()
    if y is None:
        y = torch.empty(max(A.m, 1), dtype=torch.float32, device=x.device)
    st = _lib.load().dbs_spmspv_dense(A.handle, _ptr(x), _ptr(y), _path(path), ws.handle, _stream_handle(stream))
    _lib.check("dbs_spmspv_dense", st)
    return y


def dbs_spmspv_dense_noalloc(A: DBMatrix, x, *, y, stream=None):
    """dbs_spmspv_dense_noalloc: like dbs_spmspv_dense on the pull path, but
    with the scratch in a fixed device array of the library, for callers that
    may not allocate GPU memory after start-up.  `y` must be given
    (float32[m] on the device); nothing is allocated by the call."""
    st = _lib.load().dbs_spmspv_dense_noalloc(A.handle, _ptr(x), _ptr(y), _stream_handle(stream))
    _lib.check("dbs_spmspv_dense_noalloc", st)
    return y


def dbs_spmspv_dense_noalloc_check(stream=None) -> int:
    """dbs_spmspv_dense_noalloc_check: synchronizes the stream and returns the
    status the last allocation-free call latched on the device (0 = OK)."""
    return int(_lib.load().dbs_spmspv_dense_noalloc_check(_stream_handle(stream)))


def dbs_decode_layer(A: DBMatrix, x, tau: float = 0.0, *, y=None, ws: Workspace, stream=None):
    """dbs_decode_layer: y = A x' with x' = x where |x| > tau, else 0 (dense
    CUDA float32 x, 16-byte aligned) -> dense y, pull path, one launch."""
    torch = _torch()
    if y is None:
        y = torch.empty(max(A.m, 1), dtype=torch.float32, device=x.device)
    st = _lib.load().dbs_decode_layer(A.handle, _ptr(x), float(tau), _ptr(y), ws.handle, _stream_handle(stream))
    _lib.check("dbs_decode_layer", st)
    return y


def dbs_bfs(A: DBMatrix, src: int, *, levels=None, path="auto", ws: Workspace, stream=None, sync: bool = True):
    """dbs_bfs: levels (int32 CUDA tensor, -1 unreached) and, with sync, the
    number of levels."""
    torch = _torch()
    if levels is None:
        levels = torch.empty(max(A.n, 1), dtype=torch.int32, device="cuda")
    nl = ctypes.c_int32(-1)
    st = _lib.load().dbs_bfs(A.handle, int(src), _ptr(levels), ctypes.byref(nl) if sync else None,
                             _path(path), ws.handle, _stream_handle(stream))
    _lib.check("dbs_bfs", st)
    return levels, (nl.value if sync else None)


# short names
spmspv = dbs_spmspv
spmspv_dense = dbs_spmspv_dense
decode_layer = dbs_decode_layer
bfs = dbs_bfs


class SpMVPlan:
    """dbs_spmv_plan: adaptive CSR SpMV for dense x.  The CSR arrays (CUDA
    tensors: row_ptr int64[m+1], col_idx int32[nnz], vals float32[nnz]) are
    kept referenced for the plan's lifetime."""

    def __init__(self, m: int, n: int, row_ptr, col_idx, vals, stream=None):
        torch = _torch()
        self._arrays = (row_ptr.to(torch.int64).contiguous(), col_idx.to(torch.int32).contiguous(),
                        vals.to(torch.float32).contiguous())
        rp, ci, va = self._arrays
        self.m, self.n = int(m), int(n)
        h = ctypes.c_void_p()
        st = _lib.load().dbs_spmv_plan_create(self.m, self.n, int(ci.numel()), _ptr(rp), _ptr(ci), _ptr(va),
                                              _stream_handle(stream), ctypes.byref(h))
        _lib.check("dbs_spmv_plan_create", st)
        self._h = h

    @classmethod
    def from_csr(cls, A, device="cuda", **kw) -> "SpMVPlan":
        torch = _torch()
        return cls(A.m, A.n, torch.from_numpy(np.asarray(A.row_ptr, np.int64)).to(device),
                   torch.from_numpy(np.asarray(A.col_idx, np.int32)).to(device),
                   torch.from_numpy(np.asarray(A.vals, np.float32)).to(device), **kw)

    def info(self) -> dict:
        rows = (ctypes.c_int64 * 8)()
        chunks = ctypes.c_int64(0)
        _lib.check("dbs_spmv_plan_info", _lib.load().dbs_spmv_plan_info(self._h, rows, ctypes.byref(chunks)))
        return {"lane_group_rows": {str(1 << b): rows[b] for b in range(6)}, "block_rows": rows[6],
                "split_rows": rows[7], "split_chunks": chunks.value}

    def __call__(self, x, *, y=None, stream=None):
        torch = _torch()
        if y is None:
            y = torch.empty(max(self.m, 1), dtype=torch.float32, device=x.device)
        _lib.check("dbs_spmv", _lib.load().dbs_spmv(self._h, _ptr(x), _ptr(y), _stream_handle(stream)))
        return y

    def close(self):
        if getattr(self, "_h", None):
            _lib.load().dbs_spmv_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def library_path() -> str:
    return _lib.lib_path()


def version() -> str:
    return _lib.load().dbs_version().decode()
