"""The allocation-free entry point (dbs_spmspv_dense_noalloc) against the
allocating one (dbs_spmspv_dense), through the C ABI.

Callers such as real-time serving loops, or hosts that pre-reserve a fixed
GPU memory budget, cannot call cudaMalloc after start-up; this entry point
keeps its scratch in a fixed device array of the library.  The file is named
so that pytest collects it last."""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import __graft_entry__  # noqa: E402

__graft_entry__.build()
import dynamic_sparsity_spmspv_gb300 as dbs  # noqa: E402
from dynamic_sparsity_spmspv_gb300 import _lib  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    A = synth.config("llm", "small")
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    y = torch.empty(A.m, dtype=torch.float32, device="cuda")
    for call, keep in enumerate((A.n // 10, A.n // 3)):            # two calls in a row
        xd = synth.x_relu_topk(A.n, keep, [31, call])
        x = _dev(xd)
        y.fill_(float("nan"))                                      # every row must be written
        dbs.dbs_spmspv_dense_noalloc(M, x, y=y)
        y_na = y.cpu().numpy()
        y_ref = dbs.spmspv_dense(M, x, ws=ws, path="pull").cpu().numpy()
        assert ws.check() == 0
        nz = np.nonzero(xd)[0].astype(np.int32)
        ri, rv, rs = O.spmspv(synth.SparseVec(A.n, nz, xd[nz]))
        S = np.zeros(A.m)
        S[ri] = rs
        # same tolerance the parity tests use: 1e-5 * sum_j |a_ij x_j| + 1e-30
        assert (np.abs(y_na.astype(np.float64) - y_ref) <= 1e-5 * S + 1e-30).all()
        assert oracle.tolerance_ok(y_na[ri], rv, rs).all()


def test_noalloc_rejects_too_many_columns():
    n = (1 << 22) + 16
    A = synth.csr_from_coo(4, n, [0, 1], [3, n - 1], [1.0, 2.0])
    M = dbs.DBMatrix.from_csr(A)
    y = torch.empty(4, dtype=torch.float32, device="cuda")
    with pytest.raises(dbs.DbsError) as e:
        dbs.dbs_spmspv_dense_noalloc(M, torch.zeros(n, device="cuda"), y=y)
    assert e.value.status == 1
    assert "dbs_spmspv_dense_noalloc" in _lib.PROTOTYPES
    assert ctypes.CDLL(_lib.lib_path()).dbs_spmspv_dense_noalloc is not None


def test_noalloc_allocates_nothing_and_reports_its_status():
    """Repeated calls leave the device's free memory unchanged (nothing is
    allocated per call), the status query reports success, and a matrix
    whose row count is not a multiple of 16 has its last rows written."""
    A = synth.random_csr(1003, 517, 0.05, 7)
    M = dbs.DBMatrix.from_csr(A)
    xd = synth.x_relu_topk(A.n, A.n // 4, [32, 0])
    x = _dev(xd)
    y = torch.empty(A.m, dtype=torch.float32, device="cuda")
    dbs.dbs_spmspv_dense_noalloc(M, x, y=y)            # first call on the device: set-up
    assert dbs.dbs_spmspv_dense_noalloc_check() == 0
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        y.fill_(float("nan"))
        dbs.dbs_spmspv_dense_noalloc(M, x, y=y)
        assert dbs.dbs_spmspv_dense_noalloc_check() == 0
    assert torch.cuda.mem_get_info()[0] == free0
    y_na = y.cpu().numpy()
    nz = np.nonzero(xd)[0].astype(np.int32)
    ri, rv, rs = oracle.Oracle(A).spmspv(synth.SparseVec(A.n, nz, xd[nz]))
    assert oracle.tolerance_ok(y_na[ri], rv, rs).all()
    rest = np.ones(A.m, bool)
    rest[ri] = False
    assert (y_na[rest] == 0).all()
