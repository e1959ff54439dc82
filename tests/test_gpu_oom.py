"""Allocation failures injected on the host side, through the library's
test hook (dbs_debug_fail_alloc): every allocation of dbs_matrix_build_csr
(host inputs, and device inputs with device conversion),
dbs_workspace_create and dbs_spmv_plan_create is made to fail in turn.  Each
call must return DBS_ERR_OOM, and the device's free memory afterwards must
equal its free memory before (nothing leaked).  No GPU fault is involved:
the failing cudaMalloc is never issued."""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import __graft_entry__  # noqa: E402

__graft_entry__.build()
import dynamic_sparsity_spmspv_gb300 as dbs  # noqa: E402
from dynamic_sparsity_spmspv_gb300 import _lib  # noqa: E402

# cudaMemGetInfo moves in whole pages of the driver's sub-allocator: a leak of
# any of the buffers swept here (megabytes each) is far above this slack
SLACK = 2 << 20


def _fail_alloc(k):
    prev = ctypes.c_int64(0)
    assert _lib.load().dbs_debug_fail_alloc(k, ctypes.byref(prev)) == 0
    return prev.value


def _free():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _sweep(make, close, max_k=120):
    close(make())                      # module loading and first-use costs
    base = _free()
    fired = 0
    for k in range(max_k):
        _fail_alloc(k)
        try:
            obj = make()
        except dbs.DbsError as e:
            assert e.status == 2, e                   # DBS_ERR_OOM
            assert _fail_alloc(-1) == -1               # the hook fired
            assert abs(_free() - base) <= SLACK, f"leak after failure {k}"
            fired += 1
            continue
        assert _fail_alloc(-1) >= 0                    # ran past every allocation
        close(obj)
        assert abs(_free() - base) <= SLACK
        return fired
    raise AssertionError("never got past the injected failures")


def test_matrix_build_workspace_and_plan_release_everything_on_oom():
    A = synth.config("llm", "full")
    rp = torch.from_numpy(np.asarray(A.row_ptr, np.int64)).cuda()
    ci = torch.from_numpy(np.asarray(A.col_idx, np.int32)).cuda()
    va = torch.from_numpy(np.asarray(A.vals, np.float32)).cuda()
    n_host = _sweep(lambda: dbs.DBMatrix.from_csr(A, num_threads=4), lambda M: M.close())
    n_dev = _sweep(lambda: dbs.DBMatrix(A.m, A.n, rp, ci, va, device_convert=1), lambda M: M.close())
    n_plan = _sweep(lambda: dbs.SpMVPlan(A.m, A.n, rp, ci, va), lambda p: p.close())
    assert n_host >= 10 and n_dev >= 10 and n_plan >= 8
    G = synth.config("rmat", "full")
    MG = dbs.DBMatrix.from_csr(G)
    n_ws = _sweep(lambda: dbs.Workspace(MG), lambda w: w.close())
    assert n_ws >= 10
    # and the library works normally afterwards
    ws = dbs.Workspace(MG)
    lev, nl = dbs.bfs(MG, int(synth.bfs_sources(G, 1, [3, 3])[0]), ws=ws)
    assert nl > 1 and ws.check() == 0
