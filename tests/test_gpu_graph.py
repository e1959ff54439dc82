"""Calls captured once in a CUDA graph and replayed with new inputs: every
launch keeps its grid-barrier state, counter slot and compaction tags on the
device, so replays need no host bookkeeping.  Each replay is checked against
the oracle like a direct call."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import __graft_entry__  # noqa: E402

__graft_entry__.build()
import dynamic_sparsity_spmspv_gb300 as dbs  # noqa: E402

DEV = "cuda"


def _check_sparse(O, x, sr, gi, gv):
    ri, rv, rs = O.spmspv(x, sr)
    np.testing.assert_array_equal(gi, ri)
    if sr == oracle.PLUS_TIMES:
        assert oracle.tolerance_ok(gv, rv, rs).all()


@pytest.mark.parametrize("path", ["auto", "push", "pull"])
def test_graph_replay_sparse_dense_bfs(path):
    A = synth.random_csr(3000, 3000, 0.004, 71)
    Ab = synth.random_csr(3000, 3000, 0.004, 72, valued=False)
    Ab = synth.csr_from_coo(3000, 3000, np.concatenate([np.repeat(np.arange(3000), np.diff(Ab.row_ptr)), Ab.col_idx]),
                            np.concatenate([Ab.col_idx, np.repeat(np.arange(3000), np.diff(Ab.row_ptr))]),
                            dedupe=True)   # symmetric pattern for BFS
    O, Ob = oracle.Oracle(A), oracle.Oracle(Ab)
    M, Mb = dbs.DBMatrix.from_csr(A), dbs.DBMatrix.from_csr(Ab)
    ws, wsb = dbs.Workspace(M), dbs.Workspace(Mb)
    k = 40
    x_idx = torch.zeros(k, dtype=torch.int32, device=DEV)
    x_val = torch.zeros(k, dtype=torch.float32, device=DEV)
    xd = torch.zeros(A.n, dtype=torch.float32, device=DEV)
    yi = torch.empty(A.m, dtype=torch.int32, device=DEV)
    yv = torch.empty(A.m, dtype=torch.float32, device=DEV)
    yn = torch.empty(1, dtype=torch.int64, device=DEV)
    bi = torch.empty(Ab.m, dtype=torch.int32, device=DEV)
    bn = torch.empty(1, dtype=torch.int64, device=DEV)
    yd = torch.empty(A.m, dtype=torch.float32, device=DEV)
    lev = torch.empty(Ab.n, dtype=torch.int32, device=DEV)
    src = torch.zeros(1, dtype=torch.int64)

    def load(i):
        x = synth.x_uniform(A.n, k, [73, i])
        x_idx.copy_(torch.from_numpy(x.idx))
        x_val.copy_(torch.from_numpy(x.val))
        dense = np.zeros(A.n, np.float32)
        dense[x.idx] = x.val
        xd.copy_(torch.from_numpy(dense))
        return x

    def step():
        dbs.spmspv(M, x_idx, x_val, ws=ws, y_idx=yi, y_val=yv, y_nnz=yn, path=path)
        dbs.spmspv(Mb, x_idx, None, semiring="or_and", ws=wsb, y_idx=bi, y_nnz=bn, path=path)
        dbs.spmspv_dense(M, xd, y=yd, ws=ws, path=path)
        dbs.bfs(Mb, 5, levels=lev, ws=wsb, path=path, sync=False)

    load(0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    bfs_ref = Ob.bfs_queue(5)
    for i in range(1, 6):
        x = load(i)
        g.replay()
        if i == 3:
            step()                               # direct calls between replays
        torch.cuda.synchronize()
        assert ws.check() == 0 and wsb.check() == 0
        n = int(yn.item())
        _check_sparse(O, x, oracle.PLUS_TIMES, yi[:n].cpu().numpy(), yv[:n].cpu().numpy())
        nb = int(bn.item())
        xb = synth.SparseVec(x.n, x.idx, None)
        _check_sparse(Ob, xb, oracle.OR_AND, bi[:nb].cpu().numpy(), None)
        ri, rv, rs = O.spmspv(x)
        y = yd.cpu().numpy()
        assert oracle.tolerance_ok(y[ri], rv, rs).all()
        rest = np.ones(A.m, bool)
        rest[ri] = False
        assert (y[rest] == 0).all()
        np.testing.assert_array_equal(lev.cpu().numpy(), bfs_ref)
