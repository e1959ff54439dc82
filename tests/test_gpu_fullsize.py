"""GPU parity at the workloads' full sizes, through the same API and defaults
the benchmark times.  The oracle is fast enough to check every output entry
(and every BFS level) at these sizes, so nothing is sampled."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import __graft_entry__  # noqa: E402

__graft_entry__.build()
import dynamic_sparsity_spmspv_gb300 as dbs  # noqa: E402
from test_gpu_parity import assert_parity, _t  # noqa: E402

PATHS = ("auto", "push", "pull")


@pytest.fixture(scope="module")
def full():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            A = synth.config(name, "full")
            cache[name] = (A, oracle.Oracle(A), dbs.DBMatrix.from_csr(A))
        return cache[name]
    return get


def test_er_full(full):
    A, O, M = full("er")
    ws = dbs.Workspace(M)
    for i in range(8):
        x = synth.x_uniform(A.n, 41, [43, i])          # 1% of 4096, U[-1, 1]
        for path in PATHS:
            assert_parity(A, O, M, ws, x, path=path)


def test_rmat_full_sweep_and_bfs(full):
    A, O, M = full("rmat")
    ws = dbs.Workspace(M, collect_stats=1)
    expected_path = {1e-4: 1, 1e-3: 1, 1e-2: 1, 1e-1: 2, 5e-1: 2}   # default work rule, 0.45
    for d, p_exp in expected_path.items():
        x = synth.x_uniform(A.n, int(round(d * A.n)), [44, 0, int(d * 1e6), 0], valued=False)
        for path in PATHS:
            assert_parity(A, O, M, ws, x, "or_and", path=path)
            if path == "auto":
                assert ws.stats()["path"] == p_exp, d
    for i, src in enumerate(synth.bfs_sources(A, 16, [44, 7])):
        ref = O.bfs_queue(int(src))
        for path in (PATHS if i < 2 else ("auto",)):
            lev, nl = dbs.bfs(M, int(src), ws=ws, path=path)
            np.testing.assert_array_equal(lev.cpu().numpy(), ref)
            assert nl == int(ref.max()) + 1


def test_fem_full(full):
    A, O, M = full("fem")
    assert A.nnz == 382 ** 3
    ws = dbs.Workspace(M)
    for f in (1e-3, 1e-2, 1e-1):
        x = synth.x_clusters(A.n, f, [45, int(f * 1e4)])
        for path in PATHS:
            assert_parity(A, O, M, ws, x, path=path)


def test_llm_full_dense_and_sparse_x(full):
    A, O, M = full("llm")
    assert A.nnz == 4096 * 5504
    ws = dbs.Workspace(M)
    for t in range(12):
        xd = synth.x_relu_topk(A.n, 1101, [46, t])
        nz = np.nonzero(xd)[0].astype(np.int32)
        x = synth.SparseVec(A.n, nz, xd[nz])
        ri, rv, rs = O.spmspv(x)
        for path in PATHS:
            y = dbs.spmspv_dense(M, _t(xd), ws=ws, path=path).cpu().numpy()
            assert ws.check() == 0
            assert oracle.tolerance_ok(y[ri], rv, rs).all()
            rest = np.ones(A.m, bool)
            rest[ri] = False
            assert (y[rest] == 0).all()
        if t < 3:
            for path in PATHS:
                assert_parity(A, O, M, ws, x, path=path)


def test_grid_hubs_full_bfs(full):
    A, O, M = full("grid")
    ws = dbs.Workspace(M)
    for i, src in enumerate(synth.bfs_sources(A, 8, [47, 7])):
        ref = O.bfs_queue(int(src))
        for path in (PATHS if i == 0 else ("auto",)):
            lev, nl = dbs.bfs(M, int(src), ws=ws, path=path)
            np.testing.assert_array_equal(lev.cpu().numpy(), ref)
            assert nl == int(ref.max()) + 1
    x = synth.x_uniform(A.n, A.n // 1000, [47, 1], valued=False)
    for path in PATHS:
        assert_parity(A, O, M, ws, x, "or_and", path=path)


def test_llm_full_decode_layer(full):
    """The DB-Decoding layer at the workload's full size, with the paper's
    thresholds and with the GB300 decode build (th1 = 31)."""
    A, O, M = full("llm")
    for Mb in (M, dbs.DBMatrix.from_csr(A, th1=31)):
        ws = dbs.Workspace(Mb)
        for t in range(4):
            xa = synth.x_activation(A.n, [90, t, 0])
            y = dbs.decode_layer(Mb, _t(xa), 1.6449, ws=ws).cpu().numpy()
            assert ws.check() == 0
            ref, s, touched = O.decode_layer(xa, 1.6449)
            assert oracle.tolerance_ok(y[touched], ref[touched], s[touched]).all()
            assert (y[~touched] == 0).all()


def test_grid_without_hubs_full_bfs():
    """DB-SpMSpV Section 4.2 (DB-BFS) in the long-diameter regime: the
    4096 x 4096 grid with 10 % of its edges deleted and no hubs, whose BFS
    runs thousands of levels over frontiers of a few thousand vertices.
    Levels are bit-exact against the queue BFS for the benchmark's four
    sources on the auto path and for the first source with every level
    forced to push and to pull; the level count is checked far beyond the
    first 64 levels, whose per-level statistics the device records."""
    A = synth.grid_hubs(4096, 0.10, 0, 0, seed=47)
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    for i, src in enumerate(synth.bfs_sources(A, 4, [48, 7])):
        ref = O.bfs_queue(int(src))
        assert int(ref.max()) + 1 > 1000
        for path in (PATHS if i == 0 else ("auto",)):
            lev, nl = dbs.bfs(M, int(src), ws=ws, path=path)
            assert ws.check() == 0
            np.testing.assert_array_equal(lev.cpu().numpy(), ref, err_msg=f"source {src}, {path}")
            assert nl == int(ref.max()) + 1
