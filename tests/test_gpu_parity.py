"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element.  Index, Boolean and BFS results must be bit-exact; fp32 values
must satisfy |y_gpu - y_ref| <= 1e-5 * sum_j |a_ij x_j| + 1e-30."""
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
PATHS = ("auto", "push", "pull")


def _t(a, dtype=None):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_spmspv(M, ws, x, semiring="plus_times", visited=None, path="auto"):
    yi, yv, yn = dbs.spmspv(M, _t(x.idx), _t(x.val), semiring=semiring, visited=visited, path=path, ws=ws)
    k = int(yn.item())
    assert ws.check() == 0
    return yi[:k].cpu().numpy(), None if yv is None else yv[:k].cpu().numpy()


def assert_parity(A, O, M, ws, x, semiring="plus_times", visited_rows=None, path="auto"):
    sr = oracle.PLUS_TIMES if semiring == "plus_times" else oracle.OR_AND
    vis_dev = None
    if visited_rows is not None:
        nbr = (A.m + 15) // 16
        words = np.zeros(nbr + (nbr & 1), np.uint16)
        r = np.nonzero(visited_rows)[0]
        np.bitwise_or.at(words, r // 16, (1 << (r % 16)).astype(np.uint16))
        vis_dev = _t(words.view(np.int16))
    gi, gv = run_spmspv(M, ws, x, semiring, vis_dev, path)
    ri, rv, rs = O.spmspv(x, sr, None if visited_rows is None else visited_rows.astype(np.uint8))
    np.testing.assert_array_equal(gi, ri, err_msg=f"pattern ({path})")
    if sr == oracle.PLUS_TIMES:
        ok = oracle.tolerance_ok(gv, rv, rs)
        assert ok.all(), f"{(~ok).sum()} values out of tolerance ({path}); first {np.nonzero(~ok)[0][:5]}"
    return gi, gv


@pytest.fixture(scope="module")
def small():
    out = {}
    for name in synth.CONFIG_NAMES:
        A = synth.config(name, "small")
        out[name] = (A, oracle.Oracle(A), dbs.DBMatrix.from_csr(A))
    return out


def _xs(A, valued, seed):
    n = A.n
    ks = [0, 1, 3, max(1, n // 1000), max(1, n // 100), n // 10, n // 2, n]
    return [synth.x_uniform(n, k, [seed, i], valued=valued) for i, k in enumerate(ks)]


@pytest.mark.parametrize("name", ["er", "fem", "llm"])
@pytest.mark.parametrize("path", PATHS)
def test_plus_times_small(small, name, path):
    A, O, M = small[name]
    ws = dbs.Workspace(M)
    for x in _xs(A, True, 1):
        assert_parity(A, O, M, ws, x, path=path)


@pytest.mark.parametrize("name", synth.CONFIG_NAMES)
@pytest.mark.parametrize("path", PATHS)
def test_boolean_small(small, name, path):
    A, O, M = small[name]
    ws = dbs.Workspace(M)
    rng = np.random.default_rng(3)
    for i, x in enumerate(_xs(A, False, 2)):
        vis = (rng.random(A.m) < 0.3) if i % 2 else None
        assert_parity(A, O, M, ws, x, "or_and", vis, path)


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("name", ["fem", "llm", "er"])
def test_forced_formats(name, fmt):
    A = synth.config(name, "small")
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A, force_format=fmt)
    assert M.info()["blocks_by_format"][fmt] == M.info()["nblocks"]
    ws = dbs.Workspace(M)
    for lp in (0, 8, 17):
        ws.set_opts(dbs.exec_opts(local_pull_min=lp))
        for path in PATHS:
            for x in _xs(A, True, 5)[1:6]:
                assert_parity(A, O, M, ws, x, path=path)
                assert_parity(A, O, M, ws, synth.SparseVec(x.n, x.idx, None), "or_and", path=path)


def _block_diag(pattern, copies, seed):
    """`copies` copies of a 16x16 pattern on the diagonal, distinct values."""
    rng = np.random.default_rng(seed)
    pr, pc = np.nonzero(pattern)
    k = np.arange(copies, dtype=np.int64)
    rows = (k[:, None] * 16 + pr[None, :]).ravel()
    cols = (k[:, None] * 16 + pc[None, :]).ravel()
    vals = rng.uniform(-1, 1, rows.shape[0]).astype(np.float32)
    return synth.csr_from_coo(copies * 16, copies * 16, rows, cols, vals)


@pytest.mark.parametrize("density", [0.15, 0.45, 0.75])
@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
def test_exhaustive_block_masks(fmt, density):
    """Every one of the 2^16 vector-block masks against one block pattern:
    copy k of the block on the diagonal meets x-block mask k."""
    rng = np.random.default_rng(int(density * 100) + fmt)
    pattern = rng.random((16, 16)) < density
    pattern[rng.integers(0, 16), :] |= density > 0.4          # a heavier row
    A = _block_diag(pattern, 1 << 16, fmt)
    k = np.arange(1 << 16)
    bits = ((k[:, None] >> np.arange(16)[None, :]) & 1).astype(bool)
    idx = (k[:, None] * 16 + np.arange(16)[None, :])[bits].astype(np.int32)
    val = rng.uniform(-1, 1, idx.shape[0]).astype(np.float32)
    x = synth.SparseVec(A.n, idx, val)
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A, force_format=fmt)
    ws = dbs.Workspace(M)
    for lp in (0, 8, 17):
        ws.set_opts(dbs.exec_opts(local_pull_min=lp))
        for path in ("push", "pull"):
            assert_parity(A, O, M, ws, x, path=path)
    assert_parity(A, O, M, ws, synth.SparseVec(A.n, idx, None), "or_and", path="pull")
    assert_parity(A, O, M, ws, synth.SparseVec(A.n, idx, None), "or_and", path="push")


@pytest.mark.parametrize("fmt", [-1, 0, 1, 2, 3, 4])
def test_integer_values_bit_exact(fmt):
    A = synth.random_csr(700, 650, 0.08, 9, integer_values=True)
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A, force_format=fmt)
    ws = dbs.Workspace(M)
    for path in PATHS:
        for kx in (5, 60, 650):
            x = synth.x_uniform(A.n, kx, [kx, 1], integer_values=True)
            gi, gv = run_spmspv(M, ws, x, path=path)
            ri, rv, _ = O.spmspv(x)
            np.testing.assert_array_equal(gi, ri)
            np.testing.assert_array_equal(gv.astype(np.float64), rv)


def test_single_contributor_rows_bit_exact():
    A = synth.config("er", "small")
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    for j in (0, 17, 999):
        x = synth.SparseVec(A.n, np.array([j], np.int32), np.array([0.3], np.float32))
        for path in PATHS:
            gi, gv = run_spmspv(M, ws, x, path=path)
            ri, rv, _ = O.spmspv(x)
            np.testing.assert_array_equal(gi, ri)
            np.testing.assert_array_equal(gv, rv.astype(np.float32))   # one product, rounded once


def test_activity_and_special_vectors(small):
    A, O, M = small["er"]
    ws = dbs.Workspace(M)
    for path in PATHS:
        empty = synth.SparseVec(A.n, np.zeros(0, np.int32), np.zeros(0, np.float32))
        gi, _ = run_spmspv(M, ws, empty, path=path)
        assert gi.size == 0
        z = synth.SparseVec(A.n, np.array([1, 2, 3], np.int32), np.array([0.0, -0.0, 0.0], np.float32))
        gi, _ = run_spmspv(M, ws, z, path=path)
        assert gi.size == 0
        nanx = synth.SparseVec(A.n, np.array([5], np.int32), np.array([np.nan], np.float32))
        gi, gv = run_spmspv(M, ws, nanx, path=path)
        ri, _, _ = O.spmspv(nanx)
        np.testing.assert_array_equal(gi, ri)
        assert np.isnan(gv).all()
        allx = synth.x_uniform(A.n, A.n, 4)
        assert_parity(A, O, M, ws, allx, path=path)


def test_permutation_and_identity():
    n = 1000
    rng = np.random.default_rng(1)
    perm = rng.permutation(n)
    vals = rng.uniform(0.5, 2.0, n).astype(np.float32)
    A = synth.csr_from_coo(n, n, perm, np.arange(n), vals)
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    x = synth.x_uniform(n, 300, 2)
    for path in PATHS:
        gi, gv = run_spmspv(M, ws, x, path=path)
        inv = np.empty(n, np.int64)
        inv[perm] = np.arange(n)
        exp_i = np.sort(perm[x.idx])
        np.testing.assert_array_equal(gi, exp_i)
        j = inv[gi]
        xd = np.zeros(n, np.float32)
        xd[x.idx] = x.val
        np.testing.assert_array_equal(gv, (vals[j] * xd[j]).astype(np.float32))


@pytest.mark.parametrize("th3,switch", [(0.01, 64), (0.1, 640)])
def test_selector_boundary(th3, switch):
    # nbc = 6400 column blocks: push iff N_nzblk / 6400 < th3 (the paper's 0.01
    # switches at 64 nonzero blocks, the GB300 default 0.1 at 640)
    n = 6400 * 16
    A = synth.random_csr(64, n, 0.002, 3)
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M, collect_stats=1, th3=th3, push_work_frac=0.0)     # the paper's rule
    O = oracle.Oracle(A)
    for nzb, expect in ((switch - 1, 1), (switch, 2), (switch + 1, 2), (1, 1)):
        blocks = np.arange(nzb) * (6400 // (switch + 2))           # all < 6400 column blocks
        assert len(np.unique(blocks)) == nzb and blocks.max() * 16 + 3 < n
        x = synth.SparseVec(n, (blocks * 16 + 3).astype(np.int32), np.ones(nzb, np.float32))
        assert_parity(A, O, M, ws, x)
        st = ws.stats()
        assert st["n_nzblk"] == nzb and st["path"] == expect, (nzb, st)


def test_work_based_selector():
    # push iff the blocks of the active column blocks < push_work_frac * B
    A = synth.config("fem", "small")
    M = dbs.DBMatrix.from_csr(A)
    O = oracle.Oracle(A)
    V = oracle.block_views(A)
    deg = np.diff(V["blk_col_ptr"])
    B = V["B"]
    ws = dbs.Workspace(M, collect_stats=1, push_work_frac=0.1)
    for k in (1, 3, 10, 40, 200, 1000):
        x = synth.x_uniform(A.n, k, [k, 5])
        act = np.unique(x.idx // 16)
        expect = 1 if deg[act].sum() < 0.1 * B else 2
        assert_parity(A, O, M, ws, x)
        assert ws.stats()["path"] == expect, (k, deg[act].sum(), B)


def test_stats_count_touched_nnz(small):
    A, O, M = small["fem"]
    ws = dbs.Workspace(M, collect_stats=1)
    V = oracle.block_views(A)
    for path in ("push", "pull"):
        x = synth.x_clusters(A.n, 0.05, 7)
        assert_parity(A, O, M, ws, x, path=path)
        st = ws.stats()
        active_cb = np.zeros(V["blk_col_ptr"].shape[0] - 1, bool)
        active_cb[x.idx // 16] = True
        vis = active_cb[V["blk_col_idx"]]
        assert st["visited_blocks"] == int(vis.sum())
        assert st["touched_nnz"] == int(V["blk_nnz"][vis].sum())
        assert st["x_active"] == x.k
        assert st["bytes_alg"] > 0


def test_workspace_reuse_alternating_paths(small):
    A, O, M = small["llm"]
    ws = dbs.Workspace(M)
    for i in range(12):
        x = synth.x_uniform(A.n, [3, 700, 40, 70][i % 4], [i, 9])
        assert_parity(A, O, M, ws, x, path=PATHS[i % 3])


def test_mixed_call_sequence_on_one_workspace():
    """Dense-x, sparse-x, Boolean and BFS calls interleaved on one workspace:
    each call must leave the scratch as the next one expects."""
    A = synth.random_csr(900, 900, 0.01, 21)
    A = synth.csr_from_coo(900, 900, *[np.r_[a, b] for a, b in zip(
        (np.repeat(np.arange(900), np.diff(A.row_ptr)), A.col_idx, A.vals),
        (A.col_idx, np.repeat(np.arange(900), np.diff(A.row_ptr)), A.vals))], dedupe=True)
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    ops = ["dense", "sparse", "dense", "dense", "bool", "bfs", "sparse", "dense", "bfs", "dense",
           "sparse", "sparse", "bool", "dense", "bfs", "bfs", "sparse"]
    for i, op in enumerate(ops):
        path = PATHS[i % 3]
        if op == "dense":
            xd = synth.x_relu_topk(A.n, [5, 90, 400][i % 3], [i, 77])
            nz = np.nonzero(xd)[0].astype(np.int32)
            ri, rv, rs = O.spmspv(synth.SparseVec(A.n, nz, xd[nz]))
            y = dbs.spmspv_dense(M, _t(xd), ws=ws, path=path).cpu().numpy()
            assert oracle.tolerance_ok(y[ri], rv, rs).all(), (i, op)
        elif op == "sparse":
            assert_parity(A, O, M, ws, synth.x_uniform(A.n, [3, 50, 600][i % 3], [i, 78]), path=path)
        elif op == "bool":
            x = synth.x_uniform(A.n, [7, 200, 30][i % 3], [i, 79], valued=False)
            assert_parity(A, O, M, ws, x, "or_and", path=path)
        else:
            lev, nl = dbs.bfs(M, i * 37 % A.n, ws=ws, path=path)
            np.testing.assert_array_equal(lev.cpu().numpy(), O.bfs_queue(i * 37 % A.n))
        assert ws.check() == 0


@pytest.mark.parametrize("name", ["llm", "er", "fem"])
def test_dense_x_form(small, name):
    A, O, M = small[name]
    ws = dbs.Workspace(M)
    for i, keep in enumerate((0, 1, A.n // 100 + 1, A.n // 10, A.n)):
        xd = synth.x_relu_topk(A.n, keep, [i, 3])
        nz = np.nonzero(xd)[0].astype(np.int32)
        ri, rv, rs = O.spmspv(synth.SparseVec(A.n, nz, xd[nz]))
        for path in PATHS:
            y = dbs.spmspv_dense(M, _t(xd), ws=ws, path=path).cpu().numpy()
            assert ws.check() == 0
            assert oracle.tolerance_ok(y[ri], rv, rs).all()
            rest = np.ones(A.m, bool)
            rest[ri] = False
            assert (y[rest] == 0).all()


@pytest.mark.parametrize("name", ["rmat", "grid", "fem", "er"])
@pytest.mark.parametrize("path", PATHS)
def test_bfs_small(small, name, path):
    A, O, M = small[name]
    ws = dbs.Workspace(M)
    for src in synth.bfs_sources(A, 4, [5, 1]):
        lev, nl = dbs.bfs(M, int(src), ws=ws, path=path)
        ref = O.bfs_queue(int(src))
        np.testing.assert_array_equal(lev.cpu().numpy(), ref)
        assert nl == int(ref.max()) + 1


def test_bfs_level_stats_match_frontiers(small):
    A, O, M = small["rmat"]
    ws = dbs.Workspace(M)
    src = int(synth.bfs_sources(A, 1, [9, 9])[0])
    lev, nl = dbs.bfs(M, src, ws=ws)
    st = ws.bfs_levels()
    ref = O.bfs_queue(src)
    assert len(st["frontier_blocks"]) == nl
    deg = np.diff(oracle.block_views(A)["blk_col_ptr"])      # blocks per column block
    for l in range(nl):
        cbs = np.unique(np.nonzero(ref == l)[0] // 16)
        assert st["frontier_blocks"][l] == len(cbs)
        assert st["push_work"][l] == int(deg[cbs].sum())
        assert st["path"][l] in ("push", "pull")
        assert 0 <= st["traversal_us"][l] <= st["level_us"][l]


def test_bfs_grid_closed_form():
    side = 61
    r, c = np.meshgrid(np.arange(side), np.arange(side - 1), indexing="ij")
    h = (r * side + c).ravel()
    v = (c * side + r).ravel()
    u = np.concatenate([h, v])
    w = np.concatenate([h + 1, v + side])
    A = synth.csr_from_coo(side * side, side * side, np.r_[u, w], np.r_[w, u])
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    rr, cc = np.divmod(np.arange(side * side), side)
    for src in (0, 30 * side + 30, side * side - 1):
        for path in PATHS:
            lev, nl = dbs.bfs(M, src, ws=ws, path=path)
            sr, sc = divmod(src, side)
            np.testing.assert_array_equal(lev.cpu().numpy(), np.abs(rr - sr) + np.abs(cc - sc))


def test_bfs_isolated_source_and_directed():
    A = synth.csr_from_coo(40, 40, [1, 2, 3], [0, 1, 2])     # chain 0 -> 1 -> 2 -> 3
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    O = oracle.Oracle(A)
    for src in (0, 2, 39):
        for path in PATHS:
            lev, nl = dbs.bfs(M, src, ws=ws, path=path)
            np.testing.assert_array_equal(lev.cpu().numpy(), O.bfs_queue(src))


def test_wait_timeout_is_reported_and_recovers(small):
    A, O, M = small["er"]
    ws = dbs.Workspace(M, wait_timeout_ns=50_000_000)
    ws.selftest_wait_timeout()
    assert ws.check() == 4                          # DBS_ERR_TIMEOUT, then cleared
    assert ws.check() == 0
    assert_parity(A, O, M, ws, synth.x_uniform(A.n, 30, 1))


def test_out_of_range_x_index_is_reported(small):
    """The kernel bounds-checks every listed index: an index >= n is skipped
    and latched as DBS_ERR_INVALID_ARG instead of being read."""
    A, O, M = small["er"]
    ws = dbs.Workspace(M)
    for sr, val in (("plus_times", np.array([1.0, 2.0], np.float32)), ("or_and", None)):
        dbs.spmspv(M, _t(np.array([3, A.n + 5], np.int32)), _t(val), semiring=sr, ws=ws)
        assert ws.check() == 1
        assert_parity(A, O, M, ws, synth.x_uniform(A.n, 20, 3))     # workspace usable again


def test_error_returns(small):
    A, O, M = small["rmat"]                          # pattern only
    ws = dbs.Workspace(M)
    xi = _t(np.array([1, 2], np.int32))
    with pytest.raises(dbs.DbsError) as e:
        dbs.spmspv(M, xi, _t(np.ones(2, np.float32)), ws=ws)
    assert e.value.status == 5                       # plus-times needs values
    with pytest.raises(dbs.DbsError) as e:
        dbs.spmspv(M, xi, None, semiring="or_and", path=7, ws=ws)
    assert e.value.status == 1
    B, _, MB = small["er"]
    with pytest.raises(dbs.DbsError):
        dbs.spmspv(MB, xi, None, semiring="or_and", ws=ws)   # workspace of another matrix
    with pytest.raises(dbs.DbsError):
        dbs.bfs(dbs.DBMatrix.from_csr(synth.config("llm", "small")), 0,
                ws=dbs.Workspace(dbs.DBMatrix.from_csr(synth.config("llm", "small"))))


def test_device_inputs_build_same_matrix(small):
    A, O, M = small["fem"]
    Md = dbs.DBMatrix(A.m, A.n, _t(A.row_ptr), _t(A.col_idx), _t(A.vals))
    Vh, Vd = M.export_views(), Md.export_views()
    for k in Vh:
        np.testing.assert_array_equal(Vh[k], Vd[k])
    rp, ci, va = Md.export_csr()
    np.testing.assert_array_equal(ci, A.col_idx)
    np.testing.assert_array_equal(va, A.vals)


def test_ragged_tiny_shapes():
    for m, n in [(1, 1), (1, 40), (40, 1), (17, 33), (16, 16), (15, 17)]:
        A = synth.random_csr(m, n, 0.5, m * 100 + n)
        O = oracle.Oracle(A)
        M = dbs.DBMatrix.from_csr(A)
        ws = dbs.Workspace(M)
        for path in PATHS:
            for k in (0, 1, n):
                assert_parity(A, O, M, ws, synth.x_uniform(n, k, [m, n, k]), path=path)
    E = synth.csr_from_coo(50, 50, [], [], [])
    ME = dbs.DBMatrix.from_csr(E)
    wsE = dbs.Workspace(ME)
    gi, gv = run_spmspv(ME, wsE, synth.x_uniform(50, 10, 1))
    assert gi.size == 0


@pytest.mark.parametrize("W,R", [(16, 1), (40, 3), (256, 32)])
def test_tile_shapes_do_not_change_results(W, R):
    A = synth.config("llm", "small")
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A, tile_weight=W, tile_max_row_blocks=R)
    ws = dbs.Workspace(M)
    for x in _xs(A, True, 8)[2:]:
        assert_parity(A, O, M, ws, x, path="pull")


@pytest.mark.parametrize("path", ["push", "pull"])
def test_pinned_host_vectors_in_place(small, path):
    # x read from and y written to pinned host memory by the kernels
    A, O, M = small["fem"]
    ws = dbs.Workspace(M)
    x = synth.x_clusters(A.n, 0.05, [91, 1])
    xi = torch.from_numpy(x.idx).pin_memory()
    xv = torch.from_numpy(x.val).pin_memory()
    yi = torch.empty(A.m, dtype=torch.int32).pin_memory()
    yv = torch.empty(A.m, dtype=torch.float32).pin_memory()
    yn = torch.empty(1, dtype=torch.int64).pin_memory()
    dbs.spmspv(M, xi, xv, ws=ws, path=path, y_idx=yi, y_val=yv, y_nnz=yn)
    torch.cuda.synchronize()
    assert ws.check() == 0
    k = int(yn.item())
    ri, rv, rs = O.spmspv(x)
    np.testing.assert_array_equal(yi[:k].numpy(), ri)
    assert oracle.tolerance_ok(yv[:k].numpy(), rv, rs).all()
    Ab, Ob, Mb = small["rmat"]
    wb = dbs.Workspace(Mb)
    xb = synth.x_uniform(Ab.n, Ab.n // 20, [91, 2], valued=False)
    xbi = torch.from_numpy(xb.idx).pin_memory()
    ybi = torch.empty(Ab.m, dtype=torch.int32).pin_memory()
    dbs.spmspv(Mb, xbi, None, semiring="or_and", ws=wb, path=path, y_idx=ybi, y_nnz=yn)
    torch.cuda.synchronize()
    assert wb.check() == 0
    ri, _, _ = Ob.spmspv(xb, oracle.OR_AND)
    np.testing.assert_array_equal(ybi[:int(yn.item())].numpy(), ri)
