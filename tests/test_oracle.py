"""Pins for the CPU oracle, checked against facts that do not come from the
oracle itself: numpy dense brute force, scipy's sparse SpMV and BFS distances,
closed forms (unit vectors, permutations, grid Manhattan distance), integer
exactness, and the views printed in Figure 5 of the DB-SpMSpV paper."""
import numpy as np
import pytest
import scipy.sparse as sp
import scipy.sparse.csgraph as csgraph

import oracle
import synth
from conftest import read_golden


def _brute(A, x, semiring, visited=None):
    """Dense brute force: pattern via boolean matrix algebra, values via fp64 matmul."""
    D = synth.csr_to_dense(A)
    P = np.zeros((A.m, A.n), dtype=bool)
    rows = np.repeat(np.arange(A.m), np.diff(A.row_ptr))
    P[rows, A.col_idx] = True
    active = np.zeros(A.n, dtype=bool)
    xd = np.zeros(A.n)
    if x.val is None:
        active[x.idx] = True
        xd[x.idx] = 1.0
    else:
        nz = x.val != 0
        active[x.idx[nz]] = True
        xd[x.idx[nz]] = x.val[nz].astype(np.float64)
    touched = (P & active[None, :]).any(axis=1)
    if semiring == oracle.OR_AND and visited is not None:
        touched &= ~visited.astype(bool)
    idx = np.nonzero(touched)[0]
    vals = (D[:, active] @ xd[active])[idx]
    absd = (np.abs(D[:, active]) @ np.abs(xd[active]))[idx]
    return idx, vals, absd


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("semiring", [oracle.PLUS_TIMES, oracle.OR_AND])
def test_push_matches_dense_brute_force(seed, semiring):
    rng = np.random.default_rng(seed)
    m, n = int(rng.integers(1, 70)), int(rng.integers(1, 70))
    A = synth.random_csr(m, n, float(rng.uniform(0.02, 0.5)), seed, valued=bool(seed % 3))
    x = synth.x_uniform(n, int(rng.integers(0, n + 1)), [seed, 7], valued=bool(seed % 2))
    vis = (rng.random(m) < 0.3).astype(np.uint8) if semiring == oracle.OR_AND else None
    O = oracle.Oracle(A)
    yi, yv, ya = O.spmspv(x, semiring, vis)
    bi, bv, ba = _brute(A, x, semiring, vis)
    np.testing.assert_array_equal(yi, bi)
    if semiring == oracle.PLUS_TIMES:
        np.testing.assert_allclose(yv, bv, rtol=0, atol=1e-12 * (1 + ba.max(initial=0)))
        np.testing.assert_allclose(ya, ba, rtol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_integer_values_are_exact(seed):
    A = synth.random_csr(90, 75, 0.2, seed, integer_values=True)
    x = synth.x_uniform(75, 30, [seed, 1], integer_values=True)
    yi, yv, _ = oracle.Oracle(A).spmspv(x)
    bi, bv, _ = _brute(A, x, oracle.PLUS_TIMES)
    np.testing.assert_array_equal(yi, bi)
    np.testing.assert_array_equal(yv, bv)          # small integers: exact in any order


def test_activation_mask_rule():
    """Magnitude thresholding (DB-Decoding, Sections 4.3 and 5): keep x_j
    iff |x_j| > tau.  Worked by hand: entries equal to +-tau are dropped,
    NaN is kept (it is not <= tau), +-0 never survive."""
    x = np.array([0.0, -0.0, 2.0, -2.0, 0.5, np.nan, np.inf, -1.0, 1.0, 1.0000001], np.float32)
    np.testing.assert_array_equal(oracle.activation_mask(x, 1.0), [2, 3, 5, 6, 9])
    np.testing.assert_array_equal(oracle.activation_mask(x, 0.0), [2, 3, 4, 5, 6, 7, 8, 9])
    np.testing.assert_array_equal(oracle.activation_mask(x, np.inf), [5])
    assert oracle.activation_mask(np.zeros(0, np.float32), 0.5).shape == (0,)


@pytest.mark.parametrize("seed", range(6))
def test_decode_layer_matches_dense_brute_force(seed):
    """y = A x' against a dense fp64 matvec of the thresholded activation,
    with several entries exactly at +-tau."""
    rng = np.random.default_rng(seed + 100)
    m = n = int(rng.integers(1, 60))      # square: a transposed-index mutant stays in bounds
    A = synth.random_csr(m, n, float(rng.uniform(0.05, 0.6)), seed + 100)
    tau = 0.5
    x = rng.standard_normal(n).astype(np.float32)
    x[rng.random(n) < 0.2] = np.float32(tau) * rng.choice([-1, 1])
    y, s, t = oracle.Oracle(A).decode_layer(x, tau)
    xp = np.where(np.abs(x.astype(np.float64)) > tau, x.astype(np.float64), 0.0)
    D = synth.csr_to_dense(A)
    np.testing.assert_allclose(y, D @ xp, rtol=0, atol=1e-12 * (1 + np.abs(D) @ np.abs(xp)).max())
    np.testing.assert_allclose(s, np.abs(D) @ np.abs(xp), rtol=1e-12)
    np.testing.assert_array_equal(t, (D != 0).astype(np.int64) @ (xp != 0).astype(np.int64) > 0)


@pytest.mark.parametrize("seed", range(6))
def test_spmv_csr_matches_dense_brute_force(seed):
    """Dense-input SpMV: every stored entry times x as given (zeros and
    negative entries included) against a dense fp64 matvec."""
    rng = np.random.default_rng(seed + 200)
    m = n = int(rng.integers(1, 70))         # square: an index mix-up mutant stays in bounds
    A = synth.random_csr(m, n, float(rng.uniform(0.02, 0.7)), seed + 200)
    x = rng.standard_normal(n).astype(np.float32)
    x[rng.random(n) < 0.3] = 0.0
    y, s = oracle.spmv_csr(A, x)
    D = synth.csr_to_dense(A)
    np.testing.assert_allclose(y, D @ x.astype(np.float64), rtol=0, atol=1e-12 * (1 + (np.abs(D) @ np.abs(x)).max()))
    np.testing.assert_allclose(s, np.abs(D) @ np.abs(x.astype(np.float64)), rtol=1e-12)


def test_spmv_csr_equals_spmspv_on_a_full_x():
    """With no zero in x, SpMV and SpMSpV with every index active agree on
    every row that holds an entry; rows without entries give 0."""
    A = synth.random_csr(50, 40, 0.2, 7)
    x = np.random.default_rng(8).uniform(0.5, 1.5, 40).astype(np.float32)
    y, _ = oracle.spmv_csr(A, x)
    ri, rv, _ = oracle.Oracle(A).spmspv(synth.SparseVec(40, np.arange(40, dtype=np.int32), x))
    np.testing.assert_allclose(y[ri], rv, rtol=1e-12)
    rest = np.ones(50, bool)
    rest[ri] = False
    assert (y[rest] == 0).all()


def test_unit_vector_returns_column():
    A = synth.random_csr(60, 40, 0.3, 3)
    D = synth.csr_to_dense(A)
    P = synth.csr_to_dense(synth.CSR(A.m, A.n, A.row_ptr, A.col_idx, None))
    O = oracle.Oracle(A)
    for j in range(A.n):
        x = synth.SparseVec(A.n, np.array([j], np.int32), np.array([1.0], np.float32))
        yi, yv, _ = O.spmspv(x)
        np.testing.assert_array_equal(yi, np.nonzero(P[:, j])[0])
        np.testing.assert_array_equal(yv, D[yi, j])


def test_permutation_permutes_x():
    n = 57
    rng = np.random.default_rng(0)
    perm = rng.permutation(n)
    A = synth.csr_from_coo(n, n, perm, np.arange(n), rng.uniform(0.5, 2, n))  # A[perm[j], j]
    x = synth.x_uniform(n, 20, 9)
    yi, yv, _ = oracle.Oracle(A).spmspv(x)
    expect = {}
    D = synth.csr_to_dense(A)
    for j, v in zip(x.idx, x.val):
        expect[perm[j]] = float(np.float64(D[perm[j], j]) * np.float64(v))
    assert list(yi) == sorted(expect)
    np.testing.assert_array_equal(yv, [expect[i] for i in yi])


def test_activity_rules():
    A = synth.random_csr(30, 30, 0.4, 5)
    O = oracle.Oracle(A)
    empty = synth.SparseVec(30, np.zeros(0, np.int32), np.zeros(0, np.float32))
    assert O.spmspv(empty)[0].size == 0
    zeros = synth.SparseVec(30, np.arange(5, dtype=np.int32), np.array([0.0, -0.0, 0.0, -0.0, 0.0], np.float32))
    assert O.spmspv(zeros)[0].size == 0                       # 0 and -0.0 are inactive
    xnan = synth.SparseVec(30, np.array([4], np.int32), np.array([np.nan], np.float32))
    col4 = np.nonzero(synth.csr_to_dense(A)[:, 4])[0]
    yi, yv, _ = O.spmspv(xnan)
    np.testing.assert_array_equal(yi, col4)                   # NaN is active
    assert np.isnan(yv).all()


def test_structural_pattern_keeps_cancellation():
    # y_0 = 1*1 + (-1)*1 = 0 exactly, but row 0 is still in the output pattern
    A = synth.csr_from_coo(2, 2, [0, 0], [0, 1], [1.0, -1.0])
    x = synth.SparseVec(2, np.array([0, 1], np.int32), np.array([1.0, 1.0], np.float32))
    yi, yv, ya = oracle.Oracle(A).spmspv(x)
    assert list(yi) == [0] and yv[0] == 0.0 and ya[0] == 2.0


@pytest.mark.parametrize("seed", range(5))
def test_push_equals_pull(seed):
    A = synth.random_csr(200, 150, 0.05, seed, valued=seed != 4)
    x = synth.x_uniform(150, 40, [seed, 3])
    for sr in (oracle.PLUS_TIMES, oracle.OR_AND):
        vis = np.random.default_rng(seed).integers(0, 2, 200).astype(np.uint8) if sr else None
        a = oracle.Oracle(A).spmspv(x, sr, vis)
        b = oracle.spmspv_pull(A, x, sr, vis)
        np.testing.assert_array_equal(a[0], b[0])
        if sr == oracle.PLUS_TIMES:
            np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)


def test_all_active_is_scipy_spmv():
    A = synth.config("er", "small")
    x = synth.x_uniform(A.n, A.n, 11)                          # every entry active
    yi, yv, _ = oracle.Oracle(A).spmspv(x)
    S = sp.csr_matrix((A.vals.astype(np.float64), A.col_idx, A.row_ptr), shape=(A.m, A.n))
    xd = np.zeros(A.n)
    xd[x.idx] = x.val
    ref = S @ xd
    nonempty = np.nonzero(np.diff(A.row_ptr))[0]
    np.testing.assert_array_equal(yi, nonempty)
    np.testing.assert_allclose(yv, ref[nonempty], rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------- BFS

def _grid(side):
    r, c = np.meshgrid(np.arange(side), np.arange(side - 1), indexing="ij")
    h = (r * side + c).ravel()
    v = (c * side + r).ravel()
    u = np.concatenate([h, v])
    w = np.concatenate([h + 1, v + side])
    return synth.csr_from_coo(side * side, side * side, np.concatenate([u, w]),
                              np.concatenate([w, u]))


def test_bfs_grid_is_manhattan_distance():
    side = 23
    A = _grid(side)
    O = oracle.Oracle(A)
    for src in (0, 5 * side + 7, side * side - 1):
        sr, sc = divmod(src, side)
        rr, cc = np.divmod(np.arange(side * side), side)
        expect = np.abs(rr - sr) + np.abs(cc - sc)
        np.testing.assert_array_equal(O.bfs_queue(src), expect)
        np.testing.assert_array_equal(O.bfs_spmspv(src), expect)


def test_bfs_path_star_complete_disconnected():
    n = 40
    path = synth.csr_from_coo(n, n, np.r_[np.arange(n - 1), np.arange(1, n)],
                              np.r_[np.arange(1, n), np.arange(n - 1)])
    np.testing.assert_array_equal(oracle.Oracle(path).bfs_spmspv(13), np.abs(np.arange(n) - 13))
    star = synth.csr_from_coo(n, n, np.r_[np.zeros(n - 1, int), np.arange(1, n)],
                              np.r_[np.arange(1, n), np.zeros(n - 1, int)])
    lev = oracle.Oracle(star).bfs_spmspv(5)
    assert lev[5] == 0 and lev[0] == 1 and (np.delete(lev, [0, 5]) == 2).all()
    ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    off = ii != jj
    comp = synth.csr_from_coo(n, n, ii[off], jj[off])
    lev = oracle.Oracle(comp).bfs_queue(3)
    assert lev[3] == 0 and (np.delete(lev, 3) == 1).all()
    two = synth.csr_from_coo(n, n, [0, 1], [1, 0])             # vertices 2.. isolated
    lev = oracle.Oracle(two).bfs_spmspv(0)
    assert list(lev[:2]) == [0, 1] and (lev[2:] == -1).all()


@pytest.mark.parametrize("name", ["rmat", "grid"])
def test_bfs_matches_scipy_distances(name):
    A = synth.config(name, "small")
    O = oracle.Oracle(A)
    S = sp.csr_matrix((np.ones(A.nnz), A.col_idx, A.row_ptr), shape=(A.m, A.n))
    for src in synth.bfs_sources(A, 3, 1):
        d = csgraph.shortest_path(S.T, method="D", unweighted=True, indices=int(src))
        expect = np.where(np.isinf(d), -1, d).astype(np.int32)
        np.testing.assert_array_equal(O.bfs_queue(src), expect)
        np.testing.assert_array_equal(O.bfs_spmspv(src), expect)


def test_bfs_directed_follows_columns():
    # A(1,0) stored: x_0 reaches row 1 (edge 0 -> 1); nothing reaches 0.
    A = synth.csr_from_coo(3, 3, [1, 2], [0, 1])
    O = oracle.Oracle(A)
    np.testing.assert_array_equal(O.bfs_queue(0), [0, 1, 2])
    np.testing.assert_array_equal(O.bfs_spmspv(0), [0, 1, 2])
    np.testing.assert_array_equal(O.bfs_spmspv(2), [-1, -1, 0])


# ------------------------------------------------- all-cores CPU baseline

@pytest.mark.parametrize("seed", range(5))
def test_parallel_pull_equals_push_and_serial_pull(seed):
    """The all-cores baseline's row-parallel pull gives the push oracle's
    pattern and the serial pull's values bit for bit (same order per row)."""
    A = synth.random_csr(300, 250, 0.04, seed, valued=seed != 4)
    for k in (0, 1, 60, 250):
        x = synth.x_uniform(250, k, [seed, 5, k])
        for sr in (oracle.PLUS_TIMES, oracle.OR_AND):
            vis = np.random.default_rng(seed).integers(0, 2, 300).astype(np.uint8) if sr else None
            a = oracle.Oracle(A).spmspv(x, sr, vis)
            b = oracle.spmspv_pull(A, x, sr, vis)
            c = oracle.spmspv_pull_par(A, x, sr, vis)
            np.testing.assert_array_equal(c[0], a[0])
            if sr == oracle.PLUS_TIMES:
                np.testing.assert_array_equal(c[1], b[1])
                np.testing.assert_array_equal(c[2], b[2])


@pytest.mark.parametrize("name", ["rmat", "grid"])
def test_parallel_bfs_equals_queue_bfs(name):
    A = synth.config(name, "small")
    O = oracle.Oracle(A)
    for src in synth.bfs_sources(A, 3, 2):
        np.testing.assert_array_equal(oracle.bfs_pull_par(A, int(src)), O.bfs_queue(int(src)))
    side = 19
    G = _grid(side)
    src = 4 * side + 11
    rr, cc = np.divmod(np.arange(side * side), side)
    np.testing.assert_array_equal(oracle.bfs_pull_par(G, src), np.abs(rr - 4) + np.abs(cc - 11))
    assert oracle.par_threads() >= 1


# ---------------------------------------------------------------- block views

def _fig5_matrix(bs):
    blocks = [(0, 0), (0, 1), (1, 1), (1, 2), (2, 0), (2, 1), (2, 2)]
    rng = np.random.default_rng(5)
    rows, cols = [], []
    for (rb, cb) in blocks:
        k = int(rng.integers(1, bs * bs // 2))
        flat = rng.choice(bs * bs, k, replace=False)
        rows += list(rb * bs + flat // bs)
        cols += list(cb * bs + flat % bs)
    return synth.csr_from_coo(3 * bs, 3 * bs, rows, cols, np.ones(len(rows)))


@pytest.mark.parametrize("bs", [4, 16])
def test_block_views_match_figure5(bs):
    g = read_golden("fig5_views.txt")
    V = oracle.block_views(_fig5_matrix(bs), bs=bs)
    assert V["B"] == 7
    for key in ("blk_row_ptr", "blk_col_idx", "blk_row_idx", "blk_csc2csr", "blk_col_ptr"):
        np.testing.assert_array_equal(V[key], g[key], err_msg=key)
    assert g["blk_col_ptr_printed"] != g["blk_col_ptr"]       # the printed erratum


def test_block_views_invariants_on_random():
    A = synth.random_csr(300, 200, 0.03, 1)
    V = oracle.block_views(A)
    B = V["B"]
    assert sorted(V["blk_csc2csr"]) == list(range(B))          # a permutation
    blk_row = np.repeat(np.arange(len(V["blk_row_ptr"]) - 1), np.diff(V["blk_row_ptr"]))
    np.testing.assert_array_equal(blk_row[V["blk_csc2csr"]], V["blk_row_idx"])
    col_of_q = np.repeat(np.arange(len(V["blk_col_ptr"]) - 1), np.diff(V["blk_col_ptr"]))
    np.testing.assert_array_equal(V["blk_col_idx"][V["blk_csc2csr"]], col_of_q)
    assert V["blk_nnz"].sum() == A.nnz
    # brute-force block occupancy from the dense pattern
    D = synth.csr_to_dense(A) != 0
    Db = np.pad(D, ((0, (-A.m) % 16), (0, (-A.n) % 16))).reshape((A.m + 15) // 16, 16, (A.n + 15) // 16, 16)
    occ = Db.sum(axis=(1, 3))
    rb, cb = np.nonzero(occ)
    np.testing.assert_array_equal(V["blk_col_idx"], cb)
    np.testing.assert_array_equal(V["blk_nnz"], occ[rb, cb])


def _one_block(entries):
    r, c = zip(*entries)
    return synth.csr_from_coo(16, 16, r, c, np.ones(len(r)))


def _cls(entries):
    V = oracle.block_views(_one_block(entries))
    assert V["B"] == 1
    return int(V["blk_class"][0])


def test_format_classes_by_density():
    cells = [(i // 16, i % 16) for i in range(256)]
    diag = lambda k: [(i, (i + d) % 16) for d in range(k) for i in range(16)]  # noqa: E731
    assert _cls(cells[:31]) == oracle.COO                   # 31 < th0 = 32
    assert _cls(diag(2)) == oracle.PATCHED_CSR              # 32 entries, every row/col 2
    assert _cls(diag(8)) == oracle.PATCHED_CSR              # 128 = th1, not > th1
    assert _cls(diag(8) + [(0, 8)]) == oracle.DENSE         # 129 > th1
    assert _cls(cells) == oracle.DENSE


def test_format_classes_by_skew():
    # row 0 full (16) + rows 1..15 two entries each on a band: max_row 16, max_col 3
    heavy_row = [(0, c) for c in range(16)] + [(r, (r + d) % 16) for r in range(1, 16) for d in (0, 1)]
    assert _cls(heavy_row) == oracle.FORCE_CSC              # row skew 16/3 > 2
    heavy_col = [(c, r) for (r, c) in heavy_row]
    assert _cls(heavy_col) == oracle.FORCE_CSR              # column skew dominates
    # max_row 4, max_col 2 (ratio exactly 2): not strictly above th2 -> patched CSR
    ratio2 = [(r, (r + d) % 16) for r in range(16) for d in (0, 1)] + [(0, 4), (0, 9)]
    ratio2 = sorted(set(ratio2))
    rows = np.bincount([r for r, _ in ratio2], minlength=16)
    cols = np.bincount([c for _, c in ratio2], minlength=16)
    assert rows.max() == 4 and cols.max() == 3               # hand check of the fixture
    assert _cls(ratio2) == oracle.PATCHED_CSR               # 4 / 3 < 2
    # diagonal + one more entry per column: row 0 takes columns 1..3, the
    # other columns' second entry sits one row above (column 0 on row 15):
    # every column holds 2, row 0 holds 4 -> ratio exactly 2, nnz = 32
    exact2 = [(r, r) for r in range(16)] + [(0, 1), (0, 2), (0, 3), (15, 0)] + \
             [(c - 1, c) for c in range(4, 16)]
    rows = np.bincount([r for r, _ in exact2], minlength=16)
    cols = np.bincount([c for _, c in exact2], minlength=16)
    assert len(exact2) == 32 and rows.max() == 4 and (cols == 2).all()
    assert _cls(exact2) == oracle.PATCHED_CSR               # 4 / 2 == 2, strict >
    above2 = [e for e in exact2 if e != (3, 4)] + [(0, 4)]  # row 0 holds 5, columns still 2
    assert _cls(above2) == oracle.FORCE_CSC                 # 5 / 2 > 2
    assert _cls([(c, r) for (r, c) in above2]) == oracle.FORCE_CSR


def test_tolerance_helper_rejects_a_wrong_value():
    ref = np.array([1.0, -2.0])
    S = np.array([1.0, 2.0])
    assert oracle.tolerance_ok(np.array([1.0 + 5e-6, -2.0]), ref, S).all()
    assert not oracle.tolerance_ok(np.array([1.0 + 2e-5, -2.0]), ref, S).all()
