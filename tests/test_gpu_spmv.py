"""GPU parity of the dense-input regime (adaptive CSR SpMV, dbs_spmv):
y = A x over every stored entry, against the oracle's plain CSR SpMV, with
the fp32 tolerance |y - y_ref| <= 1e-5 * sum |a x| + 1e-30 on every row
(rows without entries must be exactly 0)."""
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


def check(A, x, y):
    ref, s = oracle.spmv_csr(A, x)
    y = y.cpu().numpy()[:A.m]
    assert oracle.tolerance_ok(y, ref, s).all()
    empty = np.diff(A.row_ptr) == 0
    assert (y[empty] == 0).all()


def valued(A, seed):
    if A.vals is not None:
        return A
    v = np.random.default_rng(seed).uniform(-1, 1, A.nnz).astype(np.float32)
    return synth.CSR(A.m, A.n, A.row_ptr, A.col_idx, v)


@pytest.mark.parametrize("name", synth.CONFIG_NAMES)
def test_spmv_small_configs(name):
    A = valued(synth.config(name, "small"), 1)
    plan = dbs.SpMVPlan.from_csr(A)
    rng = np.random.default_rng(2)
    for _ in range(3):
        x = rng.standard_normal(A.n).astype(np.float32)
        x[rng.random(A.n) < 0.4] = 0.0
        check(A, x, plan(torch.from_numpy(x).to(DEV)))


def _shaped(lengths, n, seed):
    """Rows of the given lengths, distinct uniform columns, values U[-1, 1]."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for i, L in enumerate(lengths):
        rows.append(np.full(L, i))
        cols.append(rng.choice(n, size=L, replace=False))
    rows = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    cols = np.concatenate(cols) if cols else np.zeros(0, np.int64)
    vals = rng.uniform(-1, 1, rows.shape[0]).astype(np.float32)
    return synth.csr_from_coo(len(lengths), n, rows, cols, vals)


def test_spmv_every_bucket_and_boundary():
    """Row lengths at every bucket boundary (4 .. 64 / 1024 / 16384) and split
    rows of several chunks, empty rows between them; the plan's bucket counts
    follow the lengths."""
    lengths = [0, 1, 4, 5, 8, 9, 16, 17, 32, 33, 64, 65, 0, 1024, 1025, 16384, 16385, 50000, 3, 0,
               8192 * 4, 8192 * 4 + 1]
    A = _shaped(lengths, 60000, 4)
    plan = dbs.SpMVPlan.from_csr(A)
    inf = plan.info()
    L = np.array(lengths)
    lo = 0
    for b in range(6):                          # 2^b lanes for rows of up to 4 * 2^b entries (32 lanes: 1024)
        hi = 4 << b if b < 5 else 1024
        assert inf["lane_group_rows"][str(1 << b)] == int(((L > lo) & (L <= hi)).sum() + (L == 0).sum() * (b == 0)), b
        lo = hi
    assert inf["block_rows"] == int(((L > 1024) & (L <= 16384)).sum())
    assert inf["split_rows"] == int((L > 16384).sum())
    assert inf["split_chunks"] == int(sum((l + 8191) // 8192 for l in lengths if l > 16384))
    rng = np.random.default_rng(5)
    y = torch.full((A.m,), 3.0, dtype=torch.float32, device=DEV)        # stale values are overwritten
    for _ in range(4):                                                  # split-row counters reset themselves
        x = rng.standard_normal(A.n).astype(np.float32)
        plan(torch.from_numpy(x).to(DEV), y=y)
        check(A, x, y)


@pytest.mark.parametrize("b", range(5))
def test_spmv_short_row_buckets(b):
    """Thousands of rows of the 2^b-lane bucket (lengths in (2^(b+1),
    2^(b+2)], 1 to 4 entries for b = 0), every alignment of a row's first
    entry, empty rows among them, rows of wider buckets in between, columns
    outside [0, n) on some entries and a row count that leaves a ragged last
    item; integer values make the sums exact, so y must equal the oracle's
    and the plan's bucket count must follow the lengths."""
    rng = np.random.default_rng(40 + b)
    lo, hi = (1, 4) if b == 0 else ((4 << b) // 2 + 1, 4 << b)
    m, n = 5000 + 37 * b, 4096
    lengths = rng.integers(lo, hi + 1, m)
    lengths[rng.random(m) < 0.03] = 0
    other = rng.random(m) < 0.01
    lengths[other] = rng.integers(hi + 1, 2 * hi + 40, int(other.sum()))
    A = _shaped(list(lengths), n, 50 + b)
    vals = rng.integers(-3, 4, A.nnz).astype(np.float32)
    ci = A.col_idx.copy()
    ci[rng.random(A.nnz) < 0.01] = n + 3
    A = synth.CSR(A.m, A.n, A.row_ptr, ci, vals)
    below = 0 if b == 0 else hi // 2
    want = int(((lengths > below) & (lengths <= hi)).sum() + (b == 0) * (lengths == 0).sum())
    assert dbs.SpMVPlan.from_csr(A).info()["lane_group_rows"][str(1 << b)] == want
    x = rng.integers(-3, 4, n).astype(np.float32)
    y = torch.full((A.m,), 7.0, dtype=torch.float32, device=DEV)
    dbs.SpMVPlan.from_csr(A)(torch.from_numpy(x).to(DEV), y=y)
    ref, _ = oracle.spmv_csr(A, x)
    np.testing.assert_array_equal(y.cpu().numpy(), ref.astype(np.float32))


def test_spmv_integer_values_bit_exact():
    A = synth.random_csr(300, 300, 0.1, 9, integer_values=True)
    x = np.random.default_rng(9).integers(-3, 4, 300).astype(np.float32)
    y = dbs.SpMVPlan.from_csr(A)(torch.from_numpy(x).to(DEV)).cpu().numpy()
    ref, _ = oracle.spmv_csr(A, x)
    np.testing.assert_array_equal(y, ref.astype(np.float32))


def test_spmv_out_of_range_columns_and_clamped_rows():
    """Columns outside [0, n) contribute nothing; row pointers past nnz are
    clamped (no stray access, rows beyond the entries read as empty)."""
    A = synth.random_csr(100, 80, 0.1, 11)
    ci = A.col_idx.copy()
    ci[::7] = 80 + (np.arange(ci[::7].shape[0]) % 5)
    ci[3::11] = -1
    B = synth.CSR(A.m, A.n, A.row_ptr, ci, A.vals)
    x = np.random.default_rng(12).standard_normal(80).astype(np.float32)
    check(B, x, dbs.SpMVPlan.from_csr(B)(torch.from_numpy(x).to(DEV)))
    rp = A.row_ptr.copy()
    rp[60:] = A.nnz + 1000                               # past the end: clamped to nnz
    dev_rp = torch.from_numpy(rp).to(DEV)
    plan = dbs.SpMVPlan(A.m, A.n, dev_rp, torch.from_numpy(A.col_idx).to(DEV), torch.from_numpy(A.vals).to(DEV))
    y = plan(torch.from_numpy(x).to(DEV)).cpu().numpy()
    C = synth.CSR(A.m, A.n, np.minimum(rp, A.nnz), A.col_idx, A.vals)
    ref, s = oracle.spmv_csr(C, x)
    assert oracle.tolerance_ok(y, ref, s).all()


def test_spmv_empty_and_graph_replay():
    E = synth.CSR(5, 7, np.zeros(6, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32))
    y = dbs.SpMVPlan.from_csr(E)(torch.ones(7, dtype=torch.float32, device=DEV)).cpu().numpy()
    assert (y == 0).all()
    A = valued(synth.config("rmat", "small"), 13)
    plan = dbs.SpMVPlan.from_csr(A)
    x = torch.zeros(A.n, dtype=torch.float32, device=DEV)
    y = torch.empty(A.m, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan(x, y=y)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan(x, y=y)
    rng = np.random.default_rng(14)
    for _ in range(3):
        h = rng.standard_normal(A.n).astype(np.float32)
        x.copy_(torch.from_numpy(h))
        g.replay()
        torch.cuda.synchronize()
        check(A, h, y)


def test_spmv_full_size_llm_and_rmat():
    for name in ("llm", "rmat"):
        A = valued(synth.config(name, "full"), 15)
        plan = dbs.SpMVPlan.from_csr(A)
        x = np.random.default_rng(16).standard_normal(A.n).astype(np.float32)
        check(A, x, plan(torch.from_numpy(x).to(DEV)))
        if name == "rmat":
            assert plan.info()["split_rows"] > 0          # hub rows exercise the long-row split


def _dense_parity(A, O, y, xd):
    """dbs_spmspv_dense's contract: the structural product over the nonzero
    entries of x (zeros inactive), rows nothing reaches exactly 0."""
    nz = np.nonzero(xd)[0].astype(np.int32)
    ri, rv, rs = O.spmspv(synth.SparseVec(A.n, nz, xd[nz]))
    y = y.cpu().numpy()[:A.m]
    assert oracle.tolerance_ok(y[ri], rv, rs).all()
    rest = np.ones(A.m, bool)
    rest[ri] = False
    assert (y[rest] == 0).all()


@pytest.mark.parametrize("name", ["llm", "fem", "er", "rmat"])
def test_dense_x_handed_to_the_kept_spmv(name):
    """The paper's Limitations (conventional SpMV suits dense inputs): with
    dense_spmv the matrix keeps its CSR and an adaptive SpMV plan, and
    dbs_spmspv_dense computes a dense x by that SpMV -- forced ('spmv'), or
    on the auto path once the sampled nonzero fraction reaches spmv_x_frac --
    with the same structural result as the blocked paths; a sparse x stays
    on the blocked path."""
    A = valued(synth.config(name, "small"), 2)
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A, dense_spmv=1)
    assert M.info()["spmv_bytes"] > 0
    ws = dbs.Workspace(M, collect_stats=1)
    rng = np.random.default_rng(5)
    for frac in (1.0, 0.6, 0.09, 0.02, 0.0):
        xd = rng.standard_normal(A.n).astype(np.float32)
        xd[rng.random(A.n) >= frac] = 0.0
        xd[:3] = [0.0, -0.0, 1.0] if A.n >= 3 else xd[:3]
        for path in ("auto", "spmv", "pull", "push"):
            y = dbs.spmspv_dense(M, torch.from_numpy(xd).to(DEV), ws=ws, path=path)
            st = ws.stats()
            assert ws.check() == 0
            _dense_parity(A, O, y, xd)
            if path == "spmv":
                assert st["path"] == 3
            if path == "auto":
                if A.n <= 256:
                    sample = xd
                else:
                    t = np.arange(256)
                    sample = xd[(t >> 5) * (A.n // 8) + (t & 31)]
                assert (st["path"] == 3) == (np.count_nonzero(sample) >= 0.08 * sample.size), frac
    # integer values: the SpMV route is bit-exact like the blocked paths
    I = synth.random_csr(300, 200, 0.2, 7, integer_values=True)
    MI = dbs.DBMatrix.from_csr(I, dense_spmv=1)
    wsi = dbs.Workspace(MI)
    xi = rng.integers(-3, 4, I.n).astype(np.float32)
    y1 = dbs.spmspv_dense(MI, torch.from_numpy(xi).to(DEV), ws=wsi, path="spmv").cpu().numpy()
    y2 = dbs.spmspv_dense(MI, torch.from_numpy(xi).to(DEV), ws=wsi, path="pull").cpu().numpy()
    np.testing.assert_array_equal(y1, y2)
    # without the kept plan the spmv path is refused
    M0 = dbs.DBMatrix.from_csr(A)
    with pytest.raises(dbs.DbsError) as e:
        dbs.spmspv_dense(M0, torch.zeros(A.n, device=DEV), ws=dbs.Workspace(M0), path="spmv")
    assert e.value.status == 1


@pytest.mark.parametrize("name", ["fem", "llm", "rmat"])
def test_dense_x_full_size_auto_route(name):
    """Full-size FEM, LLM and R-MAT (unit weights) with an all-nonzero x: the
    auto path routes to the kept SpMV and matches the oracle; the
    one-launch graph replay of the routed call stays correct."""
    A = valued(synth.config(name, "full"), 3) if name != "rmat" else synth.CSR(
        *(lambda G: (G.m, G.n, G.row_ptr, G.col_idx, np.ones(G.nnz, np.float32)))(synth.config("rmat", "full")))
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A, dense_spmv=1)
    ws = dbs.Workspace(M, collect_stats=1)
    xd = np.random.default_rng(9).standard_normal(A.n).astype(np.float32)
    y = dbs.spmspv_dense(M, torch.from_numpy(xd).to(DEV), ws=ws)
    assert ws.stats()["path"] == 3 and ws.check() == 0
    _dense_parity(A, O, y, xd)
