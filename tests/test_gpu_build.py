"""Device-side conversion (device_convert = 1): every pass of the conversion
runs on the GPU -- blocks, formats, payloads, payload offsets, the block-CSC
view, the pull tiles and the row masks -- and the matrix must equal the host
builder's byte for byte -- every internal array -- for every workload,
forced format, pattern-only and valued inputs, ragged sizes and empty rows,
block-CSC column ranges on each side of the sort's size classes, and tile
options.  Rows whose columns are not ascending fall back to the host
conversion; bad row pointers and out-of-range or repeated columns are
rejected like on the host."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import __graft_entry__  # noqa: E402

__graft_entry__.build()
import dynamic_sparsity_spmspv_gb300 as dbs  # noqa: E402

DEV = "cuda"


def _dev(A):
    return (torch.from_numpy(np.asarray(A.row_ptr, np.int64)).to(DEV),
            torch.from_numpy(np.asarray(A.col_idx, np.int32)).to(DEV),
            None if A.vals is None else torch.from_numpy(np.asarray(A.vals, np.float32)).to(DEV))


def assert_same(A, **kw):
    host = dbs.DBMatrix.from_csr(A, **kw)
    rp, ci, va = _dev(A)
    gpu = dbs.DBMatrix(A.m, A.n, rp, ci, va, device_convert=1, **kw)
    ih, ig = host.info(), gpu.info()
    for k in ("nblocks", "ntiles", "payload_bytes", "view_bytes", "blocks_by_format", "nnz_by_format"):
        assert ih[k] == ig[k], k
    for name in dbs.DBMatrix.RAW_ARRAYS:
        np.testing.assert_array_equal(host.export_raw(name), gpu.export_raw(name), err_msg=name)
    return gpu


@pytest.mark.parametrize("name", synth.CONFIG_NAMES)
def test_device_conversion_matches_host(name):
    assert_same(synth.config(name, "small"))


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("name", ["llm", "fem", "rmat"])
def test_device_conversion_forced_formats(name, fmt):
    assert_same(synth.config(name, "small"), force_format=fmt)


def test_device_conversion_thresholds_ragged_and_empty():
    A = synth.random_csr(1003, 517, 0.3, 21)                     # ragged, mid-class blocks
    assert_same(A)
    assert_same(A, th0=8, th1=64, th2=1.5, tile_weight=16, tile_max_row_blocks=1)
    rows = np.repeat(np.arange(A.m), np.diff(A.row_ptr))
    keep = (rows // 16) % 3 != 1                                   # whole empty row blocks
    B = synth.csr_from_coo(A.m, A.n, rows[keep], A.col_idx[keep], A.vals[keep])
    assert_same(B)
    P = synth.CSR(B.m, B.n, B.row_ptr, B.col_idx, None)            # pattern only (inline blocks)
    assert_same(P)
    E = synth.CSR(40, 30, np.zeros(41, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32))
    assert_same(E)


def test_device_conversion_csc_size_classes_and_tile_windows():
    """Column blocks holding 1, 32, 33, 4096, 4097 and 9000 blocks (the
    warp rank, one shared-memory sort, and sorted chunks merged by rank),
    and more blocks than one window of the tile-start walk."""
    rng = np.random.default_rng(31)
    nrb = 9000
    m, n = 16 * nrb, 4096
    rows, cols = [], []
    for c, k in ((3, nrb), (20, 4096), (40, 4097), (60, 33), (80, 32), (100, 1)):
        rbs = np.sort(rng.choice(nrb, k, replace=False))
        rows.append(rbs * 16 + rng.integers(0, 16, k))
        cols.append(np.full(k, c))
    rr = rng.integers(0, m, 60000)
    rows.append(rr)
    cols.append(rng.integers(128, n, rr.size))
    rows, cols = np.concatenate(rows), np.concatenate(cols)
    key = np.unique(rows.astype(np.int64) * n + cols)
    rows, cols = key // n, (key % n).astype(np.int32)
    vals = rng.standard_normal(rows.size).astype(np.float32)
    A = synth.csr_from_coo(m, n, rows, cols, vals)
    M = assert_same(A)
    assert M.info()["nblocks"] > 11264
    assert_same(synth.CSR(A.m, A.n, A.row_ptr, A.col_idx, None))
    assert_same(A, tile_weight=256)
    assert_same(A, tile_weight=16, tile_max_row_blocks=1)


def test_device_conversion_rejects_bad_row_pointers():
    """The device validates the row pointers before reading any entry:
    rp[0] != 0, rp[m] != nnz, a decreasing pair and a pointer past nnz are
    DBS_ERR_INVALID_ARG, as on the host."""
    import ctypes
    from dynamic_sparsity_spmspv_gb300 import _lib

    A = synth.random_csr(300, 200, 0.05, 29)
    for mutate in ("first", "decreasing", "past_end"):
        rp = A.row_ptr.copy()
        if mutate == "first":
            rp[0] = 1
        elif mutate == "decreasing":
            rp[100] = rp[101] + 1
        else:
            rp[150] = A.nnz + 1000
        r, c, v = _dev(synth.CSR(A.m, A.n, rp, A.col_idx, A.vals))
        with pytest.raises(dbs.DbsError):
            dbs.DBMatrix(A.m, A.n, r, c, v, device_convert=1)
        with pytest.raises(dbs.DbsError):
            dbs.DBMatrix(A.m, A.n, r, c, v)
    # nnz other than rp[m] (the entry arrays are padded, so nothing is out of bounds)
    r, _, _ = _dev(A)
    c = torch.zeros(A.nnz + 8, dtype=torch.int32, device=DEV)
    v = torch.zeros(A.nnz + 8, dtype=torch.float32, device=DEV)
    c[:A.nnz] = torch.from_numpy(A.col_idx).to(DEV)
    lib = _lib.load()
    for dc in (1, 0):
        o = _lib.dbs_build_opts()
        lib.dbs_build_opts_default(ctypes.byref(o))
        o.device_convert = dc
        h = ctypes.c_void_p()
        st = lib.dbs_matrix_build_csr(A.m, A.n, A.nnz + 5, ctypes.c_void_p(r.data_ptr()),
                                      ctypes.c_void_p(c.data_ptr()), ctypes.c_void_p(v.data_ptr()), 1,
                                      ctypes.byref(o), None, ctypes.byref(h))
        assert st == 1 and not h.value


@pytest.mark.parametrize("name", ["rmat", "llm"])
def test_build_peak_device_memory(name):
    """build_peak_bytes: the host build holds the uploaded matrix alone; the
    device conversion holds the matrix plus 4 bytes per block and 12 per
    column block, or 4 per row block and 8 per merge task while the blocks
    are found, and the scan partials: the bound the header states."""
    A = synth.config(name, "full")
    rp, ci, va = _dev(A)
    for dc in (0, 1):
        M = dbs.DBMatrix(A.m, A.n, rp, ci, va, device_convert=dc)
        inf = M.info()
        B, nbr, nbc = inf["nblocks"], inf["nbr"], inf["nbc"]
        padded = inf["total_bytes"] + 4 * 8 * 16 + 8 * 16
        assert inf["build_peak_bytes"] >= inf["total_bytes"]
        if dc == 0:
            assert inf["build_peak_bytes"] <= padded + 4096
        else:
            tasks = nbr + A.nnz // 4096 + 1
            scan = 24 * ((max(B, nbc, nbr, tasks) + 4095) // 4096 + 1)
            extra = max(4 * B + 12 * nbc, 4 * (nbr + 1) + 8 * (tasks + 1))
            assert inf["build_peak_bytes"] <= padded + extra + scan + 4096, inf
        M.close()


def test_device_conversion_then_multiply_and_keep_host():
    """A device-converted matrix multiplies like the host one, and keep_host
    holds its payload too (export round trip)."""
    A = synth.config("llm", "small")
    rp, ci, va = _dev(A)
    M = dbs.DBMatrix(A.m, A.n, rp, ci, va, device_convert=1, keep_host=1)
    r2, c2, v2 = M.export_csr()
    np.testing.assert_array_equal(r2, A.row_ptr)
    np.testing.assert_array_equal(c2, A.col_idx)
    np.testing.assert_array_equal(v2.view(np.uint32), A.vals.view(np.uint32))
    Mh = dbs.DBMatrix.from_csr(A)
    x = torch.from_numpy(synth.x_activation(A.n, [3])).to(DEV)
    y1 = dbs.decode_layer(M, x, 1.0, ws=dbs.Workspace(M)).cpu().numpy()
    y2 = dbs.decode_layer(Mh, x, 1.0, ws=dbs.Workspace(Mh)).cpu().numpy()
    np.testing.assert_allclose(y1, y2, rtol=1e-6, atol=1e-6)


def test_device_conversion_unsorted_rows_fall_back_and_bad_columns_fail():
    A = synth.random_csr(200, 150, 0.1, 23)
    ci = A.col_idx.copy()
    s, e = int(A.row_ptr[5]), int(A.row_ptr[6])
    ci[s:e] = ci[s:e][::-1]                                        # one row in descending order
    U = synth.CSR(A.m, A.n, A.row_ptr, ci, A.vals)
    host = dbs.DBMatrix.from_csr(U)
    rp, c, v = _dev(U)
    gpu = dbs.DBMatrix(U.m, U.n, rp, c, v, device_convert=1)
    for name in dbs.DBMatrix.RAW_ARRAYS:
        np.testing.assert_array_equal(host.export_raw(name), gpu.export_raw(name), err_msg=name)
    for bad in (A.n, -1):
        ci2 = A.col_idx.copy()
        ci2[7] = bad
        rp, c, v = _dev(synth.CSR(A.m, A.n, A.row_ptr, ci2, A.vals))
        with pytest.raises(dbs.DbsError):
            dbs.DBMatrix(A.m, A.n, rp, c, v, device_convert=1)
    ci3 = A.col_idx.copy()
    k = int(A.row_ptr[9])
    assert A.row_ptr[10] - A.row_ptr[9] >= 2
    ci3[k + 1] = ci3[k]                                            # repeated column
    rp, c, v = _dev(synth.CSR(A.m, A.n, A.row_ptr, ci3, A.vals))
    with pytest.raises(dbs.DbsError):
        dbs.DBMatrix(A.m, A.n, rp, c, v, device_convert=1)


@pytest.mark.parametrize("name", ["rmat", "llm", "fem", "grid"])
def test_device_conversion_full_size(name):
    M = assert_same(synth.config(name, "full"))
    assert M.info()["build_seconds"] > 0


@pytest.mark.parametrize("name", ["rmat", "llm"])
def test_device_conversion_full_size_against_oracle(name):
    """A device-converted matrix against the oracle directly, not only
    against the host builder: its block views (DB-SpMSpV Section 3.2.1,
    Figure 5(b)) equal the oracle's, and its products pass the parity bar --
    Boolean SpMSpV at three densities on every path and BFS levels for the
    R-MAT graph, plus-times SpMSpV and the DB-Decoding layer (Section 4.3)
    for the LLM layer."""
    import oracle
    from test_gpu_parity import assert_parity, _t

    A = synth.config(name, "full")
    rp, ci, va = _dev(A)
    M = dbs.DBMatrix(A.m, A.n, rp, ci, va, device_convert=1)
    del rp, ci, va
    V, W = M.export_views(), oracle.block_views(A)
    assert V["B"] == W["B"]
    for k in ("blk_row_ptr", "blk_col_idx", "blk_col_ptr", "blk_row_idx", "blk_csc2csr", "blk_nnz"):
        np.testing.assert_array_equal(V[k], W[k], err_msg=k)
    np.testing.assert_array_equal(V["blk_format"], W["blk_class"])
    del V, W
    O = oracle.Oracle(A)
    ws = dbs.Workspace(M)
    if name == "rmat":
        for d in (1e-3, 1e-2, 1e-1):
            x = synth.x_uniform(A.n, int(round(d * A.n)), [60, int(d * 1e4)], valued=False)
            for path in ("auto", "push", "pull"):
                assert_parity(A, O, M, ws, x, "or_and", path=path)
        for src in synth.bfs_sources(A, 2, [60, 7]):
            lev, nl = dbs.bfs(M, int(src), ws=ws)
            ref = O.bfs_queue(int(src))
            np.testing.assert_array_equal(lev.cpu().numpy(), ref)
            assert nl == int(ref.max()) + 1
    else:
        for t in range(2):
            xd = synth.x_relu_topk(A.n, 1101, [61, t])
            nz = np.nonzero(xd)[0].astype(np.int32)
            for path in ("auto", "push", "pull"):
                assert_parity(A, O, M, ws, synth.SparseVec(A.n, nz, xd[nz]), path=path)
            xa = synth.x_activation(A.n, [62, t])
            y = dbs.decode_layer(M, _t(xa), 1.6449, ws=ws).cpu().numpy()
            assert ws.check() == 0
            ref, s, touched = O.decode_layer(xa, 1.6449)
            assert oracle.tolerance_ok(y[touched], ref[touched], s[touched]).all()
            assert (y[~touched] == 0).all()
