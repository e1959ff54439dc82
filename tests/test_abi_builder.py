"""CPU-side checks of the C ABI: the library loads, exports every function the
header declares, validates its inputs, and its host builder produces exactly
the block views, format classes and payload the oracle and the paper fix."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth
from conftest import ROOT, read_golden

import __graft_entry__

__graft_entry__.build()
import dynamic_sparsity_spmspv_gb300 as dbs  # noqa: E402
from dynamic_sparsity_spmspv_gb300 import _lib  # noqa: E402


def _header_functions():
    text = open(os.path.join(ROOT, "include", "dbspmspv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dbs_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    lib = _lib.load()
    names = _header_functions()
    assert len(names) >= 18
    for name in names:
        assert hasattr(lib, name), name
        assert name in _lib.PROTOTYPES, f"binding lacks {name}"


def test_library_is_rebuilt_after_any_source_or_header_changes(monkeypatch):
    """The in-tree build is redone when any file under csrc/ or include/ is
    newer than the library: a later modification time faked for each file in
    turn (the files themselves are not touched) must make the library stale."""
    from dynamic_sparsity_spmspv_gb300 import _build
    lib_t = os.path.getmtime(_build.LIB)
    files = [os.path.join(_build.CSRC, f) for f in os.listdir(_build.CSRC)
             if f.endswith((".cu", ".cpp", ".h", ".cuh"))]
    files += [os.path.join(_build.INCLUDE, f) for f in os.listdir(_build.INCLUDE) if f.endswith(".h")]
    assert any(f.endswith("spmv_dev.h") for f in files)
    real = os.path.getmtime
    for f in files:
        monkeypatch.setattr(os.path, "getmtime", lambda p, f=f: lib_t + 10.0 if p == f else real(p))
        assert _build._newest_input() > lib_t, f
    monkeypatch.setattr(os.path, "getmtime", real)
    assert _build._newest_input() <= lib_t


def test_status_strings_and_version():
    lib = _lib.load()
    assert lib.dbs_status_string(4) == b"DBS_ERR_TIMEOUT"
    assert lib.dbs_version().startswith(b"dbspmspv")


def test_struct_layouts_match_header_sizes():
    # sizes implied by the C declarations on LP64
    assert ctypes.sizeof(_lib.dbs_build_opts) == 48
    assert ctypes.sizeof(_lib.dbs_exec_opts) == 40
    assert ctypes.sizeof(_lib.dbs_stats) == 104
    assert ctypes.sizeof(_lib.dbs_matrix_info) == 8 * 15 + 8 * 2 * 5 + 4 * 2   # 64-bit scalars, formats, 2 int32
    o = dbs.build_opts()
    assert (o.th0, o.th1, o.th2, o.force_format) == (32, 128, 2.0, -1)
    e = dbs.exec_opts()
    assert (e.th3, e.local_pull_min, e.push_work_frac, e.spmv_x_frac) == (0.01, 0, 0.45, 0.08)
    assert o.dense_spmv == 0
    with pytest.raises(TypeError):
        dbs.build_opts(no_such_option=1)


def _host(A, **kw):
    return dbs.DBMatrix.from_csr(A, host_only=1, **kw)


@pytest.mark.parametrize("name", synth.CONFIG_NAMES)
def test_views_match_oracle(name):
    A = synth.config(name, "small")
    M = _host(A)
    V = M.export_views()
    O = oracle.block_views(A)
    assert V["B"] == O["B"]
    for k in ("blk_row_ptr", "blk_col_idx", "blk_col_ptr", "blk_row_idx", "blk_csc2csr", "blk_nnz"):
        np.testing.assert_array_equal(V[k], O[k], err_msg=k)
    np.testing.assert_array_equal(V["blk_format"], O["blk_class"])


@pytest.mark.parametrize("bs_scale", [16])
def test_views_match_figure5(bs_scale):
    g = read_golden("fig5_views.txt")
    rng = np.random.default_rng(2)
    blocks = [(0, 0), (0, 1), (1, 1), (1, 2), (2, 0), (2, 1), (2, 2)]
    rows, cols = [], []
    for rb, cb in blocks:
        flat = rng.choice(256, int(rng.integers(1, 200)), replace=False)
        rows += list(rb * 16 + flat // 16)
        cols += list(cb * 16 + flat % 16)
    A = synth.csr_from_coo(48, 48, rows, cols, rng.standard_normal(len(rows)))
    V = _host(A).export_views()
    for k in ("blk_row_ptr", "blk_col_idx", "blk_row_idx", "blk_csc2csr", "blk_col_ptr"):
        np.testing.assert_array_equal(V[k], g[k], err_msg=k)


@pytest.mark.parametrize("fmt", [-1, 0, 1, 2, 3, 4])
@pytest.mark.parametrize("name", ["er", "fem", "llm", "grid"])
def test_decode_round_trip_is_bitwise(name, fmt):
    A = synth.config(name, "small")
    M = _host(A, force_format=fmt)
    rp, ci, va = M.export_csr()
    np.testing.assert_array_equal(rp, A.row_ptr)
    np.testing.assert_array_equal(ci, A.col_idx)
    if A.vals is None:
        assert va is None
    else:
        assert va.view(np.uint32).tobytes() == A.vals.view(np.uint32).tobytes()
    inf = M.info()
    if fmt >= 0:
        assert inf["blocks_by_format"][fmt] == inf["nblocks"]
    assert sum(inf["nnz_by_format"]) == A.nnz


def test_row_mask_bit_order_matches_figure5():
    # One ForceCSR block whose row 0 holds columns 1 and 3: Figure 5 prints
    # that row_mask as 10 = 0b1010.  Read the exported payload back through
    # the decoder and check the entries land in columns 1 and 3.
    g = read_golden("fig5_views.txt")
    assert g["row_mask_example"] == [10]
    rows = [0, 0] + [r for r in range(1, 16) for _ in range(2)]
    cols = [1, 3] + [c for r in range(1, 16) for c in (r % 16, (r + 5) % 16)]
    A = synth.csr_from_coo(16, 16, rows, cols, np.arange(len(rows), dtype=np.float32) + 1)
    M = _host(A, force_format=dbs.FMT_FORCE_CSR)
    rp, ci, va = M.export_csr()
    assert list(ci[rp[0]:rp[1]]) == g["row_mask_example_cols"]


def test_tiles_respect_weight_and_span():
    A = synth.config("rmat", "small")
    for W, R in [(16, 1), (64, 8), (2048, 32)]:
        inf = _host(A, tile_weight=W, tile_max_row_blocks=R).info()
        assert inf["ntiles"] >= 1
    # paper segments: W = 16, R = 1 -> no tile spans two row blocks, so the
    # tile count is at least the number of non-empty row blocks
    V = _host(A).export_views()
    nonempty = int((np.diff(V["blk_row_ptr"]) > 0).sum())
    assert _host(A, tile_weight=16, tile_max_row_blocks=1).info()["ntiles"] >= nonempty


def test_storage_report():
    A = synth.config("llm", "small")
    inf = _host(A).info()
    assert inf["csr_csc_bytes"] == 2 * inf["csr_bytes"] - (A.m + 1) * 4 + (A.n + 1) * 4
    assert inf["total_bytes"] == inf["payload_bytes"] + inf["view_bytes"]
    assert inf["valued"] == 1 and inf["on_device"] == 0
    assert inf["build_peak_bytes"] == 0          # a host-only build touches no device memory


@pytest.mark.parametrize("bad", ["dup", "range", "rowptr", "neg"])
def test_builder_rejects_invalid_csr(bad):
    rp = np.array([0, 2, 3], np.int64)
    ci = np.array([0, 1, 2], np.int32)
    if bad == "dup":
        ci = np.array([1, 1, 2], np.int32)
    elif bad == "range":
        ci = np.array([0, 1, 7], np.int32)
    elif bad == "rowptr":
        rp = np.array([0, 3, 2], np.int64)
    elif bad == "neg":
        ci = np.array([0, -1, 2], np.int32)
    with pytest.raises(dbs.DbsError) as e:
        dbs.DBMatrix(2, 4, rp, ci, np.ones(3, np.float32), host_only=1)
    assert e.value.status == 1


def test_unsorted_rows_are_accepted():
    rp = np.array([0, 3], np.int64)
    ci = np.array([5, 0, 17], np.int32)
    va = np.array([1.0, 2.0, 3.0], np.float32)
    M = dbs.DBMatrix(1, 20, rp, ci, va, host_only=1)
    rp2, ci2, va2 = M.export_csr()
    assert list(ci2) == [0, 5, 17] and list(va2) == [2.0, 1.0, 3.0]


def test_empty_and_degenerate_shapes():
    for m, n in [(0, 0), (0, 5), (5, 0), (1, 1), (17, 33)]:
        rp = np.zeros(m + 1, np.int64)
        M = dbs.DBMatrix(m, n, rp, np.zeros(0, np.int32), np.zeros(0, np.float32), host_only=1)
        inf = M.info()
        assert inf["nblocks"] == 0 and inf["nbr"] == (m + 15) // 16


def test_export_raw_sizes_and_contents():
    A = synth.config("llm", "small")
    M = dbs.DBMatrix.from_csr(A, host_only=1, keep_host=1)
    inf = M.info()
    B, nbr, nbc = inf["nblocks"], inf["nbr"], inf["nbc"]
    sizes = {"rb_ptr": 4 * (nbr + 1), "blk_desc": 8 * B, "blk_ref": 4 * B, "cb_ptr": 4 * (nbc + 1),
             "csc_desc": 8 * B, "csc_ref": 4 * B, "payload": inf["payload_bytes"], "tiles": 16 * inf["ntiles"],
             "rb_rows": 2 * nbr}
    for name, size in sizes.items():
        assert M.export_raw(name).nbytes == size, name
    rbp = M.export_raw("rb_ptr").view(np.uint32)
    views = M.export_views()
    np.testing.assert_array_equal(rbp, views["blk_row_ptr"])
    ref = M.export_raw("blk_ref").view(np.uint32)
    fmt = views["blk_format"]
    assert (ref[fmt == 1] % 4 == 0).all()            # valued Dense blocks start on 64-byte boundaries


def test_export_raw_rejects_bad_requests():
    A = synth.config("er", "small")
    M = dbs.DBMatrix.from_csr(A, host_only=1, keep_host=1)
    lib = _lib.load()
    nb = ctypes.c_int64(0)
    assert lib.dbs_matrix_export_raw(M.handle, 99, None, 0, ctypes.byref(nb)) == 1
    assert lib.dbs_matrix_export_raw(M.handle, 0, None, 0, None) == 1
    assert lib.dbs_matrix_export_raw(M.handle, 0, None, 0, ctypes.byref(nb)) == 0 and nb.value > 0
    small = np.zeros(max(nb.value - 1, 1), np.uint8)
    assert lib.dbs_matrix_export_raw(M.handle, 0, small.ctypes.data, small.nbytes, ctypes.byref(nb)) == \
        1


def test_device_convert_with_host_inputs_is_the_host_conversion():
    """device_convert applies to device inputs only; with host arrays the
    host builder runs and the result is unchanged."""
    A = synth.config("llm", "small")
    M1 = dbs.DBMatrix.from_csr(A, host_only=1, keep_host=1)
    M2 = dbs.DBMatrix.from_csr(A, host_only=1, keep_host=1, device_convert=1)
    for name in dbs.DBMatrix.RAW_ARRAYS:
        np.testing.assert_array_equal(M1.export_raw(name), M2.export_raw(name), err_msg=name)


@pytest.mark.parametrize("name,kw", [("llm", {"tile_weight": 24}), ("rmat", {}), ("fem", {"tile_max_row_blocks": 1})])
def test_tiles_and_row_block_rows(name, kw):
    """Pull tiles cover the blocks in order within their caps, each tile's
    span names the row blocks of its first and last blocks, and every row
    block records which of its rows hold an entry."""
    A = synth.config(name, "small")
    M = dbs.DBMatrix.from_csr(A, host_only=1, keep_host=1, **kw)
    inf = M.info()
    tiles = M.export_raw("tiles").view(np.uint32).reshape(-1, 4)
    rbp = M.export_raw("rb_ptr").view(np.uint32)
    span = tiles[:, 3] & 0xFFFF
    nblk = tiles[:, 3] >> 20
    assert (tiles[1:, 0] == tiles[:-1, 0] + nblk[:-1]).all() and tiles[0, 0] == 0
    assert int(nblk.sum()) == inf["nblocks"]
    assert ((tiles[:, 0] & 1) + nblk <= 256).all() and (span >= 1).all() and (span <= 32).all()
    for t in range(tiles.shape[0]):
        p0, n, rb0, sp = int(tiles[t, 0]), int(nblk[t]), int(tiles[t, 2]), int(span[t])
        # first and last row blocks of the span hold the tile's first and last blocks
        assert rbp[rb0] <= p0 < rbp[rb0 + 1]
        assert rbp[rb0 + sp - 1] <= p0 + n - 1 < rbp[rb0 + sp]
    rows = M.export_raw("rb_rows").view(np.uint16)
    nonempty = np.diff(A.row_ptr) > 0
    want = np.zeros(inf["nbr"], np.uint32)
    for i in np.nonzero(nonempty)[0]:
        want[i // 16] |= 1 << (i % 16)
    np.testing.assert_array_equal(rows, want.astype(np.uint16))


def _fail_alloc(k):
    prev = ctypes.c_int64(0)
    assert _lib.load().dbs_debug_fail_alloc(k, ctypes.byref(prev)) == 0
    return prev.value


def test_injected_allocation_failures_in_the_host_builder():
    """Every host allocation point of the builder, made to fail in turn by
    the test hook, returns DBS_ERR_OOM (and the process stays usable); with
    the hook past the last allocation the build succeeds unchanged."""
    A = synth.config("llm", "small")
    ref = _host(A).export_raw("blk_desc")
    fired = 0
    for k in range(200):
        _fail_alloc(k)
        try:
            M = _host(A, num_threads=2)
        except dbs.DbsError as e:
            assert e.status == 2, e              # DBS_ERR_OOM
            assert _fail_alloc(-1) == -1         # the hook fired
            fired += 1
            continue
        left = _fail_alloc(-1)
        assert left >= 0                          # not reached: every point was covered
        np.testing.assert_array_equal(M.export_raw("blk_desc"), ref)
        break
    else:
        raise AssertionError("the build never got past the injected failures")
    assert fired >= 4
