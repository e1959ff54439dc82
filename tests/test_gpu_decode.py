"""GPU parity of the DB-Decoding layer (dbs_decode_layer): y = A x' with x'
the activation thresholded by magnitude, against the oracle's decode_layer.
Rows reached by an active entry must meet the fp32 tolerance
|y - y_ref| <= 1e-5 * sum |a x| + 1e-30; every other row must be exactly 0."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import __graft_entry__  # noqa: E402

__graft_entry__.build()
import dynamic_sparsity_spmspv_gb300 as dbs  # noqa: E402
from test_gpu_parity import _block_diag  # noqa: E402

DEV = "cuda"


def check(O, x, tau, y):
    ref, s, t = O.decode_layer(x, tau)
    y = y.cpu().numpy() if hasattr(y, "cpu") else y
    assert oracle.tolerance_ok(y[t], ref[t], s[t]).all()
    assert (y[~t] == 0).all()


def run(M, ws, x, tau):
    xt = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(DEV)
    y = dbs.decode_layer(M, xt, tau, ws=ws)
    assert ws.check() == 0
    return y


@pytest.mark.parametrize("name", ["llm", "er", "fem"])
def test_decode_small(name):
    A = synth.config(name, "small")
    O, M = oracle.Oracle(A), dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    rng = np.random.default_rng(5)
    for tau in (0.0, 0.5, 1.6449, 3.0, 1e9):
        for _ in range(3):
            x = rng.standard_normal(A.n).astype(np.float32)
            x[rng.random(A.n) < 0.3] = 0.0
            check(O, x, tau, run(M, ws, x, tau))


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
def test_decode_forced_formats_and_local_modes(fmt):
    A = synth.config("llm", "small")
    O, M = oracle.Oracle(A), dbs.DBMatrix.from_csr(A, force_format=fmt, tile_weight=24)
    ws = dbs.Workspace(M)
    rng = np.random.default_rng(fmt)
    for lp in (0, 8, 17):
        ws.set_opts(dbs.exec_opts(local_pull_min=lp))
        for tau in (0.0, 1.2):
            x = rng.standard_normal(A.n).astype(np.float32)
            check(O, x, tau, run(M, ws, x, tau))


def test_decode_every_block_mask():
    """All 2^16 activation masks against one dense-ish block pattern (copy k
    of the block on the diagonal meets x-block mask k); tau = 0."""
    rng = np.random.default_rng(11)
    pattern = rng.random((16, 16)) < 0.6
    A = _block_diag(pattern, 1 << 16, 3)
    k = np.arange(1 << 16)
    bits = ((k[:, None] >> np.arange(16)[None, :]) & 1).astype(bool)
    x = np.where(bits.ravel(), rng.uniform(0.5, 1.5, bits.size), 0.0).astype(np.float32)
    O = oracle.Oracle(A)
    for fmt in (1, 3, 4):
        M = dbs.DBMatrix.from_csr(A, force_format=fmt)
        check(O, x, 0.0, run(M, dbs.Workspace(M), x, 0.0))


@pytest.mark.parametrize("m,n", [(1, 1), (17, 33), (250, 1000), (1000, 250), (4099, 4111)])
def test_decode_ragged_and_empty_rows(m, n):
    """Sizes that are not multiples of 16 (ragged row and column tails),
    empty rows and empty row blocks; repeated calls into the same output
    (every row is rewritten on every call, stale values included)."""
    rng = np.random.default_rng(m * 7 + n)
    A = synth.random_csr(m, n, 0.05, m + n)
    keep = rng.random(m) < 0.7
    keep[(np.arange(m) // 16) % 5 == 3] = False           # whole empty row blocks
    rows = np.repeat(np.arange(m), np.diff(A.row_ptr))
    sel = keep[rows]
    A = synth.csr_from_coo(m, n, rows[sel], A.col_idx[sel], A.vals[sel])
    O, M = oracle.Oracle(A), dbs.DBMatrix.from_csr(A, tile_weight=16)
    ws = dbs.Workspace(M)
    y = torch.full((m,), 7.0, dtype=torch.float32, device=DEV)      # stale values must be overwritten
    for i in range(4):
        x = rng.standard_normal(n).astype(np.float32)
        dbs.decode_layer(M, torch.from_numpy(x).to(DEV), 0.7, y=y, ws=ws)
        assert ws.check() == 0
        check(O, x, 0.7, y)


@pytest.mark.parametrize("fmt", [-1, 0, 1, 2, 3, 4])
def test_decode_long_row_blocks(fmt):
    """Row blocks of more than one round of the kernel (over 1,024 blocks:
    the (block, column) pair list is refilled per round) with every column
    of a block active (16 pairs per block at tau = 0), in every format."""
    rng = np.random.default_rng(40 + fmt)
    m, n = 45, 16 * 2100 + 5
    dense = rng.random((m, n)) < 0.35
    rows, cols = np.nonzero(dense)
    A = synth.csr_from_coo(m, n, rows, cols.astype(np.int32), rng.standard_normal(rows.size).astype(np.float32))
    O = oracle.Oracle(A)
    M = dbs.DBMatrix.from_csr(A, force_format=fmt)
    ws = dbs.Workspace(M)
    assert M.info()["nblocks"] > 3 * 2 * 1024
    for tau in (0.0, 0.9):
        x = rng.standard_normal(n).astype(np.float32)
        check(O, x, tau, run(M, ws, x, tau))


def test_decode_interleaved_with_other_calls():
    """The accumulator the decoding layer borrows stays clean for sparse-x
    calls on the same workspace, and the other way round."""
    A = synth.config("llm", "small")
    O, M = oracle.Oracle(A), dbs.DBMatrix.from_csr(A, tile_weight=16)
    ws = dbs.Workspace(M)
    rng = np.random.default_rng(3)
    for i in range(4):
        x = rng.standard_normal(A.n).astype(np.float32)
        check(O, x, 1.0, run(M, ws, x, 1.0))
        xs = synth.x_uniform(A.n, 40, [31, i])
        yi, yv, yn = dbs.spmspv(M, torch.from_numpy(xs.idx).to(DEV), torch.from_numpy(xs.val).to(DEV), ws=ws)
        k = int(yn.item())
        ri, rv, rs = O.spmspv(xs)
        np.testing.assert_array_equal(yi[:k].cpu().numpy(), ri)
        assert oracle.tolerance_ok(yv[:k].cpu().numpy(), rv, rs).all()


def test_decode_argument_errors():
    A = synth.config("llm", "small")
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    x = torch.zeros(A.n + 4, dtype=torch.float32, device=DEV)
    for bad in (-0.5, float("nan")):
        with pytest.raises(dbs.DbsError):
            dbs.decode_layer(M, x[:A.n], bad, ws=ws)
    with pytest.raises(dbs.DbsError):
        dbs.decode_layer(M, x[1:A.n + 1], 0.5, ws=ws)                 # not 16-byte aligned
    P = synth.config("rmat", "small")
    Mp = dbs.DBMatrix.from_csr(P)
    with pytest.raises(dbs.DbsError):
        dbs.decode_layer(Mp, torch.zeros(P.n, dtype=torch.float32, device=DEV), 0.0, ws=dbs.Workspace(Mp))


def test_decode_graph_replay_layer_stack():
    """Four distinct layers captured once in a CUDA graph and replayed with
    new activations copied into the captured input buffers."""
    layers = [synth.llm_weight(96, 300, seed=60 + i) for i in range(4)]
    Os = [oracle.Oracle(A) for A in layers]
    Ms = [dbs.DBMatrix.from_csr(A, tile_weight=20) for A in layers]
    wss = [dbs.Workspace(M) for M in Ms]
    xs = [torch.zeros(A.n, dtype=torch.float32, device=DEV) for A in layers]
    ys = [torch.empty(A.m, dtype=torch.float32, device=DEV) for A in layers]

    def step():
        for M, ws, x, y in zip(Ms, wss, xs, ys):
            dbs.decode_layer(M, x, 1.0, y=y, ws=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    rng = np.random.default_rng(9)
    for _ in range(4):
        hs = [rng.standard_normal(A.n).astype(np.float32) for A in layers]
        for x, h in zip(xs, hs):
            x.copy_(torch.from_numpy(h))
        g.replay()
        torch.cuda.synchronize()
        for O, h, y in zip(Os, hs, ys):
            check(O, h, 1.0, y)
