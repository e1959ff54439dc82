"""Seeded generators for the five synthetic workloads and their sparse vectors.

Every generator is deterministic in its ``seed`` (numpy PCG64).  Matrices come
out as CSR with int64 row pointers, int32 column indices sorted and unique
within each row, and either float32 values or ``None`` (pattern only, used with
the Boolean semiring).  Sparse vectors come out as sorted unique int32 indices
plus float32 values (or ``None``).

Workload recipes (shapes follow the DB-SpMSpV paper's evaluation, section 5:
SuiteSparse FEM and graph matrices, R-MAT-like social graphs, BFS frontiers and
single-token LLM linear layers; the real datasets are replaced by these
synthetic stand-ins):

* ``er``     Erdos-Renyi square matrix, fixed count of distinct uniform columns
             per row, values U[-1, 1].
* ``rmat``   R-MAT graph (a, b, c, d quadrant probabilities, no noise, no
             relabelling), symmetrised, self-loops and duplicates removed,
             pattern only.
* ``fem``    27-point stencil on a g^3 grid, rows randomly permuted within
             aligned windows, values N(0, 1).
* ``llm``    pruned linear-layer weight: a fixed count of uniformly chosen kept
             columns per row, values N(0, std).
* ``grid``   2-D 4-neighbour grid with a fraction of edges deleted, plus hub
             vertices each wired to uniform random targets, pattern only.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass
class CSR:
    m: int
    n: int
    row_ptr: np.ndarray          # int64[m + 1]
    col_idx: np.ndarray          # int32[nnz]
    vals: Optional[np.ndarray]   # float32[nnz] or None (pattern only)

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])


@dataclasses.dataclass
class SparseVec:
    n: int
    idx: np.ndarray              # int32[k], sorted unique
    val: Optional[np.ndarray]    # float32[k] or None (all listed entries active)

    @property
    def k(self) -> int:
        return int(self.idx.shape[0])


def _rng(*seed) -> np.random.Generator:
    return np.random.default_rng(list(seed))


def csr_from_coo(m: int, n: int, rows, cols, vals=None, *, dedupe: bool = False) -> CSR:
    """Sort (row, col) pairs into CSR.  With ``dedupe`` repeated pairs collapse
    to one (the first value in sorted order is kept)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    key = rows * np.int64(n) + cols
    order = np.argsort(key, kind="stable")
    key = key[order]
    if vals is not None:
        vals = np.asarray(vals, dtype=np.float32)[order]
    if dedupe and key.size:
        keep = np.empty(key.shape, dtype=bool)
        keep[0] = True
        np.not_equal(key[1:], key[:-1], out=keep[1:])
        key = key[keep]
        if vals is not None:
            vals = vals[keep]
    r = key // n
    c = (key - r * n).astype(np.int32)
    counts = np.bincount(r, minlength=m).astype(np.int64)
    row_ptr = np.zeros(m + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    return CSR(m, n, row_ptr, c, vals)


def csr_to_dense(A: CSR, dtype=np.float64) -> np.ndarray:
    """Dense copy (pattern-only matrices become 0/1).  Small inputs only."""
    D = np.zeros((A.m, A.n), dtype=dtype)
    rows = np.repeat(np.arange(A.m), np.diff(A.row_ptr))
    D[rows, A.col_idx] = 1.0 if A.vals is None else A.vals.astype(dtype)
    return D


def _distinct_per_row(rng, m: int, n: int, k: int) -> np.ndarray:
    """k distinct uniform columns per row, sorted (m x k)."""
    out = np.empty((m, k), dtype=np.int32)
    step = max(1, (1 << 24) // max(n, 1))
    for r0 in range(0, m, step):
        r1 = min(m, r0 + step)
        keys = rng.random((r1 - r0, n), dtype=np.float32)
        sel = np.argpartition(keys, k - 1, axis=1)[:, :k] if k < n else np.tile(np.arange(n), (r1 - r0, 1))
        out[r0:r1] = np.sort(sel, axis=1)
    return out


def er_matrix(n: int = 4096, per_row: int = 8, seed: int = 43) -> CSR:
    rng = _rng(seed, 0)
    cols = _distinct_per_row(rng, n, n, per_row)
    row_ptr = np.arange(0, n * per_row + 1, per_row, dtype=np.int64)
    vals = rng.uniform(-1.0, 1.0, n * per_row).astype(np.float32)
    return CSR(n, n, row_ptr, cols.reshape(-1), vals)


def _sorted_unique(a: np.ndarray) -> np.ndarray:
    a = np.sort(a)
    if a.size == 0:
        return a
    keep = np.empty(a.shape, dtype=bool)
    keep[0] = True
    np.not_equal(a[1:], a[:-1], out=keep[1:])
    return a[keep]


def _symmetric_pattern(nv: int, u: np.ndarray, v: np.ndarray) -> CSR:
    u = np.asarray(u, dtype=np.int64)
    v = np.asarray(v, dtype=np.int64)
    keep = u != v
    u, v = u[keep], v[keep]
    key = _sorted_unique(np.concatenate([u * nv + v, v * nv + u]))
    r = key // nv
    c = (key - r * nv).astype(np.int32)
    counts = np.bincount(r, minlength=nv).astype(np.int64)
    row_ptr = np.zeros(nv + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    return CSR(nv, nv, row_ptr, c, None)


def rmat_graph(scale: int = 20, edge_factor: int = 16, abcd=(0.57, 0.19, 0.19, 0.05),
               seed: int = 44) -> CSR:
    rng = _rng(seed, 0)
    nv = 1 << scale
    ne = edge_factor * nv
    a, b, c, _ = abcd
    t1, t2, t3 = a, a + b, a + b + c
    u = np.zeros(ne, dtype=np.int64)
    v = np.zeros(ne, dtype=np.int64)
    for lvl in range(scale):
        r = rng.random(ne, dtype=np.float32)
        row_bit = r >= t2
        col_bit = ((r >= t1) & (r < t2)) | (r >= t3)
        bit = np.int64(1) << np.int64(scale - 1 - lvl)
        u |= row_bit.astype(np.int64) * bit
        v |= col_bit.astype(np.int64) * bit
    return _symmetric_pattern(nv, u, v)


def fem_stencil(g: int = 128, window: int = 4096, seed: int = 45) -> CSR:
    rng = _rng(seed, 0)
    n = g * g * g
    r = np.arange(n, dtype=np.int64)
    z, y, x = r // (g * g), (r // g) % g, r % g
    cols = np.full((n, 27), -1, dtype=np.int32)
    k = 0
    for dz in (-1, 0, 1):
        for dy in (-1, 0, 1):
            for dx in (-1, 0, 1):
                ok = ((z + dz >= 0) & (z + dz < g) & (y + dy >= 0) & (y + dy < g)
                      & (x + dx >= 0) & (x + dx < g))
                cols[ok, k] = (r[ok] + dz * g * g + dy * g + dx).astype(np.int32)
                k += 1
    mask = cols >= 0
    counts = mask.sum(axis=1).astype(np.int64)
    flat = cols[mask]
    old_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=old_ptr[1:])
    del cols, mask
    perm = np.empty(n, dtype=np.int64)
    for w0 in range(0, n, window):
        w1 = min(n, w0 + window)
        perm[w0:w1] = w0 + rng.permutation(w1 - w0)
    new_counts = counts[perm]
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(new_counts, out=row_ptr[1:])
    nnz = int(row_ptr[-1])
    src = np.repeat(old_ptr[:-1][perm] - row_ptr[:-1], new_counts) + np.arange(nnz, dtype=np.int64)
    col_idx = flat[src]
    vals = rng.standard_normal(nnz, dtype=np.float32)
    return CSR(n, n, row_ptr, col_idx, vals)


def llm_weight(m: int = 4096, n: int = 11008, keep_per_row: Optional[int] = None,
               std: float = 0.02, seed: int = 46) -> CSR:
    rng = _rng(seed, 0)
    k = n // 2 if keep_per_row is None else keep_per_row
    cols = _distinct_per_row(rng, m, n, k)
    row_ptr = np.arange(0, m * k + 1, k, dtype=np.int64)
    vals = (rng.standard_normal(m * k, dtype=np.float32) * np.float32(std)).astype(np.float32)
    return CSR(m, n, row_ptr, cols.reshape(-1), vals)


def grid_hubs(side: int = 4096, delete_frac: float = 0.10, n_hubs: int = 1000,
              hub_deg: int = 20000, seed: int = 47) -> CSR:
    rng = _rng(seed, 0)
    nv = side * side
    rr, cc = np.meshgrid(np.arange(side, dtype=np.int64), np.arange(side - 1, dtype=np.int64),
                         indexing="ij")
    h_u = (rr * side + cc).reshape(-1)
    h_v = h_u + 1
    v_u = (cc * side + rr).reshape(-1)
    v_v = v_u + side
    del rr, cc
    eu = np.concatenate([h_u, v_u])
    ev = np.concatenate([h_v, v_v])
    del h_u, h_v, v_u, v_v
    n_del = int(round(delete_frac * eu.shape[0]))
    keep = rng.permutation(eu.shape[0])[n_del:]
    eu, ev = eu[keep], ev[keep]
    if n_hubs > 0:
        hubs = rng.choice(nv, size=n_hubs, replace=False).astype(np.int64)
        tgt = rng.integers(0, nv, size=(n_hubs, hub_deg), dtype=np.int64)
        eu = np.concatenate([eu, np.repeat(hubs, hub_deg)])
        ev = np.concatenate([ev, tgt.reshape(-1)])
    return _symmetric_pattern(nv, eu, ev)


def random_csr(m: int, n: int, density: float, seed: int, *, valued: bool = True,
               integer_values: bool = False) -> CSR:
    """Uniform random pattern of the given density (small test inputs)."""
    rng = _rng(seed, 1)
    total = m * n
    k = int(round(density * total))
    flat = rng.choice(total, size=k, replace=False) if k else np.zeros(0, dtype=np.int64)
    rows, cols = np.divmod(np.asarray(flat, dtype=np.int64), n)
    vals = None
    if valued:
        if integer_values:
            v = rng.integers(-3, 4, size=k)
            v[v == 0] = 1
            vals = v.astype(np.float32)
        else:
            vals = rng.uniform(-1.0, 1.0, size=k).astype(np.float32)
    return csr_from_coo(m, n, rows, cols, vals)


def x_uniform(n: int, k: int, seed, *, valued: bool = True, integer_values: bool = False) -> SparseVec:
    """k distinct uniform indices; values U[-1, 1] (or small integers), or None."""
    rng = _rng(*np.atleast_1d(seed).tolist(), 2)
    k = min(k, n)
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.int32) if k else np.zeros(0, np.int32)
    val = None
    if valued:
        if integer_values:
            v = rng.integers(-3, 4, size=k)
            v[v == 0] = -1
            val = v.astype(np.float32)
        else:
            val = rng.uniform(-1.0, 1.0, size=k).astype(np.float32)
    return SparseVec(n, idx, val)


def x_clusters(n: int, frac: float, seed, cluster: int = 64, *, valued: bool = True) -> SparseVec:
    """round(frac*n/cluster) runs of `cluster` consecutive indices at uniform
    offsets in [0, n - cluster]; overlapping runs merge."""
    rng = _rng(*np.atleast_1d(seed).tolist(), 3)
    c = int(round(frac * n / cluster))
    starts = rng.integers(0, n - cluster + 1, size=c)
    idx = _sorted_unique((starts[:, None] + np.arange(cluster)[None, :]).reshape(-1)).astype(np.int32)
    val = rng.uniform(-1.0, 1.0, size=idx.shape[0]).astype(np.float32) if valued else None
    return SparseVec(n, idx, val)


def x_relu_topk(n: int, keep: int, seed) -> np.ndarray:
    """Dense activation: N(0, 1) draws with all but the `keep` largest zeroed."""
    rng = _rng(*np.atleast_1d(seed).tolist(), 4)
    v = rng.standard_normal(n, dtype=np.float32)
    out = np.zeros(n, dtype=np.float32)
    if keep > 0:
        top = np.argpartition(-v, keep - 1)[:keep]
        out[top] = v[top]
    return out


def x_activation(n: int, seed) -> np.ndarray:
    """Dense pre-threshold activation of a decoding layer: N(0, 1) float32
    (magnitude thresholding at 1.6449 keeps about 10 % of the entries)."""
    rng = _rng(*np.atleast_1d(seed).tolist(), 5)
    return rng.standard_normal(n, dtype=np.float32)


def bfs_sources(A: CSR, k: int, seed) -> np.ndarray:
    """k distinct uniform sources among vertices with at least one neighbour."""
    rng = _rng(*np.atleast_1d(seed).tolist(), 5)
    deg = np.diff(A.row_ptr)
    cand = np.nonzero(deg > 0)[0]
    k = min(k, cand.shape[0])
    return np.sort(rng.choice(cand, size=k, replace=False)).astype(np.int64)


# ----------------------------------------------------------------------------
# Named workloads.  "full" is the size the paper-shaped benchmark uses; "small"
# keeps the same structure at a size the CPU oracle finishes in seconds while
# still spanning many 16x16 blocks, several tiles and ragged tails.

CONFIG_NAMES = ("er", "rmat", "fem", "llm", "grid")


def config(name: str, size: str = "full") -> CSR:
    full = size == "full"
    if name == "er":
        return er_matrix(4096 if full else 1000, 8, seed=43)
    if name == "rmat":
        return rmat_graph(20 if full else 12, 16, seed=44)
    if name == "fem":
        return fem_stencil(128 if full else 18, 4096 if full else 512, seed=45)
    if name == "llm":
        return llm_weight(4096 if full else 200, 11008 if full else 700, seed=46)
    if name == "grid":
        if full:
            return grid_hubs(4096, 0.10, 1000, 20000, seed=47)
        return grid_hubs(90, 0.10, 6, 300, seed=47)
    raise ValueError(f"unknown workload {name!r}")
