"""Seeded synthetic workloads for the SpMSpV library and its oracle.

This package only *draws* inputs (sparsity patterns, values, sparse vectors,
BFS sources).  It holds none of the SpMSpV arithmetic, so both the CUDA path
and the CPU oracle can consume its output without sharing any method code.
"""
from .workloads import (  # noqa: F401
    CSR,
    SparseVec,
    csr_from_coo,
    csr_to_dense,
    er_matrix,
    rmat_graph,
    fem_stencil,
    llm_weight,
    grid_hubs,
    x_uniform,
    x_clusters,
    x_relu_topk,
    x_activation,
    bfs_sources,
    random_csr,
    config,
    CONFIG_NAMES,
)
