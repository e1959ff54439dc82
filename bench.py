#!/usr/bin/env python
"""Benchmark of the DB-SpMSpV hot path on one GB300 (or N replicas).

Workload (default): R-MAT scale 20 (2^20 vertices, edge factor 16, a/b/c/d =
.57/.19/.19/.05), symmetrised, duplicates and self-loops removed, pattern
only.  One step = one Boolean SpMSpV at each input density in
{0.01%, 0.1%, 1%, 10%, 50%} (auto push/pull) + one DB-BFS from the next of 16
random non-isolated sources.  Inputs are resident in HBM before timing; L2 is
flushed (256 MiB write) before every call, outside the timed regions; every
call is timed with CUDA events on its stream.

Metric: touched nnz per second (nnz of the matrix blocks whose column block
is active in x, summed over the step's SpMSpV calls and BFS levels).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same workload on its own GPU (replicas, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DENSITIES = (1e-4, 1e-3, 1e-2, 1e-1, 5e-1)
N_SOURCES = 16
POOL = 32                      # distinct x per density, cycled over the steps
FLUSH_BYTES = 256 << 20        # > 2x the 129 MB L2
METRIC = "SpMSpV touched-nnz/s and HBM GB/s vs input density (1 GB300); DB-BFS GTEPS"
UNIT = "touched-nnz/s"
WORKLOAD = ("rmat-s20-ef16 (2^20 vertices, a/b/c/d .57/.19/.19/.05, symmetrised, pattern only); "
            "Boolean SpMSpV at x density 0.01%/0.1%/1%/10%/50% + DB-BFS from 16 sources")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("kernels.cu", "format.h"):
        with open(os.path.join(ROOT, "dynamic_sparsity_spmspv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the kernel sources changed since it was captured."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic_rmat_s20.json")) as f:
            d = json.load(f)
        if d.get("kernel_source_sha256") != _kernel_source_hash():
            return None
        return d["traffic_bytes_per_launch"][kernel]["mean"]
    except Exception:
        return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons of this process's GPU, matched
    by UUID (indices differ when CUDA_VISIBLE_DEVICES remaps devices)."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.uuid = None
        try:
            import torch
            u = str(torch.cuda.get_device_properties(device).uuid)
            self.uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        self.p = None

    def start(self):
        if self.uuid is None:
            return
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out = ""
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9 or f[0].lower() != self.uuid.lower():
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "gpu_uuid": self.uuid}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None, "gpu_uuid": self.uuid}


def build_workload(scale: int, seed_tag: int):
    import synth
    A = synth.config("rmat", "full") if scale == 20 else synth.rmat_graph(scale, 16, seed=44)
    xs = {}
    for d in DENSITIES:
        k = max(1, int(round(d * A.n)))
        xs[d] = [synth.x_uniform(A.n, k, [44, seed_tag, int(d * 1e6), i], valued=False) for i in range(POOL)]
    sources = synth.bfs_sources(A, N_SOURCES, [44, 7])
    return A, xs, sources


class TouchedCounter:
    """touched nnz = sum of nnz over the blocks whose column block holds an
    active x entry; a BFS level touches the blocks of its frontier's column
    blocks.  Independent of the path taken."""

    def __init__(self, views):
        nbc = len(views["blk_col_ptr"]) - 1
        self.nbc = nbc
        self.per_cb = np.zeros(nbc, np.int64)
        np.add.at(self.per_cb, views["blk_col_idx"], views["blk_nnz"].astype(np.int64))

    def spmspv(self, idx) -> int:
        act = np.zeros(self.nbc, bool)
        act[np.asarray(idx) // 16] = True
        return int(self.per_cb[act].sum())

    def bfs(self, levels) -> int:
        reached = np.nonzero(levels >= 0)[0]
        lv = levels[reached]
        cb = reached // 16
        key = np.sort(lv.astype(np.int64) * self.nbc + cb)       # (level, column block) pairs
        if key.size:
            key = key[np.r_[True, key[1:] != key[:-1]]]
        return int(self.per_cb[key % self.nbc].sum())


def _host_cores() -> int:
    """Cores this process may run on (the oracle itself uses one)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(A, xs, sources, touched_x, touched_bfs, budget_s: float):
    """The oracle as it stands, single-threaded, on a bounded sample of the
    same step (densities cycled, then BFS sources); beside it the all-cores
    baseline -- the row-partitioned plain pull (Algorithm 1, bottom) and a
    pull-based level-synchronous BFS on OpenMP threads -- on its own sample
    of the same steps."""
    import oracle
    O = oracle.Oracle(A)

    def run(spmspv, bfs, budget):
        t_total, units, calls, bfs_runs, i = 0.0, 0, 0, 0, 0
        while t_total < budget and i < POOL:
            for d in DENSITIES:
                x = xs[d][i]
                t0 = time.perf_counter()
                spmspv(x)
                t_total += time.perf_counter() - t0
                units += touched_x[d][i]
                calls += 1
            src = int(sources[i % len(sources)])
            t0 = time.perf_counter()
            bfs(src)
            t_total += time.perf_counter() - t0
            units += touched_bfs[i % len(sources)]
            bfs_runs += 1
            i += 1
        return units / t_total, i, calls, bfs_runs, t_total

    v1, i1, c1, b1, t1 = run(lambda x: O.spmspv(x, oracle.OR_AND), O.bfs_queue, budget_s * 0.7)
    threads = oracle.par_threads()
    vp, ip, cp, bp, tp = run(lambda x: oracle.spmspv_pull_par(A, x, oracle.OR_AND),
                             lambda s: oracle.bfs_pull_par(A, s), budget_s * 0.3)
    return {"value": v1, "unit": UNIT, "cores": 1, "host_cores_available": _host_cores(), "kind": "oracle",
            "sample": f"{i1} steps: {c1} oracle SpMSpV calls (push scatter, fp64 C, 1 thread) at the 5 densities "
                      f"+ {b1} queue BFS; {t1:.1f} s of CPU time; units = the same touched nnz",
            "all_cores": {"value": vp, "unit": UNIT, "cores": threads, "kind": "oracle pull, OpenMP rows",
                          "sample": f"{ip} steps: {cp} row-parallel pulls (Algorithm 1 bottom, fp64 C, {threads} "
                                    f"threads) at the 5 densities + {bp} level-synchronous pull BFS; "
                                    f"{tp:.1f} s of wall time"}}


def reduce_over_ranks(t_ms: float, units: float, device):
    """Whole-job totals of a replicated run: the slowest rank's timed
    milliseconds and the units all ranks processed (one all-reduce each,
    on whatever process group is initialised)."""
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(t_ms)], device=device, dtype=torch.float64)
    uu = torch.tensor([float(units)], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    dist.all_reduce(uu, op=dist.ReduceOp.SUM)
    return float(tt.item()), float(uu.item())


def config_dict(world: int, n: int, nnz: int, blocks: int) -> dict:
    """The workload description both arms print (the same dict)."""
    return {"workload": WORKLOAD, "densities": list(DENSITIES), "bfs_sources": N_SOURCES,
            "x_pool_per_density": POOL,
            "l2": "GPU arm: flushed (256 MiB write) before every call, outside timing",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "matrix": {"n": int(n), "nnz": int(nnz), "blocks": int(blocks)}}


def run_reference(args):
    """--impl reference: the CPU oracle timed on this host's cores, on the
    same step as the GPU arm (one Boolean SpMSpV at each of the five
    densities plus one BFS from the next source)."""
    ws_, rank, _ = _dist()
    if rank != 0:
        return
    A, xs, sources = build_workload(args.scale, 0)
    import oracle
    O = oracle.Oracle(A)
    views = oracle.block_views(A)
    counter = TouchedCounter(views)
    steps_total = args.warmup + args.steps
    t_step, units = [], []
    for s in range(steps_total):
        i = s % POOL
        u = 0
        t0 = time.perf_counter()
        for d in DENSITIES:
            O.spmspv(xs[d][i], oracle.OR_AND)
        lev = O.bfs_queue(int(sources[s % N_SOURCES]))
        dt = time.perf_counter() - t0
        u = sum(counter.spmspv(xs[d][i].idx) for d in DENSITIES) + counter.bfs(lev)
        if s >= args.warmup:
            t_step.append(dt)
            units.append(u)
    T = sum(t_step)
    value = sum(units) / T
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * T / len(t_step), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bool", "data": "synthetic",
            "config": config_dict(ws_, A.n, A.nnz, views["B"]),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores_available": _host_cores(),
                             "kind": "oracle",
                             "sample": f"{args.steps} steps, each one oracle SpMSpV at each of the 5 densities "
                                       "plus one queue BFS (the GPU arm's step); fp64 C, 1 thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


ABLATION_FORMATS = (("auto", -1), ("coo", 0), ("force_csr", 2))


def run_configs(dbs, torch, dev, stream, flush, reps: int):
    """The other workloads at full size, default options (auto path): ER and
    FEM plus-times SpMSpV, the LLM layer with dense and sparse activations,
    FEM and LLM density sweeps with each path forced, and BFS on the grid
    with hubs and on the grid without hubs.  Per line: median kernel µs over `reps`
    calls (L2 flushed before each), touched nnz and algorithmic bytes from
    one statistics call per input, touched-nnz/s, GB/s, share of HBM."""
    import synth
    peak, _ = _peaks()
    lines = []

    def timed(call, i):
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3

    def measure(name, mode, M, ws, calls, extra):
        touched = bytes_alg = 0
        paths = set()
        ws.set_opts(dbs.exec_opts(collect_stats=1))
        for c in calls:
            c()
            st = ws.stats()
            touched += st["touched_nnz"]
            bytes_alg += st["bytes_alg"]
            paths.add({0: "-", 1: "push", 2: "pull"}.get(st["path"], "?"))
        ws.set_opts(dbs.exec_opts(collect_stats=0))
        for i in range(2):
            timed(calls[i % len(calls)], i)
        ts = [timed(calls[i % len(calls)], i) for i in range(reps)]
        us = float(np.median(ts))
        t_nnz, b_alg = touched / len(calls), bytes_alg / len(calls)
        line = {"workload": name, "mode": mode, "path": "/".join(sorted(paths)), "us": round(us, 2),
                "bytes_alg": round(b_alg), "touched_nnz_per_s": round(t_nnz / us * 1e6), "gbs": round(b_alg / us / 1e3, 1),
                "frac_of_measured_hbm": round(b_alg / us / 1e3 / peak, 4)}
        line.update(extra)
        lines.append(line)

    # ER, plus-times, 1 % active
    A = synth.config("er", "full")
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    y_idx = torch.empty(A.m, dtype=torch.int32, device=dev)
    y_val = torch.empty(A.m, dtype=torch.float32, device=dev)
    y_nnz = torch.empty(1, dtype=torch.int64, device=dev)
    xs = [synth.x_uniform(A.n, 41, [43, i]) for i in range(8)]
    xt = [(torch.from_numpy(x.idx).to(dev), torch.from_numpy(x.val).to(dev)) for x in xs]
    measure("er", "spmspv x 1%", M, ws, [lambda xi=xi, xv=xv: dbs.spmspv(M, xi, xv, ws=ws, y_idx=y_idx, y_val=y_val,
                                                                          y_nnz=y_nnz) for xi, xv in xt], {})
    ws.close(); M.close()

    # FEM, plus-times, clustered x
    A = synth.config("fem", "full")
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    y_idx = torch.empty(A.m, dtype=torch.int32, device=dev)
    y_val = torch.empty(A.m, dtype=torch.float32, device=dev)
    for f in (0.001, 0.01, 0.1):
        xs = [synth.x_clusters(A.n, f, [45, int(f * 1e4), i]) for i in range(4)]
        xt = [(torch.from_numpy(x.idx).to(dev), torch.from_numpy(x.val).to(dev)) for x in xs]
        measure("fem", f"spmspv x {f:g}", M, ws,
                [lambda xi=xi, xv=xv: dbs.spmspv(M, xi, xv, ws=ws, y_idx=y_idx, y_val=y_val, y_nnz=y_nnz)
                 for xi, xv in xt], {"density": f})
    # density sweep with both paths forced (blocks of ~3 stored entries with
    # values, against R-MAT's inline pattern blocks); from 10 % up each path
    # moves more than 64 MB, the size at which the roofline fraction is judged
    for f in (0.001, 0.01, 0.1, 0.2, 0.5):
        xs = [synth.x_clusters(A.n, f, [45, int(f * 1e4), i]) for i in range(4)]
        xt = [(torch.from_numpy(x.idx).to(dev), torch.from_numpy(x.val).to(dev)) for x in xs]
        for path in ("push", "pull"):
            measure("fem", f"spmspv x {f:g}, {path} forced", M, ws,
                    [lambda xi=xi, xv=xv, path=path: dbs.spmspv(M, xi, xv, ws=ws, path=path, y_idx=y_idx,
                                                                y_val=y_val, y_nnz=y_nnz) for xi, xv in xt],
                    {"density": f, "forced": path})
    ws.close(); M.close()

    # LLM layer: dense activations (decoding form) and the same as a sparse x
    A = synth.config("llm", "full")
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    y = torch.empty(A.m, dtype=torch.float32, device=dev)
    y_idx = torch.empty(A.m, dtype=torch.int32, device=dev)
    y_val = torch.empty(A.m, dtype=torch.float32, device=dev)
    xds = [synth.x_relu_topk(A.n, 1101, [46, t]) for t in range(8)]
    xdt = [torch.from_numpy(xd).to(dev) for xd in xds]
    measure("llm", "dense x (10% nonzero)", M, ws, [lambda x=x: dbs.spmspv_dense(M, x, y=y, ws=ws) for x in xdt], {})
    sp = []
    for xd in xds:
        nz = np.nonzero(xd)[0].astype(np.int32)
        sp.append((torch.from_numpy(nz).to(dev), torch.from_numpy(xd[nz]).to(dev)))
    measure("llm", "sparse x (1,101 entries)", M, ws,
            [lambda xi=xi, xv=xv: dbs.spmspv(M, xi, xv, ws=ws, y_idx=y_idx, y_val=y_val, y_nnz=y_nnz)
             for xi, xv in sp], {})
    # density sweep of uniform sparse x with both paths forced (Dense and
    # patched-CSR blocks of ~128 entries)
    for f in (0.001, 0.01, 0.1, 0.5):
        xs = [synth.x_uniform(A.n, max(1, int(round(f * A.n))), [47, int(f * 1e4), i]) for i in range(4)]
        xt = [(torch.from_numpy(x.idx).to(dev), torch.from_numpy(x.val).to(dev)) for x in xs]
        for path in ("push", "pull"):
            measure("llm", f"spmspv x {f:g}, {path} forced", M, ws,
                    [lambda xi=xi, xv=xv, path=path: dbs.spmspv(M, xi, xv, ws=ws, path=path, y_idx=y_idx,
                                                                y_val=y_val, y_nnz=y_nnz) for xi, xv in xt],
                    {"density": f, "forced": path})
    ws.close(); M.close()

    # grid with hubs: BFS
    A = synth.config("grid", "full")
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    levels = torch.empty(A.n, dtype=torch.int32, device=dev)
    deg = np.diff(A.row_ptr)
    srcs = synth.bfs_sources(A, 8, [47, 7])
    ts, teps, nls = [], [], []
    for i, src in enumerate(srcs):
        timed(lambda: dbs.bfs(M, int(src), levels=levels, ws=ws, sync=False), i)   # warm-up
        t = timed(lambda: dbs.bfs(M, int(src), levels=levels, ws=ws, sync=False), i)
        lv = levels.cpu().numpy()
        edges = int(deg[lv >= 0].sum()) // 2
        ts.append(t)
        teps.append(edges / t * 1e6 / 1e9)
        nls.append(int(lv.max()) + 1)
    lines.append({"workload": "grid", "mode": "bfs (8 sources)", "us": round(float(np.median(ts)), 2),
                  "gteps_harmonic": round(len(teps) / sum(1.0 / v for v in teps), 3),
                  "levels_mean": float(np.mean(nls))})
    assert ws.check() == 0
    ws.close(); M.close()

    # the same grid without hubs: thousands of levels with small frontiers
    # (the long-diameter regime), four sources
    A = synth.grid_hubs(4096, 0.10, 0, 0, seed=47)
    M = dbs.DBMatrix.from_csr(A)
    ws = dbs.Workspace(M)
    levels = torch.empty(A.n, dtype=torch.int32, device=dev)
    deg = np.diff(A.row_ptr)
    ts, teps, nls = [], [], []
    for i, src in enumerate(synth.bfs_sources(A, 4, [48, 7])):
        t = timed(lambda: dbs.bfs(M, int(src), levels=levels, ws=ws, sync=False), i)
        lv = levels.cpu().numpy()
        ts.append(t)
        teps.append(int(deg[lv >= 0].sum()) // 2 / t * 1e6 / 1e9)
        nls.append(int(lv.max()) + 1)
    lines.append({"workload": "grid (no hubs)", "mode": "bfs (4 sources)", "us": round(float(np.median(ts)), 2),
                  "gteps_harmonic": round(len(teps) / sum(1.0 / v for v in teps), 3),
                  "levels_mean": float(np.mean(nls)), "us_per_level": round(float(np.median(ts)) / float(np.mean(nls)), 2)})
    assert ws.check() == 0
    ws.close(); M.close()
    return lines


def run_ablation(dbs, torch, dev, stream, flush, reps: int):
    """Format ablation (the paper's Fig. 10 setting: pull at x density 0.1,
    plus push at 0.001): every block forced to COO or to ForceCSR, against
    the automatic choice, on the R-MAT (Boolean), FEM and LLM (fp32)
    workloads.  Median kernel time per call, algorithmic bytes, GB/s."""
    import synth
    rows = []
    for name in ("rmat", "fem", "llm"):
        A = synth.config(name, "full")
        boolean = A.vals is None
        sr = "or_and" if boolean else "plus_times"
        xs = {}
        for d in (0.1, 0.001):
            if name == "fem":
                x = synth.x_clusters(A.n, d, [70, int(d * 1e4)])
            elif name == "llm":
                xd = synth.x_relu_topk(A.n, max(1, int(round(d * A.n))), [71, int(d * 1e4)])
                nz = np.nonzero(xd)[0].astype(np.int32)
                x = synth.SparseVec(A.n, nz, xd[nz])
            else:
                x = synth.x_uniform(A.n, int(round(d * A.n)), [72, int(d * 1e4)], valued=False)
            xv = None if (boolean or x.val is None) else torch.from_numpy(x.val.astype(np.float32)).to(dev)
            xs[d] = (torch.from_numpy(x.idx).to(dev), xv)
        y_idx = torch.empty(A.m, dtype=torch.int32, device=dev)
        y_val = torch.empty(A.m, dtype=torch.float32, device=dev)
        y_nnz = torch.empty(1, dtype=torch.int64, device=dev)
        for fname, ff in ABLATION_FORMATS:
            M = dbs.DBMatrix.from_csr(A, force_format=ff)
            info = M.info()
            ws = dbs.Workspace(M, collect_stats=1)
            for d, path in ((0.1, "pull"), (0.001, "push")):
                xi, xv = xs[d]
                dbs.spmspv(M, xi, xv, semiring=sr, path=path, ws=ws, y_idx=y_idx, y_val=y_val, y_nnz=y_nnz)
                bytes_alg = ws.stats()["bytes_alg"]
                ws.set_opts(dbs.exec_opts(collect_stats=0))
                ts = []
                for i in range(reps + 2):
                    flush(i)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    dbs.spmspv(M, xi, xv, semiring=sr, path=path, ws=ws, y_idx=y_idx, y_val=y_val, y_nnz=y_nnz)
                    e1.record(stream)
                    e1.synchronize()
                    if i >= 2:
                        ts.append(e0.elapsed_time(e1))
                ws.set_opts(dbs.exec_opts(collect_stats=1))
                us = 1e3 * float(np.median(ts))
                rows.append({"workload": name, "format": fname, "density": d, "path": path,
                             "us": round(us, 2), "bytes_alg": int(bytes_alg),
                             "gbs": round(bytes_alg / us / 1e3, 1),
                             "blocks_by_format": list(info["blocks_by_format"]),
                             "payload_mb": round(info["payload_bytes"] / 1e6, 1)})
            assert ws.check() == 0
            ws.close()
            M.close()
    return rows


def run_convert(dbs, torch, reps: int):
    """Offline conversion (DB-SpMSpV Section 5.5) of each full-size workload
    from a device CSR: the host builder (download, native threads, upload)
    against the device conversion (every pass on the GPU), best wall time of
    `reps` builds each, with the most device memory each build held
    (`build_peak_bytes`)."""
    import synth
    out = []
    for name in ("rmat", "fem", "llm", "grid"):
        A = synth.config(name, "full")
        rp = torch.from_numpy(A.row_ptr).cuda()
        ci = torch.from_numpy(A.col_idx).cuda()
        va = None if A.vals is None else torch.from_numpy(A.vals).cuda()
        torch.cuda.synchronize()
        line = {"workload": name, "nnz": int(A.nnz)}
        for key, dc in (("host", 0), ("device", 1)):
            ts, inf = [], None
            for _ in range(reps):
                t0 = time.perf_counter()
                M = dbs.DBMatrix(A.m, A.n, rp, ci, va, device_convert=dc)
                torch.cuda.synchronize()
                ts.append(time.perf_counter() - t0)
                inf = M.info()
                M.close()
            line[key] = {"seconds": round(min(ts), 4), "seconds_each": [round(t, 4) for t in ts],
                         "build_peak_mb": round(inf["build_peak_bytes"] / 1e6, 1),
                         "matrix_mb": round(inf["total_bytes"] / 1e6, 1)}
        line["blocks"] = int(inf["nblocks"])
        out.append(line)
        del rp, ci, va
    return out


def run_spmv(dbs, torch, dev, flush, reps: int):
    """Dense-input regime: adaptive CSR SpMV (dbs_spmv, plan built once);
    dbs_spmspv_dense on the auto path of a matrix built with dense_spmv (which
    hands this x to the kept SpMV); and the DB-format pull forced, on the same
    matrix with a dense x (every entry nonzero, N(0,1)).  FEM rows (27
    entries) run as warp rows, LLM rows (5,504) as block rows, the R-MAT
    graph with unit weights mixes scalar and warp rows with split hub rows.
    Median µs over `reps` calls, L2 flushed before each; GB/s from the CSR
    bytes (8 B per row pointer, 8 B per entry, x and y once)."""
    import synth
    peak, _ = _peaks()
    out = []
    for name in ("fem", "llm", "rmat"):
        A = synth.config(name, "full")
        if A.vals is None:
            A = synth.CSR(A.m, A.n, A.row_ptr, A.col_idx, np.ones(A.nnz, np.float32))
        plan = dbs.SpMVPlan.from_csr(A)
        M = dbs.DBMatrix.from_csr(A, dense_spmv=1)
        ws = dbs.Workspace(M)
        x = torch.from_numpy(np.random.default_rng(17).standard_normal(A.n).astype(np.float32)).to(dev)
        y = torch.empty(A.m, dtype=torch.float32, device=dev)

        def timed(call):
            ts = []
            for i in range(reps + 2):
                flush(i)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                call()
                e1.record()
                e1.synchronize()
                if i >= 2:
                    ts.append(e0.elapsed_time(e1) * 1e3)
            return float(np.median(ts))

        us_csr = timed(lambda: plan(x, y=y))
        us_auto = timed(lambda: dbs.spmspv_dense(M, x, y=y, ws=ws))
        us_db = timed(lambda: dbs.spmspv_dense(M, x, y=y, ws=ws, path="pull"))
        csr_bytes = 8 * (A.m + 1) + 8 * A.nnz + 4 * A.n + 4 * A.m
        line = {"workload": name, "nnz": int(A.nnz), "buckets": plan.info(),
                "csr_spmv_us": round(us_csr, 2), "csr_gbs": round(csr_bytes / us_csr / 1e3, 1),
                "csr_frac_of_measured_hbm": round(csr_bytes / us_csr / 1e3 / peak, 3),
                "dense_x_auto_us": round(us_auto, 2), "db_pull_us": round(us_db, 2)}
        out.append(line)
        assert ws.check() == 0
        ws.close(); M.close(); plan.close()
    return out


DECODE_TAU = 1.6449      # |N(0,1)| > tau for 10 % of the entries


def run_decode(dbs, torch, dev, stream, n_layers: int, tokens: int):
    """DB-Decoding token step (the pages' Section 4.3 / Table 2 setting):
    `n_layers` distinct 4096 x 11008 weights, 50 % pruned per row, fp32,
    each a DB-format matrix; one token = one dbs_decode_layer per layer, the
    activation of each layer thresholded by magnitude at DECODE_TAU inside
    the kernel.  The step is captured once as a CUDA graph and replayed per
    token after the token's activations are copied into the captured input
    buffers (outside the timed replay; the e2e figure times pinned-host
    activations in and outputs out as well).  The weights total several GB,
    far above L2, so every layer streams its blocks cold.  Two builds: the
    paper's format thresholds, and th1 = 31 (every block with 32 or more
    entries Dense, column-major) -- the setting measured fastest on GB300.  cuBLAS
    dense GEMV of the same layers (fp32 and bf16, dense weights) is timed
    the same way as context."""
    import synth
    m, n = 4096, 11008
    layers = [synth.llm_weight(m, n, seed=46 + i) for i in range(n_layers)]
    acts = [[synth.x_activation(n, [90, t, l]) for l in range(n_layers)] for t in range(tokens)]
    active = float(np.mean([np.mean(np.abs(a) > DECODE_TAU) for a in acts[0]]))
    X = torch.empty(n_layers, n, dtype=torch.float32, device=dev)     # one buffer: one copy per token
    Y = torch.empty(n_layers, m, dtype=torch.float32, device=dev)
    xs, ys = list(X.unbind(0)), list(Y.unbind(0))
    acts_dev = [torch.from_numpy(np.stack(tok)).to(dev) for tok in acts]

    def capture(step):
        s2 = torch.cuda.Stream()
        s2.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s2):
            step()
        torch.cuda.current_stream().wait_stream(s2)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        return g

    def time_tokens(g, load):
        ts = []
        for t in range(tokens + 3):
            load(t % tokens)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            if t >= 3:
                ts.append(e0.elapsed_time(e1) * 1e3)
        return float(np.median(ts))

    def load_dev(t):
        X.copy_(acts_dev[t])

    out = {"workload": f"{n_layers} distinct {m}x{n} layers, 50 % pruned per row (fp32), activations N(0,1) "
                       f"thresholded by magnitude at {DECODE_TAU} inside the kernel",
           "layers": n_layers, "tokens_timed": tokens, "active_fraction": round(active, 4),
           "timing": "CUDA graph of the token step, replayed per token; weights far above L2", "builds": []}
    for name, kw in (("paper thresholds", {}), ("th1 31", {"th1": 31})):
        Ms = [dbs.DBMatrix.from_csr(A, **kw) for A in layers]
        wss = [dbs.Workspace(M) for M in Ms]

        def step():
            for M, ws, x, y in zip(Ms, wss, xs, ys):
                dbs.decode_layer(M, x, DECODE_TAU, y=y, ws=ws)

        g = capture(step)
        us = time_tokens(g, load_dev)
        row = {"build": name, "us_per_token": round(us, 1), "us_per_layer": round(us / n_layers, 2),
               "tokens_per_s": round(1e6 / us, 1), "payload_mb_per_layer": round(Ms[0].info()["payload_bytes"] / 1e6, 1)}
        if kw:
            # end to end: activations from pinned host memory, outputs back to pinned host memory
            h_in = [torch.from_numpy(np.stack(tok)).pin_memory() for tok in acts]
            h_out = torch.empty(n_layers, m, dtype=torch.float32).pin_memory()
            ts = []
            for t in range(tokens + 3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                X.copy_(h_in[t % tokens], non_blocking=True)
                g.replay()
                h_out.copy_(Y, non_blocking=True)
                e1.record()
                e1.synchronize()
                if t >= 3:
                    ts.append(e0.elapsed_time(e1) * 1e3)
            e2e = float(np.median(ts))
            row["e2e"] = {"us_per_token": round(e2e, 1), "tokens_per_s": round(1e6 / e2e, 1),
                          "h2d_bytes_per_token": 4 * n * n_layers, "d2h_bytes_per_token": 4 * m * n_layers}
        out["builds"].append(row)
        del g
        for ws in wss:
            ws.close()
        for M in Ms:
            M.close()
        torch.cuda.synchronize()
    # dense cuBLAS GEMV of the same layers on the thresholded activations
    Ws = []
    for A in layers:
        W = torch.zeros(m, n, dtype=torch.float32, device=dev)
        rows = torch.from_numpy(np.repeat(np.arange(m), np.diff(A.row_ptr))).to(dev)
        W[rows, torch.from_numpy(A.col_idx.astype(np.int64)).to(dev)] = torch.from_numpy(A.vals).to(dev)
        Ws.append(W)
    thr = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(n_layers)]

    def load_thr(t):
        for x, a in zip(thr, acts_dev[t].unbind(0)):
            x.copy_(torch.where(a.abs() > DECODE_TAU, a, torch.zeros_like(a)))

    g = capture(lambda: [torch.mv(W, x, out=y) for W, x, y in zip(Ws, thr, ys)])
    us = time_tokens(g, load_thr)
    out["dense_gemv_fp32"] = {"us_per_token": round(us, 1), "us_per_layer": round(us / n_layers, 2)}
    del g
    Wb = [W.to(torch.bfloat16) for W in Ws]
    del Ws
    thr_b = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    yb = [torch.empty(m, dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]

    def load_thr_b(t):
        for x, a in zip(thr_b, acts_dev[t].unbind(0)):
            x.copy_(torch.where(a.abs() > DECODE_TAU, a, torch.zeros_like(a)))

    g = capture(lambda: [torch.mv(W, x, out=y) for W, x, y in zip(Wb, thr_b, yb)])
    us = time_tokens(g, load_thr_b)
    out["dense_gemv_bf16"] = {"us_per_token": round(us, 1), "us_per_layer": round(us / n_layers, 2)}
    del g, Wb
    torch.cuda.synchronize()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--scale", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--path-sweep", type=int, default=8,
                    help="calls per density and forced path for the push/pull crossover table (0 = off)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the secondary lines for the ER, FEM, LLM and grid workloads")
    ap.add_argument("--decode-layers", type=int, default=32,
                    help="layers of the DB-Decoding token step (distinct 4096x11008 weights; 0 = off)")
    ap.add_argument("--decode-tokens", type=int, default=20, help="tokens timed in the decoding step")
    ap.add_argument("--spmv", type=int, default=10,
                    help="calls per point of the dense-input comparison (adaptive CSR SpMV vs DB pull; 0 = off)")
    ap.add_argument("--convert", type=int, default=2,
                    help="builds per point of the conversion comparison (host vs device; 0 = off)")
    ap.add_argument("--ablation", type=int, default=0,
                    help="calls per point of the format ablation (Auto / COO-only / CSR-only on the "
                         "R-MAT, FEM and LLM workloads) and per-level frontier histograms (0 = off)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    __graft_entry__.build()
    import dynamic_sparsity_spmspv_gb300 as dbs

    A, xs, sources = build_workload(args.scale, 0)
    M = dbs.DBMatrix.from_csr(A)
    info = M.info()
    ws = dbs.Workspace(M, collect_stats=1)
    stream = torch.cuda.current_stream()

    x_dev = {d: [torch.from_numpy(x.idx).to(dev) for x in xs[d]] for d in DENSITIES}
    y_idx = torch.empty(A.m, dtype=torch.int32, device=dev)
    y_nnz = torch.empty(1, dtype=torch.int64, device=dev)
    levels = torch.empty(A.n, dtype=torch.int32, device=dev)

    # Units: touched nnz = nnz of the blocks whose column block is active in
    # x (for BFS: in each level's frontier), from the library's block views.
    counter = TouchedCounter(M.export_views())
    # untimed pass with device statistics: algorithmic bytes and path
    touched_x = {d: [counter.spmspv(x.idx) for x in xs[d]] for d in DENSITIES}
    bytes_x = {d: [] for d in DENSITIES}
    path_x = {d: [] for d in DENSITIES}
    phase_x = {d: [] for d in DENSITIES}
    for d in DENSITIES:
        for xi in x_dev[d]:
            dbs.spmspv(M, xi, None, semiring="or_and", ws=ws, y_idx=y_idx, y_nnz=y_nnz)
            st = ws.stats()
            bytes_x[d].append(st["bytes_alg"])
            path_x[d].append(st["path"])
            phase_x[d].append(st["phase_ns"])
    touched_bfs, bytes_bfs, edges_bfs, nlev_bfs, push_lev, phase_bfs, level_bfs = [], [], [], [], [], [], []
    deg = np.diff(A.row_ptr)
    for src in sources:
        _, nl = dbs.bfs(M, int(src), levels=levels, ws=ws)
        st = ws.stats()
        bytes_bfs.append(st["bytes_alg"])
        lev = levels.cpu().numpy()
        touched_bfs.append(counter.bfs(lev))
        edges_bfs.append(int(deg[lev >= 0].sum()) // 2)
        nlev_bfs.append(nl)
        push_lev.append(st["bfs_push_levels"])
        phase_bfs.append(st["phase_ns"])
        if len(level_bfs) < 3:
            level_bfs.append(ws.bfs_levels())
    assert ws.check() == 0
    ws.set_opts(dbs.exec_opts(collect_stats=0))

    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush(i):
        flush_buf.fill_(float(i & 7))

    def step(s, ev, rec):
        i = s % POOL
        for d in DENSITIES:
            flush(s)
            e0, e1 = ev.pop(), ev.pop()
            e0.record(stream)
            dbs.spmspv(M, x_dev[d][i], None, semiring="or_and", ws=ws, y_idx=y_idx, y_nnz=y_nnz)
            e1.record(stream)
            rec.append(("spmspv", d, i, e0, e1))
        flush(s)
        e0, e1 = ev.pop(), ev.pop()
        e0.record(stream)
        dbs.bfs(M, int(sources[s % N_SOURCES]), levels=levels, ws=ws, sync=False)
        e1.record(stream)
        rec.append(("bfs", None, s % N_SOURCES, e0, e1))

    def new_events(n):
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    for s in range(args.warmup):
        step(s, new_events(12), [])
    torch.cuda.synchronize()

    calls_per_step = len(DENSITIES) + 1
    ev = new_events(2 * calls_per_step * args.steps)
    rec = []
    sampler = ClockSampler(dev)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        step(args.warmup + s, ev, rec)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    assert ws.check() == 0

    t_sp = {d: 0.0 for d in DENSITIES}
    n_sp = {d: 0 for d in DENSITIES}
    units_sp = {d: 0 for d in DENSITIES}
    bytes_sp = {d: 0 for d in DENSITIES}
    t_bfs = 0.0
    units_bfs = edges = bytes_b = 0
    for kind, d, i, e0, e1 in rec:
        ms = e0.elapsed_time(e1)
        if kind == "spmspv":
            t_sp[d] += ms
            n_sp[d] += 1
            units_sp[d] += touched_x[d][i]
            bytes_sp[d] += bytes_x[d][i]
        else:
            t_bfs += ms
            units_bfs += touched_bfs[i]
            edges += edges_bfs[i]
            bytes_b += bytes_bfs[i]
    t_total_ms = sum(t_sp.values()) + t_bfs
    units_total = sum(units_sp.values()) + units_bfs
    t_max = t_total_ms
    if world > 1:
        t_max, units_total = reduce_over_ranks(t_total_ms, units_total, dev)
    value = units_total / (t_max * 1e-3)

    peak, peak_kind = _peaks()
    per_density = []
    for d in DENSITIES:
        t = t_sp[d] / max(n_sp[d], 1)
        per_density.append({
            "density": d, "us_per_call": 1e3 * t,
            "touched_nnz_per_s": units_sp[d] / (t_sp[d] * 1e-3),
            "bytes_alg_per_call": bytes_sp[d] / max(n_sp[d], 1),
            "gbs": bytes_sp[d] / (t_sp[d] * 1e-3) / 1e9,
            "frac_of_measured_hbm": bytes_sp[d] / (t_sp[d] * 1e-3) / 1e9 / peak,
            "path": "push" if statistics.mode(path_x[d]) == 1 else "pull",
            "device_phase_us_with_stats": [round(float(np.mean([p[i] for p in phase_x[d]])) / 1e3, 2)
                                           for i in range(3)]})
    bfs_info = {"gteps_harmonic": None, "ms_per_bfs": t_bfs / args.steps,
                "gteps": edges / (t_bfs * 1e-3) / 1e9, "levels_mean": float(np.mean(nlev_bfs)),
                "push_levels_mean": float(np.mean(push_lev)),
                "gbs": bytes_b / (t_bfs * 1e-3) / 1e9,
                "device_phase_us_with_stats": [round(float(np.mean([p[i] for p in phase_bfs])) / 1e3, 2)
                                               for i in range(3)],
                "levels_first_sources": level_bfs}
    # harmonic mean of per-source GTEPS from per-call times
    per_src_t = {}
    for kind, d, i, e0, e1 in rec:
        if kind == "bfs":
            per_src_t.setdefault(i, []).append(e0.elapsed_time(e1))
    if per_src_t:
        g = [edges_bfs[i] / (np.mean(v) * 1e-3) / 1e9 for i, v in per_src_t.items()]
        bfs_info["gteps_harmonic"] = len(g) / sum(1.0 / x for x in g)

    # dominant kernel: the launch kind with the largest share of the step time
    t_spmspv_all = sum(t_sp.values())
    if t_spmspv_all >= t_bfs:
        dom, dom_bytes, dom_t, dom_n = "k_spmspv_sparse<or_and>", sum(bytes_sp.values()), t_spmspv_all, sum(n_sp.values())
    else:
        dom, dom_bytes, dom_t, dom_n = "k_bfs", bytes_b, t_bfs, args.steps
    achieved = dom_bytes / dom_n / (dom_t / dom_n * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind, "traffic": _traffic(dom),
                "bytes_alg_per_launch": dom_bytes / dom_n, "us_per_launch": 1e3 * dom_t / dom_n,
                "share_of_step": dom_t / t_total_ms}

    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bool", "data": "synthetic",
           "config": config_dict(world, A.n, A.nnz, info["nblocks"]),
           "matrix_format": {"tiles": info["ntiles"], "device_bytes": info["total_bytes"]},
           "gpu_launches": calls_per_step * args.steps,
           "roofline": roofline, "per_density": per_density, "bfs": bfs_info, "clocks": clocks,
           "wall_s_timed_region": wall}

    # Hot-L2 numbers (no flush between calls: what L2 reuse adds) and the
    # kernel's own floor: one call with an empty x (every phase, no work),
    # against which the smallest densities' µs are read.
    def back_to_back(call, n=20):
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        e1.synchronize()
        return 1e3 * e0.elapsed_time(e1) / n

    x_empty = torch.empty(0, dtype=torch.int32, device=dev)
    out["hot_l2_us_per_call"] = {str(d): round(back_to_back(
        lambda d=d: dbs.spmspv(M, x_dev[d][0], None, semiring="or_and", ws=ws, y_idx=y_idx, y_nnz=y_nnz)), 2)
        for d in DENSITIES}
    flush(0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    dbs.spmspv(M, x_empty, None, semiring="or_and", ws=ws, y_idx=y_idx, y_nnz=y_nnz)
    e1.record(stream)
    e1.synchronize()
    out["floor_us"] = {"spmspv_empty_x_l2_flushed": round(1e3 * e0.elapsed_time(e1), 2),
                       "spmspv_empty_x_back_to_back": round(back_to_back(
                           lambda: dbs.spmspv(M, x_empty, None, semiring="or_and", ws=ws, y_idx=y_idx,
                                              y_nnz=y_nnz)), 2)}
    assert ws.check() == 0

    # push/pull crossover on this GPU: forced paths, same inputs, same timing
    if args.path_sweep > 0:
        sweep = []
        for d in DENSITIES:
            row = {"density": d}
            for path in ("push", "pull"):
                ts = []
                for i in range(args.path_sweep):
                    flush(i)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    dbs.spmspv(M, x_dev[d][i % POOL], None, semiring="or_and", path=path, ws=ws,
                               y_idx=y_idx, y_nnz=y_nnz)
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1))
                row[f"{path}_us"] = round(1e3 * float(np.median(ts)), 2)
            # blocks push visits, as a share of the B blocks pull scans
            ws.set_opts(dbs.exec_opts(collect_stats=1))
            dbs.spmspv(M, x_dev[d][0], None, semiring="or_and", ws=ws, y_idx=y_idx, y_nnz=y_nnz)
            row["push_work_frac"] = round(ws.stats()["visited_blocks"] / info["nblocks"], 4)
            ws.set_opts(dbs.exec_opts(collect_stats=0))
            sweep.append(row)
        # BFS levels with every level forced to one path
        bfs_sweep = []
        for src in sources[:3]:
            lv = {}
            for path in ("push", "pull"):
                flush(0)
                dbs.bfs(M, int(src), levels=levels, path=path, ws=ws)
                lv[path] = ws.bfs_levels()
            bfs_sweep.append({"push_work_frac": [round(w / info["nblocks"], 4) for w in lv["pull"]["push_work"]],
                              "push_us": lv["push"]["level_us"], "pull_us": lv["pull"]["level_us"]})
        out["path_sweep"] = sweep
        out["bfs_path_sweep"] = bfs_sweep
        assert ws.check() == 0

    if not args.no_configs:
        out["other_workloads"] = run_configs(dbs, torch, dev, stream, flush, 10)

    if args.convert > 0:
        out["conversion"] = run_convert(dbs, torch, args.convert)

    if args.spmv > 0:
        out["dense_input"] = run_spmv(dbs, torch, dev, flush, args.spmv)

    if args.decode_layers > 0:
        out["decode"] = run_decode(dbs, torch, dev, stream, args.decode_layers, args.decode_tokens)

    if args.ablation > 0:
        out["ablation"] = run_ablation(dbs, torch, dev, stream, flush, args.ablation)
        # Fig. 3 style frontier diagnostics: per BFS level, how many of the
        # frontier's nonzero vector blocks hold 1, 2, ..., 16 active entries
        hist = []
        for src in sources[:3]:
            dbs.bfs(M, int(src), levels=levels, ws=ws)
            lv = levels.cpu().numpy()
            per = []
            for l in range(int(lv.max()) + 1):
                vb = np.nonzero(lv == l)[0] >> 4
                cnt = np.bincount(np.bincount(vb)[np.unique(vb)], minlength=17)[1:17]
                per.append(cnt.tolist())
            hist.append(per)
        out["frontier_block_histograms"] = hist

    # end to end through the public API with host buffers.  SpMSpV: x lives in
    # pinned host memory and y is written to pinned host memory; the kernels
    # read and write them in place (GB300: coherent over NVLink-C2C), so the
    # transfers happen inside each call.  BFS: levels on the device, copied to
    # pinned host memory after the call (its scattered level writes are
    # faster in HBM).  The same step with explicit staging copies and a host
    # read of y_nnz before copying y back is reported beside it.
    if not args.no_e2e:
        pin = {d: [torch.from_numpy(x.idx).pin_memory() for x in xs[d]] for d in DENSITIES}
        xbuf = torch.empty(A.n, dtype=torch.int32, device=dev)
        lev_host = torch.empty(A.n, dtype=torch.int32).pin_memory()
        yh = torch.empty(A.m, dtype=torch.int32).pin_memory()
        ynh = torch.empty(1, dtype=torch.int64).pin_memory()
        ksteps = max(10, args.steps // 4)

        def e2e_run(staged: bool):
            h2d = d2h = 0
            tot_ms, units = 0.0, 0
            for s in range(args.warmup + ksteps):
                i = s % POOL
                timed = s >= args.warmup
                step_ms = 0.0
                for d in DENSITIES:
                    flush(s)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    k = pin[d][i].numel()
                    if staged:
                        xbuf[:k].copy_(pin[d][i], non_blocking=True)
                        dbs.spmspv(M, xbuf[:k], None, semiring="or_and", ws=ws, y_idx=y_idx, y_nnz=y_nnz)
                        ynh.copy_(y_nnz, non_blocking=True)
                        stream.synchronize()
                        yh[:int(ynh.item())].copy_(y_idx[:int(ynh.item())], non_blocking=True)
                    else:
                        dbs.spmspv(M, pin[d][i], None, semiring="or_and", ws=ws, y_idx=yh, y_nnz=ynh)
                    e1.record(stream)
                    e1.synchronize()
                    step_ms += e0.elapsed_time(e1)
                    if timed:
                        h2d += 4 * k
                        d2h += 8 + 4 * int(ynh.item())
                        units += touched_x[d][i]
                flush(s)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dbs.bfs(M, int(sources[s % N_SOURCES]), levels=levels, ws=ws, sync=False)
                lev_host.copy_(levels, non_blocking=True)
                e1.record(stream)
                e1.synchronize()
                step_ms += e0.elapsed_time(e1)
                if timed:
                    d2h += 4 * A.n
                    units += touched_bfs[s % N_SOURCES]
                    tot_ms += step_ms
            return {"value": units / (tot_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d // ksteps, "d2h_bytes_per_step": d2h // ksteps,
                    "steps": ksteps, "ms_per_step": tot_ms / ksteps}

        out["e2e"] = e2e_run(False)
        out["e2e"]["transfer"] = ("SpMSpV: x read from and y written to pinned host memory by the kernels "
                                  "(NVLink-C2C); BFS: levels copied device-to-host after each call")
        staged = e2e_run(True)
        out["e2e"]["staged_copies"] = {"value": staged["value"], "ms_per_step": staged["ms_per_step"]}
        assert ws.check() == 0

    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(A, xs, sources, touched_x, touched_bfs, args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
