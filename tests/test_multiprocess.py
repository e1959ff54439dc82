"""The N > 1 launch of bench.py on CPU: one process per rank over gloo.
The path is replicated (one independent problem per GPU), so the only
cross-rank step is the final reduction -- the slowest rank's time and the
sum of the units -- and the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, u = bench.reduce_over_ranks(10.0 + rank, 1000 * (rank + 1), torch.device("cpu"))
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 11.0, 3000.0), (1, 11.0, 3000.0)]     # slowest rank's time, summed units


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--scale", "10", "--steps", "2", "--warmup", "3", "--gpus", "2"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "config"):
        assert k in d, k
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["value"] == d["value"]
    # the same workload description as the GPU arm prints
    m = d["config"]["matrix"]
    assert d["config"] == bench.config_dict(2, m["n"], m["nnz"], m["blocks"]) and m["blocks"] > 0


def test_touched_nnz_counter_matches_brute_force():
    """The bench's unit (touched nnz: nnz of the blocks in column blocks that
    hold an active x entry, summed over BFS levels) against a direct count
    over the CSR entries."""
    import numpy as np
    import oracle
    import synth
    A = synth.config("rmat", "small")
    counter = bench.TouchedCounter(oracle.block_views(A))
    col_cb = A.col_idx.astype(np.int64) // 16
    for k in (0, 1, 7, 100, 2000):
        x = synth.x_uniform(A.n, k, [5, k], valued=False)
        act = np.zeros((A.n + 15) // 16, bool)
        act[x.idx // 16] = True
        assert counter.spmspv(x.idx) == int(act[col_cb].sum())
    lv = oracle.Oracle(A).bfs_queue(int(synth.bfs_sources(A, 1, [5, 9])[0]))
    want = 0
    for L in range(int(lv.max()) + 1):
        act = np.zeros((A.n + 15) // 16, bool)
        act[np.nonzero(lv == L)[0] // 16] = True
        want += int(act[col_cb].sum())
    assert counter.bfs(lv) == want
