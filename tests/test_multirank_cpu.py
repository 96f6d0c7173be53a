"""Multi-process host logic on CPU (gloo, world size 2).

Each process of `bench.py --gpus N` runs the whole R-rank problem on its own
GPU, so the only cross-process traffic is the barrier and the max of the step
times.  These tests run that host-side logic with two CPU processes: the
reference arm under torchrun (rank 0 prints the one JSON line, the other rank
exits cleanly) and the max-over-ranks reduction.  They also run the
rank-local path's one exchange step, the all-gather of every rank's [E]
tokens_per_expert that feeds moonep_plan_rank, with one process per EP rank.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--config", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def _max_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    dist.barrier()
    v = bench.max_over_ranks(10.0 + rank * 5.0, dist)
    q.put((rank, v))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def _gather_worker(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    from combine_moonep_plan_gb300 import workloads as wl
    from combine_moonep_plan_gb300.api import gather_tokens_per_expert
    sh = wl.Shape("x", R=world, E=12, K=3, S=40, H=8, Hp=8, B=6, tp=4, weights="softmax")
    # every process draws the same seeded routing and keeps its own rank's rows
    topk, _ = wl.routing(sh, "zipf", zipf_s=1.5, seed=77)
    mine = torch.from_numpy(topk[rank].reshape(-1).astype(np.int64))
    tpe = torch.bincount(mine, minlength=sh.E).to(torch.int32)
    hist = gather_tokens_per_expert(tpe)
    q.put((rank, hist.numpy().tolist(), wl.tokens_per_expert(topk, sh.E).tolist()))
    dist.destroy_process_group()


def test_histogram_all_gather_feeds_every_rank_the_same_counts():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    (r0, h0, want0), (r1, h1, want1) = got
    assert (r0, r1) == (0, 1)
    assert h0 == h1 == want0 == want1     # [R, E], rows in rank order, on every rank
