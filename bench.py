#!/usr/bin/env python
"""Benchmark of the balanced expert-parallel hot path on one GB300 per process.

The headline is the metric plan+dispatch+combine tokens/s on the
DeepSeek-V3-shaped workload (R=8 ranks, E=256 experts, top-8, S=4096 tokens
per rank, H=7168, B=32, token_padding=128) at maxvio 1.0, the largest
configuration with a maxvio sweep and the shape of the API page's own
Buffer(...) example.

One step = one pass of every hot-path row over one batch of synthetic input:
plan -> dispatch (hidden + route weights) -> combine (the dispatched rows
stand in for the expert outputs) -> weight prefetch -> plan-reuse dispatch of
an [R, S, H] gradient -> redundant-expert gradient reduce (one projection).
CUDA events sit between the ops of every timed step; `value` = R*S tokens per
step / the mean plan+dispatch+combine time of the timed steps (the metric),
`whole_step` the same over the whole step.  Beside it, on the same routing:
the maxvio sweep, the decode-path preparation, the packed MXFP4 prefetch, the
deduplicated dispatch/combine pair (`dedup_path`), and the other workload
shapes (`configs`: Mixtral, Kimi-K2, Qwen3 decode).

  python bench.py [--gpus N --steps K --warmup W] [--config deepseek_v3]
                  [--maxvio 1.0] [--impl ours|reference]

With N > 1 (torchrun), every process runs the same workload on its own GPU
(the R emulated ranks are independent batches: weak scaling, no data-path
collective); a gloo group carries only the barrier and the max of the timings.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "plan+dispatch+combine tokens/s and effective HBM GB/s vs ~8 TB/s, per maxvio"
SWEEPS = {"tiny": [1.0], "mixtral": [0.0, 0.5, 1.0, 2.0, 3.0],
          "deepseek_v3": [0.0, 1.0, 2.0, 4.0], "kimi_k2": ["hot30", "hot9"],
          "qwen3_decode": ["uniform", "zipf1", "pad100"]}
HEADLINE = {"tiny": 1.0, "mixtral": 1.0, "deepseek_v3": 1.0, "kimi_k2": "hot30",
            "qwen3_decode": "zipf1"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="deepseek_v3")
    ap.add_argument("--extra-configs", default="mixtral,kimi_k2,qwen3_decode",
                    help="comma list of other workload shapes measured after the headline "
                         "(chain and whole step only); empty for none")
    ap.add_argument("--maxvio", default=None, help="headline routing point")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-mxfp4", action="store_true",
                    help="skip the packed-MXFP4 weight prefetch measurement")
    ap.add_argument("--no-dedup", action="store_true",
                    help="skip the deduplicated dispatch/combine measurement")
    ap.add_argument("--step-only", action="store_true",
                    help="time the step and nothing else (no sweep, chain, preparation, MXFP4, "
                         "end-to-end or CPU legs): a clean launch list for profilers")
    ap.add_argument("--sweep-steps", type=int, default=30)
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--graph", action="store_true",
                    help="capture one step in a CUDA graph and replay it in the timed region")
    ap.add_argument("--hp", type=int, default=None, help="override H' (profiling case)")
    ap.add_argument("--s", type=int, default=None, help="override S (profiling case)")
    ap.add_argument("--k", type=int, default=None, help="override K (profiling case)")
    ap.add_argument("--profile-op", default=None,
                    help="comma list of ops (plan,dispatch,combine,prefetch,reduce,"
                         "dispatch_dedup,combine_dedup,prefetch_mxfp4): "
                         "allocate only what they need and run each --steps times "
                         "(a small, self-contained case for profilers; prints timings)")
    args = ap.parse_args()
    if args.step_only:
        args.no_sweep = args.no_e2e = args.no_cpu_baseline = args.no_mxfp4 = True
        args.no_dedup = True
        args.graph = False
        args.extra_configs = ""
    return args


# ----------------------------------------------------------------- routing

def make_routing(sh, point, seed):
    from combine_moonep_plan_gb300 import workloads as wl
    if point == "hot30":
        return wl.routing(sh, "hot", hot_share=0.30, seed=seed)
    if point == "hot9":
        return wl.routing(sh, "hot", hot_share=0.09375, seed=seed)
    if point == "uniform":
        return wl.routing(sh, "uniform", seed=seed)
    if point == "zipf1":
        return wl.routing(sh, "zipf", zipf_s=1.0, seed=seed)
    if point == "pad100":
        # 100 real tokens per rank, padded to the capacity: padding routes go
        # to expert 0 (with zero weight), as the decode-path preparation does
        topk, info = wl.routing(sh, "zipf", zipf_s=1.0, seed=seed)
        topk = topk.copy()
        topk[:, 100:, :] = 0
        info = dict(info, padded_from=100,
                    maxvio=float(np.bincount(topk.reshape(-1), minlength=sh.E).max()
                                 / (sh.N / sh.E) - 1))
        return topk, info
    mv = float(point)
    if mv == 0.0 and (sh.N % sh.E == 0):
        return wl.routing(sh, "exact0", seed=seed)
    return wl.routing(sh, "zipf", target_maxvio=mv, seed=seed)


def point_label(p):
    return p if isinstance(p, str) else float(p)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, with host times."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        used = inside
        if not used and self.samples:
            # timed region shorter than the sampling period: nearest samples
            used = [min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[1]]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        sm = [num(p[0]) for p in used if num(p[0]) is not None]
        mx = [num(p[1]) for p in used if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in used for n, v in zip(names, p[4:8]) if v == "Active"})
        pw = [num(p[2]) for p in used if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(inside)}


# ------------------------------------------------------------- our arm

class Step:
    """Device-resident inputs and outputs of one hot-path step."""

    def __init__(self, buf, sh, topk_np, seed, torch):
        from combine_moonep_plan_gb300 import workloads as wl
        dev = "cuda"
        R, S, K, E, H, Hp, B = sh.R, sh.S, sh.K, sh.E, sh.H, sh.Hp, sh.B
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.sh = sh
        self.buf = buf
        self.topk = torch.from_numpy(topk_np).to(dev)
        self.tpe = torch.from_numpy(wl.tokens_per_expert(topk_np, E)).to(dev)
        self.hidden = torch.randn((R, S, H), generator=g, device=dev).to(torch.bfloat16)
        self.w_sk = torch.from_numpy(wl.route_weights(sh, seed)).to(dev)
        self.grad = torch.randn((R, S, H), generator=g, device=dev).to(torch.bfloat16)
        NvS = buf.NvS
        self.hid_nvsh = torch.empty((R * NvS, H), dtype=torch.bfloat16, device=dev)
        self.w_nvs = torch.empty((R * NvS,), dtype=torch.float32, device=dev)
        self.grad_nvsh = torch.empty((R * NvS, H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((R, S, H), dtype=torch.bfloat16, device=dev)
        self.w_back = torch.empty((R, S, K), dtype=torch.float32, device=dev)
        self.W = torch.randn((E + R * B, H, Hp), generator=g, device=dev).to(torch.bfloat16)
        self.Gh = torch.randn((E, H, Hp), generator=g, device=dev)
        self.Gs = torch.randn((R, B, H, Hp), generator=g, device=dev)
        self.plan = buf.new_plan()

    def plan_dispatch(self, rec=lambda i: None):
        b = self.buf
        b.plan(self.topk, self.tpe, plan=self.plan)
        rec(1)
        b.dispatch(self.hidden, self.w_sk, plan=self.plan, out=self.hid_nvsh,
                   weights_out=self.w_nvs)

    def run(self, events=None):
        b = self.buf
        rec = (lambda i: events[i].record()) if events else (lambda i: None)
        rec(0)
        self.plan_dispatch(rec)
        rec(2)
        b.combine(self.plan, self.hid_nvsh, self.w_nvs, out=self.out, weights_out=self.w_back)
        rec(3)
        b.prefetch_weight(self.plan, self.W)
        rec(4)
        b.dispatch(self.grad, plan=self.plan, out=self.grad_nvsh)
        rec(5)
        b.reduce_grad(self.plan, [self.Gh], [self.Gs])
        rec(6)

    LAUNCHES_PER_STEP = 6  # plan (one launch), dispatch, combine, prefetch, dispatch, reduce

    def algorithmic_bytes(self):
        """Bytes each op must move (reads + writes), per launch."""
        sh = self.sh
        R, S, K, E, H, B, Hp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B, sh.Hp
        N = R * S * K
        p = self.plan
        zfr = p.zero_fill_ranges.cpu().numpy().astype(np.int64)
        P = int((zfr[..., 1] - zfr[..., 0]).sum())
        etc = p.experts_to_copy.cpu().numpy()
        U = int((etc >= 0).sum())
        D = len(np.unique(etc[etc >= 0]))
        HHp = H * Hp
        return {
            "plan": N * 4 + R * E * 4 + N * 4 + R * (E + B) * 16,
            "dispatch": R * S * H * 2 + N * 8 + (N + P) * (H * 2 + 4),
            "prefetch": (D + U) * HHp * 2,  # each expert's row read once, U slot rows written
            "combine": N * H * 2 + N * 8 + R * S * H * 2 + N * 4,
            "grad_dispatch": R * S * H * 2 + N * 4 + (N + P) * H * 2,
            "reduce": (2 * D + 2 * U) * HHp * 4,
        }, {"P": P, "U": U, "D": D}


OPS = ["plan", "dispatch", "combine", "prefetch", "grad_dispatch", "reduce"]
CHAIN = ("plan", "dispatch", "combine")  # the metric's ops, the first three of a step


def timed_steps(step, steps, torch, dist=None):
    """Run `steps` steps with CUDA events between the ops of every step.
    Returns (ms from the first step's start to the last step's end, per-op ms
    lists, per-step plan+dispatch+combine ms list, host times of the region)."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(steps):
        step.run(evs[i])
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    total = evs[0][0].elapsed_time(evs[-1][6])
    per_op = {op: [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)]
              for j, op in enumerate(OPS)}
    chain = [evs[i][0].elapsed_time(evs[i][3]) for i in range(steps)]
    return total, per_op, chain, (t0, t1)


def time_chain(step, n, torch, graph=False):
    """plan -> dispatch -> combine back to back, timed as one chain (no
    events between the ops); ms per chain, eagerly issued or (graph=True)
    replayed from a CUDA graph of the chain."""
    b = step.buf

    def chain():
        step.plan_dispatch()
        b.combine(step.plan, step.hid_nvsh, step.w_nvs, out=step.out, weights_out=step.w_back)
    run = chain
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            chain()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain()
        run = g.replay
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        run()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def max_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_mxfp4_prefetch(buf, step, sh, steps, torch, peak):
    """The packed-MXFP4 form of the weight prefetch on the step's plan: a
    gate/up/down set [E + R*B, H, H'/2] uint8 (two 4-bit codes per byte) with
    its E8M0 block scales [E + R*B, H, H'/32] uint8, all six tensors moved by
    one launch per call."""
    rows = sh.E + sh.R * sh.B
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    ts = [torch.randint(0, 256, (rows, sh.H, sh.Hp // 2), generator=g, dtype=torch.uint8,
                        device="cuda") for _ in range(3)]
    ts += [torch.randint(0, 256, (rows, sh.H, sh.Hp // 32), generator=g, dtype=torch.uint8,
                         device="cuda") for _ in range(3)]
    for _ in range(3):
        buf.prefetch_weight(step.plan, *ts[:3], scales=ts[3:])
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        buf.prefetch_weight(step.plan, *ts[:3], scales=ts[3:])
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    cnt = step.algorithmic_bytes()[1]
    U, D = cnt["U"], cnt["D"]
    nbytes = (D + U) * 3 * (sh.H * sh.Hp // 2 + sh.H * sh.Hp // 32)
    del ts
    torch.cuda.empty_cache()
    return {"set": "gate/up/down packed MXFP4 [E+R*B, H, H'/2] uint8 + E8M0 block scales "
                   "[E+R*B, H, H'/32] uint8, one launch",
            "ms": round(ms, 5), "GB": round(nbytes / 1e9, 4), "slots_used": U,
            "GBps": round(nbytes / (ms / 1e3) / 1e9, 1) if ms > 0 else None,
            "frac_of_peak": round(nbytes / (ms / 1e3) / 1e9 / peak, 4) if ms > 0 else None}


def run_dedup(sh, step, steps, torch, peak):
    """The deduplicated data flow on the step's routing: dispatch copies only
    the primary rows and expands the duplicates in an epilogue; combine folds
    every rank's duplicates into their primaries first and then sums the
    primaries.  On one GPU both move more HBM bytes than the direct kernels;
    what they save is the rows that would cross between ranks
    (cross_rank_rows, direct vs deduplicated)."""
    from combine_moonep_plan_gb300.api import Buffer
    R, S, K, H = sh.R, sh.S, sh.K, sh.H
    buf = Buffer(S=S, H=H, K=K, E=sh.E, num_ep_ranks=R, B=sh.B, token_padding=sh.tp,
                 zero_copy_views=False, dup_records=True)
    plan = buf.plan(step.topk, step.tpe)
    y = step.hid_nvsh.clone()

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps
    ms = {
        "plan_with_dup_records": timed(lambda: buf.plan(step.topk, step.tpe, plan=plan)),
        "dispatch_dedup": timed(lambda: buf.dispatch(step.hidden, step.w_sk, plan=plan,
                                                     out=step.hid_nvsh, weights_out=step.w_nvs,
                                                     dedup=True)),
        "dispatch": timed(lambda: buf.dispatch(step.hidden, step.w_sk, plan=plan,
                                               out=step.hid_nvsh, weights_out=step.w_nvs)),
        "combine_dedup": timed(lambda: buf.combine(plan, y, step.w_nvs, out=step.out,
                                                   weights_out=step.w_back, dedup=True)),
        "combine": timed(lambda: buf.combine(plan, y, step.w_nvs, out=step.out,
                                             weights_out=step.w_back)),
    }
    status = buf.get_status()
    dst = plan.dst.cpu().numpy().astype(np.int64).reshape(R, S * K)
    g = np.where(dst >= 0, dst, -dst - 1)
    dest_rank = g // buf.NvS
    remote = dest_rank != np.arange(R)[:, None]
    dc = plan.dup_counts.cpu().numpy().astype(np.int64)
    D, Gr = int(dc[:, 0].sum()), int(dc[:, 1].sum())
    N = R * S * K
    zfr = plan.zero_fill_ranges.cpu().numpy().astype(np.int64)
    P = int((zfr[..., 1] - zfr[..., 0]).sum())
    row = H * 2
    nbytes = {
        # primaries + padding rows written, weights for every route; then the
        # epilogue reads Gr primary rows and writes D duplicate rows
        "dispatch_dedup": R * S * row + N * 8 + (N - D + P) * row + (N + P) * 4
        + (Gr + D) * row,
        "dispatch": R * S * row + N * 8 + (N + P) * (row + 4),
        # the fold reads Gr + D rows and writes Gr; the sum reads N - D rows
        "combine_dedup": (2 * Gr + D) * row + (N - D) * row + N * 12 + R * S * row,
        "combine": N * row + N * 12 + R * S * row,
    }
    ops = {}
    for k, v in ms.items():
        e = {"ms": round(v, 5)}
        if k in nbytes and v > 0:
            e["GB"] = round(nbytes[k] / 1e9, 4)
            e["frac_of_peak"] = round(nbytes[k] / (v / 1e3) / 1e9 / peak, 4)
        ops[k] = e
    buf.destroy()
    del y
    torch.cuda.empty_cache()
    return {"ops": ops, "duplicate_routes": D, "duplicate_groups": Gr, "routes": N,
            "cross_rank_rows": {"direct": int(remote.sum()),
                                "deduplicated": int((remote & (dst >= 0)).sum())},
            "device_status": status}


def run_prepare(buf, sh, steps, torch):
    """The decode-path preparation on this shape: every rank holds 3/4 of the
    capacity as real tokens (about 4 % of their ids invalid); the call pads
    the rest in place and counts tokens_per_expert."""
    R, S, K, E, H = sh.R, sh.S, sh.K, sh.E, sh.H
    g = torch.Generator(device="cuda")
    g.manual_seed(23)
    n = [S - S // 4] * R
    topk = torch.randint(0, E, (R, S, K), generator=g, device="cuda", dtype=torch.int32)
    topk[torch.rand((R, S, K), generator=g, device="cuda") < 0.04] = -1
    w = torch.rand((R, S, K), generator=g, device="cuda")
    hidden = torch.randn((R, S, H), generator=g, device="cuda").to(torch.bfloat16)
    # timed as CUDA-graph replays: the GPU time of the call, not the Python
    # wrapper's issue rate
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            buf.prepare(hidden, topk, w, num_tokens=n)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(10):
            buf.prepare(hidden, topk, w, num_tokens=n)
    graph.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / (10 * steps) * 1e3
    nbytes = R * S * K * 8 + R * E * 4 + R * (S // 4) * H * 2
    del topk, w, hidden
    return {"us": round(us, 2), "num_tokens_per_rank": n[0], "capacity": S,
            "bytes": nbytes, "GBps": round(nbytes / (us / 1e6) / 1e9, 1)}


def run_e2e(buf, sh, topk_np, seed, steps, torch, dist):
    """The metric's plan -> dispatch -> combine through the public API with
    the inputs in pinned host memory: every step copies its inputs (top-k ids,
    tokens_per_expert, hidden rows, route weights) host->device and reads the
    combined rows and the gathered route weights back.  Copies run on their
    own streams, double-buffered, so step i's compute overlaps step i+1's
    inputs and step i-1's result; the timed region spans the first input copy
    to the last result copy."""
    from combine_moonep_plan_gb300 import workloads as wl
    R, S, K, E, H = sh.R, sh.S, sh.K, sh.E, sh.H
    g = torch.Generator().manual_seed(seed)
    h_in = {
        "topk": torch.from_numpy(topk_np).pin_memory(),
        "tpe": torch.from_numpy(wl.tokens_per_expert(topk_np, E)).pin_memory(),
        "hidden": torch.randn((R, S, H), generator=g).to(torch.bfloat16).pin_memory(),
        "w_sk": torch.from_numpy(wl.route_weights(sh, seed)).pin_memory(),
    }
    h_out = [{"out": torch.empty((R, S, H), dtype=torch.bfloat16, pin_memory=True),
              "w_back": torch.empty((R, S, K), dtype=torch.float32, pin_memory=True)}
             for _ in range(2)]
    NvS = buf.NvS
    plan = buf.new_plan()
    hid_nvsh = torch.empty((R * NvS, H), dtype=torch.bfloat16, device="cuda")
    w_nvs = torch.empty((R * NvS,), dtype=torch.float32, device="cuda")
    sets = []
    for _ in range(2):
        sets.append({k: torch.empty_like(v, device="cuda") for k, v in h_in.items()} |
                    {"out": torch.empty((R, S, H), dtype=torch.bfloat16, device="cuda"),
                     "w_back": torch.empty((R, S, K), dtype=torch.float32, device="cuda")})
    bi = sum(t.numel() * t.element_size() for t in h_in.values())
    bo = sum(t.numel() * t.element_size() for t in h_out[0].values())
    compute = torch.cuda.Stream()
    h2d = torch.cuda.Stream()
    d2h = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    inputs_ready = [ev(), ev()]
    computed = [ev(), ev()]
    read_back = [ev(), ev()]
    used = [False, False]

    def run(n, timed):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        h2d.record_event(start) if timed else None
        for i in range(n):
            b = i % 2
            d = sets[b]
            with torch.cuda.stream(h2d):
                if used[b]:
                    h2d.wait_event(computed[b])      # step i-2 no longer reads this set
                for k, v in h_in.items():
                    d[k].copy_(v, non_blocking=True)
                h2d.record_event(inputs_ready[b])
            with torch.cuda.stream(compute):
                compute.wait_event(inputs_ready[b])
                if used[b]:
                    compute.wait_event(read_back[b])  # step i-2's result has been read
                buf.dispatch(d["hidden"], d["w_sk"], d["topk"], d["tpe"], out=hid_nvsh,
                             weights_out=w_nvs, plan_out=plan)
                buf.combine(plan, hid_nvsh, w_nvs, out=d["out"], weights_out=d["w_back"])
                compute.record_event(computed[b])
            with torch.cuda.stream(d2h):
                d2h.wait_event(computed[b])
                h_out[b]["out"].copy_(d["out"], non_blocking=True)
                h_out[b]["w_back"].copy_(d["w_back"], non_blocking=True)
                d2h.record_event(read_back[b])
            used[b] = True
        if timed:
            d2h.record_event(end)
        torch.cuda.synchronize()
        return start.elapsed_time(end) if timed else 0.0

    run(6, False)  # warm-up: host copies and kernels
    ms = max_over_ranks(run(steps, True), dist)
    del hid_nvsh, w_nvs, sets, plan
    torch.cuda.empty_cache()
    return ms / steps, bi, bo


class OracleChain:
    """The oracle's plan -> dispatch -> combine on the whole workload (every
    token, every hidden column), single-threaded on the host, with its
    output buffers allocated once and reused like a framework's."""

    def __init__(self, sh, topk_np, seed):
        from combine_moonep_plan_gb300 import workloads as wl
        self.sh = sh
        self.topk = topk_np
        self.tpe = wl.tokens_per_expert(topk_np, sh.E)
        self.x = wl.hidden_bf16(sh, seed)
        self.w = wl.route_weights(sh, seed)
        NvS = sh.NvS
        self.hid = np.zeros((sh.R * NvS, sh.H), np.uint16)
        self.wn = np.zeros(sh.R * NvS, np.float32)

    def step(self):
        """One pass; returns the seconds of plan, dispatch and combine."""
        import oracle
        sh = self.sh
        R, S, K, E, H, B, tp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B, sh.tp
        a = time.perf_counter()
        st, p = oracle.plan(R, E, K, S, B, tp, self.topk, self.tpe, dup_records=False)
        b = time.perf_counter()
        if st != 0:
            raise RuntimeError(f"oracle plan status {st}")
        NvS = p["NvS"]
        oracle.dispatch(R, S, K, E, B, NvS, H, p["dst"], p["zero_fill_ranges"], self.x, self.w,
                        self.hid, self.wn)
        c = time.perf_counter()
        oracle.combine(R, S, K, NvS, H, p["dst"], self.hid, self.wn)
        d = time.perf_counter()
        return {"plan": b - a, "dispatch": c - b, "combine": d - c}

    SAMPLE = "the whole workload: every token, every hidden column (plan, dispatch, combine)"


def cpu_baseline(sh, topk_np, seed, budget_s=15.0):
    """The oracle timed on the host: one untimed pass (first touch of its
    buffers), then passes until about budget_s seconds of oracle work."""
    t0 = time.perf_counter()
    ch = OracleChain(sh, topk_np, seed)
    ch.step()
    times = []
    a = time.perf_counter()
    while not times or time.perf_counter() - a < budget_s:
        times.append(ch.step())
        if len(times) >= 50:
            break
    per = {op: statistics.mean(t[op] for t in times) for op in CHAIN}
    step_s = sum(per.values())
    return {"value": R_S(sh) / step_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{OracleChain.SAMPLE}; mean of {len(times)} passes after one untimed",
            "step_s": round(step_s, 4), "op_s": {k: round(v, 4) for k, v in per.items()},
            "wall_s": round(time.perf_counter() - t0, 2), "host": host_info()}


def reference_arm(args, sh, point, topk_np, seed, dist):
    """The oracle as the reference arm: each step is one oracle pass of the
    metric's plan -> dispatch -> combine over the whole workload; ms_per_step
    is its wall time."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    steps, warm = args.steps, args.warmup
    t0 = time.perf_counter()
    ch = OracleChain(sh, topk_np, seed)
    for _ in range(warm):
        ch.step()
    a = time.perf_counter()
    per = {op: 0.0 for op in CHAIN}
    for _ in range(steps):
        for op, v in ch.step().items():
            per[op] += v
    wall = time.perf_counter() - a
    value = R_S(sh) * steps / wall
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * wall / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(sh, point),
            "op_ms": {op: round(1e3 * v / steps, 2) for op, v in per.items()},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": OracleChain.SAMPLE + "; every timed step one full pass",
                             "wall_s": round(time.perf_counter() - t0, 2), "host": host_info()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def host_info():
    """The host cores the CPU baseline runs on: count, model, memory."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and model is None:
                    model = ln.split(":", 1)[1].strip()
    except OSError:
        pass
    ram = None
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemTotal:"):
                    ram = round(int(ln.split()[1]) / 2**20, 1)
    except OSError:
        pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model, "machine": platform.machine(),
            "ram_gib": ram}


def recorded_traffic(op, config):
    """DRAM bytes per launch of `op` on `config` from profiles/traffic.md, if
    the kernel's source files are unchanged since the capture (else None).
    The table's source column lists the files joined by '+', the sha1 column
    the SHA-1 of their concatenated contents."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) < 5 or cells[0] != op or cells[1] != config:
            continue
        h = hashlib.sha1()
        for rel in cells[3].split("+"):
            src = os.path.join(ROOT, rel.strip())
            if not os.path.exists(src):
                return None
            with open(src, "rb") as f:
                h.update(f.read())
        if h.hexdigest() != cells[4]:
            return None
        return int(cells[2])
    return None


def R_S(sh):
    return sh.R * sh.S


def workload_config(sh, point):
    return {"workload": f"{sh.name}-shaped: R={sh.R} E={sh.E} K={sh.K} S={sh.S} H={sh.H} "
                        f"H'={sh.Hp} B={sh.B} token_padding={sh.tp}, routing maxvio point "
                        f"{point_label(point)}",
            "R": sh.R, "E": sh.E, "K": sh.K, "S": sh.S, "H": sh.H, "H_prime": sh.Hp, "B": sh.B,
            "token_padding": sh.tp, "maxvio_point": point_label(point), "n_proj": 1,
            "metric_ops": "plan -> dispatch(+weights) -> combine(+weights)",
            "step": "plan -> dispatch(+weights) -> combine(+weights) -> prefetch -> "
                    "plan-reuse grad dispatch -> grad reduce",
            "l2": "inputs larger than L2 (no flush): every step moves several GB",
            "dup_records": False, "global_batch": sh.R * sh.S}


def profile_ops(args, sh, point, seed):
    """Run only the named ops, allocating only what they need (profiling case)."""
    import dataclasses
    import torch
    from combine_moonep_plan_gb300 import workloads as wl
    from combine_moonep_plan_gb300.api import Buffer
    from combine_moonep_plan_gb300.build import build
    build()
    if args.hp:
        sh = dataclasses.replace(sh, Hp=args.hp)
    if args.s:
        sh = dataclasses.replace(sh, S=args.s)
    if args.k:
        sh = dataclasses.replace(sh, K=args.k)
    ops = args.profile_op.split(",")
    R, S, K, E, H, B, Hp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B, sh.Hp
    topk_np, info = make_routing(sh, point, seed)
    dedup = any(o.endswith("_dedup") for o in ops)
    buf = Buffer(S=S, H=H, K=K, E=E, num_ep_ranks=R, B=B, token_padding=sh.tp,
                 zero_copy_views=False, dup_records=dedup)
    dev = "cuda"
    topk = torch.from_numpy(topk_np).to(dev)
    plan = buf.plan(topk)
    t = {}
    if {"dispatch", "combine", "dispatch_dedup", "combine_dedup"} & set(ops):
        t["x"] = torch.randn((R, S, H), device=dev).to(torch.bfloat16)
        t["w"] = torch.from_numpy(wl.route_weights(sh, seed)).to(dev)
        t["y"] = torch.empty((R * buf.NvS, H), dtype=torch.bfloat16, device=dev)
        t["wn"] = torch.empty((R * buf.NvS,), dtype=torch.float32, device=dev)
        buf.dispatch(t["x"], t["w"], plan=plan, out=t["y"], weights_out=t["wn"])
        t["out"] = torch.empty((R, S, H), dtype=torch.bfloat16, device=dev)
        t["wb"] = torch.empty((R, S, K), dtype=torch.float32, device=dev)
    if "prefetch" in ops:
        t["W"] = torch.randn((E + R * B, H, Hp), device=dev).to(torch.bfloat16)
    if "prefetch_mxfp4" in ops:
        rows = E + R * B
        t["mx"] = [torch.randint(0, 256, (rows, H, Hp // 2), dtype=torch.uint8, device=dev)
                   for _ in range(3)]
        t["mx"] += [torch.randint(0, 256, (rows, H, Hp // 32), dtype=torch.uint8, device=dev)
                    for _ in range(3)]
    if "reduce" in ops:
        t["Gh"] = torch.randn((E, H, Hp), device=dev)
        t["Gs"] = torch.randn((R, B, H, Hp), device=dev)
    run = {"plan": lambda: buf.plan(topk, plan=plan),
           "dispatch": lambda: buf.dispatch(t["x"], t["w"], plan=plan, out=t["y"],
                                            weights_out=t["wn"]),
           "combine": lambda: buf.combine(plan, t["y"], t["wn"], out=t["out"],
                                          weights_out=t["wb"]),
           "dispatch_dedup": lambda: buf.dispatch(t["x"], t["w"], plan=plan, out=t["y"],
                                                  weights_out=t["wn"], dedup=True),
           "combine_dedup": lambda: buf.combine(plan, t["y"], t["wn"], out=t["out"],
                                                weights_out=t["wb"], dedup=True),
           "prefetch": lambda: buf.prefetch_weight(plan, t["W"]),
           "prefetch_mxfp4": lambda: buf.prefetch_weight(plan, *t["mx"][:3],
                                                         scales=t["mx"][3:]),
           "reduce": lambda: buf.reduce_grad(plan, [t["Gh"]], [t["Gs"]])}
    res = {}
    for op in ops:
        for _ in range(2):
            run[op]()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(args.steps):
            run[op]()
        ev1.record()
        torch.cuda.synchronize()
        res[op] = ev0.elapsed_time(ev1) / args.steps
    etc = plan.experts_to_copy.cpu().numpy()
    print(json.dumps({"profile_case": sh.name, "Hp": Hp, "maxvio": info["maxvio"], "ms": res,
                      "slots_used": int((etc >= 0).sum()),
                      "experts_with_copies": len(np.unique(etc[etc >= 0])),
                      "status": buf.get_status()}),
          flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = {}
    if os.path.exists(path):
        try:
            with open(path) as f:
                peaks = json.load(f)
        except Exception:
            peaks = {}
    if "hbm_gbs" in peaks:
        return float(peaks["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def summarise(step, sh, total_ms, per_op, chain, steps, peak, world=1):
    """Per-op times and rates, the metric's chain and the whole step."""
    alg, counts = step.algorithmic_bytes()
    op_ms = {op: statistics.mean(v) for op, v in per_op.items()}
    chain_ms = statistics.mean(chain)
    ops = {o: {"ms": round(op_ms[o], 5), "GB": round(alg[o] / 1e9, 4),
               "GBps": round(alg[o] / (op_ms[o] / 1e3) / 1e9, 1) if op_ms[o] > 0 else None,
               "frac_of_peak": round(alg[o] / (op_ms[o] / 1e3) / 1e9 / peak, 4)
               if op_ms[o] > 0 else None,
               "ms_p10_p50_p90": [round(float(np.percentile(per_op[o], q)), 5)
                                  for q in (10, 50, 90)]} for o in OPS}
    tokens = R_S(sh) * world
    return {
        "chain_ms": chain_ms, "tokens_per_s": tokens / (chain_ms / 1e3),
        "chain_ms_p10_p50_p90": [round(float(np.percentile(chain, q)), 5) for q in (10, 50, 90)],
        "chain_hbm_GBps": sum(alg[o] for o in CHAIN) / (chain_ms / 1e3) / 1e9,
        "whole_step": {"ms_per_step": total_ms / steps,
                       "tokens_per_s": tokens / (total_ms / steps / 1e3),
                       "hbm_GBps": sum(alg.values()) / (total_ms / steps / 1e3) / 1e9},
        "plan_frac_of_dispatch": op_ms["plan"] / op_ms["dispatch"],
        "ops": ops, "plan_counts": counts, "op_ms": op_ms, "alg": alg,
    }


def roofline_entry(op, summ, peak, peak_src, config_name):
    achieved = summ["alg"][op] / (summ["op_ms"][op] / 1e3) / 1e9
    return {"bound": "hbm", "kernel": op, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_src,
            "bytes_per_launch": summ["alg"][op], "ms_per_launch": round(summ["op_ms"][op], 5),
            "traffic": recorded_traffic(op, config_name)}


def measure_config(name, args, torch, peak, seed_idx=0, steps=None):
    """The step on another workload shape at its headline routing point:
    the metric's chain and the whole step, nothing else."""
    from combine_moonep_plan_gb300 import workloads as wl
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.SHAPES[name]
    point = HEADLINE[name]
    seed = wl.seed_for(name, seed_idx)
    topk_np, info = make_routing(sh, point, seed)
    buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                 token_padding=sh.tp, zero_copy_views=False)
    step = Step(buf, sh, topk_np, seed, torch)
    for _ in range(max(args.warmup, 3)):
        step.run()
    n = steps or max(args.steps, 20)
    total, per_op, chain, _ = timed_steps(step, n, torch, None)
    summ = summarise(step, sh, total, per_op, chain, n, peak)
    nb = max(20, min(n, 200))
    b2b = time_chain(step, nb, torch)
    b2b_graph = time_chain(step, nb, torch, graph=True) if sh.S * sh.R <= 4096 else None
    status = buf.get_status()
    out = {"workload": workload_config(sh, point)["workload"], "maxvio": round(info["maxvio"], 4),
           "plan_dispatch_combine_tokens_per_s": summ["tokens_per_s"],
           "chain_ms": round(summ["chain_ms"], 5),
           "plan_us": round(1e3 * summ["op_ms"]["plan"], 2),
           "plan_frac_of_dispatch": round(summ["plan_frac_of_dispatch"], 4),
           "dispatch_frac_of_peak": summ["ops"]["dispatch"]["frac_of_peak"],
           "combine_frac_of_peak": summ["ops"]["combine"]["frac_of_peak"],
           "whole_step": summ["whole_step"], "ops": summ["ops"], "steps": n,
           "back_to_back_chain": {
               "ms": round(b2b, 5), "tokens_per_s": R_S(sh) / (b2b / 1e3),
               "graph_ms": round(b2b_graph, 5) if b2b_graph else None},
           "device_status": status}
    del step
    buf.destroy()
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from combine_moonep_plan_gb300 import workloads as wl
    sh = wl.SHAPES[args.config]
    point = args.maxvio if args.maxvio is not None else HEADLINE[args.config]
    try:
        point = float(point)
    except (TypeError, ValueError):
        pass
    seed = wl.seed_for(sh.name, 0)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("gloo")
        dist = dist_mod

    if args.profile_op:
        profile_ops(args, sh, point, seed)
        return

    if args.impl == "reference":
        topk_np, _ = make_routing(sh, point, seed)
        line = reference_arm(args, sh, point, topk_np, seed, dist)
        if line is not None:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    import torch
    torch.cuda.set_device(local)
    from combine_moonep_plan_gb300.build import build
    build()
    from combine_moonep_plan_gb300.api import Buffer

    topk_np, rinfo = make_routing(sh, point, seed)
    buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                 token_padding=sh.tp, zero_copy_views=False)
    step = Step(buf, sh, topk_np, seed, torch)
    for _ in range(max(args.warmup, 3)):
        step.run()
    torch.cuda.synchronize()
    status = buf.get_status()
    if status != 0:
        raise SystemExit(f"device status {status} during warm-up")
    peak, peak_src = load_peaks()

    graph_ms = None
    if args.graph:
        # the whole step as one CUDA graph (the decode-sized case is
        # launch-latency bound)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step.run()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step.run()
        for _ in range(max(args.warmup, 3)):
            graph.replay()
        torch.cuda.synchronize()
        ga = torch.cuda.Event(enable_timing=True)
        gb = torch.cuda.Event(enable_timing=True)
        ga.record()
        for _ in range(args.steps):
            graph.replay()
        gb.record()
        torch.cuda.synchronize()
        graph_ms = max_over_ranks(ga.elapsed_time(gb), dist) / args.steps

    sampler = ClockSampler(local)
    time.sleep(0.3)
    total_ms, per_op, chain, (t0, t1) = timed_steps(step, args.steps, torch, dist)
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    summ = summarise(step, sh, total_ms, per_op, chain, args.steps, peak, world)
    chain_ms = max_over_ranks(summ["chain_ms"], dist)
    tokens = R_S(sh) * world
    value = tokens / (chain_ms / 1e3)
    # the dominant kernel of the metric's chain, and both graded copy ops
    dom = max(("dispatch", "combine"), key=lambda o: summ["op_ms"][o])
    roof = roofline_entry(dom, summ, peak, peak_src, sh.name)
    roof_ops = {o: roofline_entry(o, summ, peak, peak_src, sh.name) for o in ("dispatch", "combine")}
    back_to_back_ms = (time_chain(step, max(20, min(args.steps, 200)), torch)
                       if not args.step_only else None)
    chain_graph_ms = (time_chain(step, max(20, min(args.steps, 200)), torch, graph=True)
                      if args.graph else None)

    sweep = []
    if not args.no_sweep:
        for p in SWEEPS[args.config]:
            tk, info = make_routing(sh, p, seed + 1 + len(sweep))
            s2 = Step(buf, sh, tk, seed, torch)
            for _ in range(3):
                s2.run()
            tot2, po2, ch2, _ = timed_steps(s2, args.sweep_steps, torch, None)
            m = summarise(s2, sh, tot2, po2, ch2, args.sweep_steps, peak)
            sweep.append({
                "maxvio_point": point_label(p), "maxvio": round(info["maxvio"], 4),
                "plan_dispatch_combine_tokens_per_s": m["tokens_per_s"],
                "chain_hbm_GBps": round(m["chain_hbm_GBps"], 1),
                "chain_frac_of_peak": round(m["chain_hbm_GBps"] / peak, 4),
                "step_tokens_per_s": m["whole_step"]["tokens_per_s"],
                "plan_us": round(1e3 * m["op_ms"]["plan"], 2),
                "dispatch_GBps": m["ops"]["dispatch"]["GBps"],
                "combine_GBps": m["ops"]["combine"]["GBps"],
                "dispatch_frac_of_peak": m["ops"]["dispatch"]["frac_of_peak"],
                "combine_frac_of_peak": m["ops"]["combine"]["frac_of_peak"],
                "plan_frac_of_dispatch": round(m["plan_frac_of_dispatch"], 4),
                "padding_rows": m["plan_counts"]["P"], "slots_used": m["plan_counts"]["U"]})
            del s2
        torch.cuda.synchronize()

    prep = run_prepare(buf, sh, 20, torch) if not args.step_only else None
    dedup = (run_dedup(sh, step, max(10, min(args.steps, 50)), torch, peak)
             if not args.no_dedup else None)
    mxfp4 = None
    if not args.no_mxfp4:
        mxfp4 = run_mxfp4_prefetch(buf, step, sh, max(10, min(args.steps, 50)), torch, peak)

    # free the headline step before the end-to-end and the other shapes
    step_counts = summ["plan_counts"]
    del step
    torch.cuda.empty_cache()

    e2e = None
    if not args.no_e2e:
        ms_e2e, bi, bo = run_e2e(buf, sh, topk_np, seed, args.e2e_steps, torch, dist)
        e2e = {"value": tokens / (ms_e2e / 1e3), "unit": "tokens/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": args.e2e_steps,
               "ops": "plan -> dispatch -> combine through api.Buffer, inputs copied in and "
                      "the combined rows and route weights read back every step"}
    status = buf.get_status()
    buf.destroy()
    torch.cuda.empty_cache()

    configs = {}
    for name in [c for c in args.extra_configs.split(",") if c and c != args.config]:
        configs[name] = measure_config(name, args, torch, peak)

    cpu = None
    if not args.no_cpu_baseline and rank == 0:
        cpu = cpu_baseline(sh, topk_np, seed)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": chain_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(sh, point),
        "routing": {k: v for k, v in rinfo.items() if k != "hot"},
        "plan_frac_of_dispatch": summ["plan_frac_of_dispatch"],
        "chain_hbm_GBps": summ["chain_hbm_GBps"],
        "chain_frac_of_peak": summ["chain_hbm_GBps"] / peak,
        "chain_ms_p10_p50_p90": summ["chain_ms_p10_p50_p90"],
        "whole_step": summ["whole_step"],
        "back_to_back_chain": {
            "ms": round(back_to_back_ms, 5), "tokens_per_s": tokens / (back_to_back_ms / 1e3),
            "graph_ms": round(chain_graph_ms, 5) if chain_graph_ms else None,
            "note": "plan -> dispatch -> combine issued back to back with no event between "
                    "the ops"} if back_to_back_ms else None,
        "ops": summ["ops"], "plan_counts": step_counts,
        "roofline": roof, "roofline_ops": roof_ops,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": Step.LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks, "sweep": sweep, "configs": configs, "mxfp4_prefetch": mxfp4,
        "decode_prepare": prep, "dedup_path": dedup,
        "device_status": status,
    }
    if graph_ms is not None:
        line["graph_replay"] = {"ms_per_step": graph_ms,
                                "tokens_per_s": tokens / (graph_ms / 1e3)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
