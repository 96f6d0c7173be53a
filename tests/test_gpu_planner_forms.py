"""The planner's launch forms on small batches, against the oracle.

The whole-problem planner runs as one launch of G + 2 blocks that meet once
[API, Buffer.dispatch(...): the planning step; README items 1-2].  When
those blocks fit in one thread-block cluster (decode-sized batches) they are
launched as a cluster and meet at its hardware barrier; otherwise as a
cooperative launch that meets on an arrival counter.  Rank-local calls have a
counter of their own.  These tests run small batches through a fresh
dispatch (plan, then dispatch) and check against the oracle's plan and
dispatch, bit for bit (plan arrays, every valid and padding row and weight,
tail rows left as they were): repeated calls, interleaving with the other
forms on one context, CUDA-graph replay (the meeting's targets are derived
on the device, so replays need nothing from the host), and the error and
wait-limit paths.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moonep_plan_gb300 import workloads as wl
from tests.plan_checks import decode

pytestmark = pytest.mark.gpu

FIELDS = ("dst", "experts_to_copy", "cu_seqlens", "zero_fill_ranges", "remote_stats",
          "dup_counts")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moonep_plan_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _buf(sh, **kw):
    from combine_moonep_plan_gb300.api import Buffer
    return Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B, token_padding=sh.tp,
                  zero_copy_views=False, **kw)


def _inputs(sh, seed):
    x = wl.hidden_bf16(sh, seed).reshape(sh.R, sh.S, sh.H)
    w = wl.route_weights(sh, seed)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return x, w, xt, torch.from_numpy(w).cuda()


def _check(sh, topk, plan, hid, wn, x, w, tpe=None):
    R, S, K, E, H, B, tp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B, sh.tp
    st, op = oracle.plan(R, E, K, S, B, tp, topk, tpe, dup_records=False)
    assert st == 0
    for f in FIELDS:
        assert np.array_equal(getattr(plan, f).cpu().numpy(), op[f]), f
    NvS = op["NvS"]
    want = np.full((R * NvS, H), 0x7fc0, np.uint16)
    want_w = np.full(R * NvS, np.nan, np.float32)
    oracle.dispatch(R, S, K, E, B, NvS, H, op["dst"], op["zero_fill_ranges"], x.reshape(-1, H),
                    w, want, want_w)
    got, gw = _bits(hid), wn.cpu().numpy()
    for j in range(R):
        end = int(op["cu_seqlens"][j, -1])
        lo = j * NvS
        assert np.array_equal(got[lo:lo + end], want[lo:lo + end]), f"rank {j} rows"
        assert np.array_equal(gw[lo:lo + end].view(np.uint32),
                              want_w[lo:lo + end].view(np.uint32)), f"rank {j} weights"
        assert np.all((got[lo + end:lo + NvS] & 0x7f80) == 0x7f80), f"rank {j} tail written"
    return op


def _poisoned(buf, sh):
    rows = torch.full((sh.R * buf.NvS, sh.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    wts = torch.full((sh.R * buf.NvS,), float("nan"), dtype=torch.float32, device="cuda")
    return rows, wts


def _decode_shape(H=4096, S=128):
    sh = wl.SHAPES["qwen3_decode"]
    return wl.Shape("decode", R=sh.R, E=sh.E, K=sh.K, S=S, H=H, Hp=8, B=sh.B, tp=sh.tp,
                    weights=sh.weights)


CASES = [
    ("decode_full", _decode_shape(), "zipf", 1.0),
    ("decode_uniform", _decode_shape(), "uniform", None),
    ("decode_S37", _decode_shape(H=1024, S=37), "zipf", 1.5),
    ("tiny", wl.SHAPES["tiny"], "zipf", 1.2),
    ("k2_e8", wl.Shape("m", R=8, E=8, K=2, S=200, H=512, Hp=8, B=1, tp=16,
                       weights="softmax"), "zipf", 2.0),
    ("k6_r4", wl.Shape("k6", R=4, E=24, K=6, S=150, H=264, Hp=8, B=6, tp=8,
                       weights="softmax"), "zipf", 1.4),
    ("k16", wl.Shape("k16", R=8, E=64, K=16, S=48, H=128, Hp=8, B=8, tp=4,
                     weights="softmax"), "zipf", 1.1),
]


@pytest.mark.parametrize("name,sh,kind,p", CASES, ids=[c[0] for c in CASES])
def test_small_batch_plan_dispatch_equals_oracle(name, sh, kind, p):
    buf = _buf(sh)
    seed = 700 + len(name)
    topk = (wl.routing(sh, "uniform", seed=seed)[0] if kind == "uniform"
            else wl.routing(sh, "zipf", zipf_s=p, seed=seed)[0])
    tpe = wl.tokens_per_expert(topk, sh.E)
    x, w, xt, wt = _inputs(sh, seed)
    plan = buf.new_plan()
    for call in range(3):        # repeated calls: the meeting's targets move on
        rows, wts = _poisoned(buf, sh)
        buf.dispatch(xt, wt, torch.from_numpy(topk).cuda(), torch.from_numpy(tpe).cuda(),
                     out=rows, weights_out=wts, plan_out=plan)
        assert buf.get_status() == 0
        _check(sh, topk, plan, rows, wts, x, w, tpe)


def test_planner_forms_interleaved():
    """Whole-problem plans (alone and inside a fresh dispatch) and rank-local
    plans on one context, interleaved over several routings: each form keeps
    its own counters and totals, and every result equals the oracle's."""
    sh = _decode_shape(H=512)
    buf = _buf(sh)
    x, w, xt, wt = _inputs(sh, 5)
    for it in range(4):
        topk = wl.routing(sh, "zipf", zipf_s=0.8 + 0.3 * it, seed=900 + it)[0]
        tk = torch.from_numpy(topk).cuda()
        st, op = oracle.plan(sh.R, sh.E, sh.K, sh.S, sh.B, sh.tp, topk, dup_records=False)
        plain = buf.plan(tk)
        rows, wts = _poisoned(buf, sh)
        _, _, _, fresh = buf.dispatch(xt, wt, tk, out=rows, weights_out=wts)
        hist = torch.from_numpy(wl.tokens_per_expert(topk, sh.E)).cuda()
        local = buf.new_plan()
        for r in range(sh.R):
            buf.plan_rank(r, tk[r].contiguous(), hist, plan=local)
        assert buf.get_status() == 0
        for f in ("dst", "cu_seqlens", "zero_fill_ranges", "experts_to_copy"):
            assert np.array_equal(getattr(plain, f).cpu().numpy(), op[f]), f
            assert np.array_equal(getattr(local, f).cpu().numpy(), op[f]), f
        _check(sh, topk, fresh, rows, wts, x, w)


def test_plan_dispatch_combine_graph_replay():
    """plan, dispatch then combine captured once in a CUDA graph and replayed
    with new routings copied into the captured inputs: every replay equals
    the oracle's plan, dispatch and combine."""
    sh = _decode_shape(H=1024)
    buf = _buf(sh)
    x, w, xt, wt = _inputs(sh, 8)
    tk = torch.zeros((sh.R, sh.S, sh.K), dtype=torch.int32, device="cuda")
    first = wl.routing(sh, "zipf", zipf_s=1.0, seed=40)[0]
    tk.copy_(torch.from_numpy(first))
    plan = buf.new_plan()
    rows, wts = _poisoned(buf, sh)
    out = torch.empty((sh.R, sh.S, sh.H), dtype=torch.bfloat16, device="cuda")
    wback = torch.empty((sh.R, sh.S, sh.K), dtype=torch.float32, device="cuda")

    def chain():
        buf.dispatch(xt, wt, tk, out=rows, weights_out=wts, plan_out=plan)
        buf.combine(plan, rows, wts, out=out, weights_out=wback)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for rep in range(4):
        topk = wl.routing(sh, "zipf", zipf_s=0.7 + 0.4 * rep, seed=41 + rep)[0]
        tk.copy_(torch.from_numpy(topk))
        rows.fill_(float("nan"))
        wts.fill_(float("nan"))
        graph.replay()
        assert buf.get_status() == 0
        op = _check(sh, topk, plan, rows, wts, x, w)
        ref, ref_w = oracle.combine(sh.R, sh.S, sh.K, op["NvS"], sh.H, op["dst"], _bits(rows),
                                    wts.cpu().numpy())
        assert np.array_equal(_bits(out).reshape(sh.R * sh.S, sh.H), ref)
        assert np.array_equal(wback.cpu().numpy().reshape(-1, sh.K).view(np.uint32),
                              ref_w.view(np.uint32))


def test_small_batch_errors_and_wait_limit(monkeypatch):
    """A bad expert id and a wrong tokens_per_expert latch their errors; a
    planner wait that can never be satisfied (test hook) gives up, latches
    MOONEP_ERR_TIMEOUT and leaves a plan the dispatch consumes inside its
    buffers; a context without the hook then plans and dispatches
    correctly."""
    from combine_moonep_plan_gb300 import _lib
    sh = _decode_shape(H=256)
    x, w, xt, wt = _inputs(sh, 3)
    topk = wl.routing(sh, "zipf", zipf_s=1.0, seed=3)[0]
    buf = _buf(sh)
    bad = topk.copy()
    bad[2, 5, 1] = sh.E
    rows, wts = _poisoned(buf, sh)
    buf.dispatch(xt, wt, torch.from_numpy(bad).cuda(), out=rows, weights_out=wts)
    assert buf.get_status() == _lib.ERR_BAD_EXPERT
    tpe = wl.tokens_per_expert(topk, sh.E)
    tpe_bad = tpe.copy()
    tpe_bad[0, 0] += 1
    rows, wts = _poisoned(buf, sh)
    _, _, _, plan = buf.dispatch(xt, wt, torch.from_numpy(topk).cuda(),
                                 torch.from_numpy(tpe_bad).cuda(), out=rows, weights_out=wts)
    assert buf.get_status() == _lib.ERR_HIST_MISMATCH
    _check(sh, topk, plan, rows, wts, x, w)     # built from the recount
    monkeypatch.setenv("MOONEP_TEST_PLANNER_TIMEOUT", "1")
    hung = _buf(sh)
    monkeypatch.delenv("MOONEP_TEST_PLANNER_TIMEOUT")
    rows, wts = _poisoned(hung, sh)
    _, _, _, plan = hung.dispatch(xt, wt, torch.from_numpy(topk).cuda(), out=rows,
                                  weights_out=wts)
    assert hung.get_status() == _lib.ERR_TIMEOUT
    g = decode(plan.dst.cpu().numpy())
    assert g.min() >= 0 and g.max() < sh.R * hung.NvS
    rows, wts = _poisoned(buf, sh)
    _, _, _, plan = buf.dispatch(xt, wt, torch.from_numpy(topk).cuda(), out=rows,
                                 weights_out=wts)
    assert buf.get_status() == 0
    _check(sh, topk, plan, rows, wts, x, w)
