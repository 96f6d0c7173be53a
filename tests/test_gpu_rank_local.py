"""The rank-local form of the path: what each rank does when every EP rank
is its own GPU, emulated as R calls on one device.

The one exchange is the all-gather of the per-rank [E] histograms
[API, Buffer.dispatch(...): planning is collective; MoonEPCommPlan
remote_stats]; every rank then plans its own routes from the gathered
[R, E] counts (moonep_plan_rank), dispatches its own tokens into R rank
windows that are separate allocations (moonep_dispatch_rank; on R GPUs they
would be peer pointers), and gathers its tokens' rows back from those windows
(moonep_combine_rank).  The R calls together must equal the oracle's plan,
dispatch and combine bit for bit; dup_counts comes per source rank and sums
to the oracle's.  Real peer traffic between GPUs is not exercised here.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moonep_plan_gb300 import workloads as wl
from tests.plan_checks import decode

pytestmark = pytest.mark.gpu

TABLES = ("experts_to_copy", "cu_seqlens", "zero_fill_ranges", "remote_stats")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moonep_plan_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _shape(name, S, H=256):
    sh = wl.SHAPES[name]
    return wl.Shape(f"{name}_S{S}", R=sh.R, E=sh.E, K=sh.K, S=S, H=H, Hp=8, B=sh.B, tp=sh.tp,
                    weights=sh.weights)


CASES = [
    ("tiny", wl.SHAPES["tiny"], "zipf", 1.2),
    ("deepseek", _shape("deepseek_v3", 300), "zipf", 1.5),
    ("kimi_hot", _shape("kimi_k2", 256), "hot", 0.3),
    ("decode", _shape("qwen3_decode", 128, H=512), "zipf", 1.0),
    ("mixtral", _shape("mixtral", 700), "zipf", 2.0),
    ("r16_k6", wl.Shape("r16", R=16, E=64, K=6, S=90, H=64, Hp=8, B=4, tp=8,
                        weights="softmax"), "zipf", 1.3),
    ("r4_k3_small_b", wl.Shape("r4", R=4, E=16, K=3, S=77, H=136, Hp=8, B=4, tp=4,
                               weights="softmax"), "zipf", 2.5),
    # top-K that the combine stages through shared memory (2 KB and 1 KB
    # chunks), rows of several chunks
    ("r4_k5_staged", wl.Shape("r4k5", R=4, E=32, K=5, S=120, H=2048, Hp=8, B=8, tp=8,
                              weights="softmax"), "zipf", 1.2),
    ("r8_k14_staged", wl.Shape("r8k14", R=8, E=64, K=14, S=64, H=1024, Hp=8, B=8, tp=16,
                               weights="softmax"), "zipf", 1.0),
]


def _routing(sh, kind, p, seed):
    if kind == "hot":
        return wl.routing(sh, "hot", hot_share=p, seed=seed)[0]
    return wl.routing(sh, "zipf", zipf_s=p, seed=seed)[0]


@pytest.mark.parametrize("name,sh,kind,p", CASES, ids=[c[0] for c in CASES])
def test_rank_local_path_equals_oracle(name, sh, kind, p):
    from combine_moonep_plan_gb300.api import Buffer
    R, S, K, E, H, B, tp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B, sh.tp
    seed = 300 + len(name)
    topk = _routing(sh, kind, p, seed)
    hist = wl.tokens_per_expert(topk, E)            # what the all-gather delivers
    st, op = oracle.plan(R, E, K, S, B, tp, topk, hist)
    assert st == 0
    NvS = op["NvS"]
    buf = Buffer(S=S, H=H, K=K, E=E, num_ep_ranks=R, B=B, token_padding=tp,
                 zero_copy_views=False)
    hist_t = torch.from_numpy(hist).cuda()
    tk = torch.from_numpy(topk).cuda()
    plans = [buf.plan_rank(r, tk[r].contiguous(), hist_t) for r in range(R)]
    assert buf.get_status() == 0
    dup = np.zeros((R, 2), np.int64)
    for r, pl in enumerate(plans):
        assert np.array_equal(pl.dst[r].cpu().numpy(), op["dst"][r]), f"rank {r} dst"
        for f in TABLES:
            assert np.array_equal(getattr(pl, f).cpu().numpy(), op[f]), f"rank {r}: {f}"
        dup += pl.dup_counts.cpu().numpy()
    assert np.array_equal(dup, op["dup_counts"])

    # dispatch: R windows, each its own allocation, NaN-poisoned
    x = wl.hidden_bf16(sh, seed).reshape(R, S, H)
    w = wl.route_weights(sh, seed)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    wt = torch.from_numpy(w).cuda()
    wins = [torch.full((NvS, H), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(R)]
    wwins = [torch.full((NvS,), float("nan"), dtype=torch.float32, device="cuda")
             for _ in range(R)]
    for r in range(R):
        buf.dispatch_rank(plans[r], r, xt[r], wt[r], wins, wwins)
    assert buf.get_status() == 0
    want = np.full((R * NvS, H), 0x7fc0, np.uint16)
    want_w = np.full(R * NvS, np.nan, np.float32)
    oracle.dispatch(R, S, K, E, B, NvS, H, op["dst"], op["zero_fill_ranges"], x.reshape(-1, H),
                    w, want, want_w)
    nan16 = _bits(torch.tensor([float("nan")], dtype=torch.bfloat16))[0]
    for j in range(R):
        end = int(op["cu_seqlens"][j, -1])
        got = _bits(wins[j])
        assert np.array_equal(got[:end], want[j * NvS:j * NvS + end]), f"window {j}"
        assert np.all(got[end:] == nan16), f"window {j} tail written"
        gw = wwins[j].cpu().numpy()
        assert np.array_equal(gw[:end].view(np.uint32),
                              want_w[j * NvS:j * NvS + end].view(np.uint32)), f"weights {j}"

    # combine: random expert outputs in the windows, rank by rank
    rng = np.random.default_rng(seed)
    y = wl.bf16_bits_from_f32(rng.standard_normal((R * NvS, H)).astype(np.float32))
    ywins = [torch.from_numpy(y[j * NvS:(j + 1) * NvS].view(np.int16).copy())
             .view(torch.bfloat16).cuda() for j in range(R)]
    for r in range(R):
        out, wb = buf.combine_rank(plans[r], r, ywins, wwins)
        ref, ref_w = oracle.combine(R, S, K, NvS, H, op["dst"], y, want_w,
                                    tokens=np.arange(r * S, (r + 1) * S))
        assert np.array_equal(_bits(out), ref), f"rank {r} combine"
        assert np.array_equal(wb.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))
    assert buf.get_status() == 0
    buf.destroy()


def test_rank_local_and_whole_planner_interleave():
    """Rank-local calls keep their own counters and totals: a whole-problem
    plan, the R rank-local plans and another whole-problem plan of another
    routing on one context are each right."""
    from combine_moonep_plan_gb300.api import Buffer
    sh = _shape("deepseek_v3", 200)
    buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                 token_padding=sh.tp, zero_copy_views=False)
    for it in range(3):
        topk = _routing(sh, "zipf", 1.2 + 0.3 * it, 500 + it)
        hist = wl.tokens_per_expert(topk, sh.E)
        st, op = oracle.plan(sh.R, sh.E, sh.K, sh.S, sh.B, sh.tp, topk)
        tk = torch.from_numpy(topk).cuda()
        whole = buf.plan(tk)
        ht = torch.from_numpy(hist).cuda()
        local = buf.new_plan()
        for r in range(sh.R):
            buf.plan_rank(r, tk[r].contiguous(), ht, plan=local)
        assert buf.get_status() == 0
        for f in ("dst",) + TABLES:
            assert np.array_equal(getattr(whole, f).cpu().numpy(), op[f]), f
            assert np.array_equal(getattr(local, f).cpu().numpy(), op[f]), f


def test_rank_local_histogram_mismatch_and_refusals():
    from combine_moonep_plan_gb300 import _lib
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.SHAPES["tiny"]
    topk = _routing(sh, "zipf", 1.2, 9)
    hist = wl.tokens_per_expert(topk, sh.E)
    buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B, token_padding=sh.tp,
                 zero_copy_views=False)
    tk = torch.from_numpy(topk).cuda()
    bad = hist.copy()
    e = int(np.argmax(bad[1]))
    bad[1, e] -= 1                    # one route moved to another expert: totals
    bad[1, (e + 1) % sh.E] += 1       # still sum to S*K, rank 1's row is wrong
    buf.plan_rank(1, tk[1].contiguous(), torch.from_numpy(bad).cuda())
    assert buf.get_status() == _lib.ERR_HIST_MISMATCH
    # the next call plans correctly
    p = buf.plan_rank(0, tk[0].contiguous(), torch.from_numpy(hist).cuda())
    assert buf.get_status() == 0
    st, op = oracle.plan(sh.R, sh.E, sh.K, sh.S, sh.B, sh.tp, topk)
    assert np.array_equal(p.dst[0].cpu().numpy(), op["dst"][0])
    with pytest.raises(_lib.MoonepError):
        buf.plan_rank(sh.R, tk[0].contiguous(), torch.from_numpy(hist).cuda())
    dbuf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                  token_padding=sh.tp, zero_copy_views=False, dup_records=True)
    with pytest.raises(_lib.MoonepError):
        dbuf.plan_rank(0, tk[0].contiguous(), torch.from_numpy(hist).cuda())
