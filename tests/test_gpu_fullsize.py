"""Parity at the five workload shapes' full sizes, in the launch configuration
bench.py uses.

* the plan is compared with the oracle's bit for bit (every field);
* dispatch is checked in full on the device as the scatter it is (every
  route's row equals its token's row, every padding row and weight is zero,
  every route weight lands), and against the oracle on sampled tokens;
* combine is checked against the oracle on sampled tokens (the oracle computes
  them one by one from the gathered rows) and, in full, by the closed form
  combine(dispatch(x)) = K*x;
* prefetch in full (every used slot equals its home row, unused slots keep
  their checksum); gradient reduce against the oracle on sampled columns.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moonep_plan_gb300 import workloads as wl
from tests.plan_checks import decode

pytestmark = pytest.mark.gpu

POINTS = [("tiny", "zipf1.2"), ("mixtral", 1.0), ("mixtral", 3.0), ("deepseek_v3", 2.0),
          ("deepseek_v3", 0.0), ("kimi_k2", "hot30"), ("qwen3_decode", "zipf1")]


def _routing(sh, point, seed):
    if point == "hot30":
        return wl.routing(sh, "hot", hot_share=0.30, seed=seed)[0]
    if point == "zipf1":
        return wl.routing(sh, "zipf", zipf_s=1.0, seed=seed)[0]
    if point == "zipf1.2":
        return wl.routing(sh, "zipf", zipf_s=1.2, seed=seed)[0]
    if point == 0.0:
        return wl.routing(sh, "exact0", seed=seed)[0]
    return wl.routing(sh, "zipf", target_maxvio=float(point), seed=seed)[0]


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moonep_plan_gb300 import build
    build.build()
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,point", POINTS, ids=[f"{n}-{p}" for n, p in POINTS])
def test_full_size_parity(name, point):
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.SHAPES[name]
    R, S, K, E, H, Hp, B, tp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.Hp, sh.B, sh.tp
    seed = wl.seed_for(name, 7)
    topk = _routing(sh, point, seed)
    tpe = wl.tokens_per_expert(topk, E)
    st, op = oracle.plan(R, E, K, S, B, tp, topk, tpe, dup_records=False)
    assert st == 0
    NvS = op["NvS"]

    buf = Buffer(S=S, H=H, K=K, E=E, num_ep_ranks=R, B=B, token_padding=tp,
                 zero_copy_views=False)
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn((R, S, H), generator=g, device=dev).to(torch.bfloat16)
    w = torch.from_numpy(wl.route_weights(sh, seed)).to(dev)
    out = torch.full((R * NvS, H), float("nan"), dtype=torch.bfloat16, device=dev)
    wout = torch.full((R * NvS,), float("nan"), dtype=torch.float32, device=dev)
    hid, wn, cu, plan = buf.dispatch(x, w, torch.from_numpy(topk).to(dev),
                                     torch.from_numpy(tpe).to(dev), out=out, weights_out=wout)
    assert buf.get_status() == 0

    # plan: bit-exact with the oracle
    for f in ("dst", "experts_to_copy", "cu_seqlens", "zero_fill_ranges", "remote_stats",
              "dup_counts"):
        assert np.array_equal(getattr(plan, f).cpu().numpy(), op[f]), f

    # dispatch: the full scatter, on the device
    gidx = torch.from_numpy(decode(op["dst"]).reshape(-1)).to(dev)
    tok = torch.arange(R * S, device=dev).repeat_interleave(K)
    xf = x.reshape(R * S, H)
    for c0 in range(0, gidx.numel(), 1 << 16):
        c1 = c0 + (1 << 16)
        assert torch.equal(hid[gidx[c0:c1]].view(torch.int16), xf[tok[c0:c1]].view(torch.int16))
    assert torch.equal(wn[gidx].view(torch.int32), w.reshape(-1).view(torch.int32))
    zfr = op["zero_fill_ranges"]
    pad = np.concatenate([np.arange(j * NvS + a, j * NvS + b) for j in range(R)
                          for a, b in zfr[j] if b > a] or [np.zeros(0, np.int64)])
    if len(pad):
        pt = torch.from_numpy(pad).to(dev)
        assert torch.all(hid[pt].view(torch.int16) == 0)
        assert torch.all(wn[pt].view(torch.int32) == 0)
    # sampled tokens against the oracle's dispatch of those tokens' rows
    rng = np.random.default_rng(seed)
    toks = np.unique(rng.integers(0, R * S, 256))
    rows = decode(op["dst"]).reshape(R * S, K)[toks]
    got = _bits(hid[torch.from_numpy(rows.reshape(-1)).to(dev)]).reshape(len(toks), K, H)
    xs = _bits(xf[torch.from_numpy(toks).to(dev)])
    sub_dst = np.arange(len(toks) * K, dtype=np.int32).reshape(1, -1)
    want = oracle.dispatch(1, len(toks), K, 0, 0, len(toks) * K, H, sub_dst,
                           np.zeros((1, 0, 2), np.int32), xs)
    assert np.array_equal(got.reshape(-1, H), want)

    # combine: sampled tokens via the oracle, plus the closed form in full
    y = torch.randn((R * NvS, H), generator=g, device=dev).to(torch.bfloat16)
    cout, cw = buf.combine(plan, y, wn)
    assert buf.get_status() == 0
    ysub = _bits(y[torch.from_numpy(rows.reshape(-1)).to(dev)])
    want, _ = oracle.combine(1, len(toks), K, len(toks) * K, H,
                             np.arange(len(toks) * K, dtype=np.int32), ysub)
    assert np.array_equal(_bits(cout.reshape(R * S, H)[torch.from_numpy(toks).to(dev)]), want)
    assert torch.equal(cw.reshape(-1).view(torch.int32), w.reshape(-1).view(torch.int32))
    if K & (K - 1) == 0:
        ident, _ = buf.combine(plan, hid)
        assert torch.equal(ident.float(), x.float() * K)
    del y, out, wout, cout, cw, hid, wn, x

    # prefetch: every used slot equals its home row; unused slots untouched
    etc = op["experts_to_copy"]
    W = torch.randn((E + R * B, H, Hp), generator=g, device=dev).to(torch.bfloat16)
    W32 = W.view(E + R * B, -1).view(torch.int32)

    def checksums():
        return torch.stack([W32[i].to(torch.int64).sum() for i in range(E + R * B)]).cpu()
    before = checksums()
    buf.prefetch_weight(plan, W)
    after = checksums()
    for j in range(R):
        for b in range(B):
            row = E + j * B + b
            if etc[j, b] >= 0:
                assert torch.equal(W[row].view(torch.int16), W[etc[j, b]].view(torch.int16))
            else:
                assert before[row] == after[row]
    del W, W32

    # gradient reduce: sampled column windows against the oracle
    HHp = H * Hp
    Gh = torch.randn((E, H, Hp), generator=g, device=dev)
    Gs = torch.randn((R, B, H, Hp), generator=g, device=dev)
    wins = [(0, 4096), (HHp // 2 - 2048, HHp // 2 + 2048), (HHp - 4096, HHp)]
    gh0 = [Gh.view(E, -1)[:, a:b].cpu().numpy().copy() for a, b in wins]
    gs0 = [Gs.view(R * B, -1)[:, a:b].cpu().numpy().copy() for a, b in wins]
    buf.reduce_grad(plan, [Gh], [Gs])
    assert buf.get_status() == 0
    for (a, b), gh, gs in zip(wins, gh0, gs0):
        oracle.reduce(R, E, B, etc.reshape(-1), gh, gs, b - a)
        assert np.array_equal(Gh.view(E, -1)[:, a:b].cpu().numpy().view(np.uint32),
                              gh.view(np.uint32))
        assert np.array_equal(Gs.view(R * B, -1)[:, a:b].cpu().numpy().view(np.uint32),
                              gs.view(np.uint32))
    buf.destroy()


@pytest.mark.parametrize("name,point", [("deepseek_v3", 2.0), ("kimi_k2", "hot30")])
def test_full_size_mxfp4_prefetch(name, point):
    """A full-size packed MXFP4 gate/up/down set with its E8M0 block scales
    ([E + R*B, H, H'/2] and [E + R*B, H, H'/32] uint8), one launch: every used
    slot equals its source expert's row, every unused slot and home row keeps
    its checksum."""
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.SHAPES[name]
    R, E, B, H, Hp = sh.R, sh.E, sh.B, sh.H, sh.Hp
    seed = wl.seed_for(name, 9)
    topk = _routing(sh, point, seed)
    st, op = oracle.plan(R, E, sh.K, sh.S, B, sh.tp, topk, wl.tokens_per_expert(topk, E),
                         dup_records=False)
    assert st == 0
    etc = op["experts_to_copy"]
    buf = Buffer(S=sh.S, H=H, K=sh.K, E=E, num_ep_ranks=R, B=B, token_padding=sh.tp,
                 zero_copy_views=False)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    rows = E + R * B
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    ts = [torch.randint(0, 256, (rows, H, Hp // 2), generator=g, device="cuda",
                        dtype=torch.uint8) for _ in range(3)]
    ts += [torch.randint(0, 256, (rows, H, Hp // 32), generator=g, device="cuda",
                         dtype=torch.uint8) for _ in range(3)]

    def sums(t):
        return t.view(rows, -1).view(torch.int32).to(torch.int64).sum(dim=1).cpu()
    before = [sums(t) for t in ts]
    buf.prefetch_weight(plan, *ts[:3], scales=ts[3:])
    assert buf.get_status() == 0
    for t, b0 in zip(ts, before):
        after = sums(t)
        for j in range(R):
            for b in range(B):
                row = E + j * B + b
                if etc[j, b] >= 0:
                    assert torch.equal(t[row], t[etc[j, b]])
                else:
                    assert after[row] == b0[row]
        assert torch.equal(after[:E], b0[:E])
        del t
    del ts
    buf.destroy()


def test_full_size_three_projections():
    """The gate/up/down case at the DeepSeek-V3 shape's full size (three bf16
    [E + R*B, H, H'] weight tensors, 15 GB each, in one prefetch call; three
    projections of fp32 gradients in one reduce call): every used slot equals
    its home row, unused slots keep their contents, and the reduce matches the
    oracle on sampled column windows of every projection."""
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.SHAPES["deepseek_v3"]
    R, E, B, H, Hp = sh.R, sh.E, sh.B, sh.H, sh.Hp
    seed = wl.seed_for("deepseek_v3", 13)
    topk = _routing(sh, 2.0, seed)
    st, op = oracle.plan(R, E, sh.K, sh.S, B, sh.tp, topk, wl.tokens_per_expert(topk, E),
                         dup_records=False)
    assert st == 0
    etc = op["experts_to_copy"]
    buf = Buffer(S=sh.S, H=H, K=sh.K, E=E, num_ep_ranks=R, B=B, token_padding=sh.tp,
                 zero_copy_views=False)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    rows = E + R * B
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    Ws = []
    for _ in range(3):
        w = torch.empty((rows, H, Hp), dtype=torch.bfloat16, device="cuda")
        w.normal_(generator=g)
        Ws.append(w)
    unused = [E + j * B + b for j in range(R) for b in range(B) if etc[j, b] < 0]
    ui = torch.tensor(unused, dtype=torch.int64, device="cuda")

    def unused_sums(w):
        w32 = w.view(rows, -1).view(torch.int32)
        return torch.stack([w32[i].to(torch.int64).sum() for i in unused]).cpu() \
            if unused else torch.zeros(0, dtype=torch.int64)
    before = [unused_sums(w) for w in Ws]
    buf.prefetch_weight(plan, *Ws)
    assert buf.get_status() == 0
    for w, b0 in zip(Ws, before):
        for j in range(R):
            for b in range(B):
                if etc[j, b] >= 0:
                    assert torch.equal(w[E + j * B + b].view(torch.int16),
                                       w[etc[j, b]].view(torch.int16))
        assert torch.equal(unused_sums(w), b0)
    del Ws, ui
    torch.cuda.empty_cache()

    HHp = H * Hp
    Gh = [torch.empty((E, H, Hp), device="cuda").normal_(generator=g) for _ in range(3)]
    Gs = [torch.empty((R, B, H, Hp), device="cuda").normal_(generator=g) for _ in range(3)]
    wins = [(0, 2048), (HHp // 3, HHp // 3 + 2048), (HHp - 2048, HHp)]
    gh0 = [[t.view(E, -1)[:, a:b].cpu().numpy().copy() for a, b in wins] for t in Gh]
    gs0 = [[t.view(R * B, -1)[:, a:b].cpu().numpy().copy() for a, b in wins] for t in Gs]
    buf.reduce_grad(plan, Gh, Gs)
    assert buf.get_status() == 0
    for p in range(3):
        for (a, b), gh, gs in zip(wins, gh0[p], gs0[p]):
            oracle.reduce(R, E, B, etc.reshape(-1), gh, gs, b - a)
            assert np.array_equal(Gh[p].view(E, -1)[:, a:b].cpu().numpy().view(np.uint32),
                                  gh.view(np.uint32))
            assert np.array_equal(Gs[p].view(R * B, -1)[:, a:b].cpu().numpy().view(np.uint32),
                                  gs.view(np.uint32))
    del Gh, Gs
    buf.destroy()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("R,E,K,S,B,H", [(8, 160, 6, 4096, 20, 5120), (8, 512, 10, 2048, 64, 2048),
                                         (8, 128, 3, 8192, 16, 4096)])
def test_full_size_other_top_k(R, E, K, S, B, H):
    """Top-K values outside the five workload shapes (top-6 with 160 experts,
    top-10 with 512, top-3), at full batch sizes: the single-launch planner
    with whole-token warp chunks (several tiles per rank) against the oracle's
    plan bit for bit, the dispatch scatter in full on the device, and the
    combine by its closed form in fp32 (K copies of a row add exactly)."""
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.Shape("topk", R=R, E=E, K=K, S=S, H=H, Hp=64, B=B, tp=128, weights="softmax")
    seed = 4242 + K
    topk = wl.routing(sh, "zipf", target_maxvio=1.5, seed=seed)[0]
    tpe = wl.tokens_per_expert(topk, E)
    st, op = oracle.plan(R, E, K, S, B, 128, topk, tpe, dup_records=False)
    assert st == 0
    buf = Buffer(S=S, H=H, K=K, E=E, num_ep_ranks=R, B=B, token_padding=128,
                 zero_copy_views=False)
    dev = "cuda"
    x = torch.randn((R, S, H), device=dev).to(torch.bfloat16)
    hid, _, _, plan = buf.dispatch(x, None, torch.from_numpy(topk).to(dev),
                                   torch.from_numpy(tpe).to(dev))
    assert buf.get_status() == 0
    for f in ("dst", "experts_to_copy", "cu_seqlens", "zero_fill_ranges", "remote_stats",
              "dup_counts"):
        assert np.array_equal(getattr(plan, f).cpu().numpy(), op[f]), f
    gidx = torch.from_numpy(decode(op["dst"]).reshape(-1)).to(dev)
    tok = torch.arange(R * S, device=dev).repeat_interleave(K)
    xf = x.reshape(R * S, H)
    for c0 in range(0, gidx.numel(), 1 << 16):
        c1 = c0 + (1 << 16)
        assert torch.equal(hid[gidx[c0:c1]].view(torch.int16), xf[tok[c0:c1]].view(torch.int16))
    out, _ = buf.combine(plan, hid)
    assert torch.equal(out.view(torch.int16), (x.float() * K).to(torch.bfloat16).view(torch.int16))
    buf.destroy()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,point", [("deepseek_v3", 1.0), ("kimi_k2", "hot30")])
def test_full_size_plan_reuse_dispatch(name, point):
    """Combine-backward dispatch at full size, launched as bench.py launches
    it: a bf16 [R, S, H] gradient dispatched with a clone of the forward plan
    and no weights [API, Buffer.dispatch with a saved plan].  Every row of
    every rank is compared with the oracle's dispatch on two column windows
    (the first and last 64 columns: dispatch moves columns independently);
    tail rows keep their poison in full; the forward's route weights are
    left as they were."""
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.SHAPES[name]
    R, S, K, E, H, B, tp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B, sh.tp
    seed = wl.seed_for(name, 11)
    topk = _routing(sh, point, seed)
    st, op = oracle.plan(R, E, K, S, B, tp, topk, None, dup_records=False)
    assert st == 0
    NvS = op["NvS"]
    buf = Buffer(S=S, H=H, K=K, E=E, num_ep_ranks=R, B=B, token_padding=tp,
                 zero_copy_views=False)
    dev = "cuda"
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    x = torch.randn((R, S, H), generator=gen, device=dev).to(torch.bfloat16)
    w = torch.from_numpy(wl.route_weights(sh, seed)).to(dev)
    hid, wn, _, plan = buf.dispatch(x, w, torch.from_numpy(topk).to(dev))
    saved = plan.clone()
    del hid
    torch.cuda.synchronize()
    wn0 = wn.clone()
    grad = torch.randn((R, S, H), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.full((R * NvS, H), float("nan"), dtype=torch.bfloat16, device=dev)
    nan_bits = int(out[0, 0].view(torch.int16).item())
    buf.dispatch(grad, plan=saved, out=out)
    assert buf.get_status() == 0
    assert torch.equal(wn.view(torch.int32), wn0.view(torch.int32))
    ends = op["cu_seqlens"][:, -1]
    for c0 in (0, H - 64):
        gcols = _bits(grad.reshape(R * S, H)[:, c0:c0 + 64].contiguous())
        want = oracle.dispatch(R, S, K, E, B, NvS, 64, op["dst"], op["zero_fill_ranges"], gcols)
        got = _bits(out[:, c0:c0 + 64].contiguous())
        for j in range(R):
            lo = j * NvS
            assert np.array_equal(got[lo:lo + ends[j]], want[lo:lo + ends[j]]), (c0, j)
    for j in range(R):
        tail = out[j * NvS + int(ends[j]):(j + 1) * NvS].view(torch.int16)
        assert torch.all(tail == nan_bits), f"rank {j} tail written"
    del out, grad, x, wn, wn0
