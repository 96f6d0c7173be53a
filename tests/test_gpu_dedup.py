"""GPU parity of the deduplicated data flow (dispatch with an expand epilogue,
combine with a duplicate prologue) against the oracle.

* moonep_dispatch_dedup: bit-exact with the oracle's dispatch (every route's
  row, every padding row, every weight) and with moonep_dispatch;
* moonep_combine_dedup: the folded rows bit-exact with the oracle's
  fold_duplicates, the output bit-exact with the oracle's fold followed by
  combine_primaries (both sides add in the same order in fp32 and round once
  per step);
* the closed form of the combine of a dispatch: every duplicate row equals
  its primary, so for top-2 the fold (x + x) and the sum stay exact and
  combine(dispatch(x)) = 2x; with more routes a fold of three or more copies
  of x rounds, and the result stays within 2^-7 * K|x| of K*x;
* full size (DeepSeek-V3 shape): the whole scatter on the device and sampled
  tokens through the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moonep_plan_gb300 import workloads as wl
from tests.plan_checks import decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moonep_plan_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    torch.cuda.empty_cache()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _shape(name, S, H):
    sh = wl.SHAPES[name]
    return wl.Shape(f"{name}_S{S}_H{H}", R=sh.R, E=sh.E, K=sh.K, S=S, H=H, Hp=64, B=sh.B,
                    tp=sh.tp, weights=sh.weights)


CASES = [
    # (shape, S, H, routing): several 4 KB / 2 KB chunks and a ragged tail
    ("deepseek_v3", 64, 4104, "uniform"),
    ("deepseek_v3", 48, 512, "zipf"),
    ("kimi_k2", 32, 1032, "hot"),
    ("mixtral", 128, 2056, "zipf"),
    ("qwen3_decode", 24, 776, "exact0"),
    ("tiny", 64, 256, "zipf"),
]


def _routing(sh, kind, seed):
    if kind == "uniform":
        return wl.routing(sh, "uniform", seed=seed)[0]
    if kind == "zipf":
        return wl.routing(sh, "zipf", zipf_s=1.2, seed=seed)[0]
    if kind == "hot":
        return wl.routing(sh, "hot", hot_share=0.3, seed=seed)[0]
    if kind == "exact0":
        return wl.routing(sh, "exact0", seed=seed)[0]
    raise ValueError(kind)


def _check_identity(got, x, K):
    """combine(dispatch(x)) against K*x: exact for K <= 2 (a fold adds x + x),
    else within the folds' roundings (half an ulp of each rank's partial
    sum, at most 2^-8 * K|x| together) and the final rounding (2^-8 * K|x|)."""
    if K <= 2:
        assert np.array_equal(got, x * K)
    else:
        assert np.all(np.abs(got - x * K) <= np.abs(x) * K * 2.0 ** -7)


def _buffer(sh, dup=True):
    from combine_moonep_plan_gb300.api import Buffer
    return Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                  token_padding=sh.tp, zero_copy_views=False, dup_records=dup)


@pytest.mark.parametrize("name,S,H,kind", CASES, ids=[f"{c[0]}-S{c[1]}-H{c[2]}-{c[3]}"
                                                     for c in CASES])
def test_dedup_parity(name, S, H, kind):
    sh = _shape(name, S, H)
    seed = wl.seed_for(name, 31) + S
    _dedup_parity(sh, _routing(sh, kind, seed), seed)


@pytest.mark.parametrize("seed", range(12))
def test_dedup_random_small_configs(seed):
    """Random R, E, K (including K outside the specialised set, so the generic
    combine runs in its primaries-only form), S, B, token_padding and H, with
    repeated experts inside a token (many duplicates on one rank)."""
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.integers(1, 9))
    L = int(rng.integers(1, 9))
    E = R * L
    K = int(rng.choice([2, 3, 4, 5, 6, 8, 12]))
    S = int(rng.integers(1, 400))
    B = L + int(rng.integers(0, 3))
    tp = int(rng.choice([1, 2, 8, 16]))
    H = int(rng.choice([8, 64, 136, 2056]))
    sh = wl.Shape("rand", R=R, E=E, K=K, S=S, H=H, Hp=16, B=B, tp=tp, weights="softmax")
    p = rng.random(E) ** 4
    topk = rng.choice(E, size=(R, S, K), p=p / p.sum()).astype(np.int32)
    _dedup_parity(sh, topk, seed)


def _dedup_parity(sh, topk, seed):
    R, S, K, E, B, tp, H = sh.R, sh.S, sh.K, sh.E, sh.B, sh.tp, sh.H
    tpe = wl.tokens_per_expert(topk, E)
    st, op = oracle.plan(R, E, K, S, B, tp, topk, tpe)
    assert st == 0
    NvS = op["NvS"]
    buf = _buffer(sh)
    x = wl.hidden_bf16(sh, seed)
    w = wl.route_weights(sh, seed)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).reshape(R, S, H).cuda()
    wt = torch.from_numpy(w).cuda()
    plan = buf.plan(torch.from_numpy(topk).cuda(), torch.from_numpy(tpe).cuda())

    # dispatch: dedup and plain into NaN-poisoned buffers
    def run_dispatch(dedup):
        out = torch.full((R * NvS, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        wout = torch.full((R * NvS,), float("nan"), dtype=torch.float32, device="cuda")
        buf.dispatch(xt, wt, plan=plan, out=out, weights_out=wout, dedup=dedup)
        assert buf.get_status() == 0
        return out, wout
    hd, wd = run_dispatch(True)
    hp, wp = run_dispatch(False)
    want = np.full((R * NvS, H), 0x7fc0, np.uint16)
    want_w = np.full(R * NvS, np.nan, np.float32)
    oracle.dispatch(R, S, K, E, B, NvS, H, op["dst"], op["zero_fill_ranges"], x, w, want,
                    want_w)
    got = _bits(hd)
    touched = np.zeros(R * NvS, bool)
    touched[decode(op["dst"]).reshape(-1)] = True
    for j in range(R):
        for a, b in op["zero_fill_ranges"][j]:
            touched[j * NvS + a:j * NvS + b] = True
    assert np.array_equal(got[touched], want[touched]), "deduplicated dispatch differs"
    assert np.array_equal(wd.cpu().numpy()[touched].view(np.uint32),
                          want_w[touched].view(np.uint32))
    # bit for bit the plain dispatch, NaN poison of the tail included
    assert torch.equal(hd.view(torch.int16), hp.view(torch.int16))
    assert torch.equal(wd.view(torch.int32), wp.view(torch.int32))

    # combine: random expert outputs, padding and tail NaN-poisoned
    rng = np.random.default_rng(seed + 5)
    y = wl.bf16_bits_from_f32(rng.standard_normal((R * NvS, H)).astype(np.float32))
    valid = np.zeros(R * NvS, bool)
    valid[decode(op["dst"]).reshape(-1)] = True
    y[~valid] = 0x7fc1
    wy = rng.standard_normal(R * NvS).astype(np.float32)
    yt = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda()
    cout, cw = buf.combine(plan, yt, torch.from_numpy(wy).cuda(), dedup=True)
    assert buf.get_status() == 0
    yf = y.copy()
    oracle.fold_duplicates(R, S, K, NvS, H, op["dst"], yf)
    assert np.array_equal(_bits(yt), yf), "folded rows differ from the oracle's fold"
    ot, ow = oracle.combine_primaries(R, S, K, NvS, H, op["dst"], yf, wy)
    assert np.array_equal(_bits(cout).reshape(R * S, H), ot), "deduplicated combine differs"
    assert np.array_equal(cw.cpu().numpy().reshape(R * S, K).view(np.uint32), ow.view(np.uint32))
    # against the plain combine: the folds' roundings (half an ulp of each
    # rank's partial sum) and the two final roundings, 3 * 2^-8 * sum |y| at
    # most
    plain, _ = oracle.combine(R, S, K, NvS, H, op["dst"], y)
    yv = oracle.bf16_to_f32(y)
    g = decode(op["dst"]).reshape(R * S, K)
    bound = np.abs(yv[g]).sum(axis=1) * 3 * 2.0 ** -8
    diff = np.abs(oracle.bf16_to_f32(ot) - oracle.bf16_to_f32(plain))
    assert np.all(diff <= bound + 1e-30)

    # closed form of combine(dispatch(x)) through the deduplicated path
    ident, _ = buf.combine(plan, hd, dedup=True)
    _check_identity(ident.float().cpu().numpy(), oracle.bf16_to_f32(x).reshape(R, S, H), K)
    buf.destroy()


def test_dedup_needs_dup_records():
    from combine_moonep_plan_gb300._lib import MoonepError
    sh = _shape("tiny", 16, 64)
    buf = _buffer(sh, dup=False)
    topk = _routing(sh, "zipf", 3)
    tpe = wl.tokens_per_expert(topk, sh.E)
    xt = torch.zeros((sh.R, sh.S, sh.H), dtype=torch.bfloat16, device="cuda")
    hid, _, _, plan = buf.dispatch(xt, None, torch.from_numpy(topk).cuda(),
                                   torch.from_numpy(tpe).cuda())
    with pytest.raises(MoonepError):
        buf.dispatch(xt, plan=plan, dedup=True)
    with pytest.raises(MoonepError):
        buf.combine(plan, hid, dedup=True)
    assert buf.get_status() == 0
    buf.destroy()


def test_dedup_single_route_is_plain():
    """K = 1 has no duplicates: both deduplicated calls equal the plain ones."""
    sh = wl.Shape("k1", R=4, E=16, K=1, S=96, H=520, Hp=64, B=4, tp=8, weights="softmax")
    R, S, K, E, H = sh.R, sh.S, sh.K, sh.E, sh.H
    topk = _routing(sh, "zipf", 11)
    tpe = wl.tokens_per_expert(topk, E)
    buf = _buffer(sh)
    x = torch.randn((R, S, H), device="cuda").bfloat16()
    plan = buf.plan(torch.from_numpy(topk).cuda(), torch.from_numpy(tpe).cuda())
    assert buf.get_status() == 0
    assert int(plan.dup_counts.sum()) == 0
    a, _, _, _ = buf.dispatch(x, plan=plan, dedup=True)
    b, _, _, _ = buf.dispatch(x, plan=plan)
    rows = torch.from_numpy(decode(plan.dst.cpu().numpy()).reshape(-1)).cuda()
    assert torch.equal(a[rows].view(torch.int16), b[rows].view(torch.int16))
    y = torch.randn((R * buf.NvS, H), device="cuda").bfloat16()
    c1, _ = buf.combine(plan, y.clone(), dedup=True)
    c2, _ = buf.combine(plan, y)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert buf.get_status() == 0
    buf.destroy()


def test_dedup_full_size_deepseek():
    """DeepSeek-V3 shape at full size (S = 4096, H = 7168, K = 8 over 8 ranks)."""
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.SHAPES["deepseek_v3"]
    R, S, K, E, H, B, tp = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B, sh.tp
    seed = wl.seed_for("deepseek_v3", 41)
    topk = wl.routing(sh, "zipf", target_maxvio=2.0, seed=seed)[0]
    tpe = wl.tokens_per_expert(topk, E)
    st, op = oracle.plan(R, E, K, S, B, tp, topk, tpe)
    assert st == 0
    NvS = op["NvS"]
    buf = Buffer(S=S, H=H, K=K, E=E, num_ep_ranks=R, B=B, token_padding=tp,
                 zero_copy_views=False, dup_records=True)
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn((R, S, H), generator=g, device=dev).to(torch.bfloat16)
    w = torch.from_numpy(wl.route_weights(sh, seed)).to(dev)
    plan = buf.plan(torch.from_numpy(topk).to(dev), torch.from_numpy(tpe).to(dev))
    for f in ("dst", "dup_counts"):
        assert np.array_equal(getattr(plan, f).cpu().numpy(), op[f]), f
    out = torch.full((R * NvS, H), float("nan"), dtype=torch.bfloat16, device=dev)
    wout = torch.full((R * NvS,), float("nan"), dtype=torch.float32, device=dev)
    hid, wn, _, _ = buf.dispatch(x, w, plan=plan, out=out, weights_out=wout, dedup=True)
    assert buf.get_status() == 0
    # the whole scatter on the device
    dst = op["dst"]
    gidx = torch.from_numpy(decode(dst).reshape(-1)).to(dev)
    tok = torch.arange(R * S, device=dev).repeat_interleave(K)
    xf = x.reshape(R * S, H)
    for c0 in range(0, gidx.numel(), 1 << 16):
        c1 = c0 + (1 << 16)
        assert torch.equal(hid[gidx[c0:c1]].view(torch.int16), xf[tok[c0:c1]].view(torch.int16))
    assert torch.equal(wn[gidx].view(torch.int32), w.reshape(-1).view(torch.int32))
    pad = np.concatenate([np.arange(j * NvS + a, j * NvS + b) for j in range(R)
                          for a, b in op["zero_fill_ranges"][j] if b > a])
    pt = torch.from_numpy(pad).to(dev)
    assert torch.all(hid[pt].view(torch.int16) == 0)
    del out, wout

    # combine: sampled tokens re-laid out as a small problem for the oracle
    y = torch.randn((R * NvS, H), generator=g, device=dev).to(torch.bfloat16)
    y0 = y.clone()
    cout, _ = buf.combine(plan, y, dedup=True)
    assert buf.get_status() == 0
    rng = np.random.default_rng(seed)
    toks = np.unique(rng.integers(0, R * S, 96))
    n = len(toks)
    gt = decode(dst).reshape(R * S, K)[toks]            # global rows of the sampled routes
    dt = dst.reshape(R * S, K)[toks]
    NvS2 = n * K
    # row of route (i, k) in the small problem: same rank, position i*K + k
    g2 = (gt // NvS) * NvS2 + np.arange(NvS2).reshape(n, K)
    d2 = np.where(dt >= 0, g2, -(g2 + 1)).astype(np.int32)
    y2 = np.zeros((R * NvS2, H), np.uint16)
    y2[g2.reshape(-1)] = _bits(y0[torch.from_numpy(gt.reshape(-1)).to(dev)])
    oracle.fold_duplicates(1, n, K, NvS2, H, d2, y2)
    want, _ = oracle.combine_primaries(1, n, K, NvS2, H, d2, y2)
    assert np.array_equal(_bits(cout.reshape(R * S, H)[torch.from_numpy(toks).to(dev)]), want)
    # the sampled primaries hold the oracle's folds
    prim = dt >= 0
    got_f = _bits(y[torch.from_numpy(gt[prim]).to(dev)])
    assert np.array_equal(got_f, y2[g2[prim]])
    ident, _ = buf.combine(plan, hid, dedup=True)
    err = (ident.float() - x.float() * K).abs()
    assert bool((err <= x.float().abs() * K * 2.0 ** -7).all())
    buf.destroy()
