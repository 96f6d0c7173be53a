"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer and bit-copy outputs (plan arrays, dispatched rows, route weights,
prefetched weights) must match bit for bit.  Combine must match to within one
bf16 ulp and the gradient reduce to within 1e-6 relative (both sides add in
the same order in fp32, so both are in fact expected to be bit-exact and the
tests also report exactness).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moonep_plan_gb300 import workloads as wl
from tests.plan_checks import check_plan, decode

pytestmark = pytest.mark.gpu

PLAN_FIELDS = ("dst", "experts_to_copy", "cu_seqlens", "zero_fill_ranges", "remote_stats",
               "dup_counts")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_moonep_plan_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _buffer(cfg, H=64, dup=True, views=True):
    from combine_moonep_plan_gb300.api import Buffer
    return Buffer(S=cfg["S"], H=H, K=cfg["K"], E=cfg["E"], num_ep_ranks=cfg["R"], B=cfg["B"],
                  token_padding=cfg["tp"], zero_copy_views=views, dup_records=dup)


def _oracle_plan(cfg, topk, tpe=None):
    return oracle.plan(cfg["R"], cfg["E"], cfg["K"], cfg["S"], cfg["B"], cfg["tp"], topk, tpe)


def _cmp_plan(gp, op, cfg):
    for f in PLAN_FIELDS:
        g = getattr(gp, f).cpu().numpy()
        assert np.array_equal(g, op[f]), f"plan field {f} differs"
    if gp.dup_groups is not None:
        dg = gp.dup_groups.cpu().numpy()
        dl = gp.dup_loffs.cpu().numpy()
        for j in range(cfg["R"]):
            ng, nd = op["dup_counts"][j, 1], op["dup_counts"][j, 0]
            assert np.array_equal(dg[j, :ng], op["dup_groups"][j, :ng])
            assert np.array_equal(dl[j, :nd], op["dup_loffs"][j, :nd])


def _cfg_of(sh):
    return dict(R=sh.R, E=sh.E, K=sh.K, S=sh.S, B=sh.B, tp=sh.tp)


def _small(name, S):
    sh = wl.SHAPES[name]
    return wl.Shape(f"{name}_S{S}", R=sh.R, E=sh.E, K=sh.K, S=S, H=min(sh.H, 512),
                    Hp=64, B=sh.B, tp=sh.tp, weights=sh.weights)


def _routing(sh, kind, seed):
    if kind == "exact0":
        return wl.routing(sh, "exact0", seed=seed)[0]
    if kind == "uniform":
        return wl.routing(sh, "uniform", seed=seed)[0]
    if kind == "zipf":
        return wl.routing(sh, "zipf", zipf_s=1.2, seed=seed)[0]
    if kind == "zipf_hard":
        return wl.routing(sh, "zipf", zipf_s=3.0, seed=seed)[0]
    if kind == "hot":
        return wl.routing(sh, "hot", hot_share=0.3, seed=seed)[0]
    if kind == "hot_group0":
        return wl.routing(sh, "hot", hot_share=0.3, hot_group0=True, seed=seed)[0]
    raise ValueError(kind)


def _full_pipeline(sh, topk, seed, *, dup=True, check_invariants=True):
    """Plan, dispatch (+weights), combine (+weights) on the GPU and the oracle."""
    cfg = _cfg_of(sh)
    R, S, K, E, H = sh.R, sh.S, sh.K, sh.E, sh.H
    tpe = wl.tokens_per_expert(topk, E)
    st, op = _oracle_plan(cfg, topk, tpe)
    assert st == 0
    if check_invariants and S:
        check_plan(cfg, topk, op, max_records=256)
    buf = _buffer(cfg, H=H, dup=dup)
    x = wl.hidden_bf16(sh, seed)
    w = wl.route_weights(sh, seed)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).reshape(R, S, H).cuda()
    wt = torch.from_numpy(w).cuda()
    tk = torch.from_numpy(topk).cuda()
    tp = torch.from_numpy(tpe).cuda()
    NvS = buf.NvS
    assert NvS == op["NvS"]
    # poison the outputs so untouched rows are visible
    out = torch.full((R * NvS, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    wout = torch.full((R * NvS,), float("nan"), dtype=torch.float32, device="cuda")
    hid, wn, cu, plan = buf.dispatch(xt, wt, tk, tp, out=out, weights_out=wout)
    assert buf.get_status() == 0
    _cmp_plan(plan, op, cfg)
    assert torch.equal(cu, plan.cu_seqlens)
    # dispatch parity
    want = np.full((R * NvS, H), 0x7fc0, np.uint16)
    want_w = np.full(R * NvS, np.nan, np.float32)
    oracle.dispatch(R, S, K, E, sh.B, NvS, H, op["dst"], op["zero_fill_ranges"], x, w, want,
                    want_w)
    got = hid.view(torch.int16).cpu().numpy().view(np.uint16)
    touched = np.zeros(R * NvS, bool)
    touched[decode(op["dst"]).reshape(-1)] = True
    for j in range(R):
        for a, b in op["zero_fill_ranges"][j]:
            touched[j * NvS + a:j * NvS + b] = True
    assert np.array_equal(got[touched], want[touched]), "dispatched rows differ"
    gw = wn.cpu().numpy()
    assert np.array_equal(gw[touched].view(np.uint32), want_w[touched].view(np.uint32))
    # tail rows untouched (still NaN poison)
    if (~touched).any():
        assert np.all(np.isnan(gw[~touched]))
        tail = got[~touched]
        assert np.all((tail & 0x7f80) == 0x7f80)
    # combine parity on random expert outputs with NaN-poisoned padding/tail
    rng = np.random.default_rng(seed + 17)
    y = wl.bf16_bits_from_f32(rng.standard_normal((R * NvS, H)).astype(np.float32))
    valid = np.zeros(R * NvS, bool)
    valid[decode(op["dst"]).reshape(-1)] = True
    y[~valid] = 0x7fc1
    wy = rng.standard_normal(R * NvS).astype(np.float32)
    wy[~valid] = np.nan
    ot, ow = oracle.combine(R, S, K, NvS, H, op["dst"], y, wy)
    yt = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda()
    cout, cw = buf.combine(plan, yt, torch.from_numpy(wy).cuda())
    assert buf.get_status() == 0
    gc = cout.view(torch.int16).cpu().numpy().view(np.uint16).reshape(R * S, H)
    _assert_bf16_close(gc, ot)
    assert np.array_equal(cw.cpu().numpy().reshape(R * S, K).view(np.uint32), ow.view(np.uint32))
    # identity expert: combine(dispatch(x)) == K * x for K a power of two
    if K & (K - 1) == 0:
        ident, _ = buf.combine(plan, hid)
        ref = oracle.bf16_to_f32(x).reshape(R, S, H) * K
        assert np.array_equal(ident.float().cpu().numpy(), ref)
    return buf, plan, op


def _assert_bf16_close(got, want):
    """Within one bf16 ulp (the accuracy bound for combine); exact is the norm."""
    if np.array_equal(got, want):
        return
    g = got.astype(np.int32)
    w = want.astype(np.int32)
    # ordered integer representation of bf16
    g = np.where(g & 0x8000, 0x8000 - g, g)
    w = np.where(w & 0x8000, 0x8000 - w, w)
    diff = np.abs(g - w)
    assert diff.max() <= 1, f"combine differs by {diff.max()} bf16 ulp"


# ------------------------------------------------------------------ cases

@pytest.mark.parametrize("kind", ["zipf", "exact0", "uniform", "zipf_hard", "hot"])
def test_tiny_full_pipeline(kind):
    sh = wl.SHAPES["tiny"]
    seeds = {"zipf": 1001, "exact0": 1002, "uniform": 1003, "zipf_hard": 1004, "hot": 1005}
    topk = _routing(sh, kind, seeds[kind])
    _full_pipeline(sh, topk, 3)


@pytest.mark.parametrize("name", ["mixtral", "deepseek_v3", "kimi_k2", "qwen3_decode"])
@pytest.mark.parametrize("kind", ["zipf", "zipf_hard", "hot_group0", "exact0"])
def test_scaled_shapes_pipeline(name, kind):
    # S chosen so S*K spans several 2048-route planner tiles plus a ragged tail
    S = {"mixtral": 2100, "deepseek_v3": 600, "kimi_k2": 600, "qwen3_decode": 128}[name]
    sh = _small(name, S)
    topk = _routing(sh, kind, 7)
    _full_pipeline(sh, topk, 11, check_invariants=(name == "qwen3_decode"))


@pytest.mark.parametrize("seed", range(24))
def test_random_small_configs(seed):
    """Random R, E, K (including K outside the specialised set), S, B >= E/R,
    token_padding and H, skewed routing with repeated experts inside a token."""
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 9))
    L = int(rng.integers(1, 9))
    E = R * L
    K = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 12]))
    S = int(rng.integers(1, 700))
    B = L + int(rng.integers(0, 3))
    tp = int(rng.choice([1, 2, 3, 8, 16, 128]))
    H = int(rng.choice([8, 64, 136, 264]))
    sh = wl.Shape("rand", R=R, E=E, K=K, S=S, H=H, Hp=16, B=B, tp=tp, weights="softmax")
    p = rng.random(E) ** 4
    topk = rng.choice(E, size=(R, S, K), p=p / p.sum()).astype(np.int32)
    _full_pipeline(sh, topk, seed)


@pytest.mark.parametrize("K", [6, 7, 16, 32])
def test_wide_and_odd_top_k(K):
    """K that divides 32 (16, 32: a token's routes fill half or all of a warp
    on the single-launch planner) and K that does not (6, 7: the tile path)."""
    sh = wl.Shape("k", R=4, E=64, K=K, S=97, H=72, Hp=16, B=16, tp=8, weights="softmax")
    rng = np.random.default_rng(K)
    p = rng.random(sh.E) ** 3
    topk = np.stack([np.stack([rng.choice(sh.E, K, replace=False, p=p / p.sum())
                               for _ in range(sh.S)]) for _ in range(sh.R)]).astype(np.int32)
    _full_pipeline(sh, topk, K)


@pytest.mark.parametrize("K", [5, 7, 10, 14, 20])
def test_staged_combine_full_width_rows(K):
    """Top-K without a register-tuned combine: 14 KB rows (H = 7168) in 2 KB
    (K <= 13) or 1 KB chunks staged through shared memory, with enough
    tokens that every block takes several units (on 152 SMs the top-7 and
    top-14 grids are a multiple of the chunks per row, the case where one
    block sits out)."""
    sh = wl.Shape("staged", R=4, E=32, K=K, S=48, H=7168, Hp=16, B=8, tp=16, weights="softmax")
    rng = np.random.default_rng(300 + K)
    p = rng.random(sh.E) ** 2
    topk = np.stack([np.stack([rng.choice(sh.E, K, replace=False, p=p / p.sum())
                               for _ in range(sh.S)]) for _ in range(sh.R)]).astype(np.int32)
    _full_pipeline(sh, topk, 40 + K)


@pytest.mark.parametrize("block", range(4))
def test_random_wide_configs(block):
    """100 random shapes (up to 16 ranks, top-1..16, 1..12 experts per rank,
    token_padding 1..128, rows of 16 bytes to 4 KB, mild to sharp skew): the
    plan and its duplicate records bit for bit with the oracle, the whole
    dispatch scatter and its deduplicated form, the route weights, and the
    combine of the dispatched rows (K copies add exactly in fp32)."""
    for seed in range(25 * block, 25 * (block + 1)):
        rng = np.random.default_rng(777000 + seed)
        R = int(rng.integers(1, 17))
        L = int(rng.integers(1, 13))
        E = R * L
        K = int(rng.integers(1, 17))
        S = int(rng.integers(1, 1500))
        B = L + int(rng.integers(0, 3))
        tp = int(rng.choice([1, 2, 4, 8, 16, 64, 128]))
        H = int(rng.choice([8, 16, 64, 520, 1024, 2056]))
        p = rng.random(E) ** float(rng.choice([1, 4, 8]))
        topk = rng.choice(E, size=(R, S, K), p=p / p.sum()).astype(np.int32)
        tpe = wl.tokens_per_expert(topk, E)
        cfg = dict(R=R, E=E, K=K, S=S, B=B, tp=tp)
        st, op = _oracle_plan(cfg, topk, tpe)
        assert st == 0
        buf = _buffer(cfg, H=H, views=False)
        x = torch.from_numpy(rng.standard_normal((R, S, H)).astype(np.float32)).bfloat16().cuda()
        w = torch.from_numpy(rng.random((R, S, K)).astype(np.float32)).cuda()
        hid, wn, _, plan = buf.dispatch(x, w, torch.from_numpy(topk).cuda(),
                                        torch.from_numpy(tpe).cuda())
        assert buf.get_status() == 0, cfg
        _cmp_plan(plan, op, cfg)
        g = torch.from_numpy(decode(op["dst"]).reshape(-1)).cuda()
        tok = torch.arange(R * S, device="cuda").repeat_interleave(K)
        assert torch.equal(hid[g].view(torch.int16), x.reshape(-1, H)[tok].view(torch.int16)), cfg
        assert torch.equal(wn[g], w.reshape(-1)), cfg
        hd, _, _, _ = buf.dispatch(x, w, plan=plan, dedup=True)
        assert torch.equal(hd[g].view(torch.int16), hid[g].view(torch.int16)), cfg
        out, wb = buf.combine(plan, hid, wn)
        assert torch.equal(out.view(torch.int16), (x.float() * K).bfloat16().view(torch.int16)), cfg
        assert torch.equal(wb, w), cfg
        assert buf.get_status() == 0, cfg
        buf.destroy()


def test_planner_tables_near_the_default_shared_memory_limit():
    """Tables of 48,400 bytes: under 48 KB, but over 48 KB with the kernel's
    static shared memory, so the limit must be raised explicitly (a launch
    error before)."""
    sh = wl.Shape("smem48", R=16, E=192, K=12, S=387, H=64, Hp=8, B=13, tp=4,
                  weights="softmax")
    buf, _, _ = _full_pipeline(sh, _routing(sh, "zipf", 114), 114)
    buf.destroy()


def test_contexts_of_different_table_sizes_coexist():
    """The planner's shared-memory limit is per kernel and process-wide: a
    context with smaller tables created later must not lower it under an
    earlier context's need."""
    big = wl.Shape("big", R=8, E=768, K=8, S=64, H=64, Hp=8, B=96, tp=8, weights="softmax")
    mid = wl.Shape("mid", R=8, E=256, K=8, S=64, H=64, Hp=8, B=32, tp=8, weights="softmax")
    tb, tm = _routing(big, "zipf", 5), _routing(mid, "zipf", 6)
    bb, bm = _buffer(_cfg_of(big)), _buffer(_cfg_of(mid))
    pb = bb.plan(torch.from_numpy(tb).cuda())
    pm = bm.plan(torch.from_numpy(tm).cuda())
    pb = bb.plan(torch.from_numpy(tb).cuda(), plan=pb)
    assert bb.get_status() == 0 and bm.get_status() == 0
    for sh, topk, p in ((big, tb, pb), (mid, tm, pm)):
        st, op = _oracle_plan(_cfg_of(sh), topk)
        assert st == 0 and np.array_equal(p.dst.cpu().numpy(), op["dst"])
    bb.destroy()
    bm.destroy()


@pytest.mark.parametrize("K", [2, 6, 8])
def test_tile_path_planner(K):
    """Tables too large for the single-launch planner's shared memory
    (E = 1536) take the three-kernel tile path; it must give the same plan."""
    sh = wl.Shape("tilepath", R=8, E=1536, K=K, S=96, H=64, Hp=8, B=192, tp=8,
                  weights="softmax")
    _full_pipeline(sh, _routing(sh, "zipf", 40 + K), 40 + K)


def test_largest_tables():
    """The largest expert table the library takes (E = 4096, R = 64, B = 64,
    K = 8): the planner's tables no longer fit in shared memory, so the tile
    path runs with its balance tables in global memory."""
    sh = wl.Shape("max", R=64, E=4096, K=8, S=16, H=16, Hp=8, B=64, tp=16, weights="softmax")
    topk = _routing(sh, "zipf_hard", 51)
    _full_pipeline(sh, topk, 51, dup=False, check_invariants=True)


def test_zero_slots():
    """B = 0: a routing that never overflows a home group plans without slots;
    one that does reports MOONEP_ERR_SLOTS."""
    from combine_moonep_plan_gb300 import _lib
    sh = wl.Shape("b0", R=4, E=16, K=2, S=64, H=32, Hp=8, B=0, tp=4, weights="softmax")
    topk, _ = wl.routing(sh, "exact0", seed=3)
    buf, plan, op = _full_pipeline(sh, topk, 3)
    assert plan.experts_to_copy.numel() == 0
    buf.destroy()
    skew = _routing(sh, "zipf_hard", 4)
    st, _ = _oracle_plan(_cfg_of(sh), skew)
    assert st == -4
    buf = _buffer(_cfg_of(sh), H=32)
    buf.plan(torch.from_numpy(skew).cuda())
    assert buf.get_status() == _lib.ERR_SLOTS
    buf.destroy()


def test_all_routes_to_one_expert():
    sh = wl.Shape("one", R=4, E=8, K=2, S=300, H=64, Hp=16, B=2, tp=8, weights="softmax")
    topk = np.zeros((4, 300, 2), np.int32)
    buf, plan, op = _full_pipeline(sh, topk, 1)
    assert np.all(op["experts_to_copy"][1:, 0] == 0)


def test_k1_tp1():
    sh = wl.Shape("k1", R=3, E=6, K=1, S=1000, H=32, Hp=8, B=2, tp=1, weights="softmax")
    topk = _routing(sh, "zipf_hard", 5)
    _full_pipeline(sh, topk, 2)


def test_empty_tokens():
    cfg = dict(R=2, E=4, K=2, S=0, B=2, tp=4)
    buf = _buffer(cfg, H=16)
    tk = torch.zeros((2, 0, 2), dtype=torch.int32, device="cuda")
    plan = buf.plan(tk)
    assert buf.get_status() == 0
    assert torch.all(plan.cu_seqlens == 0) and torch.all(plan.experts_to_copy == -1)
    # every copy call, direct and deduplicated, takes the empty batch
    x = torch.zeros((2, 0, 16), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((2, 0, 2), dtype=torch.float32, device="cuda")
    for dedup in (False, True):
        rows, wn, _, _ = buf.dispatch(x, w, plan=plan, dedup=dedup)
        out, wb = buf.combine(plan, rows, wn, dedup=dedup)
        assert out.shape == (2, 0, 16) and wb.shape == (2, 0, 2)
    assert buf.get_status() == 0


# ----------------------------------------------------- plan properties

def test_plan_is_deterministic_and_clone_matches():
    sh = _small("deepseek_v3", 512)
    topk = _routing(sh, "zipf_hard", 3)
    buf = _buffer(_cfg_of(sh), H=64)
    tk = torch.from_numpy(topk).cuda()
    p1 = buf.plan(tk)
    p2 = buf.plan(tk)
    c = p1.clone()
    torch.cuda.synchronize()
    for f in PLAN_FIELDS + ("dup_groups", "dup_loffs"):
        assert torch.equal(getattr(p1, f), getattr(p2, f)), f
        assert torch.equal(getattr(p1, f), getattr(c, f)), f


def test_plan_reuse_dispatch_equals_fresh():
    """Combine-backward: a gradient dispatched with the forward plan lands on
    the same rows as a fresh dispatch of the same tensor would."""
    sh = _small("kimi_k2", 300)
    topk = _routing(sh, "hot", 4)
    buf = _buffer(_cfg_of(sh), H=sh.H)
    tk = torch.from_numpy(topk).cuda()
    x = torch.randn(sh.R, sh.S, sh.H, device="cuda").bfloat16()
    g = torch.randn(sh.R, sh.S, sh.H, device="cuda").bfloat16()
    _, _, cu, plan = buf.dispatch(x, None, tk)
    saved = plan.clone()
    a, wa, cu2, _ = buf.dispatch(g, plan=saved)
    assert cu2 is None and wa is None
    b, _, _, _ = buf.dispatch(g, None, tk)
    # compare every written row (valid and padding); the tail is unspecified
    ends = plan.cu_seqlens[:, -1].cpu().tolist()
    for j, end in enumerate(ends):
        lo = j * buf.NvS
        assert torch.equal(a[lo:lo + end].view(torch.int16), b[lo:lo + end].view(torch.int16))


@pytest.mark.parametrize("name,kind,S", [("kimi_k2", "hot", 300), ("deepseek_v3", "zipf", 257),
                                         ("tiny", "zipf", 64)])
def test_plan_reuse_dispatch_matches_oracle(name, kind, S):
    """Combine-backward dispatch [API, Buffer.dispatch with a saved plan;
    Buffer.combine backward]: an independent [R, S, H] gradient dispatched
    with a clone of the forward plan and no weights equals the oracle's
    dispatch of that gradient (weights absent) on every valid and padding
    row; tail rows keep their poison, and the forward's zero-copy rows and
    route weights stay as the forward left them."""
    sh = _small(name, S) if name != "tiny" else wl.SHAPES["tiny"]
    topk = _routing(sh, kind, 31)
    cfg = _cfg_of(sh)
    buf = _buffer(cfg, H=sh.H, dup=False, views=True)
    tk = torch.from_numpy(topk).cuda()
    x = torch.randn(sh.R, sh.S, sh.H, device="cuda").bfloat16()
    w = torch.rand(sh.R, sh.S, sh.K, device="cuda")
    hid, wn, _, plan = buf.dispatch(x, w, tk, zero_copy=True, router_weights_zero_copy=True)
    saved = plan.clone()
    torch.cuda.synchronize()
    hid0, wn0 = hid.clone(), wn.clone()
    g = torch.randn(sh.R, sh.S, sh.H, device="cuda").bfloat16()
    poison = torch.full((sh.R * buf.NvS, sh.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    out, wout, cu, _ = buf.dispatch(g, plan=saved, out=poison)
    assert out.data_ptr() == poison.data_ptr() and wout is None and cu is None
    assert buf.get_status() == 0
    st, op = _oracle_plan(cfg, topk)
    assert st == 0
    NvS = op["NvS"]
    gb = g.view(torch.int16).cpu().numpy().view(np.uint16).reshape(sh.R * sh.S, sh.H)
    want = np.full((sh.R * NvS, sh.H), 0x7fc0, np.uint16)
    oracle.dispatch(sh.R, sh.S, sh.K, sh.E, sh.B, NvS, sh.H, op["dst"], op["zero_fill_ranges"],
                    gb, None, want)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    nan_bits = int(torch.tensor(float("nan"), dtype=torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    for j in range(sh.R):
        end = int(op["cu_seqlens"][j, -1])
        lo = j * NvS
        assert np.array_equal(got[lo:lo + end], want[lo:lo + end]), f"rank {j} rows differ"
        assert np.all(got[lo + end:lo + NvS] == nan_bits), f"rank {j} tail written"
    assert torch.equal(hid.view(torch.int16), hid0.view(torch.int16))
    assert torch.equal(wn.view(torch.int32), wn0.view(torch.int32))


def test_zero_copy_views():
    sh = wl.SHAPES["tiny"]
    topk = _routing(sh, "zipf", 2)
    buf = _buffer(_cfg_of(sh), H=sh.H)
    x = torch.randn(sh.R, sh.S, sh.H, device="cuda").bfloat16()
    w = torch.rand(sh.R, sh.S, sh.K, device="cuda")
    hid, wn, _, plan = buf.dispatch(x, w, torch.from_numpy(topk).cuda(), zero_copy=True,
                                    router_weights_zero_copy=True)
    assert hid.data_ptr() == buf.hidden_nvsh_buffer_view().data_ptr()
    assert wn.data_ptr() == buf.router_weight_buffer_view().data_ptr()
    v1 = buf.hidden_nvsh_buffer_view(1)
    assert v1.data_ptr() == hid.data_ptr() + buf.NvS * sh.H * 2
    assert torch.equal(v1, hid[buf.NvS:2 * buf.NvS])


# ------------------------------------------------- prefetch and reduce

@pytest.mark.parametrize("name,kind", [("tiny", "zipf"), ("deepseek_v3", "zipf_hard"),
                                       ("kimi_k2", "hot_group0"), ("mixtral", "zipf_hard")])
def test_prefetch_and_reduce_parity(name, kind):
    sh = wl.SHAPES[name] if name == "tiny" else _small(name, 256)
    cfg = _cfg_of(sh)
    topk = _routing(sh, kind, 9)
    st, op = _oracle_plan(cfg, topk)
    assert st == 0
    etc = op["experts_to_copy"]
    assert (etc >= 0).any()
    buf = _buffer(cfg, H=64)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    H, Hp = 64, 40                    # HHp = 2560: several 64 KB-chunk boundaries
    rows = sh.E + sh.R * sh.B
    rng = np.random.default_rng(1)
    Ws = [rng.integers(0, 65535, (rows, H * Hp), dtype=np.uint16) for _ in range(3)]
    Wt = [torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).reshape(rows, H, Hp).cuda()
          for W in Ws]
    buf.prefetch_weight(plan, *Wt)
    for W, t in zip(Ws, Wt):
        oracle.prefetch(sh.R, sh.E, sh.B, etc, W, H * Hp)
        assert np.array_equal(t.view(torch.int16).cpu().numpy().view(np.uint16).reshape(rows, -1), W)
    Gh = [rng.standard_normal((sh.E, H * Hp)).astype(np.float32) for _ in range(2)]
    Gs = [rng.standard_normal((sh.R * sh.B, H * Hp)).astype(np.float32) for _ in range(2)]
    Ght = [torch.from_numpy(g).reshape(sh.E, H, Hp).cuda() for g in Gh]
    Gst = [torch.from_numpy(g).reshape(sh.R, sh.B, H, Hp).cuda() for g in Gs]
    buf.reduce_grad(plan, Ght, Gst)
    assert buf.get_status() == 0
    for gh, gs, ght, gst in zip(Gh, Gs, Ght, Gst):
        oracle.reduce(sh.R, sh.E, sh.B, etc, gh, gs, H * Hp)
        got_h = ght.cpu().numpy().reshape(sh.E, -1)
        got_s = gst.cpu().numpy().reshape(sh.R * sh.B, -1)
        rel = np.abs(got_h - gh) / np.maximum(np.abs(gh), 1e-30)
        assert rel.max() <= 1e-6
        assert np.array_equal(got_h.view(np.uint32), gh.view(np.uint32)), "reduce not bit-exact"
        assert np.array_equal(got_s.view(np.uint32), gs.view(np.uint32))


@pytest.mark.parametrize("name,kind", [("tiny", "zipf"), ("deepseek_v3", "hot"),
                                       ("kimi_k2", "hot")])
def test_prefetch_mxfp4_set_parity(name, kind):
    """A packed MXFP4 gate/up/down set with its E8M0 block scales, one launch:
    every tensor byte-identical to the oracle's byte-row prefetch."""
    sh = wl.SHAPES[name] if name == "tiny" else _small(name, 256)
    cfg = _cfg_of(sh)
    topk = _routing(sh, kind, 11)
    st, op = _oracle_plan(cfg, topk)
    assert st == 0
    etc = op["experts_to_copy"]
    assert (etc >= 0).any()
    buf = _buffer(cfg, H=64)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    H, Hp = 64, 2080                  # packed row 66,560 B: crosses a 64 KB unit
    rows = sh.E + sh.R * sh.B
    rng = np.random.default_rng(3)
    packed = [rng.integers(0, 256, (rows, H * Hp // 2), dtype=np.uint8) for _ in range(3)]
    scales = [rng.integers(0, 256, (rows, H * Hp // 32), dtype=np.uint8) for _ in range(3)]
    pt = [torch.from_numpy(a).reshape(rows, H, Hp // 2).cuda() for a in packed]
    stt = [torch.from_numpy(a).reshape(rows, H, Hp // 32).cuda() for a in scales]
    buf.prefetch_weight(plan, *pt, scales=stt)
    assert buf.get_status() == 0
    for a, t in zip(packed + scales, pt + stt):
        oracle.prefetch_bytes(sh.R, sh.E, sh.B, etc, a, a.shape[1])
        assert np.array_equal(t.cpu().numpy().reshape(rows, -1), a)


def test_prefetch_rows_odd_row_sizes():
    """Rows that are not 16-byte multiples (and a tensor on an odd address)
    take the byte path; a row size of 0 is skipped."""
    sh = wl.SHAPES["tiny"]
    cfg = _cfg_of(sh)
    topk = _routing(sh, "zipf", 12)
    st, op = _oracle_plan(cfg, topk)
    etc = op["experts_to_copy"]
    buf = _buffer(cfg, H=64)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    rows = sh.E + sh.R * sh.B
    rng = np.random.default_rng(4)
    arrs = [rng.integers(0, 256, (rows, n), dtype=np.uint8) for n in (3, 40, 65537)]
    ts = [torch.from_numpy(a).cuda() for a in arrs]
    big = torch.from_numpy(rng.integers(0, 256, rows * 48 + 1, dtype=np.uint8)).cuda()
    odd = big[1:].view(rows, 48)      # 48-byte rows on an odd base
    odd_np = odd.cpu().numpy().copy()
    empty = torch.empty((rows, 0), dtype=torch.uint8, device="cuda")
    buf.prefetch_rows(plan, ts + [odd, empty])
    assert buf.get_status() == 0
    for a, t in zip(arrs + [odd_np], ts + [odd]):
        oracle.prefetch_bytes(sh.R, sh.E, sh.B, etc, a, a.shape[1])
        assert np.array_equal(t.cpu().numpy(), a)
    with pytest.raises(ValueError):
        buf.prefetch_weight(plan, ts[0], ts[1], scales=[ts[2]])


# --------------------------------------------------- concurrent contexts

def test_two_contexts_on_two_streams():
    """Two contexts plan and dispatch at the same time on two streams (their
    single-launch planners overlap on the GPU); each result equals the
    oracle's."""
    from combine_moonep_plan_gb300.api import Buffer
    shapes = [_small("deepseek_v3", 256), _small("kimi_k2", 192)]
    runs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i, sh in enumerate(shapes):
        topk = _routing(sh, "zipf_hard", 60 + i)
        buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                     token_padding=sh.tp, zero_copy_views=False)
        x = torch.randn((sh.R, sh.S, sh.H), device="cuda").bfloat16()
        runs.append((sh, topk, buf, torch.from_numpy(topk).cuda(), x))
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):
        outs = []
        for (sh, topk, buf, tk, x), st in zip(runs, streams):
            with torch.cuda.stream(st):
                hid, wn, cu, plan = buf.dispatch(x, None, tk)
                outs.append((plan, hid))
    torch.cuda.synchronize()
    for (sh, topk, buf, tk, x), (plan, hid) in zip(runs, outs):
        assert buf.get_status() == 0
        st_, op = _oracle_plan(_cfg_of(sh), topk)
        _cmp_plan(plan, op, _cfg_of(sh))
        g = torch.from_numpy(decode(op["dst"]).reshape(-1)).cuda()
        tok = torch.arange(sh.R * sh.S, device="cuda").repeat_interleave(sh.K)
        assert torch.equal(hid[g].view(torch.int16), x.reshape(-1, sh.H)[tok].view(torch.int16))
        buf.destroy()


# ------------------------------------------------------------ SM cap

def test_sm_cap_gives_identical_results(monkeypatch):
    """A context capped to 16 SMs (by its config, or by MOONEP_NUM_SMS) moves
    the same bytes to the same places as one using every SM."""
    from combine_moonep_plan_gb300.api import Buffer
    sh = _small("deepseek_v3", 128)
    topk = torch.from_numpy(_routing(sh, "zipf_hard", 41)).cuda()
    x = torch.randn((sh.R, sh.S, sh.H), device="cuda").bfloat16()
    w = torch.rand((sh.R, sh.S, sh.K), device="cuda")
    rows = sh.E + sh.R * sh.B
    W = torch.randn((rows, sh.H, sh.Hp), device="cuda").bfloat16()
    results = []
    for how in ("all", "config", "env"):
        if how == "env":
            monkeypatch.setenv("MOONEP_NUM_SMS", "16")
        buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                     token_padding=sh.tp, zero_copy_views=False,
                     num_sms=16 if how == "config" else None)
        monkeypatch.delenv("MOONEP_NUM_SMS", raising=False)
        assert buf.num_sms == (16 if how != "all" else torch.cuda.get_device_properties(0).multi_processor_count)
        # the tail rows after the last segment are unspecified: start from zeros
        hid0 = torch.zeros((sh.R * buf.NvS, sh.H), dtype=torch.bfloat16, device="cuda")
        wn0 = torch.zeros((sh.R * buf.NvS,), dtype=torch.float32, device="cuda")
        hid, wn, cu, plan = buf.dispatch(x, w, topk, out=hid0, weights_out=wn0)
        out, wb = buf.combine(plan, hid, wn)
        Wc = W.clone()
        buf.prefetch_weight(plan, Wc)
        assert buf.get_status() == 0
        results.append((hid.clone(), wn.clone(), out.clone(), wb.clone(), Wc))
        buf.destroy()
    for other in results[1:]:
        for a, b in zip(results[0], other):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


# ------------------------------------------------------------ canaries

def test_guard_rows_around_every_output_stay_untouched():
    """Every output buffer sits between guard rows holding a fixed bit
    pattern; after prepare, plan, dispatch, combine, prefetch (bf16 and byte
    rows) and reduce the guards still hold it."""
    sh = wl.SHAPES["tiny"]
    cfg = _cfg_of(sh)
    R, S, K, E, H, B = sh.R, sh.S, sh.K, sh.E, sh.H, sh.B
    buf = _buffer(cfg, H=H, views=False)
    NvS = buf.NvS
    gr = 4
    dev = "cuda"

    def guarded(rows, cols, dtype, fill):
        big = torch.empty((rows + 2 * gr, cols), dtype=dtype, device=dev)
        big.view(torch.uint8).view(torch.int8).fill_(0x5A) if dtype == torch.uint8 else \
            big.view(torch.int16).fill_(0x5A5A)
        inner = big[gr:gr + rows]
        if fill is not None:
            inner.copy_(fill)
        return big, inner

    def guards_ok(big):
        v = big.view(torch.uint8)
        return bool((v[:gr] == 0x5A).all() and (v[-gr:] == 0x5A).all())

    topk = _routing(sh, "zipf", 31)
    g = torch.Generator(device=dev).manual_seed(31)
    x_big, x = guarded(R * S, H, torch.bfloat16,
                       torch.randn((R * S, H), generator=g, device=dev).bfloat16())
    tk_big = torch.empty((R * S + 2 * gr, K), dtype=torch.int32, device=dev)
    tk_big.view(torch.uint8).fill_(0x5A)
    tk = tk_big[gr:gr + R * S]
    tk.copy_(torch.from_numpy(topk.reshape(R * S, K)))
    w_big = torch.empty((R * S + 2 * gr, K), dtype=torch.float32, device=dev)
    w_big.view(torch.uint8).fill_(0x5A)
    w = w_big[gr:gr + R * S]
    w.copy_(torch.from_numpy(wl.route_weights(sh, 31).reshape(R * S, K)))
    tpe = buf.prepare(x.view(R, S, H), tk.view(R, S, K), w.view(R, S, K), num_tokens=[S - 5, S])
    out_big, out = guarded(R * NvS, H, torch.bfloat16, None)
    wo_big = torch.empty(R * NvS + 2 * gr * 4, dtype=torch.float32, device=dev)
    wo_big.view(torch.uint8).fill_(0x5A)
    wo = wo_big[gr * 4:gr * 4 + R * NvS]
    hid, wn, cu, plan = buf.dispatch(x.view(R, S, H), w.view(R, S, K), tk.view(R, S, K), tpe,
                                     out=out, weights_out=wo)
    c_big, c = guarded(R * S, H, torch.bfloat16, None)
    cw_big = torch.empty((R * S + 2 * gr, K), dtype=torch.float32, device=dev)
    cw_big.view(torch.uint8).fill_(0x5A)
    cw = cw_big[gr:gr + R * S]
    buf.combine(plan, hid, wn, out=c.view(R, S, H), weights_out=cw.view(R, S, K))
    rows = E + R * B
    W_big, W = guarded(rows, H * sh.Hp, torch.bfloat16,
                       torch.randn((rows, H * sh.Hp), generator=g, device=dev).bfloat16())
    buf.prefetch_weight(plan, W.view(rows, H, sh.Hp))
    P_big, P = guarded(rows, 48, torch.uint8,
                       torch.randint(0, 256, (rows, 48), generator=g, device=dev,
                                     dtype=torch.uint8))
    buf.prefetch_rows(plan, [P])
    Gh_big = torch.empty((E + 2 * gr, H * sh.Hp), dtype=torch.float32, device=dev)
    Gs_big = torch.empty((R * B + 2 * gr, H * sh.Hp), dtype=torch.float32, device=dev)
    for t in (Gh_big, Gs_big):
        t.view(torch.uint8).fill_(0x5A)
    Gh_big[gr:gr + E].normal_(generator=g)
    Gs_big[gr:gr + R * B].normal_(generator=g)
    buf.reduce_grad(plan, [Gh_big[gr:gr + E].view(E, H, sh.Hp)],
                    [Gs_big[gr:gr + R * B].view(R, B, H, sh.Hp)])
    assert buf.get_status() == 0
    for name, big in (("hidden", x_big), ("topk", tk_big), ("weights", w_big),
                      ("dispatched rows", out_big), ("dispatched weights", wo_big),
                      ("combined rows", c_big), ("combined weights", cw_big),
                      ("bf16 weights", W_big), ("byte rows", P_big), ("grads", Gh_big),
                      ("slot grads", Gs_big)):
        assert guards_ok(big), f"guard rows around the {name} were written"
    buf.destroy()


# ------------------------------------------------------------- errors

def test_device_errors_latch_status_without_faulting():
    from combine_moonep_plan_gb300 import _lib
    sh = wl.SHAPES["tiny"]
    cfg = _cfg_of(sh)
    topk = _routing(sh, "zipf", 1)
    buf = _buffer(cfg, H=sh.H)
    x = torch.randn(sh.R, sh.S, sh.H, device="cuda").bfloat16()
    bad = topk.copy()
    bad[1, 3, 1] = sh.E + 5
    _, _, _, plan = buf.dispatch(x, None, torch.from_numpy(bad).cuda())
    out, _ = buf.combine(plan, buf.hidden_nvsh_buffer_view())
    assert buf.get_status() == _lib.ERR_BAD_EXPERT
    bad[1, 3, 1] = -4
    buf.plan(torch.from_numpy(bad).cuda())
    assert buf.get_status() == _lib.ERR_BAD_EXPERT
    tpe = wl.tokens_per_expert(topk, sh.E)
    tpe[0, 2] += 1
    buf.plan(torch.from_numpy(topk).cuda(), torch.from_numpy(tpe).cuda())
    assert buf.get_status() == _lib.ERR_HIST_MISMATCH
    # the context still works afterwards
    _full_pipeline(sh, topk, 5)


def test_slots_error_when_b_too_small():
    from combine_moonep_plan_gb300 import _lib
    cfg = dict(R=2, E=4, K=1, S=4, B=1, tp=1)
    topk = np.array([[[0], [0], [0], [0]], [[0], [0], [1], [1]]], np.int32)
    buf = _buffer(cfg, H=16)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    assert buf.get_status() == _lib.ERR_SLOTS
    assert torch.all(plan.experts_to_copy == -1)
    x = torch.randn(2, 4, 16, device="cuda").bfloat16()
    buf.dispatch(x, plan=plan)
    buf.combine(plan, buf.hidden_nvsh_buffer_view())
    assert buf.get_status() == 0


def test_destroy_is_idempotent():
    from combine_moonep_plan_gb300 import _lib
    buf = _buffer(dict(R=2, E=4, K=2, S=8, B=2, tp=2), H=16)
    buf.destroy()
    buf.destroy()
    assert buf.destroyed
    with pytest.raises(_lib.MoonepError):
        buf.plan(torch.zeros((2, 8, 2), dtype=torch.int32, device="cuda"))


def test_planner_wait_limit_reports_timeout(monkeypatch):
    """The planner's blocks wait for one another with a time limit.  A test
    hook makes the arrival wait unsatisfiable; every block must give up, latch
    MOONEP_ERR_TIMEOUT and leave a plan every later kernel can still consume
    without leaving its buffers."""
    from combine_moonep_plan_gb300 import _lib
    monkeypatch.setenv("MOONEP_TEST_PLANNER_TIMEOUT", "1")
    sh = wl.SHAPES["tiny"]
    buf = _buffer(_cfg_of(sh), H=sh.H)
    monkeypatch.delenv("MOONEP_TEST_PLANNER_TIMEOUT")
    topk = _routing(sh, "zipf", 8)
    x = torch.randn(sh.R, sh.S, sh.H, device="cuda").bfloat16()
    _, _, _, plan = buf.dispatch(x, None, torch.from_numpy(topk).cuda())
    buf.combine(plan, buf.hidden_nvsh_buffer_view())
    assert buf.get_status() == _lib.ERR_TIMEOUT
    g = decode(plan.dst.cpu().numpy())
    assert g.min() >= 0 and g.max() < sh.R * buf.NvS
    # a context created without the hook plans normally
    _full_pipeline(sh, topk, 8)


@pytest.mark.parametrize("R,L,K,S,tp", [(40, 2, 2, 100, 4), (64, 1, 4, 40, 8), (33, 3, 8, 64, 16)])
def test_many_ranks(R, L, K, S, tp):
    """More than 32 ranks: the chain and segment scans take their wide paths."""
    E = R * L
    sh = wl.Shape("wide", R=R, E=E, K=K, S=S, H=64, Hp=8, B=L, tp=tp, weights="softmax")
    topk = _routing(sh, "zipf_hard", R)
    _full_pipeline(sh, topk, R, check_invariants=False)
