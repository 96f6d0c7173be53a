"""The decode path: padding to a pooled static capacity, then the hot path.

vLLM's prepare/finalize page pads each step's batch to the capacity of a
buffer taken from a pool of power-of-two capacities, mapping invalid
(negative) expert ids to expert 0 with zero weight.  Here the padding runs in
place on the device (moonep_prepare); its result, and the plan, dispatch and
combine that follow, must equal the oracle's prepare -> plan -> dispatch ->
combine bit for bit (combine within one bf16 ulp, exact in practice).
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


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _batch(rng, R, S, K, E, H, n, bad_ids=False):
    """Capacity-sized inputs: rank r's first n[r] rows hold its tokens (about
    4 % of their ids negative), the rest is garbage the padding must replace."""
    topk = rng.integers(0, E, (R, S, K)).astype(np.int32)
    topk[rng.random((R, S, K)) < 0.04] = -1
    rows = np.arange(S)[None, :] >= np.asarray(n)[:, None]
    topk[rows] = rng.integers(-7, 3 * E, (int(rows.sum()), K)).astype(np.int32)
    if bad_ids:  # left for the planner to report (a full rank keeps it)
        topk[-1, 0, 0] = E + 1
    w = rng.random((R, S, K)).astype(np.float32)
    hidden = wl.bf16_bits_from_f32(rng.standard_normal((R, S, H)).astype(np.float32))
    hidden[rows] = 0x7fc1
    return topk, w, hidden


def _to_dev(topk, w, hidden):
    return (torch.from_numpy(topk.copy()).cuda(), torch.from_numpy(w.copy()).cuda(),
            torch.from_numpy(hidden.view(np.int16).copy()).view(torch.bfloat16).cuda())


@pytest.mark.parametrize("R,S,K,E,H,B", [(2, 64, 2, 8, 256, 4), (8, 128, 8, 128, 512, 16),
                                         (3, 37, 4, 12, 40, 4)])
def test_prepare_matches_oracle(R, S, K, E, H, B):
    from combine_moonep_plan_gb300.api import Buffer
    rng = np.random.default_rng(R * 100 + S)
    n = rng.integers(0, S + 1, R)
    n[0], n[-1] = 0, S
    topk, w, hidden = _batch(rng, R, S, K, E, H, n, bad_ids=True)
    buf = Buffer(S=S, H=H, K=K, E=E, num_ep_ranks=R, B=B, token_padding=8,
                 zero_copy_views=False)
    tk, wt, xt = _to_dev(topk, w, hidden)
    tpe = buf.prepare(xt, tk, wt, num_tokens=n)
    want_tpe = oracle.prepare(R, S, K, E, H, n, hidden, topk, w)
    assert np.array_equal(tk.cpu().numpy(), topk)
    assert np.array_equal(wt.cpu().numpy().view(np.uint32), w.view(np.uint32))
    assert np.array_equal(_bits(xt), hidden)
    assert np.array_equal(tpe.cpu().numpy(), want_tpe)
    # without counts or hidden: only the ids and weights change
    topk2, w2, _ = _batch(rng, R, S, K, E, H, n)
    tk2, wt2, _ = _to_dev(topk2, w2, hidden)
    assert buf.prepare(None, tk2, wt2, num_tokens=None, tokens_per_expert=False) is None
    oracle.prepare(R, S, K, E, H, None, None, topk2, w2, want_tpe=False)
    assert np.array_equal(tk2.cpu().numpy(), topk2)
    assert np.array_equal(wt2.cpu().numpy().view(np.uint32), w2.view(np.uint32))
    assert buf.get_status() == 0
    buf.destroy()


def test_decode_steps_through_the_pool():
    """Steps of 3, 20, 100 and 128 tokens on a Qwen3-decode-shaped group
    (R=8, E=128, K=8, B=16, token_padding=16, H cut to 512): each takes the
    pool's power-of-two buffer, prepares in place, then plans (with the
    prepared tokens_per_expert), dispatches and combines; every output equals
    the oracle's."""
    from combine_moonep_plan_gb300.api import BufferPool
    R, K, E, H, B, tp = 8, 8, 128, 512, 16, 16
    pool = BufferPool(max_tokens_per_rank=128, min_tokens=16, H=H, K=K, E=E, num_ep_ranks=R,
                      B=B, token_padding=tp, zero_copy_views=False)
    rng = np.random.default_rng(77)
    used = set()
    for n_max in (3, 20, 100, 128, 20):
        cap, buf = pool.get(n_max)
        used.add(cap)
        assert cap == pool.capacity_for(n_max) and buf.S == cap
        n = rng.integers(0, n_max + 1, R)
        n[rng.integers(R)] = n_max
        topk, w, hidden = _batch(rng, R, cap, K, E, H, n)
        tk, wt, xt = _to_dev(topk, w, hidden)
        tpe = buf.prepare(xt, tk, wt, num_tokens=n)
        want_tpe = oracle.prepare(R, cap, K, E, H, n, hidden, topk, w)
        assert np.array_equal(tpe.cpu().numpy(), want_tpe)
        st, op = oracle.plan(R, E, K, cap, B, tp, topk, want_tpe)
        assert st == 0
        hid, wn, cu, plan = buf.dispatch(xt, wt, tk, tpe)
        assert buf.get_status() == 0
        for f in FIELDS:
            assert np.array_equal(getattr(plan, f).cpu().numpy(), op[f]), f
        NvS = op["NvS"]
        want = np.zeros((R * NvS, H), np.uint16)
        want_w = np.zeros(R * NvS, np.float32)
        oracle.dispatch(R, cap, K, E, B, NvS, H, op["dst"], op["zero_fill_ranges"], hidden, w,
                        want, want_w)
        rows = np.zeros(R * NvS, bool)
        rows[decode(op["dst"]).reshape(-1)] = True
        for j in range(R):
            for a, b in op["zero_fill_ranges"][j]:
                rows[j * NvS + a:j * NvS + b] = True
        assert np.array_equal(_bits(hid)[rows], want[rows])
        assert np.array_equal(wn.cpu().numpy()[rows].view(np.uint32), want_w[rows].view(np.uint32))
        # padded routes carry zero weight and zero rows
        pad = np.arange(cap)[None, :] >= n[:, None]
        pad_rows = decode(op["dst"]).reshape(R, cap, K)[pad].reshape(-1)
        assert np.all(want[pad_rows] == 0) and np.all(want_w[pad_rows] == 0)
        y = wl.bf16_bits_from_f32(rng.standard_normal((R * NvS, H)).astype(np.float32))
        ot, ow = oracle.combine(R, cap, K, NvS, H, op["dst"], y, want_w)
        yt = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda()
        cout, cw = buf.combine(plan, yt, wn)
        assert buf.get_status() == 0
        assert np.array_equal(_bits(cout).reshape(R * cap, H), ot)
        assert np.array_equal(cw.cpu().numpy().reshape(R * cap, K).view(np.uint32),
                              ow.view(np.uint32))
    assert pool.capacities == sorted(used) == [16, 32, 128]
    pool.destroy()
