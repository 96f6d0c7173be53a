"""GPU parity on values that only the fixed summation orders reproduce.

The oracle's orders are pinned on the CPU by hand-worked fp32 ties; here the
same kind of values go through the kernels:

* combine: route k of every token holds -2^20 (k = 0), 2^-4 (0 < k < K-1)
  or 2^20 (k = K-1), scaled per column by a power of two.  In k order the
  small terms land exactly below 2^20 and survive ((K-2)*2^-4); any order
  that adds 2^20 before them drops them at the tie.  Every K the library
  specialises (2, 3, 4, 6, 8) and the shared-memory staged kernel in both of
  its chunk sizes (5, 10, 12 with 2 KB, 14, 16, 24 with 1 KB) [vLLM,
  finalize(): the unweighted K-sum, accumulated in k order in fp32].
* the deduplicated combine's fold and primaries sum, on the same values
  [API, Buffer.combine: duplicates accumulated into primaries in fp32].
* gradient reduce: home 2^24, then slots 1.0, -2^24, 1.0, ... in (rank,
  slot) order [API, Buffer.reduce_grad].
Each result must equal the oracle's bit for bit.
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


def _f2b(v):
    return np.asarray(v, np.float32).view(np.uint32) >> 16


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _tie_rows(dst, K, NvS_total, H):
    """y [R*NvS, H] bf16 bits: route k's row holds the k-th tie value times
    2^(c % 5) in column c; rows no route names hold NaN."""
    vals = np.full(K, 2.0 ** -4)
    vals[0], vals[-1] = -2.0 ** 20, 2.0 ** 20
    scale = 2.0 ** (np.arange(H) % 5)
    y = np.full((NvS_total, H), 0x7fc0, np.uint16)
    g = decode(dst).reshape(-1, K)
    for k in range(K):
        y[g[:, k]] = _f2b((vals[k] * scale).astype(np.float32))[None, :]
    return y


@pytest.mark.parametrize("K", [2, 3, 4, 5, 6, 8, 10, 12, 14, 16, 24])
@pytest.mark.parametrize("dedup", [False, True])
def test_combine_order_sensitive_values(K, dedup):
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.Shape(f"k{K}", R=4, E=16, K=K, S=96, H=136, Hp=8, B=4, tp=8, weights="softmax")
    rng = np.random.default_rng(100 + K)
    # experts drawn with repeats allowed inside a token, so a rank often
    # holds several routes of one token (duplicate groups to fold)
    topk = rng.integers(0, sh.E, (sh.R, sh.S, K)).astype(np.int32)
    st, op = oracle.plan(sh.R, sh.E, K, sh.S, sh.B, sh.tp, topk)
    assert st == 0
    NvS = op["NvS"]
    buf = Buffer(S=sh.S, H=sh.H, K=K, E=sh.E, num_ep_ranks=sh.R, B=sh.B, token_padding=sh.tp,
                 zero_copy_views=False, dup_records=dedup)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    y = _tie_rows(op["dst"], K, sh.R * NvS, sh.H)
    yt = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).cuda()
    out, _ = buf.combine(plan, yt, dedup=dedup)
    assert buf.get_status() == 0
    if dedup:
        oracle.fold_duplicates(sh.R, sh.S, K, NvS, sh.H, op["dst"], y)
        want, _ = oracle.combine_primaries(sh.R, sh.S, K, NvS, sh.H, op["dst"], y)
        assert np.array_equal(_bits(yt), y), "folded rows differ"
    else:
        want, _ = oracle.combine(sh.R, sh.S, K, NvS, sh.H, op["dst"], y)
        # the k-order value itself, not only agreement with the oracle
        scale = 2.0 ** (np.arange(sh.H) % 5)
        assert np.array_equal(oracle.bf16_to_f32(want),
                              np.broadcast_to(((K - 2) * 2.0 ** -4 * scale).astype(np.float32)
                                              if K > 2 else np.zeros(sh.H, np.float32),
                                              want.shape))
    assert np.array_equal(_bits(out).reshape(sh.R * sh.S, sh.H), want)


def test_reduce_order_sensitive_values():
    from combine_moonep_plan_gb300.api import Buffer
    sh = wl.Shape("r", R=8, E=16, K=4, S=128, H=8, Hp=8, B=2, tp=4, weights="softmax")
    rng = np.random.default_rng(5)
    # routes 0-2 of every token to expert 0 (repeats are separate routes):
    # expert 0 gets 6 S*K worth of routes, so five receivers hold a copy
    topk = rng.integers(2, sh.E, (sh.R, sh.S, sh.K)).astype(np.int32)
    topk[:, :, :3] = 0
    st, op = oracle.plan(sh.R, sh.E, sh.K, sh.S, sh.B, sh.tp, topk)
    assert st == 0
    etc = op["experts_to_copy"].reshape(-1)
    counts = np.bincount(etc[etc >= 0], minlength=sh.E)
    buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B, token_padding=sh.tp,
                 zero_copy_views=False)
    plan = buf.plan(torch.from_numpy(topk).cuda())
    HHp = 4096
    Gh = np.full((sh.E, HHp), 2.0 ** 24, np.float32)
    Gs = np.zeros((sh.R * sh.B, HHp), np.float32)
    # the i-th slot (in (rank, slot) order) of each expert: 1, -2^24, 1, -2^24...
    seen = np.zeros(sh.E, int)
    for i, e in enumerate(etc):
        if e >= 0:
            Gs[i] = 1.0 if seen[e] % 2 == 0 else -2.0 ** 24
            seen[e] += 1
    Gs[:, 1::2] *= -1          # the mirrored case in odd columns
    Gh[:, 1::2] *= -1
    Ght = torch.from_numpy(Gh.copy()).reshape(sh.E, HHp).cuda()
    Gst = torch.from_numpy(Gs.copy()).reshape(sh.R, sh.B, HHp).cuda()
    buf.reduce_grad(plan, [Ght], [Gst])
    assert buf.get_status() == 0
    oracle.reduce(sh.R, sh.E, sh.B, etc, Gh, Gs, HHp)
    assert np.array_equal(Ght.cpu().numpy().view(np.uint32), Gh.view(np.uint32))
    assert np.array_equal(Gst.cpu().numpy().reshape(sh.R * sh.B, HHp).view(np.uint32),
                          Gs.view(np.uint32))
    # expert 0's copies in order: 2^24 + 1 ties back to 2^24, - 2^24 gives 0,
    # and so on, one fp32 rounding per add
    acc = np.float32(2.0 ** 24)
    for i in range(counts[0]):
        acc = np.float32(acc + np.float32(1.0 if i % 2 == 0 else -2.0 ** 24))
    assert counts[0] >= 3 and Ght[0, 0].item() == acc
