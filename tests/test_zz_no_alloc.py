"""moonep_plan_noalloc: the planner for callers that cannot allocate.

Frameworks whose caching allocator owns all device memory, and host paths
that cannot take cudaMalloc's implicit synchronisation, cannot create a
context or a plan object.  This entry point takes caller-allocated outputs and
keeps its intermediate tables in a fixed file-scope device array.  Its plan
must equal the one moonep_plan writes for the same inputs, bit for bit (the
plan is integer data, the tolerance every plan test uses), on two calls in a
row, since the second call reuses the scratch the first left behind, and
equal the oracle's plan; one case runs in a fresh process where this entry
point is the only planner ever called.

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_moonep_plan_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FIELDS = ("dst", "experts_to_copy", "cu_seqlens", "zero_fill_ranges", "remote_stats",
          "dup_counts")


@pytest.fixture(scope="module")
def lib():
    from combine_moonep_plan_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from combine_moonep_plan_gb300 import _lib
    return _lib.load()


def _noalloc(lib, sh, topk, tpe=None):
    from combine_moonep_plan_gb300._lib import MoonepConfig
    R, S, K, E, B = sh.R, sh.S, sh.K, sh.E, sh.B
    cfg = MoonepConfig(R=R, E=E, K=K, S=S, H=sh.H, B=B, token_padding=sh.tp, num_sms=0)
    dev = "cuda"
    out = {
        "dst": torch.full((R, S * K), -7, dtype=torch.int32, device=dev),
        "experts_to_copy": torch.full((R, B), -7, dtype=torch.int32, device=dev),
        "cu_seqlens": torch.full((R, E + B), -7, dtype=torch.int32, device=dev),
        "zero_fill_ranges": torch.full((R, E + B, 2), -7, dtype=torch.int32, device=dev),
        "remote_stats": torch.full((R, 2), -7, dtype=torch.int32, device=dev),
        "dup_counts": torch.full((R, 2), -7, dtype=torch.int32, device=dev),
    }
    status = torch.full((1,), -7, dtype=torch.int32, device=dev)
    tk = torch.from_numpy(topk).to(dev)
    tp = torch.from_numpy(tpe).to(dev) if tpe is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.moonep_plan_noalloc(ctypes.byref(cfg), tk.data_ptr(),
                                 tp.data_ptr() if tp is not None else None,
                                 *[out[f].data_ptr() for f in FIELDS], status.data_ptr(), stream)
    torch.cuda.synchronize()
    return rc, out, int(status.item())


def _reference(sh, topk, tpe=None):
    from combine_moonep_plan_gb300.api import Buffer
    buf = Buffer(S=sh.S, H=sh.H, K=sh.K, E=sh.E, num_ep_ranks=sh.R, B=sh.B,
                 token_padding=sh.tp, zero_copy_views=False)
    plan = buf.plan(torch.from_numpy(topk).cuda(),
                    torch.from_numpy(tpe).cuda() if tpe is not None else None)
    assert buf.get_status() == 0
    ref = {f: getattr(plan, f).clone() for f in FIELDS}
    buf.destroy()
    return ref


def _shape(name, S):
    sh = wl.SHAPES[name]
    return wl.Shape(name, R=sh.R, E=sh.E, K=sh.K, S=S, H=sh.H, Hp=sh.Hp, B=sh.B, tp=sh.tp,
                    weights=sh.weights)


def test_noalloc_plan_matches_moonep_plan_twice(lib):
    """Two calls in a row with different routings and sizes: each equals the
    context-based planner's output and the oracle's plan.  The calls come
    before any context of that shape exists."""
    import oracle
    cases = [(_shape("deepseek_v3", 4096), "zipf", 21),
             (_shape("kimi_k2", 600), "hot", 22),
             (wl.SHAPES["tiny"], "zipf", 23)]
    for sh, kind, seed in cases:
        if kind == "hot":
            topk, _ = wl.routing(sh, "hot", hot_share=0.3, seed=seed)
        else:
            topk, _ = wl.routing(sh, "zipf", zipf_s=1.5, seed=seed)
        tpe = wl.tokens_per_expert(topk, sh.E)
        outs = []
        for call in range(2):
            rc, out, status = _noalloc(lib, sh, topk, tpe)
            assert rc == 0 and status == 0, (rc, status)
            outs.append(out)
        ref = _reference(sh, topk, tpe)
        st, want = oracle.plan(sh.R, sh.E, sh.K, sh.S, sh.B, sh.tp, topk, tpe, dup_records=False)
        assert st == 0
        for call, out in enumerate(outs):
            for f in FIELDS:
                assert torch.equal(out[f], ref[f]), f"{sh.name} call {call}: {f} differs"
                assert np.array_equal(out[f].cpu().numpy(), want[f]), \
                    f"{sh.name} call {call}: {f} differs from the oracle"


FRESH_CHILD = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
from combine_moonep_plan_gb300 import _lib, workloads as wl
lib = _lib.load()
res = {{}}
for i, (R, E, K, S, B, tp) in enumerate({shapes!r}):
    sh = wl.Shape("s%d" % i, R=R, E=E, K=K, S=S, H=8, Hp=8, B=B, tp=tp, weights="softmax")
    topk, _ = wl.routing(sh, "zipf", zipf_s=1.4, seed=40 + i)
    cfg = _lib.MoonepConfig(R=R, E=E, K=K, S=S, H=8, B=B, token_padding=tp, num_sms=0)
    out = [torch.full(n, -7, dtype=torch.int32, device="cuda")
           for n in ((R, S * K), (R, B), (R, E + B), (R, E + B, 2), (R, 2), (R, 2))]
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    tk = torch.from_numpy(topk).cuda()
    rc = lib.moonep_plan_noalloc(ctypes.byref(cfg), tk.data_ptr(), None,
                                 *[o.data_ptr() for o in out], status.data_ptr(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    res["rc%d" % i] = np.array([rc, int(status.item())])
    res["topk%d" % i] = topk
    for n, o in zip({fields!r}, out):
        res["%s%d" % (n, i)] = o.cpu().numpy()
np.savez({path!r}, **res)
"""


def test_noalloc_first_planner_of_a_fresh_process(lib, tmp_path):
    """A process whose only planner is this entry point: shapes whose
    planner tables grow with R (same E) and with B, each compared with the
    oracle's plan.  No context exists in that process, so nothing else has
    set the planner kernels' shared-memory limits for these shapes."""
    import os
    import subprocess
    import sys
    import oracle
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    shapes = [(8, 384, 8, 64, 48, 16), (16, 384, 8, 64, 24, 16), (32, 384, 8, 32, 12, 16),
              (8, 384, 8, 64, 96, 16), (4, 64, 4, 96, 16, 8)]
    path = str(tmp_path / "fresh.npz")
    code = FRESH_CHILD.format(root=root, shapes=shapes, fields=FIELDS, path=path)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stderr[-3000:]
    got = np.load(path)
    for i, (R, E, K, S, B, tp) in enumerate(shapes):
        rc, status = got[f"rc{i}"]
        assert rc == 0 and status == 0, (i, rc, status)
        st, want = oracle.plan(R, E, K, S, B, tp, got[f"topk{i}"], None, dup_records=False)
        assert st == 0
        for f in FIELDS:
            assert np.array_equal(got[f"{f}{i}"], want[f]), f"shape {i}: {f} differs from the oracle"


def test_noalloc_reports_errors_and_limits(lib):
    from combine_moonep_plan_gb300 import _lib
    sh = wl.SHAPES["tiny"]
    topk, _ = wl.routing(sh, "zipf", zipf_s=1.2, seed=5)
    bad = topk.copy()
    bad[0, 1, 0] = sh.E
    rc, _, status = _noalloc(lib, sh, bad)
    assert rc == 0 and status == _lib.ERR_BAD_EXPERT
    # the next call starts clean
    rc, out, status = _noalloc(lib, sh, topk)
    assert rc == 0 and status == 0
    ref = _reference(sh, topk)
    assert all(torch.equal(out[f], ref[f]) for f in FIELDS)
    # tables beyond the fixed scratch are refused up front, with nothing launched
    big = _shape("kimi_k2", 1 << 15)
    rc, _, _ = _noalloc(lib, big, np.zeros((big.R, big.S, big.K), np.int32))
    assert rc == _lib.ERR_INVALID_ARG
