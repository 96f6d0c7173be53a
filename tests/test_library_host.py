"""Host-side checks of the C-ABI library (no GPU needed).

The library must build for sm_103a, load, and export every entry point that
include/moonep.h declares; host-only calls (sizes, argument validation, error
text) must behave as documented.
"""
import ctypes
import os
import re

import pytest

from combine_moonep_plan_gb300 import build as lib_build
from combine_moonep_plan_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    from combine_moonep_plan_gb300 import _lib
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moonep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moonep_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from combine_moonep_plan_gb300 import _lib
    declared = _declared()
    assert "moonep_plan" in declared and "moonep_dispatch" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(_lib.EXPORTS) == declared


def test_query_sizes_matches_formula(lib):
    from combine_moonep_plan_gb300._lib import MoonepConfig
    for sh in wl.SHAPES.values():
        cfg = MoonepConfig(R=sh.R, E=sh.E, K=sh.K, S=sh.S, H=sh.H, B=sh.B,
                           token_padding=sh.tp, num_sms=0)
        nvs, nvsp = ctypes.c_int(), ctypes.c_int()
        sb = ctypes.c_size_t()
        assert lib.moonep_query_sizes(ctypes.byref(cfg), ctypes.byref(nvs), ctypes.byref(nvsp),
                                      ctypes.byref(sb)) == 0
        assert nvs.value == sh.NvS == nvsp.value
        assert sb.value > 0


@pytest.mark.parametrize("bad", [
    dict(E=7), dict(R=0), dict(K=0), dict(K=33), dict(H=12), dict(token_padding=0),
    dict(B=-1), dict(S=-1), dict(R=65, E=65)])
def test_invalid_configs_rejected(lib, bad):
    from combine_moonep_plan_gb300._lib import MoonepConfig, ERR_INVALID_ARG
    base = dict(R=2, E=8, K=2, S=64, H=256, B=4, token_padding=8, num_sms=0)
    base.update(bad)
    cfg = MoonepConfig(**base)
    assert lib.moonep_query_sizes(ctypes.byref(cfg), None, None, None) == ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.moonep_ctx_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == ERR_INVALID_ARG
    assert not h.value


def test_null_arguments_rejected(lib):
    from combine_moonep_plan_gb300._lib import ERR_INVALID_ARG
    assert lib.moonep_ctx_create(None, 0, None) == ERR_INVALID_ARG
    assert lib.moonep_plan(None, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_dispatch(None, None, None, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_combine(None, None, None, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_dispatch_dedup(None, None, None, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_combine_dedup(None, None, None, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_ctx_destroy(None) == 0          # idempotent on NULL
    assert lib.moonep_hidden_view(None, 0) is None
    assert lib.moonep_plan_destroy(None) == 0
    assert lib.moonep_prepare(None, None, None, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_prefetch_rows(None, None, 1, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_plan_rank(None, 0, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_dispatch_rank(None, None, 0, None, None, None, None, None) == ERR_INVALID_ARG
    assert lib.moonep_combine_rank(None, None, 0, None, None, None, None, None) == ERR_INVALID_ARG


def test_buffer_pool_capacities():
    """Smallest power of two holding the step's tokens, within [min, max]
    [vLLM MoonEPBufferPool.capacity_for]; no buffer exists before get()."""
    from combine_moonep_plan_gb300.api import BufferPool
    pool = BufferPool(max_tokens_per_rank=4096, min_tokens=16, H=64, K=2, E=8, num_ep_ranks=2)
    ns = (0, 1, 2, 3, 16, 17, 100, 128, 129, 4095, 4096, 5000)
    assert [pool.capacity_for(n) for n in ns] == [16, 16, 16, 16, 16, 32, 128, 128, 256,
                                                  4096, 4096, 4096]
    pool2 = BufferPool(max_tokens_per_rank=100)
    assert [pool2.capacity_for(n) for n in (0, 1, 2, 3, 64, 65, 99, 100, 101)] == \
        [1, 1, 2, 4, 64, 100, 100, 100, 100]
    assert pool.capacities == [] and pool2.capacities == []
    pool.destroy()


@pytest.mark.parametrize("mn,mx", [(1, 100), (16, 4096), (10, 1000), (7, 7), (3, 64)])
def test_buffer_pool_rule_as_stated(mn, mx):
    """Every token count against the rule's words: a power of two that holds
    the tokens, the smallest such, then kept within [min, max].  So the
    capacity is min, max or a power of two; it holds the batch whenever the
    batch fits at all; and no smaller power of two inside the bounds holds it."""
    from combine_moonep_plan_gb300.api import BufferPool
    pool = BufferPool(max_tokens_per_rank=mx, min_tokens=mn, H=64, K=2, E=8, num_ep_ranks=2)
    pow2 = [1 << i for i in range(24)]
    for n in range(0, mx + 20):
        cap = pool.capacity_for(n)
        assert mn <= cap <= mx
        assert cap in (mn, mx) or cap in pow2
        if n <= mx:
            assert cap >= n
        smaller = [p for p in pow2 if max(n, 1) <= p < cap and mn <= p]
        assert not smaller, (n, cap, smaller)
        if cap not in (mn, mx):
            assert cap // 2 < n          # the smallest power of two holding n
    with pytest.raises(ValueError):
        pool.get(mx + 1)
    with pytest.raises(ValueError):
        BufferPool(max_tokens_per_rank=8, min_tokens=9)


def test_strerror_texts(lib):
    for code in range(-8, 1):
        assert lib.moonep_strerror(code)
    assert b"unknown" in lib.moonep_strerror(-99)


def test_binding_fails_loudly_without_library(tmp_path):
    from combine_moonep_plan_gb300 import _lib
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(RuntimeError, match="no CPU fallback"):
            _lib.load(str(tmp_path / "missing.so"))
    finally:
        _lib._lib = saved
