"""CPU oracle for the balanced expert-parallel hot path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The product library never does.  The arithmetic
lives in ``moonep_oracle.c`` (plain single-threaded C); this module compiles it
with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moonep_oracle.c")
_HDR = os.path.join(_HERE, "moonep_oracle.h")
_LIB = os.path.join(_HERE, "libmoonep_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID_ARG, ERR_BAD_EXPERT, ERR_HIST_MISMATCH, ERR_SLOTS, ERR_NOMEM = 0, -1, -2, -3, -4, -5


def compile_c(src: str, out: str, include_dir: str = _HERE) -> str:
    """gcc a C source of the oracle into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-I", include_dir, "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        compile_c(_SRC, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    i64 = ctypes.c_int64
    ci = ctypes.c_int
    lib.mo_nvs.restype = i64
    lib.mo_nvs.argtypes = [ci] * 6
    lib.mo_plan.restype = ci
    lib.mo_plan.argtypes = [ci] * 6 + [vp] * 10
    lib.mo_dispatch.restype = None
    lib.mo_dispatch.argtypes = [ci] * 5 + [i64] * 4 + [vp] * 6
    lib.mo_combine.restype = None
    lib.mo_combine.argtypes = [ci] * 3 + [i64] * 4 + [vp, vp, i64, vp, vp, vp, vp]
    lib.mo_prefetch.restype = None
    lib.mo_prefetch.argtypes = [ci] * 3 + [vp, i64, i64, i64, vp]
    lib.mo_fold_duplicates.restype = None
    lib.mo_fold_duplicates.argtypes = [ci] * 3 + [i64] * 4 + [vp, vp]
    lib.mo_combine_primaries.restype = None
    lib.mo_combine_primaries.argtypes = [ci] * 3 + [i64] * 4 + [vp, vp, i64, vp, vp, vp, vp]
    lib.mo_prepare.restype = None
    lib.mo_prepare.argtypes = [ci] * 4 + [i64] + [vp] * 5
    lib.mo_prefetch_bytes.restype = None
    lib.mo_prefetch_bytes.argtypes = [ci] * 3 + [vp, i64, i64, i64, vp]
    lib.mo_reduce.restype = None
    lib.mo_reduce.argtypes = [ci] * 3 + [vp, i64, i64, i64, vp, vp]
    lib.mo_f32_to_bf16.restype = ctypes.c_uint16
    lib.mo_f32_to_bf16.argtypes = [ctypes.c_float]
    return lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class Oracle:
    """ctypes front end of one compiled copy of the oracle."""

    OK, ERR_INVALID_ARG, ERR_BAD_EXPERT = OK, ERR_INVALID_ARG, ERR_BAD_EXPERT
    ERR_HIST_MISMATCH, ERR_SLOTS, ERR_NOMEM = ERR_HIST_MISMATCH, ERR_SLOTS, ERR_NOMEM

    def __init__(self, path):
        self.path = path
        self.lib = _bind(path)

    def nvs(self, R, E, K, S, B, tp) -> int:
        return int(self.lib.mo_nvs(R, E, K, S, B, tp))

    def plan(self, R, E, K, S, B, tp, topk, tpe=None, dup_records=True):
        """Balanced plan.  Returns (status, dict of numpy int32 arrays)."""
        NvS = self.nvs(R, E, K, S, B, tp)
        topk = np.ascontiguousarray(topk, dtype=np.int32).reshape(R, S * K)
        if tpe is not None:
            tpe = np.ascontiguousarray(tpe, dtype=np.int32).reshape(R, E)
        out = {
            "dst": np.zeros((R, S * K), np.int32),
            "experts_to_copy": np.zeros((R, B), np.int32),
            "cu_seqlens": np.zeros((R, E + B), np.int32),
            "zero_fill_ranges": np.zeros((R, E + B, 2), np.int32),
            "remote_stats": np.zeros((R, 2), np.int32),
            "dup_counts": np.zeros((R, 2), np.int32),
        }
        if dup_records:
            out["dup_groups"] = np.zeros((R, NvS, 3), np.int32)
            out["dup_loffs"] = np.zeros((R, NvS), np.int32)
        st = self.lib.mo_plan(R, E, K, S, B, tp, _ptr(topk), _ptr(tpe),
                              _ptr(out["dst"]), _ptr(out["experts_to_copy"]),
                              _ptr(out["cu_seqlens"]), _ptr(out["zero_fill_ranges"]),
                              _ptr(out["remote_stats"]), _ptr(out["dup_counts"]),
                              _ptr(out.get("dup_groups")), _ptr(out.get("dup_loffs")))
        out["NvS"] = NvS
        return int(st), out

    def dispatch(self, R, S, K, E, B, NvS, H, dst, zfr, hidden, w_sk=None,
                 out=None, w_out=None, c0=0, c1=None):
        """hidden [R*S, H] uint16 bf16 bits -> out [R*NvS, H] (in place)."""
        c1 = H if c1 is None else c1
        dst = np.ascontiguousarray(dst, dtype=np.int32)
        zfr = np.ascontiguousarray(zfr, dtype=np.int32)
        if out is None:
            out = np.zeros((R * NvS, H), np.uint16)
        self.lib.mo_dispatch(R, S, K, E, B, NvS, H, c0, c1, _ptr(dst), _ptr(zfr),
                             _ptr(hidden), _ptr(w_sk), _ptr(out), _ptr(w_out))
        return out

    def combine(self, R, S, K, NvS, H, dst, y, w_nvs=None, tokens=None, c0=0,
                c1=None):
        """y [R*NvS, H] uint16 -> (out [ntok, H] uint16, w_out [ntok, K])."""
        c1 = H if c1 is None else c1
        dst = np.ascontiguousarray(dst, dtype=np.int32)
        if tokens is not None:
            tokens = np.ascontiguousarray(tokens, dtype=np.int64)
            ntok = len(tokens)
        else:
            ntok = R * S
        out = np.zeros((ntok, H), np.uint16)
        w_out = np.zeros((ntok, K), np.float32) if w_nvs is not None else None
        self.lib.mo_combine(R, S, K, NvS, H, c0, c1, _ptr(dst), _ptr(tokens), ntok,
                            _ptr(y), _ptr(w_nvs), _ptr(out), _ptr(w_out))
        return out, w_out

    def prefetch(self, R, E, B, etc, W, HHp, c0=0, c1=None):
        """W [E + R*B, HHp] uint16, modified in place."""
        c1 = HHp if c1 is None else c1
        etc = np.ascontiguousarray(etc, dtype=np.int32)
        self.lib.mo_prefetch(R, E, B, _ptr(etc), HHp, c0, c1, _ptr(W))
        return W

    def fold_duplicates(self, R, S, K, NvS, H, dst, y, c0=0, c1=None):
        """Duplicate prologue, in place on y [R*NvS, H] uint16."""
        c1 = H if c1 is None else c1
        dst = np.ascontiguousarray(dst, dtype=np.int32)
        assert y.dtype == np.uint16 and y.flags["C_CONTIGUOUS"]
        self.lib.mo_fold_duplicates(R, S, K, NvS, H, c0, c1, _ptr(dst), _ptr(y))
        return y

    def combine_primaries(self, R, S, K, NvS, H, dst, y, w_nvs=None, tokens=None, c0=0,
                          c1=None):
        """Combine over primary routes: (out [ntok, H] uint16, w_out [ntok, K])."""
        c1 = H if c1 is None else c1
        dst = np.ascontiguousarray(dst, dtype=np.int32)
        if tokens is not None:
            tokens = np.ascontiguousarray(tokens, dtype=np.int64)
            ntok = len(tokens)
        else:
            ntok = R * S
        out = np.zeros((ntok, H), np.uint16)
        w_out = np.zeros((ntok, K), np.float32) if w_nvs is not None else None
        self.lib.mo_combine_primaries(R, S, K, NvS, H, c0, c1, _ptr(dst), _ptr(tokens), ntok,
                                      _ptr(y), _ptr(w_nvs), _ptr(out), _ptr(w_out))
        return out, w_out

    def prepare(self, R, S, K, E, H, ntok, hidden, topk, w=None, want_tpe=True):
        """Decode-path padding in place (hidden [R,S,H] uint16 or None, topk
        [R,S,K] int32, w [R,S,K] fp32 or None); returns tokens_per_expert
        [R,E] or None."""
        nt = None if ntok is None else np.ascontiguousarray(ntok, dtype=np.int32)
        tpe = np.zeros((R, E), np.int32) if want_tpe else None
        assert topk.dtype == np.int32 and topk.flags["C_CONTIGUOUS"]
        self.lib.mo_prepare(R, S, K, E, H, _ptr(nt), _ptr(hidden), _ptr(topk), _ptr(w),
                            _ptr(tpe))
        return tpe

    def prefetch_bytes(self, R, E, B, etc, W, row_bytes, c0=0, c1=None):
        """W [E + R*B, row_bytes] uint8 (packed MXFP4, block scales, any row
        format seen as bytes), modified in place."""
        c1 = row_bytes if c1 is None else c1
        etc = np.ascontiguousarray(etc, dtype=np.int32)
        assert W.dtype == np.uint8 and W.shape[-1] == row_bytes
        self.lib.mo_prefetch_bytes(R, E, B, _ptr(etc), row_bytes, c0, c1, _ptr(W))
        return W

    def reduce(self, R, E, B, etc, Gh, Gs, HHp, c0=0, c1=None):
        """Gh [E, HHp] fp32, Gs [R*B, HHp] fp32, modified in place."""
        c1 = HHp if c1 is None else c1
        etc = np.ascontiguousarray(etc, dtype=np.int32)
        self.lib.mo_reduce(R, E, B, _ptr(etc), HHp, c0, c1, _ptr(Gh), _ptr(Gs))
        return Gh, Gs

    def f32_to_bf16(self, values):
        v = np.asarray(values, dtype=np.float32).reshape(-1)
        return np.array([self.lib.mo_f32_to_bf16(float(x)) for x in v], dtype=np.uint16)

    @staticmethod
    def bf16_to_f32(bits):
        return bf16_to_f32(bits)


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def nvs(*a, **k):
    return _default().nvs(*a, **k)


def plan(*a, **k):
    return _default().plan(*a, **k)


def dispatch(*a, **k):
    return _default().dispatch(*a, **k)


def combine(*a, **k):
    return _default().combine(*a, **k)


def prefetch(*a, **k):
    return _default().prefetch(*a, **k)


def prefetch_bytes(*a, **k):
    return _default().prefetch_bytes(*a, **k)


def prepare(*a, **k):
    return _default().prepare(*a, **k)


def fold_duplicates(*a, **k):
    return _default().fold_duplicates(*a, **k)


def combine_primaries(*a, **k):
    return _default().combine_primaries(*a, **k)


def reduce(*a, **k):
    return _default().reduce(*a, **k)


def f32_to_bf16(values):
    return _default().f32_to_bf16(values)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)
