"""Seeded synthetic workloads for the balanced expert-parallel hot path.

This module only *generates inputs*: expert routings (top-k expert ids), route
weights, bf16 hidden rows and expert weight / gradient tensors.  It holds none
of the planner's, dispatch's or combine's arithmetic, so both the CUDA path and
the CPU oracle can draw their inputs from it.

Shapes follow the MoonEP tensor contract ("MoonEP Public API Visual Guide",
section "Buffer.dispatch(...)": hidden_sh [S, H] bf16, route_weights_sk [S, K]
fp32, topk_experts_sk [S, K] int32, tokens_per_expert [E] int32), with a leading
R axis because the R expert-parallel ranks are emulated as R partitions of one
device.

Router imbalance is measured as in the MoonEP README ("Performance"):
maxvio = max_e(T_e / T_bar) - 1 with T_bar = R*S*K / E the per-expert load under
perfect balance.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "Shape", "SHAPES", "routing", "route_weights", "hidden_bf16", "maxvio",
    "tokens_per_expert", "seed_for", "bf16_bits_from_f32",
]


@dataclasses.dataclass(frozen=True)
class Shape:
    """One workload shape.  Field names follow the MoonEP notation table."""
    name: str
    R: int          # expert-parallel ranks (logical partitions of one GPU)
    E: int          # experts in the EP group
    K: int          # routes per token
    S: int          # tokens per source rank
    H: int          # hidden size (bf16 elements per row)
    Hp: int         # trailing expert-weight dimension H'
    B: int          # prefetch slots per rank
    tp: int         # token_padding
    weights: str    # route-weight recipe: "softmax" or "sigmoid"

    @property
    def L(self) -> int:
        return self.E // self.R

    @property
    def C(self) -> int:
        return self.S * self.K

    @property
    def N(self) -> int:
        return self.R * self.S * self.K

    @property
    def NvS(self) -> int:
        tp = self.tp
        raw = self.C + (self.L + self.B) * (tp - 1)
        return (raw + tp - 1) // tp * tp


SHAPES = {
    "tiny": Shape("tiny", R=2, E=8, K=2, S=64, H=256, Hp=128, B=4, tp=8,
                  weights="softmax"),
    "mixtral": Shape("mixtral", R=8, E=8, K=2, S=8192, H=4096, Hp=14336, B=1,
                     tp=128, weights="softmax"),
    "deepseek_v3": Shape("deepseek_v3", R=8, E=256, K=8, S=4096, H=7168, Hp=2048,
                         B=32, tp=128, weights="sigmoid"),
    "kimi_k2": Shape("kimi_k2", R=8, E=384, K=8, S=4096, H=7168, Hp=2048, B=48,
                     tp=128, weights="sigmoid"),
    "qwen3_decode": Shape("qwen3_decode", R=8, E=128, K=8, S=128, H=4096, Hp=1536,
                          B=16, tp=16, weights="softmax"),
}

_SHAPE_INDEX = {n: i for i, n in enumerate(SHAPES)}


def seed_for(shape_name: str, sweep_idx: int) -> int:
    """Seed = 1000 * config index + sweep index."""
    return 1000 * _SHAPE_INDEX.get(shape_name, 9) + sweep_idx


def maxvio(topk: np.ndarray, E: int) -> float:
    """max_e(T_e / T_bar) - 1 over all ranks' routes (README, "Performance")."""
    t = np.bincount(topk.reshape(-1).astype(np.int64), minlength=E)
    return float(t.max() * E / topk.size - 1.0)


def tokens_per_expert(topk: np.ndarray, E: int) -> np.ndarray:
    """Per-source-rank histogram [R, E] int32 (the caller-side bincount)."""
    R = topk.shape[0]
    out = np.zeros((R, E), dtype=np.int32)
    for r in range(R):
        out[r] = np.bincount(topk[r].reshape(-1).astype(np.int64), minlength=E)
    return out


def _perm(E: int, rng: np.random.Generator) -> np.ndarray:
    return rng.permutation(E)


def _gumbel_topk(logp: np.ndarray, g: np.ndarray, K: int) -> np.ndarray:
    """K distinct experts per token: top-K of log p + Gumbel noise."""
    key = g + logp[None, :]
    idx = np.argpartition(-key, K - 1, axis=1)[:, :K]
    # order the K picks by descending key (a router's top-k order)
    kk = np.take_along_axis(key, idx, axis=1)
    o = np.argsort(-kk, axis=1, kind="stable")
    return np.take_along_axis(idx, o, axis=1)


def _zipf_logp(E: int, s: float, perm: np.ndarray) -> np.ndarray:
    return -s * np.log(perm.astype(np.float64) + 1.0)


def _hot_logp(E: int, hot: np.ndarray, h: float) -> np.ndarray:
    lp = np.zeros(E)
    lp[hot] = h
    return lp


def _bisect(fn, target: float, lo: float, hi: float, tol: float, iters: int = 60):
    """Find x in [lo, hi] with fn(x) within tol of target (fn increasing)."""
    best = None
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        v, out = fn(mid)
        if best is None or abs(v - target) < abs(best[0] - target):
            best = (v, out, mid)
        if abs(v - target) <= tol:
            return v, out, mid
        if v < target:
            lo = mid
        else:
            hi = mid
    return best


def routing(shape: Shape, kind: str = "zipf", *, target_maxvio: float | None = None,
            zipf_s: float | None = None, hot_share: float | None = None,
            hot_group0: bool = False, seed: int = 0, tol: float = 0.02):
    """Seeded top-k expert ids [R, S, K] int32 plus a description dict.

    kinds:
      * "exact0": maxvio = 0 exactly; token t = r*S + s takes experts
        perm((t*K + k) mod E), k < K (distinct when K <= E).
      * "zipf": p_e proportional to (perm(e)+1)^-s, K distinct picks per token
        by Gumbel-top-K.  Either zipf_s is given, or s is bisected until the
        realized maxvio is within tol of target_maxvio.
      * "hot": 4 hot experts (perm[0:4], or experts 0..3 when hot_group0) with a
        log-weight bisected until they receive hot_share of all routes; the rest
        uniform.
      * "uniform": zipf with s = 0.
    """
    R, S, K, E = shape.R, shape.S, shape.K, shape.E
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = _perm(E, rng)
    T = R * S
    info = {"kind": kind, "seed": seed}
    if kind == "exact0":
        t = np.arange(T, dtype=np.int64)[:, None]
        k = np.arange(K, dtype=np.int64)[None, :]
        ids = perm[(t * K + k) % E]
        topk = ids.reshape(R, S, K).astype(np.int32)
        info["maxvio"] = maxvio(topk, E)
        return topk, info
    g = rng.gumbel(size=(T, E))
    if kind == "uniform":
        kind, zipf_s = "zipf", 0.0
    if kind == "zipf":
        def ev(s):
            ids = _gumbel_topk(_zipf_logp(E, s, perm), g, K)
            tk = ids.reshape(R, S, K).astype(np.int32)
            return maxvio(tk, E), tk
        if zipf_s is not None:
            mv, topk = ev(zipf_s)
            info.update(zipf_s=zipf_s, maxvio=mv)
            return topk, info
        assert target_maxvio is not None
        mv, topk, s = _bisect(ev, target_maxvio, 0.0, 12.0, tol)
        info.update(zipf_s=s, maxvio=mv, target_maxvio=target_maxvio)
        return topk, info
    if kind == "hot":
        share = 0.30 if hot_share is None else hot_share
        hot = np.arange(4) if hot_group0 else perm[:4]

        def ev(h):
            ids = _gumbel_topk(_hot_logp(E, hot, h), g, K)
            tk = ids.reshape(R, S, K).astype(np.int32)
            frac = float(np.isin(tk, hot).mean())
            return frac, tk
        fr, topk, h = _bisect(ev, share, 0.0, 30.0, 0.002)
        info.update(hot=[int(x) for x in hot], hot_share=fr, hot_logweight=h,
                    maxvio=maxvio(topk, E))
        return topk, info
    raise ValueError(kind)


def route_weights(shape: Shape, seed: int) -> np.ndarray:
    """Route weights [R, S, K] fp32: softmax of N(0,1) logits over the K picks,
    or sigmoid(N(0,1)) scores normalised over the K picks."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    z = rng.standard_normal((shape.R, shape.S, shape.K))
    if shape.weights == "softmax":
        z = np.exp(z - z.max(axis=-1, keepdims=True))
    else:
        z = 1.0 / (1.0 + np.exp(-z))
    w = z / z.sum(axis=-1, keepdims=True)
    return w.astype(np.float32)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 for use as *inputs*, returned as uint16 bits.
    Uses torch's CPU conversion (input generation only)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def hidden_bf16(shape_or_dims, seed: int, rows: int | None = None,
                cols: int | None = None) -> np.ndarray:
    """N(0,1) hidden rows rounded to bf16, as uint16 bits [rows, cols]."""
    if isinstance(shape_or_dims, Shape):
        rows = shape_or_dims.R * shape_or_dims.S if rows is None else rows
        cols = shape_or_dims.H if cols is None else cols
    rng = np.random.Generator(np.random.PCG64(seed + 104729))
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    return bf16_bits_from_f32(x)


def describe(shape: Shape) -> dict:
    d = dataclasses.asdict(shape)
    d.update(L=shape.L, C=shape.C, N=shape.N, NvS=shape.NvS)
    return d
