"""Seeded synthetic inputs for the grouped MoE backward GEMMs.

This module holds no arithmetic of the method itself: it only draws random
tensors and token splits with the shapes and distributions of the five
workloads, and rounds fp32 draws to bf16 (the input dtype of the quantizer).
Both the CUDA path's tests and the oracle consume what it returns.

Workloads (sizes from the wgrad page's default shape and the benchmark set):

* ``wgrad_tiny``   E=2, M=256, expert_off={0,128,256}, N=K=256
* ``dgrad_4096``   rows=4096, out=in=1024, E=8, multinomial split
* ``wgrad_8192``   M=N=K=8192, E=8, 1024 tokens per expert (the wgrad page's
                   default WGRAD_M/N/K/E)
* ``wgrad_skew``   M=16384, E=32, N=4096, K=2048, Zipf(1.2) counts rounded to
                   multiples of 128 with at least one empty expert, 1% of
                   elements x50
* ``moe_ffn_pair`` E=64, hidden=4096, ffn=1536, 8192 tokens routed top-8
                   (65536 rows): wgrad N=1536, K=4096 and dgrad 1536 -> 4096
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_f32(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (rng.standard_normal(size=shape, dtype=np.float64) * std).astype(np.float32)


def offsets_from_counts(counts) -> np.ndarray:
    off = np.zeros(len(counts) + 1, dtype=np.int32)
    off[1:] = np.cumsum(np.asarray(counts, dtype=np.int64))
    return off


def multinomial_counts(rng: np.random.Generator, total: int, E: int) -> np.ndarray:
    """Token-by-token uniform categorical draws over E experts."""
    return rng.multinomial(total, [1.0 / E] * E).astype(np.int64)


def zipf_counts(seed: int, total: int, E: int, s: float = 1.2, quantum: int = 128):
    """Per-expert weights v_i ~ Zipf(s); counts = round(total*v/sum(v)/quantum)*quantum,
    the remainder put on the largest expert; re-seed until at least one expert is empty."""
    sd = seed
    while True:
        rng = np.random.default_rng(sd)
        v = rng.zipf(s, size=E).astype(np.float64)
        c = np.rint(total * v / v.sum() / quantum).astype(np.int64) * quantum
        c[int(np.argmax(c))] += total - int(c.sum())
        if (c == 0).any() and (c >= 0).all():
            return c, sd
        sd += 1


@dataclass
class WgradCase:
    """Inputs of one grouped MXFP8 wgrad: g [M, N] and x [M, K] as bf16 bits."""
    name: str
    M: int
    N: int
    K: int
    E: int
    expert_off: np.ndarray
    g_bf16: np.ndarray
    x_bf16: np.ndarray
    meta: dict = field(default_factory=dict)


@dataclass
class DgradCase:
    """Inputs of one grouped fp32 dgrad: dy [rows, out_f], W [E, out_f, in_f]."""
    name: str
    rows: int
    out_f: int
    in_f: int
    E: int
    expert_off: np.ndarray
    dy: np.ndarray
    W: np.ndarray
    meta: dict = field(default_factory=dict)


def wgrad_random(M: int, N: int, K: int, counts, seed: int = 0, outlier_frac: float = 0.0,
                 outlier_mul: float = 50.0, name: str = "wgrad_random") -> WgradCase:
    """g, x ~ N(0,1) (fp32, then bf16), optional Bernoulli outliers scaled by outlier_mul."""
    counts = np.asarray(counts, dtype=np.int64)
    assert counts.sum() == M
    rng = np.random.default_rng(seed)
    g = normal_f32(rng, (M, N))
    x = normal_f32(rng, (M, K))
    if outlier_frac > 0:
        g *= np.where(rng.random((M, N)) < outlier_frac, outlier_mul, 1.0).astype(np.float32)
        x *= np.where(rng.random((M, K)) < outlier_frac, outlier_mul, 1.0).astype(np.float32)
    return WgradCase(name, M, N, K, len(counts), offsets_from_counts(counts),
                     bf16_bits_from_f32(g), bf16_bits_from_f32(x), {"counts": counts.tolist()})


def dgrad_random(rows: int, out_f: int, in_f: int, counts, seed: int = 0,
                 w_std: float | None = None, name: str = "dgrad_random") -> DgradCase:
    counts = np.asarray(counts, dtype=np.int64)
    assert counts.sum() == rows
    E = len(counts)
    rng = np.random.default_rng(seed)
    dy = normal_f32(rng, (rows, out_f))
    W = normal_f32(rng, (E, out_f, in_f), std=(w_std if w_std is not None else out_f ** -0.5))
    return DgradCase(name, rows, out_f, in_f, E, offsets_from_counts(counts), dy, W,
                     {"counts": counts.tolist()})


# ------------------------------------------------------------- the workloads
def wgrad_tiny(seed: int = 0) -> WgradCase:
    return wgrad_random(256, 256, 256, [128, 128], seed=seed, name="wgrad_tiny")


def dgrad_4096(seed: int = 0) -> DgradCase:
    counts = multinomial_counts(np.random.default_rng(seed), 4096, 8)
    return dgrad_random(4096, 1024, 1024, counts, seed=seed, w_std=1.0 / 32, name="dgrad_4096")


def wgrad_8192(seed: int = 0) -> WgradCase:
    return wgrad_random(8192, 8192, 8192, [1024] * 8, seed=seed, name="wgrad_8192")


def wgrad_skew(seed: int = 0) -> WgradCase:
    counts, used = zipf_counts(seed, 16384, 32)
    case = wgrad_random(16384, 4096, 2048, counts, seed=seed, outlier_frac=0.01,
                        name="wgrad_skew")
    case.meta["zipf_seed"] = used
    return case


def moe_routing(seed: int, tokens: int, E: int, top_k: int):
    """Top-k distinct experts per token, uniform: the first top_k entries of a uniformly
    random permutation of the experts (argsort of uniform keys).  Routed rows are sorted
    by (expert, token).  Returns (token_of_row, counts)."""
    rng = np.random.default_rng(seed)
    choice = np.argsort(rng.random((tokens, E)), axis=1)[:, :top_k]
    tok = np.repeat(np.arange(tokens, dtype=np.int64), top_k)
    exp = choice.reshape(-1)
    order = np.lexsort((tok, exp))
    counts = np.bincount(exp, minlength=E).astype(np.int64)
    return tok[order], counts


def moe_ffn_pair(seed: int = 0, tokens: int = 8192, E: int = 64, hidden: int = 4096,
                 ffn: int = 1536, top_k: int = 8):
    """The MoE FFN up-projection backward pair: routed rows gathered from hidden
    states; wgrad (N=ffn, K=hidden) and fp32 dgrad dx = dy . W[e] (ffn -> hidden)."""
    token_of_row, counts = moe_routing(seed, tokens, E, top_k)
    rows = int(counts.sum())
    rng = np.random.default_rng(seed + 1)
    hidden_states = normal_f32(rng, (tokens, hidden))
    dy = normal_f32(rng, (rows, ffn))
    W = normal_f32(rng, (E, ffn, hidden), std=ffn ** -0.5)
    off = offsets_from_counts(counts)
    hidden_bf16 = bf16_bits_from_f32(hidden_states)
    wg = WgradCase("moe_ffn_pair.wgrad", rows, ffn, hidden, E, off, bf16_bits_from_f32(dy),
                   hidden_bf16[token_of_row],
                   {"counts": counts.tolist(), "hidden_bf16": hidden_bf16,
                    "token_of_row": token_of_row.astype(np.int32)})
    dg = DgradCase("moe_ffn_pair.dgrad", rows, ffn, hidden, E, off, dy, W,
                   {"counts": counts.tolist()})
    return wg, dg


def moe_ffn_slice(seed: int = 0) -> DgradCase:
    """A 16-expert slice of the MoE FFN pair's fp32 data gradient (2048 tokens, top-8 of 16
    experts: 16384 routed rows, ffn 1536 -> hidden 4096, 0.8 GB on the device), small enough
    for a full profiler capture of the CTA-pair dgrad kernel.  Not one of the workload
    configurations."""
    dg = moe_ffn_pair(seed, tokens=2048, E=16)[1]
    dg.name = "moe_ffn_slice.dgrad"
    return dg


WORKLOADS = ("wgrad_tiny", "dgrad_4096", "wgrad_8192", "wgrad_skew", "moe_ffn_pair")
