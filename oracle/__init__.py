"""Plain fp64 CPU oracle for the grouped MoE backward GEMMs.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``moe_grouped_gemm_wgrad_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, no blocking); this module
compiles it with gcc on first use and wraps it with ctypes over numpy arrays.
Each function's docstring names the passage of the pages it restates:

* wgrad page: "tinygrad/extra/thunder/amd/grouped_mxfp8_wgrad.cpp"
* dgrad page: "oarust ... grouped_gemm_m_data_backward.slang"
* post-attn page: vLLM "models/minimax_m3/amd/mono/kernels/post_attn" (the
  saturating clamp of its MXFP8 quantizer, mx8_q)
* OCP "OFP8 Formats" v1.0 and "Microscaling Formats (MX)" v1.0 for the codecs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (plain gcc, no -ffast-math,
    no FMA contraction, so x86 and aarch64 give the same results)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, u8, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_uint8, ctypes.c_double
            lib.orc_e4m3_decode.argtypes = [u8]
            lib.orc_e4m3_decode.restype = dbl
            lib.orc_e4m3_encode_rne_satfinite.argtypes = [dbl]
            lib.orc_e4m3_encode_rne_satfinite.restype = u8
            lib.orc_e8m0_decode.argtypes = [u8]
            lib.orc_e8m0_decode.restype = dbl
            lib.orc_mx_scale_byte.argtypes = [dbl]
            lib.orc_mx_scale_byte.restype = u8
            lib.orc_mx_scale_byte_ceil448.argtypes = [dbl]
            lib.orc_mx_scale_byte_ceil448.restype = u8
            lib.orc_padded_starts.argtypes = [P, i32, P]
            lib.orc_padded_starts.restype = None
            lib.orc_mxfp8_quantize.argtypes = [P, i32, i32, P, i32, i64, i32, P, P]
            lib.orc_mxfp8_quantize.restype = None
            lib.orc_grouped_wgrad.argtypes = [P, P, P, P, P, i32, i32, i32, i64, P]
            lib.orc_grouped_wgrad.restype = None
            lib.orc_grouped_wgrad_element.argtypes = [P, P, P, P, P, i32, i64, i32, i32, i32]
            lib.orc_grouped_wgrad_element.restype = dbl
            lib.orc_expert_for_row_scan.argtypes = [P, i32, i32]
            lib.orc_expert_for_row_scan.restype = i32
            lib.orc_expert_for_row_bsearch.argtypes = [P, i32, i32]
            lib.orc_expert_for_row_bsearch.restype = i32
            lib.orc_grouped_dgrad.argtypes = [P, P, P, i32, i32, i32, i32, P, P]
            lib.orc_grouped_dgrad.restype = None
            lib.orc_grouped_dgrad_element.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P]
            lib.orc_grouped_dgrad_element.restype = dbl
            lib.orc_grouped_dgrad_page_f32.argtypes = [P, P, P, i32, i32, i32, i32, i32, P]
            lib.orc_grouped_dgrad_page_f32.restype = None
            lib.orc_mxfp8_quantize_rows.argtypes = [P, i32, i32, P, i32, i64, i32, P, P]
            lib.orc_mxfp8_quantize_rows.restype = None
            lib.orc_mx_dot.argtypes = [P, P, P, P, i32]
            lib.orc_mx_dot.restype = dbl
            lib.orc_grouped_fprop_mx.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, P]
            lib.orc_grouped_fprop_mx.restype = None
            lib.orc_grouped_dgrad_mx.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, i64, P]
            lib.orc_grouped_dgrad_mx.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _off(expert_off) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(expert_off, dtype=np.int32))


# ------------------------------------------------------------------ codecs
def e4m3_decode(b: int) -> float:
    """OCP OFP8 E4M3 value of one byte (NaN for S.1111.111)."""
    return _load().orc_e4m3_decode(int(b) & 0xFF)


def e4m3_encode(v: float) -> int:
    """Round-to-nearest-even to E4M3, saturating at +-448 (post-attn page, mx8_q clamp)."""
    return int(_load().orc_e4m3_encode_rne_satfinite(float(v)))


def e8m0_decode(b: int) -> float:
    """OCP MX E8M0 value 2^(b-127)."""
    return _load().orc_e8m0_decode(int(b) & 0xFF)


def mx_scale_byte(amax: float) -> int:
    """E8M0 byte of 2^(floor(log2 amax) - 8), clamped to the E8M0 range; 0 for amax 0."""
    return int(_load().orc_mx_scale_byte(float(amax)))


def mx_scale_byte_ceil448(amax: float) -> int:
    """The post-attn page's RoundUp rule: exponent of ceil_pow2(amax * fp32(1/448)), in [1, 254]."""
    return int(_load().orc_mx_scale_byte_ceil448(float(amax)))


SCALE_FLOOR = 0     # OCP MX rule 2^(floor(log2 amax) - 8)
SCALE_CEIL_448 = 1  # the post-attn page's RoundUp rule


def padded_starts(expert_off) -> np.ndarray:
    """P[e]: start of expert e's 128-padded segment in the quantized token axis."""
    off = _off(expert_off)
    E = off.size - 1
    P = np.zeros(E + 1, dtype=np.int64)
    _load().orc_padded_starts(_ptr(off), E, _ptr(P))
    return P


def token_capacity(M: int, E: int) -> int:
    """Smallest padded token axis that fits any split of M tokens over E experts."""
    return (M + 127 * E + 127) // 128 * 128


# ---------------------------------------------------------------- quantize
def mxfp8_quantize(src_bf16_bits: np.ndarray, expert_off, Mcap: int | None = None,
                   rule: int = SCALE_FLOOR):
    """MXFP8 quantization along the token axis (wgrad page: A = g^T, B = x^T in e4m3
    with e8m0 scales per 32 tokens).  ``src_bf16_bits`` is uint16 [M, C]; ``rule`` picks
    the scale rule (SCALE_FLOOR or SCALE_CEIL_448).

    Returns (q [C, Mcap] uint8, sc [C, Mcap/32] uint8) in the plain layout."""
    src = np.ascontiguousarray(src_bf16_bits, dtype=np.uint16)
    M, C = src.shape
    off = _off(expert_off)
    E = off.size - 1
    if Mcap is None:
        Mcap = token_capacity(M, E)
    q = np.empty((C, Mcap), dtype=np.uint8)
    sc = np.empty((C, Mcap // 32), dtype=np.uint8)
    _load().orc_mxfp8_quantize(_ptr(src), M, C, _ptr(off), E, Mcap, int(rule), _ptr(q), _ptr(sc))
    return q, sc


# ------------------------------------------------------------------- wgrad
def grouped_wgrad(gq, gs, xq, xs, expert_off) -> np.ndarray:
    """fp64 grad_w [E*N, K] = per expert g_e^T x_e over its tokens (wgrad page)."""
    off = _off(expert_off)
    E = off.size - 1
    N, Mcap = gq.shape
    K = xq.shape[0]
    out = np.empty((E * N, K), dtype=np.float64)
    _load().orc_grouped_wgrad(_ptr(gq), _ptr(gs), _ptr(xq), _ptr(xs), _ptr(off), E, N, K,
                              Mcap, _ptr(out))
    return out


def grouped_wgrad_element(gq, gs, xq, xs, expert_off, e: int, n: int, k: int) -> float:
    """One element grad_w[e*N + n, k] of :func:`grouped_wgrad`."""
    off = _off(expert_off)
    return _load().orc_grouped_wgrad_element(_ptr(gq), _ptr(gs), _ptr(xq), _ptr(xs), _ptr(off),
                                             off.size - 1, gq.shape[1], e, n, k)


# ------------------------------------------------------------------- dgrad
def expert_for_row_scan(expert_off, row: int) -> int:
    """The dgrad page's expert_for_row (linear scan)."""
    off = _off(expert_off)
    return int(_load().orc_expert_for_row_scan(_ptr(off), off.size - 1, row))


def expert_for_row_bsearch(expert_off, row: int) -> int:
    """Binary-search restatement of the same rule."""
    off = _off(expert_off)
    return int(_load().orc_expert_for_row_bsearch(_ptr(off), off.size - 1, row))


def grouped_dgrad(dy: np.ndarray, W: np.ndarray, expert_off):
    """fp64 dx[r] = dy[r] . W[e(r)] and bound = |dy| . |W[e(r)]| (dgrad page)."""
    dy = np.ascontiguousarray(dy, dtype=np.float32)
    W = np.ascontiguousarray(W, dtype=np.float32)
    off = _off(expert_off)
    rows, out_f = dy.shape
    E, _, in_f = W.shape
    dx = np.empty((rows, in_f), dtype=np.float64)
    bound = np.empty((rows, in_f), dtype=np.float64)
    _load().orc_grouped_dgrad(_ptr(dy), _ptr(W), _ptr(off), E, rows, out_f, in_f, _ptr(dx),
                              _ptr(bound))
    return dx, bound


def grouped_dgrad_element(dy: np.ndarray, W: np.ndarray, expert_off, r: int, k: int):
    """(dx[r, k], bound[r, k]) of :func:`grouped_dgrad`, one element."""
    off = _off(expert_off)
    rows, out_f = dy.shape
    E, _, in_f = W.shape
    b = ctypes.c_double(0.0)
    v = _load().orc_grouped_dgrad_element(_ptr(dy), _ptr(W), _ptr(off), E, rows, out_f, in_f,
                                          r, k, ctypes.c_void_p(ctypes.addressof(b)))
    return v, b.value


def grouped_dgrad_page_f32(dy: np.ndarray, W: np.ndarray, expert_off, fused: bool = True):
    """The dgrad page's fp32 formulation (32-row groups, running fp32 sums over the
    output features; fused multiply-add or product-then-add).  A cross-check of
    :func:`grouped_dgrad`, not the definition.  Returns fp32 dx [rows, in_f]."""
    dy = np.ascontiguousarray(dy, dtype=np.float32)
    W = np.ascontiguousarray(W, dtype=np.float32)
    off = _off(expert_off)
    rows, out_f = dy.shape
    E, _, in_f = W.shape
    dx = np.empty((rows, in_f), dtype=np.float32)
    _load().orc_grouped_dgrad_page_f32(_ptr(dy), _ptr(W), _ptr(off), E, rows, out_f, in_f,
                                       1 if fused else 0, _ptr(dx))
    return dx


# ------------------------------------------- forward and data-gradient GEMMs (MXFP8)
def mxfp8_quantize_rows(src_bf16_bits: np.ndarray, expert_off, Mcap: int | None = None,
                        rule: int = SCALE_FLOOR):
    """Row-wise MXFP8 quantization along the hidden axis (post-attn page: each token's
    activations staged as MXFP8 with one e8m0 byte per 32 hidden features).  Rows of
    expert e go to padded rows P[e] + (r - off[e]).

    Returns (q [Mcap, C] uint8, sc [Mcap, C/32] uint8) in the plain layout."""
    src = np.ascontiguousarray(src_bf16_bits, dtype=np.uint16)
    M, C = src.shape
    off = _off(expert_off)
    E = off.size - 1
    if Mcap is None:
        Mcap = token_capacity(M, E)
    q = np.empty((Mcap, C), dtype=np.uint8)
    sc = np.empty((Mcap, C // 32), dtype=np.uint8)
    _load().orc_mxfp8_quantize_rows(_ptr(src), M, C, _ptr(off), E, Mcap, int(rule), _ptr(q),
                                    _ptr(sc))
    return q, sc


def mx_dot(aq, as_, bq, bs) -> float:
    """sum_l deq(a)[l] deq(b)[l] of two MXFP8 vectors (one scale per 32 elements)."""
    aq, as_, bq, bs = (np.ascontiguousarray(v, dtype=np.uint8) for v in (aq, as_, bq, bs))
    L = aq.size
    assert bq.size == L and as_.size == L // 32 and bs.size == L // 32
    return float(_load().orc_mx_dot(_ptr(aq), _ptr(as_), _ptr(bq), _ptr(bs), L))


def grouped_fprop_mx(xq, xs, wq, ws, expert_off, w_off, M: int) -> np.ndarray:
    """fp64 y[r, n] = deq(x)[r] . deq(W)[e(r), n] over the hidden axis (post-attn page's
    expert GEMMs, forward).  x row-wise quantized [Mcap, K]; W row-wise quantized stacked
    [Mw, K] with expert e's rows from the padded start of ``w_off``."""
    off, woff = _off(expert_off), _off(w_off)
    E = off.size - 1
    Mcap, K = xq.shape
    N = int(woff[1] - woff[0])
    out = np.empty((M, N), dtype=np.float64)
    _load().orc_grouped_fprop_mx(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), _ptr(off), _ptr(woff),
                                 E, M, N, K, Mcap, _ptr(out))
    return out


def grouped_dgrad_mx(dyq, dys, wtq, wts, expert_off, w_off, M: int) -> np.ndarray:
    """fp64 dx[r, k] = sum_n deq(dy)[r, n] deq(W)[e(r), n, k] (dgrad page, MXFP8 operands).
    dy row-wise quantized [Mcap, N]; W quantized along n per expert (the token-axis
    quantizer on W stacked [E*N, K] with ``w_off``): wtq [K, Mw]."""
    off, woff = _off(expert_off), _off(w_off)
    E = off.size - 1
    Mcap, N = dyq.shape
    K, Mw = wtq.shape
    out = np.empty((M, K), dtype=np.float64)
    _load().orc_grouped_dgrad_mx(_ptr(dyq), _ptr(dys), _ptr(wtq), _ptr(wts), _ptr(off),
                                 _ptr(woff), E, M, N, K, Mcap, Mw, _ptr(out))
    return out


# ------------------------------------------------ full-size references by matmul
# The same definitions, for outputs too large for the loops above: each expert's operands
# are decoded exactly into fp64 with this oracle's own E4M3 and E8M0 decoders (per byte,
# and per 32-element block for the scale), and numpy's fp64 matrix product forms the sums.
# A product of two decoded MXFP8 values is exact in fp64, so these differ from the loop
# versions only in the order of the fp64 additions (pinned against them on small cases).
_tables = None


def _decode_tables():
    """(E4M3 value of every byte, E8M0 value of every byte), from the decoders above."""
    global _tables
    if _tables is None:
        _tables = (np.array([e4m3_decode(b) for b in range(256)], dtype=np.float64),
                   np.array([e8m0_decode(b) for b in range(256)], dtype=np.float64))
    return _tables


def dequantize_token_axis(q, sc, t0: int, count: int) -> np.ndarray:
    """fp64 [C, count]: columns t0 .. t0+count-1 of a token-axis operand (q [C, Mcap],
    plain scales sc [C, Mcap/32]) decoded and multiplied by their 32-token block's scale.
    t0 is a multiple of 32 (an expert's padded start)."""
    e4m3, e8m0 = _decode_tables()
    assert t0 % 32 == 0
    vals = e4m3[q[:, t0:t0 + count]]
    nb = (count + 31) // 32
    scale = e8m0[sc[:, t0 // 32:t0 // 32 + nb]]
    vals *= np.repeat(scale, 32, axis=1)[:, :count]
    return vals


def dequantize_rows(q, sc, p0: int, count: int) -> np.ndarray:
    """fp64 [count, C]: rows p0 .. p0+count-1 of a row-wise operand (q [Mcap, C], plain
    scales sc [Mcap, C/32]) decoded and multiplied by their 32-column block's scale."""
    e4m3, e8m0 = _decode_tables()
    vals = e4m3[q[p0:p0 + count]]
    vals *= np.repeat(e8m0[sc[p0:p0 + count]], 32, axis=1)
    return vals


def grouped_wgrad_by_expert(gq, gs, xq, xs, expert_off):
    """Yields (e, fp64 grad_w[e] [N, K]) for every expert: the wgrad page's per-expert
    g_e^T x_e over its tokens, as a matrix product of the decoded slices.  An expert
    without tokens yields None (its rows are zero by definition)."""
    off = _off(expert_off)
    P = padded_starts(off)
    for e in range(off.size - 1):
        c = int(off[e + 1] - off[e])
        if c == 0:
            yield e, None
            continue
        G = dequantize_token_axis(gq, gs, int(P[e]), c)
        X = dequantize_token_axis(xq, xs, int(P[e]), c)
        yield e, G @ X.T


def grouped_dgrad_by_expert(dy: np.ndarray, W: np.ndarray, expert_off):
    """Yields (e, r0, r1, dx[r0:r1] fp64, bound[r0:r1] fp64) for every expert with rows:
    the dgrad page's dx[r] = dy[r] . W[e(r)] for the rows the expert owns, and
    bound = |dy| . |W[e]|."""
    off = _off(expert_off)
    for e in range(off.size - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        d = dy[r0:r1].astype(np.float64)
        w = W[e].astype(np.float64)
        yield e, r0, r1, d @ w, np.abs(d) @ np.abs(w)


def grouped_fprop_mx_by_expert(xq, xs, wq, ws, expert_off, w_off):
    """Yields (e, r0, r1, y[r0:r1] fp64) for every expert with rows: the forward
    y[r, n] = deq(x)[r] . deq(W)[e, n] of :func:`grouped_fprop_mx` as a matrix product."""
    off, woff = _off(expert_off), _off(w_off)
    P, Pw = padded_starts(off), padded_starts(woff)
    N = int(woff[1] - woff[0])
    for e in range(off.size - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        X = dequantize_rows(xq, xs, int(P[e]), r1 - r0)
        Wd = dequantize_rows(wq, ws, int(Pw[e]), N)
        yield e, r0, r1, X @ Wd.T


def grouped_dgrad_mx_by_expert(dyq, dys, wtq, wts, expert_off, w_off):
    """Yields (e, r0, r1, dx[r0:r1] fp64) for every expert with rows: the MXFP8 data
    gradient dx[r, k] = sum_n deq(dy)[r, n] deq(W)[e, n, k] of :func:`grouped_dgrad_mx`
    as a matrix product."""
    off, woff = _off(expert_off), _off(w_off)
    P, Pw = padded_starts(off), padded_starts(woff)
    N = int(woff[1] - woff[0])
    for e in range(off.size - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        D = dequantize_rows(dyq, dys, int(P[e]), r1 - r0)
        Wt = dequantize_token_axis(wtq, wts, int(Pw[e]), N)
        yield e, r0, r1, D @ Wt.T
