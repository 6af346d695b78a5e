"""Pins of the CPU oracle against what the pages and the number formats fix.

Each check is independent of the oracle's own code: hand-derived fixtures
(tests/golden), library decoders (torch.float8_e4m3fn), numpy fp64 matmul as the
dense special case, and invariants of the definitions (segmentation, power-of-two
scaling, error bounds).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import synth
from conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(a):
    return synth.bf16_bits_from_f32(np.asarray(a, dtype=np.float32))


def _torch_deq(q, sc):
    """Dequantize with torch's float8_e4m3fn decoder and numpy's ldexp (independent
    of the oracle's codecs).  q [C, Mcap] uint8, sc [C, Mcap/32] uint8 -> fp64."""
    vals = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scale = np.ldexp(1.0, sc.astype(np.int64) - 127)
    return vals * np.repeat(scale, 32, axis=1)


# ------------------------------------------------------------------ codecs
def test_e4m3_decode_matches_torch_all_bytes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    for b in range(256):
        got = oracle.e4m3_decode(b)
        if np.isnan(ref[b]):
            assert np.isnan(got), b
        else:
            assert got == ref[b], (b, got, ref[b])
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_encode_roundtrip_every_finite_byte():
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(b)) == b, hex(b)


def test_e4m3_encode_golden_examples():
    g = _golden("e4m3_e8m0_examples.json")
    for ex in g["encode_rne"]:
        assert oracle.e4m3_encode(ex["value"]) == int(ex["byte"], 16), ex


def test_e4m3_encode_matches_torch_rne_sweep():
    rng = np.random.default_rng(123)
    # magnitudes over the whole e4m3 range incl. subnormals, midpoints and near-ties
    mags = np.concatenate([
        np.exp2(rng.uniform(-12, np.log2(448.0), 20000)),
        np.array([oracle.e4m3_decode(b) for b in range(0x7E)]),
    ])
    mids = np.array([(oracle.e4m3_decode(b) + oracle.e4m3_decode(b + 1)) / 2 for b in range(0x7E)])
    vals = np.concatenate([mags, -mags, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_e8m0_decode():
    for b in range(255):
        assert oracle.e8m0_decode(b) == 2.0 ** (b - 127)
    assert np.isnan(oracle.e8m0_decode(255))


def test_scale_byte_golden_and_power_of_two_shift():
    g = _golden("e4m3_e8m0_examples.json")
    for ex in g["scale_byte"]:
        assert oracle.mx_scale_byte(ex["amax"]) == ex["byte"], ex
    rng = np.random.default_rng(5)
    for amax in rng.uniform(0.01, 100, 200):
        b = oracle.mx_scale_byte(amax)
        for j in (-5, -1, 1, 7):
            assert oracle.mx_scale_byte(amax * 2.0 ** j) == b + j
        # the scaled block maximum lands in [256, 512): the top binade of e4m3 and the next
        assert 256 <= amax * 2.0 ** (127 - b) < 512


# ---------------------------------------------------------------- quantize
def test_quantize_hand_example():
    g = _golden("wgrad_hand_2x2.json")
    one = g["one_expert"]
    for name, key_q, key_s in (("g", "g_q_cols", "g_scale_bytes"), ("x", "x_q_cols", "x_scale_bytes")):
        q, sc = oracle.mxfp8_quantize(_bf16(g[name]), one["expert_off"], Mcap=128)
        for c in range(2):
            assert [hex(v) for v in q[c, :2]] == [s.lower() for s in one[key_q][c]]
            assert sc[c, 0] == one[key_s][c]
        assert not q[:, 2:].any() and not sc[:, 1:].any()


def test_quantize_layout_padding_and_block_restart():
    counts = [0, 33, 128, 1, 0, 200]
    M, C = sum(counts), 8
    case = synth.wgrad_random(M, C, C, counts, seed=3)
    q, sc = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    P = oracle.padded_starts(case.expert_off)
    assert P.tolist() == [0, 0, 128, 256, 384, 384, 640]
    v = synth.bf16_bits_to_f32(case.g_bf16).astype(np.float64)
    deq = _torch_deq(q, sc)
    off = case.expert_off
    for e in range(len(counts)):
        cnt = off[e + 1] - off[e]
        seg = deq[:, P[e]:P[e] + cnt].T  # [cnt, C]
        src = v[off[e]:off[e + 1]]
        # per-block scale is the MX rule on that expert's own 32-token blocks
        for j in range((cnt + 31) // 32):
            blk = src[32 * j:32 * j + 32]
            for c in range(C):
                assert sc[c, P[e] // 32 + j] == oracle.mx_scale_byte(np.abs(blk[:, c]).max())
        # element error: half an e4m3 ulp, or saturation at 448 * scale
        if cnt:
            s = np.ldexp(1.0, np.repeat(sc[:, P[e] // 32:P[e] // 32 + (cnt + 31) // 32].astype(int) - 127, 32, axis=1)[:, :cnt].T)
            sat = np.abs(src) >= 448 * s
            assert np.all(np.abs(seg[sat]) == 448 * s[sat])
            err = np.abs(seg - src)[~sat]
            lim = np.maximum(np.abs(src) * 2.0 ** -4, s * 2.0 ** -10)[~sat]
            assert np.all(err <= lim)
        # padding of the segment is zero, values and scales
        end = P[e + 1]
        assert not q[:, P[e] + cnt:end].any()
        assert not sc[:, (P[e] + cnt + 31) // 32:end // 32].any()
    assert not q[:, P[-1]:].any()


def test_quantize_power_of_two_input_scaling():
    case = synth.wgrad_random(96, 16, 16, [40, 56], seed=9)
    q0, s0 = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    v = synth.bf16_bits_to_f32(case.g_bf16) * np.float32(8.0)
    q1, s1 = oracle.mxfp8_quantize(synth.bf16_bits_from_f32(v), case.expert_off)
    assert np.array_equal(q0, q1)
    nz = (s0 != 0)
    assert np.array_equal(s1[nz].astype(int), s0[nz].astype(int) + 3)


# ------------------------------------------------------------------- wgrad
def test_wgrad_hand_example_one_and_two_experts():
    g = _golden("wgrad_hand_2x2.json")
    for key in ("one_expert", "two_experts"):
        off = g[key]["expert_off"]
        gq, gs = oracle.mxfp8_quantize(_bf16(g["g"]), off)
        xq, xs = oracle.mxfp8_quantize(_bf16(g["x"]), off)
        out = oracle.grouped_wgrad(gq, gs, xq, xs, off)
        assert out.tolist() == g[key]["grad_w"]
    two = np.array(g["two_experts"]["grad_w"])
    assert np.array_equal(two[:2] + two[2:], np.array(g["one_expert"]["grad_w"]))


@pytest.mark.parametrize("counts", [[100, 0, 37, 200], [0, 0, 64], [1, 129, 31]])
def test_wgrad_equals_dense_matmul_per_expert(counts):
    M, N, K = sum(counts), 24, 40
    case = synth.wgrad_random(M, N, K, counts, seed=11)
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    out = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    gd, xd = _torch_deq(gq, gs), _torch_deq(xq, xs)
    P = oracle.padded_starts(case.expert_off)
    for e, cnt in enumerate(counts):
        ref = gd[:, P[e]:P[e] + cnt] @ xd[:, P[e]:P[e] + cnt].T
        np.testing.assert_allclose(out[e * N:(e + 1) * N], ref, rtol=1e-13, atol=1e-12)
        if cnt == 0:
            assert not out[e * N:(e + 1) * N].any()
    for e in range(len(counts)):
        n, k = (3 * e + 1) % N, (7 * e + 2) % K
        assert oracle.grouped_wgrad_element(gq, gs, xq, xs, case.expert_off, e, n, k) == out[e * N + n, k]


def test_wgrad_segments_sum_to_single_expert_when_32_aligned():
    counts = [64, 32, 0, 96]
    M, N, K = sum(counts), 16, 24
    case = synth.wgrad_random(M, N, K, counts, seed=13)
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    out = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off).reshape(len(counts), N, K)
    one = [0, M]
    gq1, gs1 = oracle.mxfp8_quantize(case.g_bf16, one)
    xq1, xs1 = oracle.mxfp8_quantize(case.x_bf16, one)
    dense = oracle.grouped_wgrad(gq1, gs1, xq1, xs1, one)
    np.testing.assert_allclose(out.sum(0), dense, rtol=1e-12, atol=1e-12)


def test_wgrad_scales_exactly_with_power_of_two():
    counts = [50, 70]
    case = synth.wgrad_random(120, 16, 16, counts, seed=17)
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    base = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    g4 = synth.bf16_bits_from_f32(synth.bf16_bits_to_f32(case.g_bf16) * np.float32(4.0))
    gq4, gs4 = oracle.mxfp8_quantize(g4, case.expert_off)
    assert np.array_equal(oracle.grouped_wgrad(gq4, gs4, xq, xs, case.expert_off), 4.0 * base)


# ------------------------------------------------------------------- dgrad
def test_expert_for_row_golden_and_scan_equals_bsearch():
    g = _golden("dgrad_hand.json")["expert_for_row"]
    for r, e in zip(g["rows"], g["expert"]):
        assert oracle.expert_for_row_scan(g["expert_off"], r) == e
        assert oracle.expert_for_row_bsearch(g["expert_off"], r) == e
    rng = np.random.default_rng(2)
    for _ in range(50):
        E = int(rng.integers(1, 12))
        counts = rng.integers(0, 5, E)
        if counts.sum() == 0:
            counts[-1] = 1
        off = synth.offsets_from_counts(counts)
        for r in range(int(counts.sum())):
            e = oracle.expert_for_row_scan(off, r)
            assert e == oracle.expert_for_row_bsearch(off, r)
            assert off[e] <= r < off[e + 1]


def test_dgrad_hand_example():
    g = _golden("dgrad_hand.json")["dgrad_2x2"]
    dx, bound = oracle.grouped_dgrad(np.array(g["dy"], np.float32), np.array(g["W"], np.float32),
                                     g["expert_off"])
    assert dx.tolist() == g["dx"] and bound.tolist() == g["bound"]


def test_dgrad_equals_dense_matmul_rows():
    counts = [7, 0, 40, 1, 0]
    case = synth.dgrad_random(sum(counts), 24, 20, counts, seed=4)
    dx, bound = oracle.grouped_dgrad(case.dy, case.W, case.expert_off)
    off = case.expert_off
    dy, W = case.dy.astype(np.float64), case.W.astype(np.float64)
    for e, cnt in enumerate(counts):
        ref = dy[off[e]:off[e + 1]] @ W[e]
        np.testing.assert_allclose(dx[off[e]:off[e + 1]], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(bound[off[e]:off[e + 1]], np.abs(dy[off[e]:off[e + 1]]) @ np.abs(W[e]),
                                   rtol=1e-12, atol=1e-12)
    assert np.all(np.abs(dx) <= bound * (1 + 1e-12))
    v, b = oracle.grouped_dgrad_element(case.dy, case.W, off, 10, 3)
    assert v == dx[10, 3] and b == bound[10, 3]


def test_dgrad_single_expert_is_dense_gemm():
    case = synth.dgrad_random(33, 16, 12, [33], seed=8)
    dx, _ = oracle.grouped_dgrad(case.dy, case.W, case.expert_off)
    np.testing.assert_allclose(dx, case.dy.astype(np.float64) @ case.W[0].astype(np.float64),
                               rtol=1e-12, atol=1e-12)


# Offsets 0,7,7,47,48,48,148: rows 0-31 and 32-63 straddle expert boundaries (each row
# looks up its own expert), rows 64-147 fall in 32-row groups of one expert.
@pytest.mark.parametrize("counts,out_f,in_f,seed", [
    ([7, 0, 40, 1, 0, 100], 48, 20, 21),
    ([64, 32, 0, 33], 1536, 8, 22),   # long sums: the MoE FFN pair's 1536 output features
    ([200], 64, 16, 23),              # one expert: every group takes the shortcut
])
def test_dgrad_page_fp32_formulation_within_tolerance(counts, out_f, in_f, seed):
    """The dgrad page's own fp32 arithmetic (group shortcut, sequential fp32 sums, fused or
    not) lands within 1e-5 * sum|dy||W| of the fp64 definition: the tolerance admits the
    page's result, and an indexing slip in either formulation would not."""
    case = synth.dgrad_random(sum(counts), out_f, in_f, counts, seed=seed)
    dx, bound = oracle.grouped_dgrad(case.dy, case.W, case.expert_off)
    for fused in (True, False):
        got = oracle.grouped_dgrad_page_f32(case.dy, case.W, case.expert_off, fused)
        assert got.dtype == np.float32 and got.shape == dx.shape
        err = np.abs(got.astype(np.float64) - dx)
        assert np.all(err <= 1e-5 * bound), float((err / np.maximum(bound, 1e-300)).max())
    # Rows of the straddling groups differ from what the group's first expert would give.
    if len(counts) > 1:
        off = case.expert_off
        r = int(off[1])  # first row after expert 0
        wrong = case.dy[r].astype(np.float64) @ case.W[0].astype(np.float64)
        assert np.abs(wrong - dx[r]).max() > 1e-3 * np.abs(dx[r]).max()


# ------------------------------------------------------ RoundUp scale rule
def test_ceil448_scale_golden_and_bracket():
    g = _golden("e4m3_e8m0_examples.json")["scale_byte_ceil448"]
    for ex in g["examples"]:
        assert oracle.mx_scale_byte_ceil448(ex["amax"]) == ex["byte"], ex
    rng = np.random.default_rng(6)
    for amax in np.exp2(rng.uniform(-30, 30, 500)):
        amax = float(np.float32(amax))
        b = oracle.mx_scale_byte_ceil448(amax)
        assert 1 <= b <= 254
        # the power of two is the smallest with 448 * 2^(b-127) >= amax, up to fp32 rounding
        assert 448.0 * 2.0 ** (b - 127) >= amax * (1 - 2.0 ** -22)
        assert 448.0 * 2.0 ** (b - 128) < amax * (1 + 2.0 ** -22)


def test_quantize_ceil448_never_saturates_and_rounds_to_nearest():
    counts = [40, 0, 97]
    case = synth.wgrad_random(sum(counts), 16, 16, counts, seed=12, outlier_frac=0.05)
    q, sc = oracle.mxfp8_quantize(case.g_bf16, case.expert_off, rule=oracle.SCALE_CEIL_448)
    P = oracle.padded_starts(case.expert_off)
    v = synth.bf16_bits_to_f32(case.g_bf16).astype(np.float64)
    deq = _torch_deq(q, sc)
    off = case.expert_off
    for e, cnt in enumerate(counts):
        if not cnt:
            continue
        seg = deq[:, P[e]:P[e] + cnt].T
        src = v[off[e]:off[e + 1]]
        s = np.ldexp(1.0, np.repeat(sc[:, P[e] // 32:P[e] // 32 + (cnt + 31) // 32].astype(int) - 127, 32, axis=1)[:, :cnt].T)
        assert np.all(np.abs(src) <= 448 * s * (1 + 2.0 ** -22))  # no value beyond the range
        err = np.abs(seg - src)
        assert np.all(err <= np.maximum(np.abs(src) * 2.0 ** -4, s * 2.0 ** -10))
        # the padding blocks of the segment keep byte 0
        assert not sc[:, (P[e] + cnt + 31) // 32:P[e + 1] // 32].any()
