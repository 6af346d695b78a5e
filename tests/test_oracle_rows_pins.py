"""Pins of the oracle's row-wise MXFP8 quantizer and of its grouped forward and
data-gradient MXFP8 GEMMs against what does not come from those functions: the MX
worked example fixed by the scale rule, the token-axis quantizer (pinned on its own)
applied to the transpose, torch's float8_e4m3fn decoder with numpy fp64 matmul as the
dense special case, the wgrad oracle through the transpose identity, and the fp32
dgrad oracle on dequantized operands.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import synth


def _bf16(a):
    return synth.bf16_bits_from_f32(np.asarray(a, dtype=np.float32))


def _torch_deq_rows(q, sc):
    """[R, L] e4m3 bytes with [R, L/32] e8m0 bytes -> fp64, via torch's decoder."""
    vals = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=1)


def test_rows_hand_example():
    """One 32-element row with amax 3: the MX rule gives 2^(floor(log2 3) - 8) = 2^-7, byte
    120; 3 * 2^7 = 384 = 1.5 * 2^8 is e4m3 0.1111.100 = 0x7C, 1 * 2^7 = 128 is 0.1110.000
    = 0x70, -0.5 * 2^7 = -64 is 1.1101.000 = 0xE8, 0.01 * 2^7 = 1.28 rounds to 1.25 =
    0.0111.010 = 0x3A."""
    row = np.zeros((1, 32), dtype=np.float32)
    row[0, :4] = [3.0, 1.0, -0.5, 0.01]
    q, sc = oracle.mxfp8_quantize_rows(_bf16(row), [0, 1], Mcap=128)
    assert sc[0, 0] == 120
    assert [int(v) for v in q[0, :4]] == [0x7C, 0x70, 0xE8, 0x3A]
    assert not q[0, 4:].any() and not q[1:].any() and not sc[1:].any()


@pytest.mark.parametrize("rule", [oracle.SCALE_FLOOR, oracle.SCALE_CEIL_448])
def test_rows_equal_token_axis_quantizer_of_transpose(rule):
    """Quantizing row r along its hidden axis is quantizing column r of the transpose
    along its (single-expert) token axis."""
    counts = [37, 0, 128, 5]
    M, C = sum(counts), 96
    case = synth.wgrad_random(M, C, 32, counts, seed=21)
    q, sc = oracle.mxfp8_quantize_rows(case.g_bf16, case.expert_off, rule=rule)
    qt, sct = oracle.mxfp8_quantize(np.ascontiguousarray(case.g_bf16.T), [0, C], rule=rule)
    P = oracle.padded_starts(case.expert_off)
    off = case.expert_off
    for e in range(len(counts)):
        for i in range(counts[e]):
            r, p = off[e] + i, P[e] + i
            assert np.array_equal(q[p], qt[r, :C])
            assert np.array_equal(sc[p], sct[r, :C // 32])
        # padding rows of the expert's 128-row segment are zero
        end = P[e + 1] if e + 1 < len(P) else q.shape[0]
        assert not q[P[e] + counts[e]:end].any() and not sc[P[e] + counts[e]:end].any()


@pytest.mark.parametrize("counts", [[100, 0, 37, 200], [0, 0, 64], [1, 129, 31]])
def test_fprop_equals_dense_matmul_per_expert(counts):
    M, N, K, E = sum(counts), 24, 64, len(counts)
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((M, K)))
    W = _bf16(rng.standard_normal((E * N, K)) * 0.1)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    w_off = np.arange(E + 1, dtype=np.int32) * N
    xq, xs = oracle.mxfp8_quantize_rows(x, off)
    wq, ws = oracle.mxfp8_quantize_rows(W, w_off)
    y = oracle.grouped_fprop_mx(xq, xs, wq, ws, off, w_off, M)
    xd, wd = _torch_deq_rows(xq, xs), _torch_deq_rows(wq, ws)
    P, Pw = oracle.padded_starts(off), oracle.padded_starts(w_off)
    for e, cnt in enumerate(counts):
        ref = xd[P[e]:P[e] + cnt] @ wd[Pw[e]:Pw[e] + N].T
        np.testing.assert_allclose(y[off[e]:off[e + 1]], ref, rtol=1e-13, atol=1e-12)


def test_fprop_of_transposes_is_the_wgrad():
    """g^T x contracted over tokens: with x' = g^T (rows = features of g) and W' = x^T as a
    single expert, the forward GEMM over the token axis is the one-expert wgrad exactly
    (the same exact products summed in the same order)."""
    M, N, K = 96, 16, 40
    case = synth.wgrad_random(M, N, K, [M], seed=8)
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    ref = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    aq, as_ = oracle.mxfp8_quantize_rows(np.ascontiguousarray(case.g_bf16.T), [0, N])
    bq, bs = oracle.mxfp8_quantize_rows(np.ascontiguousarray(case.x_bf16.T), [0, K])
    y = oracle.grouped_fprop_mx(aq, as_, bq, bs, [0, N], [0, K], N)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("counts", [[70, 0, 61, 3], [128, 128], [0, 5]])
def test_dgrad_mx_equals_fp32_dgrad_oracle_on_dequantized_operands(counts):
    """dx = dy W[e(r)] on MXFP8 operands is the fp32 dgrad oracle applied to the
    dequantized values (each exact in fp32), summed in the same order."""
    M, N, K, E = sum(counts), 64, 48, len(counts)
    rng = np.random.default_rng(9)
    dy = _bf16(rng.standard_normal((M, N)))
    W = _bf16(rng.standard_normal((E * N, K)) / 8.0)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    w_off = np.arange(E + 1, dtype=np.int32) * N
    dyq, dys = oracle.mxfp8_quantize_rows(dy, off)
    wtq, wts = oracle.mxfp8_quantize(W, w_off)  # along n per expert: [K, Mw]
    dx = oracle.grouped_dgrad_mx(dyq, dys, wtq, wts, off, w_off, M)
    P, Pw = oracle.padded_starts(off), oracle.padded_starts(w_off)
    dyd = _torch_deq_rows(dyq, dys)
    wd = _torch_deq_rows(wtq, wts)  # [K, Mw]
    dy_rows = np.zeros((M, N), dtype=np.float64)
    for e in range(E):
        dy_rows[off[e]:off[e + 1]] = dyd[P[e]:P[e] + counts[e]]
    W3 = np.stack([wd[:, Pw[e]:Pw[e] + N].T for e in range(E)])  # [E, N, K]
    assert np.array_equal(dy_rows.astype(np.float32).astype(np.float64), dy_rows)
    assert np.array_equal(W3.astype(np.float32).astype(np.float64), W3)
    ref, _ = oracle.grouped_dgrad(dy_rows.astype(np.float32), W3.astype(np.float32), off)
    assert np.array_equal(dx, ref)
    for e, cnt in enumerate(counts):  # and the dense special case per expert
        np.testing.assert_allclose(dx[off[e]:off[e + 1]], dy_rows[off[e]:off[e + 1]] @ W3[e],
                                   rtol=1e-13, atol=1e-12)


def test_mx_dot_matches_numpy():
    rng = np.random.default_rng(3)
    a = _bf16(rng.standard_normal((1, 128)))
    b = _bf16(rng.standard_normal((1, 128)) * 1e3)
    aq, as_ = oracle.mxfp8_quantize_rows(a, [0, 1])
    bq, bs = oracle.mxfp8_quantize_rows(b, [0, 1])
    ref = float((_torch_deq_rows(aq[:1], as_[:1]) @ _torch_deq_rows(bq[:1], bs[:1]).T)[0, 0])
    assert oracle.mx_dot(aq[0], as_[0], bq[0], bs[0]) == pytest.approx(ref, rel=1e-14)
