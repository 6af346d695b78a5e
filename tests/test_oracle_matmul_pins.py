"""Pins of the oracle's full-size references (per-expert matrix products of exactly decoded
operands) against its plain loop versions, which are pinned on their own: on ragged,
empty-expert and single-token cases the two differ only by fp64 summation order.  Also
pins the decode helpers against torch's float8_e4m3fn decoder."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import synth


def _close(a, b, scale):
    """Equal up to fp64 summation order: |a - b| <= 1e-12 * scale."""
    assert a.shape == b.shape
    assert np.all(np.abs(a - b) <= 1e-12 * scale), np.max(np.abs(a - b))


def test_decode_helpers_match_torch_decoder():
    rng = np.random.default_rng(5)
    C, Mcap = 64, 256
    q = rng.integers(0, 256, (C, Mcap), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0  # no NaN codes (never produced by the quantizer)
    sc = rng.integers(100, 150, (C, Mcap // 32), dtype=np.uint8)
    ref = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref *= np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=1)
    assert np.array_equal(oracle.dequantize_token_axis(q, sc, 128, 100), ref[:, 128:228])
    qr = np.ascontiguousarray(q[:, :64])        # [64 rows, 64 columns]
    scr = np.ascontiguousarray(sc[:, :2])       # [64 rows, 2 blocks]
    refr = torch.from_numpy(qr).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    refr *= np.repeat(np.ldexp(1.0, scr.astype(np.int64) - 127), 32, axis=1)
    assert np.array_equal(oracle.dequantize_rows(qr, scr, 7, 20), refr[7:27])


@pytest.mark.parametrize("counts,N,K", [
    ([0, 1, 129, 300, 33], 256, 256),   # empty first, single token, ragged
    ([31, 0, 64, 0], 128, 256),          # empty in the middle and last
    ([200], 128, 128),
])
def test_wgrad_by_expert_equals_loop_oracle(counts, N, K):
    case = synth.wgrad_random(sum(counts), N, K, counts, seed=sum(counts) + 3, outlier_frac=0.01)
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    ref = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    seen = []
    for e, blk in oracle.grouped_wgrad_by_expert(gq, gs, xq, xs, case.expert_off):
        seen.append(e)
        part = ref[e * N:(e + 1) * N]
        if blk is None:
            assert counts[e] == 0 and not part.any()
        else:
            _close(blk, part, np.max(np.abs(part)) * counts[e] + 1e-300)
    assert seen == list(range(len(counts)))


@pytest.mark.parametrize("counts", [[0, 70, 61, 0], [257], [1, 127, 128, 129, 31, 0, 97]])
def test_dgrad_by_expert_equals_loop_oracle(counts):
    case = synth.dgrad_random(sum(counts), 64, 256, counts, seed=len(counts) + 11)
    ref, bound = oracle.grouped_dgrad(case.dy, case.W, case.expert_off)
    covered = np.zeros(case.rows, dtype=bool)
    for e, r0, r1, dx, bd in oracle.grouped_dgrad_by_expert(case.dy, case.W, case.expert_off):
        assert r1 - r0 == counts[e]
        _close(dx, ref[r0:r1], bound[r0:r1])
        _close(bd, bound[r0:r1], bound[r0:r1])
        covered[r0:r1] = True
    assert covered.all()


def _mx_case(counts, N, K, seed):
    rng = np.random.default_rng(seed)
    E = len(counts)
    x = synth.bf16_bits_from_f32(rng.standard_normal((sum(counts), K)).astype(np.float32))
    W = synth.bf16_bits_from_f32((rng.standard_normal((E * N, K)) / 16).astype(np.float32))
    return x, W, synth.offsets_from_counts(np.asarray(counts)), synth.offsets_from_counts(np.full(E, N))


@pytest.mark.parametrize("counts", [[70, 0, 61, 3], [0, 33, 128, 1, 0, 200]])
def test_fprop_mx_by_expert_equals_loop_oracle(counts):
    N, K = 256, 128
    x, W, off, w_off = _mx_case(counts, N, K, seed=sum(counts))
    xq, xs = oracle.mxfp8_quantize_rows(x, off)
    wq, ws = oracle.mxfp8_quantize_rows(W, w_off)
    ref = oracle.grouped_fprop_mx(xq, xs, wq, ws, off, w_off, x.shape[0])
    rows = 0
    for e, r0, r1, y in oracle.grouped_fprop_mx_by_expert(xq, xs, wq, ws, off, w_off):
        _close(y, ref[r0:r1], np.max(np.abs(ref)) * K)
        rows += r1 - r0
    assert rows == x.shape[0]


@pytest.mark.parametrize("counts", [[70, 0, 61, 3], [0, 33, 128, 1, 0, 200]])
def test_dgrad_mx_by_expert_equals_loop_oracle(counts):
    N, K = 128, 256
    rng = np.random.default_rng(sum(counts) + 1)
    E = len(counts)
    dy = synth.bf16_bits_from_f32(rng.standard_normal((sum(counts), N)).astype(np.float32))
    W = synth.bf16_bits_from_f32((rng.standard_normal((E * N, K)) / 16).astype(np.float32))
    off = synth.offsets_from_counts(np.asarray(counts))
    w_off = synth.offsets_from_counts(np.full(E, N))
    dyq, dys = oracle.mxfp8_quantize_rows(dy, off)
    wtq, wts = oracle.mxfp8_quantize(W, w_off)
    ref = oracle.grouped_dgrad_mx(dyq, dys, wtq, wts, off, w_off, dy.shape[0])
    rows = 0
    for e, r0, r1, dx in oracle.grouped_dgrad_mx_by_expert(dyq, dys, wtq, wts, off, w_off):
        _close(dx, ref[r0:r1], np.max(np.abs(ref)) * N)
        rows += r1 - r0
    assert rows == dy.shape[0]
