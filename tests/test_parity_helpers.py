"""The full-size parity checkers on the CPU: an output rounded from the oracle's own
result passes, and planted mistakes fail -- one element off by more than the tolerance,
a non-zero row of an expert without tokens, a non-finite element, a row of the wrong
expert.  The GPU parity tests rely on these checkers at the workloads' full sizes."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import synth
from helpers import check_rows_full, check_wgrad_full, oracle_quantize_by_expert


def _wgrad_case():
    counts = [0, 300, 129, 0, 31]
    case = synth.wgrad_random(sum(counts), 256, 512, counts, seed=7, outlier_frac=0.01)
    Mcap = oracle.token_capacity(case.M, case.E)
    ops = oracle_quantize_by_expert(case.g_bf16, case.expert_off, Mcap)
    ops += oracle_quantize_by_expert(case.x_bf16, case.expert_off, Mcap)
    ref = oracle.grouped_wgrad(*ops, case.expert_off)
    return case, ops, ref


def test_quantize_by_expert_equals_one_call():
    counts = [0, 300, 129, 0, 31]
    case = synth.wgrad_random(sum(counts), 256, 128, counts, seed=8)
    Mcap = oracle.token_capacity(case.M, case.E)
    q, sc = oracle.mxfp8_quantize(case.g_bf16, case.expert_off, Mcap)
    q2, sc2 = oracle_quantize_by_expert(case.g_bf16, case.expert_off, Mcap)
    assert np.array_equal(q, q2) and np.array_equal(sc, sc2)
    q, sc = oracle.mxfp8_quantize_rows(case.g_bf16, case.expert_off, Mcap)
    q2, sc2 = oracle_quantize_by_expert(case.g_bf16, case.expert_off, Mcap, rows=True)
    assert np.array_equal(q, q2) and np.array_equal(sc, sc2)


def test_wgrad_checker_passes_rounded_oracle_and_catches_planted_mistakes():
    case, ops, ref = _wgrad_case()
    good = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16)
    check_wgrad_full(good, ops, case.expert_off, case.N, case.K)
    N = case.N
    bad = good.clone()
    bad[1 * N + 17, 300] = float(ref[N + 17, 300]) * 1.05 + 1.0   # one element far off
    with pytest.raises(AssertionError):
        check_wgrad_full(bad, ops, case.expert_off, case.N, case.K)
    bad = good.clone()
    bad[3 * N + 5, 0] = 2.0 ** -20                                 # an empty expert's row
    with pytest.raises(AssertionError):
        check_wgrad_full(bad, ops, case.expert_off, case.N, case.K)
    bad = good.clone()
    bad[4 * N, 3] = float("nan")
    with pytest.raises(AssertionError):
        check_wgrad_full(bad, ops, case.expert_off, case.N, case.K)
    bad = good.clone()
    bad[1 * N:2 * N] = good[2 * N:3 * N]                           # another expert's rows
    with pytest.raises(AssertionError):
        check_wgrad_full(bad, ops, case.expert_off, case.N, case.K)


def test_rows_checker_passes_rounded_oracle_and_catches_planted_mistakes():
    counts = [70, 0, 61, 3]
    rng = np.random.default_rng(9)
    N, K = 256, 128
    x = synth.bf16_bits_from_f32(rng.standard_normal((sum(counts), K)).astype(np.float32))
    W = synth.bf16_bits_from_f32((rng.standard_normal((4 * N, K)) / 16).astype(np.float32))
    off = synth.offsets_from_counts(np.asarray(counts))
    w_off = synth.offsets_from_counts(np.full(4, N))
    xq, xs = oracle.mxfp8_quantize_rows(x, off)
    wq, ws = oracle.mxfp8_quantize_rows(W, w_off)
    ref = oracle.grouped_fprop_mx(xq, xs, wq, ws, off, w_off, x.shape[0])
    good = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16)
    blocks = lambda: oracle.grouped_fprop_mx_by_expert(xq, xs, wq, ws, off, w_off)  # noqa: E731
    check_rows_full(good, blocks(), x.shape[0], N)
    bad = good.clone()
    bad[80, 7] = float(ref[80, 7]) * 1.1 + 1.0
    with pytest.raises(AssertionError):
        check_rows_full(bad, blocks(), x.shape[0], N)


def test_dgrad_threads_equals_one_call():
    counts = [0, 300, 129, 0, 31]
    case = synth.dgrad_random(sum(counts), 64, 256, counts, seed=10)
    from helpers import oracle_dgrad_threads

    d1, b1 = oracle.grouped_dgrad(case.dy, case.W, case.expert_off)
    d2, b2 = oracle_dgrad_threads(case.dy, case.W, case.expert_off)
    assert np.array_equal(d1, d2) and np.array_equal(b1, b2)
