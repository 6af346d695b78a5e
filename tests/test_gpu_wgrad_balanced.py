"""The load-balanced grouped wgrad (split-K over tokens, dynamic scheduling) against the
oracle: within 8e-3 |ref| + 1e-3 rms(ref), deterministic from call to call, workspace
counters back at zero after every call."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import mgw, synth
from helpers import (bf16_to_f64, check_wgrad_full, dev_bf16, dev_i32, full_case,
                     full_oracle_operands, oracle_quantize_by_expert, wgrad_tol)

pytestmark = pytest.mark.gpu

HEADER = 256  # workspace header bytes (item and CTA counters)


def _operands(case):
    off = dev_i32(case.expert_off)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Mcap = mgw.token_capacity(case.M, case.E)
    if case.M > 0:
        g, x = dev_bf16(case.g_bf16), dev_bf16(case.x_bf16)
    else:
        g = torch.empty((0, case.N), dtype=torch.bfloat16, device="cuda")
        x = torch.empty((0, case.K), dtype=torch.bfloat16, device="cuda")
    gq, gs = mgw.mxfp8_quantize(g, off, Mcap=Mcap, status=status)
    xq, xs = mgw.mxfp8_quantize(x, off, Mcap=Mcap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return off, gq, gs, xq, xs


def _counters_zero(ws):
    """The header and the tile counters (4 bytes per partial slot) are zero."""
    slots = (ws.numel() - HEADER) // (128 * 256 * 4 + 4)
    head = ws[:HEADER + 4 * slots]
    return not bool(head.any())


def _run(case, ws, ops=None):
    off, gq, gs, xq, xs = ops or _operands(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((case.E * case.N, case.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    mgw.grouped_wgrad_mxfp8_balanced(gq, gs, xq, xs, off, case.M, ws, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    return out


def _check_full(case, ws):
    out = bf16_to_f64(_run(case, ws))
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    ref = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    err = np.abs(out - ref)
    tol = wgrad_tol(ref)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{len(bad)} of {ref.size} outside tolerance; first {bad[:5].tolist()} "
                           f"got {out[tuple(bad[0])]} ref {ref[tuple(bad[0])]}")
    counts = np.diff(case.expert_off)
    for e in np.nonzero(counts == 0)[0]:
        assert not out[e * case.N:(e + 1) * case.N].any()
    assert _counters_zero(ws)


@pytest.fixture(scope="module")
def ws():
    return mgw.wgrad_workspace(8, 256, 256)


# With few tiles the target item length is its floor of 8 chunks, so experts longer than
# 8 chunks are split: 16 chunks -> 2 parts, 40 -> 5, 157 -> 16 (the cap).
CASES = [
    ("split_2_and_5", lambda: synth.wgrad_random(7000, 256, 256, [1000, 2000, 0, 4000], seed=41)),
    ("one_tile_split_16", lambda: synth.wgrad_random(20100, 128, 256, [20000, 100], seed=42)),
    ("ragged_tails", lambda: synth.wgrad_random(3333, 128, 512, [1111, 0, 2222], seed=43)),
    ("small_no_split", lambda: synth.wgrad_random(463, 256, 512, [0, 1, 129, 300, 33], seed=44)),
    ("many_experts", lambda: synth.wgrad_random(
        int(np.random.default_rng(45).integers(0, 300, 96).sum()), 128, 256,
        np.random.default_rng(45).integers(0, 300, 96), seed=45)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_balanced_matches_oracle(name, make, ws):
    _check_full(make(), ws)


def test_balanced_is_deterministic(ws):
    case = synth.wgrad_random(9000, 128, 256, [8000, 1000], seed=46)
    ops = _operands(case)
    a = _run(case, ws, ops)
    b = _run(case, ws, ops)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_balanced_header_only_workspace_schedules_without_splits():
    ws_small = torch.zeros(HEADER, dtype=torch.uint8, device="cuda")
    _check_full(synth.wgrad_random(5000, 256, 256, [4000, 1000], seed=47), ws_small)


def test_balanced_small_workspace_limits_splits():
    """Room for 8 partial tiles only: the split factors shrink until they fit."""
    ws8 = torch.zeros(HEADER + 256 + 8 * 128 * 256 * 4, dtype=torch.uint8, device="cuda")
    _check_full(synth.wgrad_random(7000, 256, 256, [1000, 2000, 0, 4000], seed=48), ws8)


def test_balanced_no_tokens_and_bad_offsets(ws):
    case = synth.wgrad_random(0, 128, 256, [0, 0, 0], seed=1)
    out = _run(case, ws)
    assert not bool(out.float().abs().sum())
    assert _counters_zero(ws)
    case = synth.wgrad_random(300, 128, 256, [100, 200], seed=2)
    off, gq, gs, xq, xs = _operands(case)
    bad = dev_i32([0, 100, 250])  # does not end at M
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((2 * 128, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    mgw.grouped_wgrad_mxfp8_balanced(gq, gs, xq, xs, bad, case.M, ws, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mgw.MGW_DEV_BAD_OFFSETS
    assert bool((out == 3.0).all())
    assert _counters_zero(ws)


def test_balanced_matches_oracle_more_items_than_sms(ws):
    """More items than SMs (1024 x 2048 per expert), one long expert split, every output
    element against the oracle."""
    case = synth.wgrad_random(6000, 1024, 2048, [5000, 0, 900, 100], seed=49)
    out = _run(case, ws)
    ops = oracle_quantize_by_expert(case.g_bf16, case.expert_off, mgw.token_capacity(case.M, case.E))
    ops += oracle_quantize_by_expert(case.x_bf16, case.expert_off, mgw.token_capacity(case.M, case.E))
    check_wgrad_full(out, ops, case.expert_off, case.N, case.K)
    assert _counters_zero(ws)


@pytest.mark.slow
def test_balanced_skewed_workload_full_size(ws):
    """The skewed-routing workload (27 of 32 experts empty, one expert of 12544 tokens
    split over token ranges): every output element against the oracle, rms over the whole
    output, one element per output tile from the plain loop oracle."""
    case = full_case("wgrad_skew")
    out = _run(case, ws)
    check_wgrad_full(out, full_oracle_operands("wgrad_skew"), case.expert_off, case.N, case.K)
    assert _counters_zero(ws)


def test_balanced_max_experts(ws):
    """512 experts (the balanced kernel's limit): mostly empty, one long enough to be split."""
    counts = np.zeros(512, dtype=np.int64)
    counts[[3, 100, 400, 511]] = [2000, 33, 129, 1]
    case = synth.wgrad_random(int(counts.sum()), 128, 256, counts, seed=52)
    _check_full(case, ws)
