"""Grouped fp32 dgrad (3xTF32) on the GPU against the fp64 oracle.

Tolerance (from the workload definition): |gpu - ref| <= 1e-5 * sum_n |dy||W|.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import mgw, synth
from helpers import dev_i32, full_case, oracle_dgrad_threads

pytestmark = pytest.mark.gpu


def _gpu_dgrad(case):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dx = torch.full((case.rows, case.in_f), float("nan"), dtype=torch.float32, device="cuda")
    dy = torch.from_numpy(case.dy).cuda()
    mgw.grouped_dgrad_f32(dy, torch.from_numpy(case.W).cuda(), dev_i32(case.expert_off), out=dx,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    return dx


CASES = [
    ("mixed", lambda: synth.dgrad_random(300, 64, 256, [0, 1, 130, 0, 169], seed=31)),
    ("single_expert", lambda: synth.dgrad_random(257, 32, 512, [257], seed=32)),
    ("tile_edges", lambda: synth.dgrad_random(513, 96, 256, [1, 127, 128, 129, 31, 0, 97], seed=33)),
    ("many_experts", lambda: synth.dgrad_random(
        int(np.random.default_rng(34).integers(0, 50, 40).sum()), 128, 256,
        np.random.default_rng(34).integers(0, 50, 40), seed=34)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_dgrad_matches_oracle(name, make):
    case = make()
    dx = _gpu_dgrad(case).cpu().numpy().astype(np.float64)
    ref, bound = oracle.grouped_dgrad(case.dy, case.W, case.expert_off)
    bad = np.argwhere(~(np.abs(dx - ref) <= 1e-5 * bound))
    assert bad.size == 0, (len(bad), bad[:5].tolist(), dx[tuple(bad[0])], ref[tuple(bad[0])])


def test_dgrad_no_rows():
    case = synth.dgrad_random(0, 32, 256, [0, 0], seed=1)
    dx = _gpu_dgrad(case)
    assert dx.numel() == 0


def _check_by_expert(case, dx):
    """Every row of dx against the oracle's per-expert fp64 product, within 1e-5 times
    sum_n |dy||W| of the element."""
    worst, where = 0.0, None
    rows = 0
    for e, r0, r1, ref, bound in oracle.grouped_dgrad_by_expert(case.dy, case.W, case.expert_off):
        got = dx[r0:r1].cpu().numpy().astype(np.float64)
        ratio = np.abs(got - ref) / bound
        assert np.isfinite(ratio).all(), f"expert {e}: non-finite output"
        i = int(np.argmax(ratio))
        if ratio.flat[i] > worst:
            worst, where = float(ratio.flat[i]), (e, r0 + i // ref.shape[1], i % ref.shape[1])
        rows += r1 - r0
    assert rows == case.rows
    assert worst <= 1e-5, f"worst |gpu - ref| / sum|dy||W| = {worst} at (expert, row, col) {where}"


def test_dgrad_4096_full():
    """4096 rows split 8 ways by a multinomial draw (no boundary on a tile edge): every
    output element against the plain loop oracle."""
    case = synth.dgrad_4096()
    dx = _gpu_dgrad(case).cpu().numpy().astype(np.float64)
    ref, bound = oracle_dgrad_threads(case.dy, case.W, case.expert_off)
    bad = np.argwhere(~(np.abs(dx - ref) <= 1e-5 * bound))
    assert bad.size == 0, (len(bad), bad[:5].tolist())


@pytest.mark.slow
def test_dgrad_moe_ffn_pair_full():
    """The MoE FFN pair's data gradient (65536 routed rows, 1536 -> 4096, 64 experts):
    every output element against the oracle's per-expert fp64 product."""
    case = full_case("moe_ffn_pair.dgrad")
    _check_by_expert(case, _gpu_dgrad(case))


def test_dgrad_bad_offsets_reported_and_output_untouched():
    case = synth.dgrad_random(64, 32, 256, [32, 32], seed=1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dx = torch.full((64, 256), 7.0, dtype=torch.float32, device="cuda")
    mgw.grouped_dgrad_f32(torch.from_numpy(case.dy).cuda(), torch.from_numpy(case.W).cuda(),
                          dev_i32([0, 40, 30]), out=dx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mgw.MGW_DEV_BAD_OFFSETS
    assert bool((dx == 7.0).all())


def test_dgrad_max_experts():
    rng = np.random.default_rng(46)
    counts = np.where(rng.random(1024) < 0.2, rng.integers(1, 30, 1024), 0)
    case = synth.dgrad_random(int(counts.sum()), 32, 256, counts, seed=46)
    dx = _gpu_dgrad(case).cpu().numpy().astype(np.float64)
    ref, bound = oracle.grouped_dgrad(case.dy, case.W, case.expert_off)
    assert np.all(np.abs(dx - ref) <= 1e-5 * bound)


def test_dgrad_wide_pair_tiles_ragged():
    """8192 rows, 64 -> 4096 features, 8 ragged experts (one empty, one of 3 rows): enough
    work for the 256-column pair tiles; every element against the loop oracle."""
    counts = [3, 2000, 0, 1500, 777, 1, 2400, 1511]
    case = synth.dgrad_random(sum(counts), 64, 4096, counts, seed=35)
    dx = _gpu_dgrad(case).cpu().numpy().astype(np.float64)
    ref, bound = oracle_dgrad_threads(case.dy, case.W, case.expert_off)
    bad = np.argwhere(~(np.abs(dx - ref) <= 1e-5 * bound))
    assert bad.size == 0, (len(bad), bad[:5].tolist())


@pytest.mark.parametrize("counts,out_f,in_f", [
    ([0, 1, 300, 0, 2, 511], 32, 512),                       # single-SM kernel, one 32-wide chunk
    ([0, 1, 3000, 0, 2, 2500, 1, 0], 32, 4096),              # CTA pairs, one 32-wide chunk
    ([1, 255, 256, 257, 0, 513, 1023, 1], 64, 8192),         # CTA pairs, tile-edge counts
], ids=["single_sm_one_chunk", "pairs_one_chunk", "pairs_tile_edges"])
def test_dgrad_edge_shapes(counts, out_f, in_f):
    """Shortest reduction (one raw chunk: two 16-wide operand stages), one-row and empty
    experts at both ends, counts one off the 128- and 256-row tile edges; on both kernels
    (the pair kernel when there are at least four rounds of 256-row pair tiles)."""
    case = synth.dgrad_random(sum(counts), out_f, in_f, counts, seed=38)
    dx = _gpu_dgrad(case).cpu().numpy().astype(np.float64)
    ref, bound = oracle_dgrad_threads(case.dy, case.W, case.expert_off)
    bad = np.argwhere(~(np.abs(dx - ref) <= 1e-5 * bound))
    assert bad.size == 0, (len(bad), bad[:5].tolist())


@pytest.mark.parametrize("counts,out_f,in_f", [
    ([100, 0, 156], 64, 256),                      # single-SM kernel
    ([0, 1, 3000, 0, 2, 2500, 1, 0], 32, 4096),    # CTA pairs
], ids=["single_sm", "cta_pairs"])
def test_dgrad_device_time_limit_reports_and_context_survives(monkeypatch, counts, out_f, in_f):
    """A raw stage that never fills makes the dgrad kernel's bounded waits run out: the call
    reports MGW_DEV_TIMEOUT in the status word instead of hanging, and the context stays
    usable.  The stage is dropped by the test build of the library (libmgw_testhooks.so,
    MGW_TEST_DROP_LOAD=1); libmgw.so has no such switch."""
    from moe_grouped_gemm_wgrad_gb300 import build

    hooks = mgw.bind(ctypes.CDLL(build.LIB_TESTHOOKS))
    case = synth.dgrad_random(sum(counts), out_f, in_f, counts, seed=39)
    dy = torch.from_numpy(case.dy).cuda()
    W = torch.from_numpy(case.W).cuda()
    off = dev_i32(case.expert_off)
    dx = torch.zeros((case.rows, case.in_f), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    monkeypatch.setenv("MGW_TEST_DROP_LOAD", "1")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = hooks.mgw_grouped_dgrad_f32(p(dy), p(W), p(off), case.E, case.rows, case.out_f, case.in_f,
                                     p(dx), p(status),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mgw.MGW_OK
    torch.cuda.synchronize()
    assert int(status.item()) & mgw.MGW_DEV_TIMEOUT
    # the product library ignores the variable, and the next call is correct
    got = _gpu_dgrad(case).cpu().numpy().astype(np.float64)
    ref, bound = oracle_dgrad_threads(case.dy, case.W, case.expert_off)
    assert (np.abs(got - ref) <= 1e-5 * bound).all()
