"""Grouped fp32 dgrad (3xTF32) on the GPU against the fp64 oracle.

Tolerance (from the workload definition): |gpu - ref| <= 1e-5 * sum_n |dy||W|.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import mgw, synth
from helpers import dev_i32

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


def _check_sampled(case, n_samples=2000, seed=0):
    dx = _gpu_dgrad(case)
    rng = np.random.default_rng(seed)
    rs = rng.integers(0, case.rows, n_samples)
    ks = rng.integers(0, case.in_f, n_samples)
    # rows on expert boundaries and their neighbours
    edges = np.clip(np.concatenate([case.expert_off[1:-1] + d for d in (-1, 0, 1)]), 0, case.rows - 1)
    rs[:min(len(edges), 500)] = edges[:500]
    got = dx[torch.as_tensor(rs, device="cuda"), torch.as_tensor(ks, device="cuda")].cpu().numpy()
    for r, k, gv in zip(rs, ks, got):
        ref, bound = oracle.grouped_dgrad_element(case.dy, case.W, case.expert_off, int(r), int(k))
        assert abs(float(gv) - ref) <= 1e-5 * bound, (int(r), int(k), float(gv), ref, bound)
    assert bool(torch.isfinite(dx).all())


def test_dgrad_4096_sampled():
    _check_sampled(synth.dgrad_4096())


@pytest.mark.slow
def test_dgrad_moe_ffn_pair_sampled():
    _check_sampled(synth.moe_ffn_pair()[1], n_samples=1000)


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
