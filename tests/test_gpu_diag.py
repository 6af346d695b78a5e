"""The diagnostic library (libmgw_diag.so, include/mgw_diag.h) on the GPU: the same results
as libmgw.so bit for bit, against the oracle; no bounds report on valid calls; and a
work-item timeline with one record per (CTA, work item) of the instrumented kernels."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import mgw, synth
from helpers import bf16_to_f64, dev_bf16, dev_i32, oracle_dgrad_threads, wgrad_tol

pytestmark = pytest.mark.gpu


def _wgrad(case):
    off = dev_i32(case.expert_off)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Mcap = mgw.token_capacity(case.M, case.E)
    gq, gs = mgw.mxfp8_quantize(dev_bf16(case.g_bf16), off, Mcap=Mcap, status=status)
    xq, xs = mgw.mxfp8_quantize(dev_bf16(case.x_bf16), off, Mcap=Mcap, status=status)
    out = torch.full((case.E * case.N, case.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, off, case.M, out=out, status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


def _dgrad(case):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dx = torch.full((case.rows, case.in_f), float("nan"), dtype=torch.float32, device="cuda")
    mgw.grouped_dgrad_f32(torch.from_numpy(case.dy).cuda(), torch.from_numpy(case.W).cuda(),
                          dev_i32(case.expert_off), out=dx, status=status)
    torch.cuda.synchronize()
    return dx, int(status.item())


def _check_timeline(recs, kernel, items_expected, ctas_per_item):
    recs = [r for r in recs if r["kernel"] == kernel]
    assert len(recs) == len(items_expected) * ctas_per_item, (len(recs), len(items_expected))
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    per_item = {}
    for r in recs:
        assert r["t_done_ns"] >= r["t_wait_ns"] > 0, r
        assert r["sm"] < nsm, r
        per_item.setdefault(r["item"], []).append(r["cta"])
    assert sorted(per_item) == sorted(items_expected)
    for it, ctas in per_item.items():
        assert len(ctas) == ctas_per_item, (it, ctas)
        if ctas_per_item == 2:  # the two CTAs of one cluster
            assert sorted(ctas)[0] % 2 == 0 and sorted(ctas)[1] == sorted(ctas)[0] + 1
    # one CTA's epilogue works its items one after the other: each item's wait starts after
    # the previous item's stores were issued
    by_cta = {}
    for r in recs:
        by_cta.setdefault(r["cta"], []).append(r)
    for rs in by_cta.values():
        rs.sort(key=lambda r: r["t_wait_ns"])
        for a, b in zip(rs, rs[1:]):
            assert b["t_wait_ns"] >= a["t_done_ns"], (a, b)


def test_diag_wgrad_pair_same_results_and_timeline():
    case = synth.wgrad_random(463, 256, 512, [0, 1, 129, 300, 33], seed=21)
    ref_out, st = _wgrad(case)
    assert st == 0
    with mgw.diagnostic_library():
        mgw.diag_timeline_reset()
        out, st = _wgrad(case)
        recs = mgw.diag_timeline()
    assert st == 0, st  # no MGW_DEV_BOUNDS on a valid call
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off, None)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off, None)
    ref = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    assert (np.abs(bf16_to_f64(out) - ref) <= wgrad_tol(ref)).all()
    # items of the CTA-pair kernel: (expert in order of the schedule) x (N/256 x K/256 tiles);
    # empty experts' tiles are written by the zero warp and carry no record
    per_expert = (case.N // 256) * (case.K // 256)
    nonempty = int((np.diff(case.expert_off) > 0).sum())
    recs_w = [r for r in recs if r["kernel"] == "grouped_wgrad_pair_kernel"]
    assert len(recs_w) == 2 * nonempty * per_expert
    _check_timeline(recs, "grouped_wgrad_pair_kernel", sorted({r["item"] for r in recs_w}), 2)


@pytest.mark.parametrize("counts,out_f,in_f,kernel,tile_rows,ctas", [
    ([0, 1, 130, 0, 169], 64, 256, "grouped_dgrad_kernel", 128, 1),
    ([3, 2000, 0, 1500, 777, 1, 2400, 1511], 64, 4096, "grouped_dgrad_pair_kernel", 256, 2),
], ids=["single_sm", "cta_pairs"])
def test_diag_dgrad_same_results_and_timeline(counts, out_f, in_f, kernel, tile_rows, ctas):
    case = synth.dgrad_random(sum(counts), out_f, in_f, counts, seed=36)
    ref_dx, st = _dgrad(case)
    assert st == 0
    with mgw.diagnostic_library():
        mgw.diag_timeline_reset()
        dx, st = _dgrad(case)
        recs = mgw.diag_timeline()
    assert st == 0, st
    assert torch.equal(dx, ref_dx)
    ref, bound = oracle_dgrad_threads(case.dy, case.W, case.expert_off)
    assert (np.abs(dx.cpu().numpy().astype(np.float64) - ref) <= 1e-5 * bound).all()
    tiles = sum(-(-c // tile_rows) for c in counts) * (in_f // 256)
    _check_timeline(recs, kernel, list(range(tiles)), ctas)


def test_diag_timeline_reset_and_product_switch_back():
    case = synth.dgrad_random(300, 64, 256, [0, 1, 130, 0, 169], seed=37)
    with mgw.diagnostic_library() as lib:
        _dgrad(case)
        assert len(mgw.diag_timeline()) > 0
        mgw.diag_timeline_reset()
        assert mgw.diag_timeline() == []
        assert mgw.load() is lib
    assert mgw.load() is not lib
    assert not hasattr(mgw.load(), "mgw_diag_timeline")
