"""The no-allocation entry point of the load-balanced wgrad, for callers that cannot
allocate device memory (it runs on a workspace the library owns): the same result as the
entry points that take caller memory, within 8e-3 |ref| + 1e-3 rms(ref), on calls made
back to back; the oracle's result; identical from call to call; no device memory taken by
repeated calls.  Collected last, after every other GPU test, and self-contained, so it
also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import mgw, synth
from helpers import bf16_to_f64, check_wgrad_full, dev_bf16, dev_i32, oracle_quantize_by_expert, wgrad_tol

pytestmark = pytest.mark.gpu


def _operands(case):
    off = dev_i32(case.expert_off)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Mcap = mgw.token_capacity(case.M, case.E)
    gq, gs = mgw.mxfp8_quantize(dev_bf16(case.g_bf16), off, Mcap=Mcap, status=status)
    xq, xs = mgw.mxfp8_quantize(dev_bf16(case.x_bf16), off, Mcap=Mcap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return off, gq, gs, xq, xs


def _call(case, ops, out):
    off, gq, gs, xq, xs = ops
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mgw.grouped_wgrad_mxfp8_balanced_noalloc(gq, gs, xq, xs, off, case.M, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    return out


def test_noalloc_matches_oracle_deterministic_and_allocates_nothing():
    # split experts (16 and 32 chunks with a target item length of 8 chunks) and an empty one
    case = synth.wgrad_random(7000, 256, 256, [1000, 2000, 0, 4000], seed=61)
    ops = _operands(case)
    out = torch.empty((case.E * case.N, case.K), dtype=torch.bfloat16, device="cuda")
    first = _call(case, ops, out).clone()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        again = _call(case, ops, out)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    assert torch.cuda.mem_get_info()[0] == free0
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    ref = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    got = bf16_to_f64(first)
    assert (np.abs(got - ref) <= wgrad_tol(ref)).all()
    assert not got[2 * case.N:3 * case.N].any()


def test_noalloc_single_tile_split_many_ways():
    case = synth.wgrad_random(20100, 128, 256, [20000, 100], seed=62)
    ops = _operands(case)
    out = torch.empty((case.E * case.N, case.K), dtype=torch.bfloat16, device="cuda")
    got = bf16_to_f64(_call(case, ops, out))
    gq, gs = oracle.mxfp8_quantize(case.g_bf16, case.expert_off)
    xq, xs = oracle.mxfp8_quantize(case.x_bf16, case.expert_off)
    ref = oracle.grouped_wgrad(gq, gs, xq, xs, case.expert_off)
    assert (np.abs(got - ref) <= wgrad_tol(ref)).all()


def test_noalloc_matches_caller_workspace_entry_points_on_consecutive_calls():
    """Two no-allocation calls in a row against the balanced entry point with a caller
    workspace and the static entry point, on operands with a split expert."""
    case = synth.wgrad_random(7000, 256, 512, [4000, 0, 2900, 100], seed=63)
    off, gq, gs, xq, xs = ops = _operands(case)
    shape = (case.E * case.N, case.K)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = mgw.wgrad_workspace(case.E, case.N, case.K)
    ref_bal = mgw.grouped_wgrad_mxfp8_balanced(gq, gs, xq, xs, off, case.M, ws, status=status)
    ref_static = mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, off, case.M, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rb, rs = bf16_to_f64(ref_bal), bf16_to_f64(ref_static)
    for _ in range(2):
        got = bf16_to_f64(_call(case, ops, torch.empty(shape, dtype=torch.bfloat16, device="cuda")))
        assert (np.abs(got - rb) <= wgrad_tol(rb)).all()
        assert (np.abs(got - rs) <= wgrad_tol(rs)).all()


def test_noalloc_more_than_64_tiles_per_expert_schedules_without_splits():
    """2048 x 2048 per expert is 128 output tiles: splitting any expert would need more than
    the library workspace's 128 partial slots, so no expert is split and the call runs on
    the dynamic schedule alone.  Every output element against the oracle."""
    case = synth.wgrad_random(6200, 2048, 2048, [6000, 0, 200], seed=64)
    ops = _operands(case)
    out = torch.full((case.E * case.N, case.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    _call(case, ops, out)
    Mcap = mgw.token_capacity(case.M, case.E)
    oops = oracle_quantize_by_expert(case.g_bf16, case.expert_off, Mcap)
    oops += oracle_quantize_by_expert(case.x_bf16, case.expert_off, Mcap)
    check_wgrad_full(out, oops, case.expert_off, case.N, case.K)


def test_noalloc_in_a_second_context_and_back():
    """The library looks its workspace up per CUDA context: with a second (non-primary)
    driver context current, a call on buffers of that context uses that context's copy of
    the array, and the next call back in the primary context uses the primary's again.  The
    three results are the same bits."""
    import ctypes

    case = synth.wgrad_random(7000, 256, 256, [1000, 2000, 0, 4000], seed=61)
    ops = _operands(case)
    out = torch.empty((case.E * case.N, case.K), dtype=torch.bfloat16, device="cuda")
    first = _call(case, ops, out).clone()
    host = [t.cpu().contiguous() for t in ops]  # off, gq, gs, xq, xs
    Mcap = mgw.token_capacity(case.M, case.E)
    cu = ctypes.CDLL("libcuda.so.1")
    dev = ctypes.c_int()
    assert cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
    ctx = ctypes.c_void_p()
    assert cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev) == 0  # pushed: now current
    ptrs = []
    try:
        def dalloc(nbytes):
            p = ctypes.c_uint64()
            assert cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)) == 0
            ptrs.append(p)
            return p

        dops = []
        for t in host:
            nbytes = t.numel() * t.element_size()
            p = dalloc(nbytes)
            assert cu.cuMemcpyHtoD_v2(p, ctypes.c_void_p(t.data_ptr()), ctypes.c_size_t(nbytes)) == 0
            dops.append(p)
        d_off, d_gq, d_gs, d_xq, d_xs = dops
        d_out = dalloc(out.numel() * 2)
        d_status = dalloc(4)
        assert cu.cuMemsetD32_v2(d_status, ctypes.c_uint(0), ctypes.c_size_t(1)) == 0
        V = lambda p: ctypes.c_void_p(p.value)  # noqa: E731
        rc = mgw.load().mgw_grouped_wgrad_mxfp8_balanced_noalloc(
            V(d_gq), V(d_gs), V(d_xq), V(d_xs), V(d_off), case.E, case.M, case.N, case.K, Mcap,
            V(d_out), V(d_status), None)
        assert rc == 0, rc
        assert cu.cuCtxSynchronize() == 0
        got = torch.empty((case.E * case.N, case.K), dtype=torch.int16)
        status = ctypes.c_int(-1)
        assert cu.cuMemcpyDtoH_v2(ctypes.c_void_p(got.data_ptr()), d_out, ctypes.c_size_t(got.numel() * 2)) == 0
        assert cu.cuMemcpyDtoH_v2(ctypes.byref(status), d_status, ctypes.c_size_t(4)) == 0
        assert status.value == 0
        assert torch.equal(got, first.view(torch.int16).cpu())
    finally:
        for p in ptrs:
            cu.cuMemFree_v2(p)
        assert cu.cuCtxDestroy_v2(ctx) == 0  # popped: the primary context is current again
    again = _call(case, ops, torch.empty_like(out))
    assert torch.equal(again.view(torch.int16), first.view(torch.int16))
