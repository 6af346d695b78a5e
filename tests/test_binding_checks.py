"""The Python binding's own checks, on CPU.

A stand-in for libmgw.so records which entry points are reached; CPU tensors stand in for
device tensors.  Every binding accepts correctly sized operands, and rejects undersized
buffers, wrong dtypes, mismatched shapes, short expert_off arrays and mixed devices with
MgwError before any call reaches the library (the library itself sees only pointers)."""
import contextlib

import pytest
import torch

from moe_grouped_gemm_wgrad_gb300 import mgw


class FakeLib:
    def __init__(self):
        self.calls = []

    def mgw_mxfp8_token_capacity(self, M, E):
        return (M + 127 * E + 127) // 128 * 128

    def mgw_mxfp8_scale_bytes(self, C, Mcap):
        return C * Mcap // 32

    def mgw_status_string(self, st):
        return b"stand-in"

    def __getattr__(self, name):
        if not name.startswith("mgw_"):
            raise AttributeError(name)

        def call(*args):
            self.calls.append(name)
            return 0
        return call


@pytest.fixture
def lib(monkeypatch):
    fake = FakeLib()
    monkeypatch.setattr(mgw, "load", lambda: fake)
    monkeypatch.setattr(mgw, "_on_cuda", lambda t: True)
    monkeypatch.setattr(mgw, "_device", lambda dev: contextlib.nullcontext())
    monkeypatch.setattr(mgw, "_stream", lambda s: None)
    return fake


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def i32(*vals):
    return torch.tensor(vals, dtype=torch.int32)


def st():
    return torch.zeros(1, dtype=torch.int32)


def _rejects(lib, fn, *args, **kw):
    with pytest.raises(mgw.MgwError):
        fn(*args, **kw)
    assert lib.calls == []


M, E, N, K = 64, 2, 128, 256
MCAP = 384                       # token capacity of 64 tokens over 2 experts
OFF = (0, 32, 64)


def test_quantize(lib):
    q, sc = mgw.mxfp8_quantize(bf(M, N), i32(*OFF), status=st())
    assert q.shape == (N, MCAP) and sc.numel() == N * MCAP // 32
    assert lib.calls == ["mgw_mxfp8_quantize"]
    lib.calls.clear()
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N), i32(*OFF), MCAP, u8(N, MCAP - 128))     # q short
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N), i32(*OFF), MCAP, None, u8(N * MCAP // 32 - 1))
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N), i32(*OFF), MCAP, torch.zeros((N, MCAP), dtype=torch.int8))
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N), i32(0))                                 # no expert
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N, 1), i32(*OFF))                           # not 2-D
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N), i32(*OFF), status=f32(1))              # status dtype
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N), i32(*OFF), status=torch.zeros(0, dtype=torch.int32))
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N)[:, ::2], i32(*OFF))                     # strided


def test_quantize_gather(lib):
    q, _ = mgw.mxfp8_quantize_gather(bf(16, N), torch.zeros(M, dtype=torch.int32), i32(*OFF))
    assert q.shape == (N, MCAP) and lib.calls == ["mgw_mxfp8_quantize_gather"]
    lib.calls.clear()
    _rejects(lib, mgw.mxfp8_quantize_gather, bf(16, N), torch.zeros((M, 1), dtype=torch.int32), i32(*OFF))
    _rejects(lib, mgw.mxfp8_quantize_gather, bf(16, N), torch.zeros(M, dtype=torch.int64), i32(*OFF))


def _wgrad_ops(mcap_x=MCAP):
    return u8(N, MCAP), u8(N * MCAP // 32), u8(K, mcap_x), u8(K * mcap_x // 32)


def test_wgrad(lib):
    gq, gs, xq, xs = _wgrad_ops()
    out = mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, i32(*OFF), M, status=st())
    assert out.shape == (E * N, K) and out.dtype == torch.bfloat16
    mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, i32(*OFF), M, out=bf(E * N * K))   # any shape, enough room
    assert lib.calls == ["mgw_grouped_wgrad_mxfp8"] * 2
    lib.calls.clear()
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq, gs, *_wgrad_ops(MCAP + 128)[2:], i32(*OFF), M)
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq, gs[:-1], xq, xs, i32(*OFF), M)
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq, gs, xq, xs[:-1], i32(*OFF), M)
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq, gs, xq, xs, i32(*OFF), M, out=bf(E * N - 1, K))
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq, gs, xq, xs, i32(*OFF), M, out=f32(E * N, K))
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq.view(-1), gs, xq, xs, i32(*OFF), M)
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq, gs, xq, xs, i32(*OFF).view(1, 3), M)


def test_wgrad_balanced_and_noalloc(lib):
    gq, gs, xq, xs = _wgrad_ops()
    mgw.grouped_wgrad_mxfp8_balanced(gq, gs, xq, xs, i32(*OFF), M, u8(4096))
    mgw.grouped_wgrad_mxfp8_balanced_noalloc(gq, gs, xq, xs, i32(*OFF), M)
    assert lib.calls == ["mgw_grouped_wgrad_mxfp8_balanced", "mgw_grouped_wgrad_mxfp8_balanced_noalloc"]
    lib.calls.clear()
    _rejects(lib, mgw.grouped_wgrad_mxfp8_balanced, gq, gs, xq, xs, i32(*OFF), M, f32(1024))
    _rejects(lib, mgw.grouped_wgrad_mxfp8_balanced_noalloc, gq, gs, xq, xs, i32(*OFF), M, out=bf(1))


def test_dgrad_f32(lib):
    dx = mgw.grouped_dgrad_f32(f32(M, 32), f32(E, 32, K), i32(*OFF), status=st())
    assert dx.shape == (M, K) and dx.dtype == torch.float32
    assert lib.calls == ["mgw_grouped_dgrad_f32"]
    lib.calls.clear()
    _rejects(lib, mgw.grouped_dgrad_f32, f32(M, 32), f32(E, 64, K), i32(*OFF))          # out_f differs
    _rejects(lib, mgw.grouped_dgrad_f32, f32(M, 32), f32(E, 32, K), i32(0, 16, 32, 64))  # E+1 != 3
    _rejects(lib, mgw.grouped_dgrad_f32, f32(M, 32), f32(E, 32, K), i32(*OFF), out=f32(M, K - 1))
    _rejects(lib, mgw.grouped_dgrad_f32, f32(M, 32), f32(E * 32, K), i32(*OFF))         # W not 3-D
    _rejects(lib, mgw.grouped_dgrad_f32, bf(M, 32), f32(E, 32, K), i32(*OFF))


def test_quantize_rows(lib):
    q, sc = mgw.mxfp8_quantize_rows(bf(M, K), i32(*OFF))
    assert q.shape == (MCAP, K) and sc.numel() == K * MCAP // 32
    mgw.mxfp8_quantize_rows(bf(16, K), i32(*OFF), row_index=torch.zeros(M, dtype=torch.int32))
    assert lib.calls == ["mgw_mxfp8_quantize_rows"] * 2
    lib.calls.clear()
    _rejects(lib, mgw.mxfp8_quantize_rows, bf(M, K), i32(*OFF), MCAP, u8(MCAP - 1, K))
    _rejects(lib, mgw.mxfp8_quantize_rows, bf(M, K), i32(*OFF), MCAP, None, u8(K * MCAP // 32 - 1))


def test_fprop(lib):
    Mw = 256                                   # 2 experts x N=128 rows of W, 128-padded
    xq, xs = u8(MCAP, K), u8(K * MCAP // 32)
    wq, ws = u8(Mw, K), u8(K * Mw // 32)
    y = mgw.grouped_fprop_mxfp8(xq, xs, wq, ws, i32(*OFF), M, N, status=st())
    assert y.shape == (M, N) and lib.calls == ["mgw_grouped_fprop_mxfp8"]
    lib.calls.clear()
    _rejects(lib, mgw.grouped_fprop_mxfp8, xq, xs, u8(Mw, K // 2), ws, i32(*OFF), M, N)
    _rejects(lib, mgw.grouped_fprop_mxfp8, xq, xs, wq, ws[:-1], i32(*OFF), M, N)
    _rejects(lib, mgw.grouped_fprop_mxfp8, xq, xs[:-1], wq, ws, i32(*OFF), M, N)
    _rejects(lib, mgw.grouped_fprop_mxfp8, xq, xs, wq, ws, i32(*OFF), M, N, out=bf(M - 1, N))


def test_dgrad_mx(lib):
    Mw = 256
    dyq, dys = u8(MCAP, N), u8(N * MCAP // 32)
    wtq, wts = u8(K, Mw), u8(K * Mw // 32)
    dx = mgw.grouped_dgrad_mxfp8(dyq, dys, wtq, wts, i32(*OFF), M)
    assert dx.shape == (M, K) and lib.calls == ["mgw_grouped_dgrad_mxfp8"]
    lib.calls.clear()
    _rejects(lib, mgw.grouped_dgrad_mxfp8, dyq, dys[:-1], wtq, wts, i32(*OFF), M)
    _rejects(lib, mgw.grouped_dgrad_mxfp8, dyq, dys, wtq, wts[:-1], i32(*OFF), M)
    _rejects(lib, mgw.grouped_dgrad_mxfp8, dyq, dys, wtq, wts, i32(*OFF), M, out=bf(M, K - 1))


def test_mixed_devices_rejected(lib):
    gq, gs, xq, xs = _wgrad_ops()
    other = torch.zeros(xs.shape, dtype=torch.uint8, device="meta")
    _rejects(lib, mgw.grouped_wgrad_mxfp8, gq, gs, xq, other, i32(*OFF), M)
    _rejects(lib, mgw.mxfp8_quantize, bf(M, N), i32(*OFF), status=torch.zeros(1, dtype=torch.int32, device="meta"))
