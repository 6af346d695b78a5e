"""Row-wise MXFP8 quantization (bit-exact) and the grouped MXFP8 forward and data-gradient
GEMMs (within 8e-3 |ref| + 1e-3 rms(ref), ref the fp64 oracle before bf16 rounding) on
the GPU against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import mgw, synth
from helpers import (atoms_to_plain, bf16_to_f64, check_rows_full, dev_bf16, dev_i32, full_case,
                     oracle_quantize_by_expert, wgrad_tol)

pytestmark = pytest.mark.gpu


def _bits(rng, shape, std=1.0):
    return synth.bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _off(counts):
    return synth.offsets_from_counts(np.asarray(counts))


def _quant_rows(bits, off, Mcap=None, rule=0, row_index=None):
    """GPU row-wise quantization -> (q [Mcap, C], plain scales [Mcap, C/32], Mcap, status)."""
    C = bits.shape[1]
    M = len(row_index) if row_index is not None else bits.shape[0]
    E = len(off) - 1
    if Mcap is None:
        Mcap = mgw.token_capacity(M, E)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = dev_bf16(bits) if bits.shape[0] > 0 else torch.empty((0, C), dtype=torch.bfloat16, device="cuda")
    ri = dev_i32(row_index) if row_index is not None else None
    q, sc = mgw.mxfp8_quantize_rows(src, dev_i32(off), Mcap, status=status, scale_rule=rule, row_index=ri)
    torch.cuda.synchronize()
    return q, sc, Mcap, int(status.item())


def _assert_rows_exact(bits, off, Mcap=None, rule=0):
    q, sc, Mcap, st = _quant_rows(bits, off, Mcap, rule)
    assert st == 0
    oq, osc = oracle.mxfp8_quantize_rows(bits, off, Mcap, rule=rule)
    qn = q.cpu().numpy()
    bad = np.argwhere(qn != oq)
    assert bad.size == 0, f"{len(bad)} e4m3 bytes differ, first at {bad[:5].tolist()}"
    plain = atoms_to_plain(sc.cpu().numpy(), Mcap, bits.shape[1])
    bad = np.argwhere(plain != osc)
    assert bad.size == 0, f"{len(bad)} scale bytes differ, first at {bad[:5].tolist()}"
    return q, sc, oq, osc, Mcap


# ------------------------------------------------------------- quantize_rows
@pytest.mark.parametrize("counts,C", [
    ([128, 128], 256),
    ([0, 33, 128, 1, 0, 200], 128),    # empty, ragged, exact, single-row experts
    ([0, 0, 0, 5], 384),               # C % 256 == 128: a half segment
    ([1000], 1536),
    ([31, 32, 33, 127, 129], 128),
])
def test_quantize_rows_matches_oracle(counts, C):
    rng = np.random.default_rng(sum(counts) + C)
    _assert_rows_exact(_bits(rng, (sum(counts), C)), _off(counts))


def test_quantize_rows_ceil448_rule():
    rng = np.random.default_rng(2)
    bits = _bits(rng, (300, 256), std=3.0)
    bits[5, :32] = 0  # an all-zero block of a real row: byte 1 under this rule
    _assert_rows_exact(bits, _off([100, 0, 200]), rule=oracle.SCALE_CEIL_448)


def test_quantize_rows_special_values():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((200, 128)).astype(np.float32)
    v[0, 0:32] = 0.0
    v[1, 0:32] = -0.0
    v[2, 0:32] = np.float32(1e-40)       # subnormal in bf16
    v[3, 0:32] = np.float32(3.0e38)      # near the bf16 maximum
    v[3, 5] = np.float32(-3.3e38)
    v[4, 32:64] = 1.9                    # 1.9 * 2^8 saturates to 448
    v[5, 64:96] = np.float32(2.0 ** -130)
    v[6, 96:128] = rng.choice([-1.0, 1.0], 32) * np.float32(2.0 ** 20)
    _assert_rows_exact(synth.bf16_bits_from_f32(v), _off([150, 50]))


def test_quantize_rows_larger_capacity_is_zero_filled():
    rng = np.random.default_rng(4)
    _assert_rows_exact(_bits(rng, (200, 128)), _off([150, 50]), Mcap=1024)


def test_quantize_rows_no_rows():
    _assert_rows_exact(np.zeros((0, 128), dtype=np.uint16), _off([0, 0, 0]))


def test_quantize_rows_gather_matches_oracle():
    rng = np.random.default_rng(12)
    hidden = _bits(rng, (300, 256))
    counts = [70, 0, 129, 41]
    idx = rng.integers(0, 300, size=sum(counts)).astype(np.int32)  # with repeats
    off = _off(counts)
    q, sc, Mcap, st = _quant_rows(hidden, off, row_index=idx)
    assert st == 0
    oq, osc = oracle.mxfp8_quantize_rows(hidden[idx], off, Mcap)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(atoms_to_plain(sc.cpu().numpy(), Mcap, 256), osc)


def test_quantize_rows_gather_bad_indices_give_zero_rows():
    rng = np.random.default_rng(13)
    hidden = _bits(rng, (64, 128))
    idx = rng.integers(0, 64, size=100).astype(np.int32)
    idx[[3, 50, 99]] = [-1, 64, 1 << 30]
    off = _off([60, 40])
    q, sc, Mcap, st = _quant_rows(hidden, off, row_index=idx)
    assert st & mgw.MGW_DEV_BAD_INDEX
    src = hidden[np.clip(idx, 0, 63)].copy()
    src[[3, 50, 99]] = 0
    oq, osc = oracle.mxfp8_quantize_rows(src, off, Mcap)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(atoms_to_plain(sc.cpu().numpy(), Mcap, 128), osc)


# ------------------------------------------------------------ the two GEMMs
def _fprop_case(counts, N, K, seed):
    rng = np.random.default_rng(seed)
    E = len(counts)
    x = _bits(rng, (sum(counts), K))
    W = _bits(rng, (E * N, K), std=K ** -0.5)
    return x, W, _off(counts), synth.offsets_from_counts(np.full(E, N))


def _run_fprop(x, W, off, w_off, N):
    M = x.shape[0]
    xq, xs, Mcap, st = _quant_rows(x, off)
    wq, ws, Mw, st2 = _quant_rows(W, w_off)
    assert st == 0 and st2 == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mgw.grouped_fprop_mxfp8(xq, xs, wq, ws, dev_i32(off), M, N, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y, (xq, xs, Mcap), (wq, ws, Mw)


@pytest.mark.parametrize("counts,N,K", [
    ([128, 128], 256, 256),
    ([0, 33, 128, 1, 0, 200], 512, 128),
    ([300], 256, 384),
    ([31, 97, 129, 0], 256, 1536),
])
def test_fprop_matches_oracle(counts, N, K):
    x, W, off, w_off = _fprop_case(counts, N, K, seed=sum(counts) + N + K)
    y, _, _ = _run_fprop(x, W, off, w_off, N)
    xq, xs = oracle.mxfp8_quantize_rows(x, off)
    wq, ws = oracle.mxfp8_quantize_rows(W, w_off)
    ref = oracle.grouped_fprop_mx(xq, xs, wq, ws, off, w_off, x.shape[0])
    got = bf16_to_f64(y)
    err = np.abs(got - ref)
    tol = wgrad_tol(ref)
    assert (err <= tol).all(), f"max excess {np.max(err - tol)} at {np.unravel_index(np.argmax(err - tol), err.shape)}"


def _dgrad_case(counts, N, K, seed):
    rng = np.random.default_rng(seed)
    E = len(counts)
    dy = _bits(rng, (sum(counts), N))
    W = _bits(rng, (E * N, K), std=N ** -0.5)  # W [E, N, K] stacked
    return dy, W, _off(counts), synth.offsets_from_counts(np.full(E, N))


def _run_dgrad_mx(dy, W, off, w_off):
    M = dy.shape[0]
    dyq, dys, Mcap, st = _quant_rows(dy, off)
    assert st == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wtq, wts = mgw.mxfp8_quantize(dev_bf16(W), dev_i32(w_off), status=status)
    dx = mgw.grouped_dgrad_mxfp8(dyq, dys, wtq, wts, dev_i32(off), M, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dx, (dyq, dys, Mcap), (wtq, wts)


@pytest.mark.parametrize("counts,N,K", [
    ([128, 128], 128, 256),
    ([70, 0, 61, 3], 256, 512),
    ([0, 33, 128, 1, 0, 200], 384, 256),
])
def test_dgrad_mx_matches_oracle(counts, N, K):
    dy, W, off, w_off = _dgrad_case(counts, N, K, seed=sum(counts) + N + K + 1)
    dx, _, (wtq, wts) = _run_dgrad_mx(dy, W, off, w_off)
    dyq, dys = oracle.mxfp8_quantize_rows(dy, off)
    owtq, owts = oracle.mxfp8_quantize(W, w_off)
    Mw = owtq.shape[1]
    assert np.array_equal(wtq.cpu().numpy(), owtq)
    assert np.array_equal(atoms_to_plain(wts.cpu().numpy(), K, Mw), owts)
    ref = oracle.grouped_dgrad_mx(dyq, dys, owtq, owts, off, w_off, dy.shape[0])
    got = bf16_to_f64(dx)
    err = np.abs(got - ref)
    tol = wgrad_tol(ref)
    assert (err <= tol).all(), f"max excess {np.max(err - tol)}"


def test_fprop_more_items_than_sms():
    """~270 items over the SMs: every CTA takes several; every output element checked."""
    rng = np.random.default_rng(31)
    counts = synth.multinomial_counts(rng, 8192, 8)
    N, K = 1024, 256
    x, W, off, w_off = _fprop_case(list(counts), N, K, seed=32)
    y, _, _ = _run_fprop(x, W, off, w_off, N)
    xq, xs = oracle.mxfp8_quantize_rows(x, off)
    wq, ws = oracle.mxfp8_quantize_rows(W, w_off)
    check_rows_full(y, oracle.grouped_fprop_mx_by_expert(xq, xs, wq, ws, off, w_off), x.shape[0], N)


def test_fprop_no_rows_and_bad_offsets():
    rng = np.random.default_rng(3)
    W = _bits(rng, (2 * 256, 128))
    w_off = _off([256, 256])
    wq, ws, Mw, _ = _quant_rows(W, w_off)
    Mcap = mgw.token_capacity(0, 2)
    xq = torch.zeros((Mcap, 128), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((mgw.scale_bytes(128, Mcap),), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    mgw.grouped_fprop_mxfp8(xq, xs, wq, ws, dev_i32([0, 0, 0]), 0, 256, out=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # offsets that do not end at M: reported, output untouched
    M = 100
    Mcap = mgw.token_capacity(M, 2)
    xq = torch.zeros((Mcap, 128), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((mgw.scale_bytes(128, Mcap),), dtype=torch.uint8, device="cuda")
    y = torch.full((M, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    mgw.grouped_fprop_mxfp8(xq, xs, wq, ws, dev_i32([0, 60, 90]), M, 256, out=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mgw.MGW_DEV_BAD_OFFSETS
    assert bool((y == 7.0).all())


@pytest.mark.slow
def test_moe_ffn_pair_forward_and_mx_dgrad_full_size():
    """The MoE FFN pair at full size (65536 routed rows of 8192 tokens over 64 experts,
    hidden 4096, ffn 1536): forward y = x W[e]^T with x gathered from the hidden states,
    and dx = dy W[e], both in MXFP8.  Every quantized operand is compared bit for bit with
    the oracle's, and every output element with the oracle's per-expert product (rms over
    the whole output)."""
    wg, dg = full_case("moe_ffn_pair"), full_case("moe_ffn_pair.dgrad")
    off = wg.expert_off
    E, N, K = wg.E, wg.N, wg.K              # N = ffn 1536, K = hidden 4096
    M = wg.M
    Wb = synth.bf16_bits_from_f32(dg.W.reshape(E * N, K))
    w_off = synth.offsets_from_counts(np.full(E, N))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_off = dev_i32(off)
    Mcap = mgw.token_capacity(M, E)
    xq, xs = mgw.mxfp8_quantize_rows(dev_bf16(wg.meta["hidden_bf16"]), d_off, Mcap, status=status,
                                     row_index=dev_i32(wg.meta["token_of_row"]))
    Wd = dev_bf16(Wb)
    wq, ws = mgw.mxfp8_quantize_rows(Wd, dev_i32(w_off), status=status)
    y = mgw.grouped_fprop_mxfp8(xq, xs, wq, ws, d_off, M, N, status=status)
    dyq, dys = mgw.mxfp8_quantize_rows(dev_bf16(wg.g_bf16), d_off, Mcap, status=status)
    wtq, wts = mgw.mxfp8_quantize(Wd, dev_i32(w_off), status=status)
    dx = mgw.grouped_dgrad_mxfp8(dyq, dys, wtq, wts, d_off, M, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    del Wd
    Mw, Mw2 = wq.shape[0], wtq.shape[1]
    oxq, oxs = oracle_quantize_by_expert(wg.x_bf16, off, Mcap, rows=True)
    owq, ows = oracle_quantize_by_expert(Wb, w_off, Mw, rows=True)
    assert np.array_equal(xq.cpu().numpy(), oxq) and np.array_equal(wq.cpu().numpy(), owq)
    assert np.array_equal(atoms_to_plain(xs.cpu().numpy(), Mcap, K), oxs)
    assert np.array_equal(atoms_to_plain(ws.cpu().numpy(), Mw, K), ows)
    del xq, wq
    check_rows_full(y, oracle.grouped_fprop_mx_by_expert(oxq, oxs, owq, ows, off, w_off), M, N)
    del oxq, owq
    odq, ods = oracle_quantize_by_expert(wg.g_bf16, off, Mcap, rows=True)
    owtq, owts = oracle_quantize_by_expert(Wb, w_off, Mw2)
    assert np.array_equal(dyq.cpu().numpy(), odq) and np.array_equal(wtq.cpu().numpy(), owtq)
    assert np.array_equal(atoms_to_plain(wts.cpu().numpy(), K, Mw2), owts)
    check_rows_full(dx, oracle.grouped_dgrad_mx_by_expert(odq, ods, owtq, owts, off, w_off), M, K)


def test_forward_and_mx_dgrad_max_experts():
    """1024 experts (the library's limit), most with no rows, a few ragged: parity of the
    row-wise quantizer and both GEMMs on every output element."""
    rng = np.random.default_rng(91)
    counts = np.zeros(1024, dtype=np.int64)
    counts[[0, 5, 511, 1023]] = [40, 1, 130, 7]
    N, K = 256, 256
    x, W, off, w_off = _fprop_case(list(counts), N, K, seed=92)
    _assert_rows_exact(x, off)
    y, _, _ = _run_fprop(x, W, off, w_off, N)
    xq, xs = oracle.mxfp8_quantize_rows(x, off)
    wq, ws = oracle.mxfp8_quantize_rows(W, w_off)
    ref = oracle.grouped_fprop_mx(xq, xs, wq, ws, off, w_off, x.shape[0])
    assert (np.abs(bf16_to_f64(y) - ref) <= wgrad_tol(ref)).all()
    dy, W2, off2, w_off2 = _dgrad_case(list(counts), 128, 256, seed=93)
    dx, _, _ = _run_dgrad_mx(dy, W2, off2, w_off2)
    dyq, dys = oracle.mxfp8_quantize_rows(dy, off2)
    wtq, wts = oracle.mxfp8_quantize(W2, w_off2)
    ref2 = oracle.grouped_dgrad_mx(dyq, dys, wtq, wts, off2, w_off2, dy.shape[0])
    assert (np.abs(bf16_to_f64(dx) - ref2) <= wgrad_tol(ref2)).all()
