"""MXFP8 quantization on the GPU against the oracle: bit-exact e4m3 and e8m0 bytes."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_gemm_wgrad_gb300 import mgw, synth
from helpers import atoms_to_plain, dev_bf16, dev_i32, full_case, full_oracle_operands

pytestmark = pytest.mark.gpu


def _run(bits: np.ndarray, off, Mcap=None):
    M, C = bits.shape
    E = len(off) - 1
    if Mcap is None:
        Mcap = mgw.token_capacity(M, E)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = dev_bf16(bits) if M > 0 else torch.empty((0, C), dtype=torch.bfloat16, device="cuda")
    q, sc = mgw.mxfp8_quantize(src, dev_i32(off), Mcap=Mcap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return q.cpu().numpy(), sc.cpu().numpy(), Mcap


def _check(bits, off, Mcap=None):
    q, sc, Mcap = _run(bits, off, Mcap)
    oq, osc = oracle.mxfp8_quantize(bits, off, Mcap)
    C = bits.shape[1]
    bad = np.argwhere(q != oq)
    assert bad.size == 0, f"{len(bad)} e4m3 bytes differ, first at {bad[:5].tolist()}"
    plain = atoms_to_plain(sc, C, Mcap)
    bad = np.argwhere(plain != osc)
    assert bad.size == 0, f"{len(bad)} scale bytes differ, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("counts,C", [
    ([128, 128], 256),                 # the tiny workload's split
    ([0, 33, 128, 1, 0, 200], 128),    # empty, ragged, exact, single-token experts
    ([0, 0, 0, 5], 256),
    ([1000], 384),                     # one expert, several 128-token chunks
    ([31, 32, 33, 127, 129], 128),     # block and chunk boundaries
])
def test_quantize_random_matches_oracle(counts, C):
    case = synth.wgrad_random(sum(counts), C, 128, counts, seed=sum(counts) + C)
    _check(case.g_bf16, case.expert_off)


def test_quantize_no_tokens():
    bits = np.zeros((0, 128), dtype=np.uint16)
    _check(bits, [0, 0, 0])


def test_quantize_larger_capacity_is_zero_filled():
    case = synth.wgrad_random(200, 128, 128, [150, 50], seed=4)
    _check(case.g_bf16, case.expert_off, Mcap=1024)


def test_quantize_special_values():
    """Zeros of both signs, bf16 subnormals, the largest bf16, exact powers of two,
    values that land on e4m3 rounding ties and saturating blocks."""
    rng = np.random.default_rng(7)
    M, C = 256, 128
    v = rng.standard_normal((M, C)).astype(np.float32)
    v[0:32, 0] = 0.0
    v[0:32, 1] = -0.0
    v[0:32, 2] = np.float32(1e-40)       # subnormal in bf16
    v[5, 2] = np.float32(-3e-39)
    v[0:32, 3] = np.float32(3.0e38)      # near the bf16 maximum
    v[7, 3] = np.float32(-3.3e38)
    v[32:64, 4] = 1.0
    v[40, 4] = 1.0625 * 256 / 256        # tie after scaling (scale byte 119 -> x256)
    v[32:64, 5] = 1.9                    # 1.9 * 2^8 saturates to 448
    v[32:64, 6] = np.float32(2.0 ** -130)
    v[64:96, 7] = rng.choice([-1.0, 1.0], 32) * np.float32(2.0 ** 20)
    bits = synth.bf16_bits_from_f32(v)
    _check(bits, [0, 100, 256])


def _assert_equal(q, sc, oq, osc, C, Mcap):
    bad = np.argwhere(q != oq)
    assert bad.size == 0, f"{len(bad)} e4m3 bytes differ, first at {bad[:5].tolist()}"
    bad = np.argwhere(atoms_to_plain(sc, C, Mcap) != osc)
    assert bad.size == 0, f"{len(bad)} scale bytes differ, first at {bad[:5].tolist()}"


@pytest.mark.slow
@pytest.mark.parametrize("name", ["wgrad_8192", "wgrad_skew", "moe_ffn_pair"])
def test_quantize_full_size_workloads(name):
    """Every byte of both operands of the full-size workloads (x of the MoE FFN pair also
    gathered straight from the hidden states by the routing map) against the oracle's
    quantization of the same workload."""
    case = full_case(name)
    gq, gs, xq, xs = full_oracle_operands(name)
    q, sc, Mcap = _run(case.g_bf16, case.expert_off)
    _assert_equal(q, sc, gq, gs, case.N, Mcap)
    q, sc, _ = _run(case.x_bf16, case.expert_off)
    _assert_equal(q, sc, xq, xs, case.K, Mcap)
    if "hidden_bf16" in case.meta:  # x gathered from the hidden states by the routing map
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        q, sc = mgw.mxfp8_quantize_gather(dev_bf16(case.meta["hidden_bf16"]),
                                          dev_i32(case.meta["token_of_row"]),
                                          dev_i32(case.expert_off), Mcap=Mcap, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _assert_equal(q.cpu().numpy(), sc.cpu().numpy(), xq, xs, case.K, Mcap)


def test_quantize_bad_offsets_reported_and_output_untouched():
    case = synth.wgrad_random(64, 128, 128, [32, 32], seed=1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for off in ([0, 40, 30], [1, 32, 64], [0, 32, 63]):
        Mcap = mgw.token_capacity(64, 2)
        q = torch.full((128, Mcap), 0xAB, dtype=torch.uint8, device="cuda")
        sc = torch.full((mgw.scale_bytes(128, Mcap),), 0xCD, dtype=torch.uint8, device="cuda")
        status.zero_()
        mgw.mxfp8_quantize(dev_bf16(case.g_bf16), dev_i32(off), Mcap=Mcap, q=q, scales=sc, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & mgw.MGW_DEV_BAD_OFFSETS
        assert bool((q == 0xAB).all()) and bool((sc == 0xCD).all())


def test_quantize_max_experts():
    rng = np.random.default_rng(45)
    counts = np.where(rng.random(1024) < 0.2, rng.integers(1, 70, 1024), 0)
    case = synth.wgrad_random(int(counts.sum()), 256, 128, counts, seed=45)
    _check(case.g_bf16, case.expert_off)


@pytest.mark.parametrize("counts,C", [([128, 128], 256), ([0, 33, 128, 1, 0, 200], 128),
                                      ([31, 32, 33, 127, 129], 128)])
def test_quantize_ceil448_rule_matches_oracle(counts, C):
    case = synth.wgrad_random(sum(counts), C, 128, counts, seed=sum(counts) + 7, outlier_frac=0.02)
    M, E = sum(counts), len(counts)
    Mcap = mgw.token_capacity(M, E)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, sc = mgw.mxfp8_quantize(dev_bf16(case.g_bf16), dev_i32(case.expert_off), Mcap=Mcap,
                               status=status, scale_rule=mgw.SCALE_CEIL_448)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    oq, osc = oracle.mxfp8_quantize(case.g_bf16, case.expert_off, Mcap, rule=oracle.SCALE_CEIL_448)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(atoms_to_plain(sc.cpu().numpy(), C, Mcap), osc)


def _routed_case(tokens, C, E, top_k, seed):
    token_of_row, counts = synth.moe_routing(seed, tokens, E, top_k)
    rng = np.random.default_rng(seed + 100)
    hidden = synth.bf16_bits_from_f32(synth.normal_f32(rng, (tokens, C)))
    return hidden, token_of_row.astype(np.int32), synth.offsets_from_counts(counts)


@pytest.mark.parametrize("tokens,C,E,top_k", [(300, 256, 8, 2), (1000, 128, 16, 4), (64, 384, 3, 3)])
def test_quantize_gather_matches_oracle_on_routed_rows(tokens, C, E, top_k):
    hidden, rows, off = _routed_case(tokens, C, E, top_k, seed=tokens + C)
    M = rows.size
    Mcap = mgw.token_capacity(M, E)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, sc = mgw.mxfp8_quantize_gather(dev_bf16(hidden), dev_i32(rows), dev_i32(off), Mcap=Mcap,
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    oq, osc = oracle.mxfp8_quantize(np.ascontiguousarray(hidden[rows]), off, Mcap)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(atoms_to_plain(sc.cpu().numpy(), C, Mcap), osc)


def test_quantize_gather_bad_indices_zero_rows_and_status():
    hidden, rows, off = _routed_case(200, 128, 4, 2, seed=5)
    bad = rows.copy()
    bad[[0, 17, 250]] = [-1, 200, 10 ** 6]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M = rows.size
    Mcap = mgw.token_capacity(M, 4)
    q, sc = mgw.mxfp8_quantize_gather(dev_bf16(hidden), dev_i32(bad), dev_i32(off), Mcap=Mcap,
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mgw.MGW_DEV_BAD_INDEX
    src = np.ascontiguousarray(hidden[np.clip(bad, 0, 199)])
    src[[0, 17, 250]] = 0
    oq, osc = oracle.mxfp8_quantize(src, off, Mcap)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(atoms_to_plain(sc.cpu().numpy(), 128, Mcap), osc)


def test_quantize_gather_no_tokens():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hidden = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    q, sc = mgw.mxfp8_quantize_gather(hidden, torch.zeros(0, dtype=torch.int32, device="cuda"),
                                      dev_i32([0, 0, 0]), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and not bool(q.any()) and not bool(sc.any())
