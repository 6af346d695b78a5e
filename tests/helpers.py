"""Shared test helpers: device transfer, the scale-atom index map and tolerances.

The atom index map is written here independently of the library: for feature c
and padded token t of a C-feature operand, the e8m0 byte sits in 512-byte atoms
ordered by 128-token chunk, then 128-feature tile; inside an atom, feature c%128
= r0 + 32*r1 and 32-token block kb = (t%128)//32 sit at 16*r0 + 4*r1 + kb.
"""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def dev_i32(a, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(dev)


def atom_offsets(C: int, Mcap: int) -> np.ndarray:
    """[C, Mcap/32] array: byte offset in the atom buffer of (feature c, block j)."""
    c = np.arange(C, dtype=np.int64)[:, None]
    j = np.arange(Mcap // 32, dtype=np.int64)[None, :]
    t = 32 * j
    return ((t // 128) * (C // 128) + c // 128) * 512 + (c % 32) * 16 + ((c % 128) // 32) * 4 + (t % 128) // 32


def atoms_to_plain(atoms: np.ndarray, C: int, Mcap: int) -> np.ndarray:
    return np.asarray(atoms).reshape(-1)[atom_offsets(C, Mcap)]


def wgrad_tol(ref: np.ndarray, rms: float | None = None) -> np.ndarray:
    """|gpu - ref| <= 8e-3 |ref| + 1e-3 rms(ref)."""
    if rms is None:
        rms = float(np.sqrt(np.mean(np.square(ref)))) if ref.size else 0.0
    return 8e-3 * np.abs(ref) + 1e-3 * rms


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


# ------------------------------------------------------------- full-size parity
WGRAD_REL, WGRAD_ABS = 8e-3, 1e-3   # |gpu - ref| <= 8e-3 |ref| + 1e-3 rms(ref)
DGRAD_BOUND = 1e-5                   # |gpu - ref| <= 1e-5 sum_n |dy||W|


def _threads():
    import os

    return max(1, min(16, os.cpu_count() or 1))


def oracle_quantize_by_expert(bits: np.ndarray, expert_off, Mcap: int, rows: bool = False,
                              rule: int = 0):
    """The oracle's quantizer (token-axis, or row-wise with ``rows``) applied to each
    expert's own rows and assembled at its padded start P[e]: blocks never cross experts, so
    this equals one call over all experts.  Experts run on threads (the C oracle releases
    the GIL)."""
    import concurrent.futures as cf

    import oracle

    off = np.asarray(expert_off, dtype=np.int64)
    P = oracle.padded_starts(off)
    C = bits.shape[1]
    if rows:
        q = np.zeros((Mcap, C), dtype=np.uint8)
        sc = np.zeros((Mcap, C // 32), dtype=np.uint8)
    else:
        q = np.zeros((C, Mcap), dtype=np.uint8)
        sc = np.zeros((C, Mcap // 32), dtype=np.uint8)

    def one(e):
        c = int(off[e + 1] - off[e])
        if c == 0:
            return
        cap = (c + 127) // 128 * 128
        src = np.ascontiguousarray(bits[off[e]:off[e + 1]])
        p = int(P[e])
        if rows:
            qe, se = oracle.mxfp8_quantize_rows(src, [0, c], cap, rule=rule)
            q[p:p + cap] = qe
            sc[p:p + cap] = se
        else:
            qe, se = oracle.mxfp8_quantize(src, [0, c], cap, rule=rule)
            q[:, p:p + cap] = qe
            sc[:, p // 32:(p + cap) // 32] = se

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(len(off) - 1)))
    return q, sc


def check_wgrad_full(out, ops, expert_off, N: int, K: int, seed: int = 0):
    """Every element of a grouped wgrad output (device bf16 [E*N, K]) against the oracle:
    the per-expert matrix-product reference for the whole output, with rms(ref) taken over
    the whole output (experts without tokens count as zeros), exact zeros for experts
    without tokens, and one element of every 128 x 256 output tile of every expert with
    tokens recomputed by the plain loop oracle (which the matrix-product reference must
    also match there).  ``ops`` are the oracle's quantized operands (plain scale layout)."""
    import oracle

    gq, gs, xq, xs = ops
    off = np.asarray(expert_off, dtype=np.int64)
    E = len(off) - 1
    rng = np.random.default_rng(seed)
    sumsq = 0.0
    worst, where = -np.inf, None
    samples = []   # (e, n, k, got, ref from the product)
    for e, ref in oracle.grouped_wgrad_by_expert(gq, gs, xq, xs, off):
        got = out[e * N:(e + 1) * N].float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), f"expert {e}: non-finite output"
        if ref is None:
            assert not got.any(), f"expert {e} has no tokens but non-zero rows"
            continue
        sumsq += float(np.dot(ref.ravel(), ref.ravel()))
        slack = np.abs(got - ref) - WGRAD_REL * np.abs(ref)
        i = int(np.argmax(slack))
        if slack.flat[i] > worst:
            worst, where = float(slack.flat[i]), (e, *np.unravel_index(i, ref.shape))
        ns = (np.arange(N // 128)[:, None] * 128 + rng.integers(0, 128, (N // 128, K // 256))).ravel()
        ks = (np.arange(K // 256)[None, :] * 256 + rng.integers(0, 256, (N // 128, K // 256))).ravel()
        samples += [(e, int(n), int(k), got[n, k], ref[n, k]) for n, k in zip(ns, ks)]
    rms = float(np.sqrt(sumsq / (E * N * K)))
    assert worst <= WGRAD_ABS * rms, (f"worst excess over 8e-3|ref| is {worst} > 1e-3 rms "
                                      f"= {WGRAD_ABS * rms} at (expert, n, k) {where}")
    for e, n, k, got, ref_mm in samples:
        ref = oracle.grouped_wgrad_element(gq, gs, xq, xs, off, e, n, k)
        assert abs(ref - ref_mm) <= 1e-9 * rms, (e, n, k, ref, ref_mm)  # fp64 summation order only
        assert abs(got - ref) <= WGRAD_REL * abs(ref) + WGRAD_ABS * rms, (e, n, k, got, ref)
    return rms


def check_rows_full(out, blocks, rows: int, cols: int):
    """Every element of a row-grouped output (device [rows, cols]) against per-expert
    references ``blocks`` yielding (e, r0, r1, ref), under the wgrad tolerance with rms over
    the whole output."""
    sumsq = 0.0
    worst, where = -np.inf, None
    covered = 0
    for e, r0, r1, ref in blocks:
        got = out[r0:r1].float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), f"expert {e}: non-finite output"
        sumsq += float(np.dot(ref.ravel(), ref.ravel()))
        slack = np.abs(got - ref) - WGRAD_REL * np.abs(ref)
        i = int(np.argmax(slack))
        if slack.flat[i] > worst:
            worst, where = float(slack.flat[i]), (e, r0 + np.unravel_index(i, ref.shape)[0],
                                                  np.unravel_index(i, ref.shape)[1])
        covered += r1 - r0
    assert covered == rows
    rms = float(np.sqrt(sumsq / (rows * cols)))
    assert worst <= WGRAD_ABS * rms, (f"worst excess {worst} > 1e-3 rms = {WGRAD_ABS * rms} "
                                      f"at (expert, row, col) {where}")
    return rms


_CASES = {}


def full_case(name: str):
    """A full-size workload by name (cached per process): wgrad_8192, wgrad_skew,
    moe_ffn_pair (its wgrad case), moe_ffn_pair.dgrad, dgrad_4096."""
    from moe_grouped_gemm_wgrad_gb300 import synth

    if name not in _CASES:
        if name.startswith("moe_ffn_pair"):
            wg, dg = synth.moe_ffn_pair()
            _CASES["moe_ffn_pair"], _CASES["moe_ffn_pair.dgrad"] = wg, dg
        else:
            _CASES[name] = getattr(synth, name)()
    return _CASES[name]


_OPS = {}


def full_oracle_operands(name: str):
    """The oracle's token-axis quantization of a full-size wgrad workload's g and x
    (cached per process): (gq, gs, xq, xs) in the plain scale layout."""
    import oracle

    if name not in _OPS:
        case = full_case(name)
        Mcap = oracle.token_capacity(case.M, case.E)
        gq, gs = oracle_quantize_by_expert(case.g_bf16, case.expert_off, Mcap)
        xq, xs = oracle_quantize_by_expert(case.x_bf16, case.expert_off, Mcap)
        _OPS[name] = (gq, gs, xq, xs)
    return _OPS[name]


def oracle_dgrad_threads(dy: np.ndarray, W: np.ndarray, expert_off):
    """The plain loop dgrad oracle applied to each expert's own rows on threads (the C
    oracle releases the GIL) and assembled: (dx fp64, bound fp64), equal to one call."""
    import concurrent.futures as cf

    import oracle

    off = np.asarray(expert_off, dtype=np.int64)
    rows, in_f = dy.shape[0], W.shape[2]
    dx = np.zeros((rows, in_f))
    bound = np.zeros((rows, in_f))

    def one(e):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            return
        # split long experts into row slices of at most 128 rows to use every thread
        for s0 in range(r0, r1, 128):
            s1 = min(r1, s0 + 128)
            d, b = oracle.grouped_dgrad(dy[s0:s1], W[e:e + 1], [0, s1 - s0])
            dx[s0:s1], bound[s0:s1] = d, b

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(len(off) - 1)))
    return dx, bound
