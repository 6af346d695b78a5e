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
