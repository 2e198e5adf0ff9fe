"""Helpers shared by the GPU tests: run the CUDA path, run the oracle, compare.

The pass criterion is elementwise |D_gpu - D_ref| <= 2^-7 (|D_ref| + 1), with
D_ref the CPU oracle's bf16 result.  Integer-valued inputs (every partial sum an
exact integer below 2^24) are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_bf16_gemm_persistent_gb300 import inputs

TOL = 2.0 ** -7


def f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> float:
    g, r = f64(got_bits), f64(ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    err = np.abs(g - r)
    bad = ~(err <= TOL * (np.abs(r) + 1.0))     # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} entries out of tolerance; first at {i}: "
                             f"gpu={g[i]!r} ref={r[i]!r}; max|err|={np.nanmax(err)!r}")
    return float(err.max()) if err.size else 0.0


def assert_bitexact(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> None:
    neq = got_bits != ref_bits
    if neq.any():
        i = tuple(np.argwhere(neq)[0])
        raise AssertionError(f"{what}: {int(neq.sum())} entries differ; first at {i}: "
                             f"gpu={f64(got_bits)[i]!r} ref={f64(ref_bits)[i]!r}")


def ulp_hist(got_bits: np.ndarray, ref64: np.ndarray) -> dict:
    """bf16-ULP distance of D from bf16_rne(float64 result): a diagnostic, not a gate."""
    r = oracle.f64_to_bf16(ref64).astype(np.int32)
    g = np.asarray(got_bits).astype(np.int32)
    # ordered integer view of bf16 patterns (sign-magnitude -> two's complement order)
    def key(x):
        return np.where(x & 0x8000, -(x & 0x7fff), x & 0x7fff)
    d = np.abs(key(g) - key(r))
    vals, counts = np.unique(np.minimum(d, 8), return_counts=True)
    return {int(v): int(c) for v, c in zip(vals, counts)}


def bits(t: torch.Tensor) -> np.ndarray:
    return inputs.to_bits(t)


def int_tensor(shape, seed, lo=-2, hi=2, device="cpu"):
    return inputs.randint_bf16(shape, seed=seed, lo=lo, hi=hi, device=device)
