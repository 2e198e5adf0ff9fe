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


def within_one_ulp_frac(got_bits: np.ndarray, ref64: np.ndarray) -> float:
    h = ulp_hist(got_bits, ref64)
    return sum(v for k, v in h.items() if k <= 1) / max(1, sum(h.values()))


def _gather(t: torch.Tensor, idx: np.ndarray) -> np.ndarray:
    return bits(t[torch.from_numpy(idx).to(t.device)])


def check_pairs(kind: str, D: torch.Tensor, ops: dict, i: np.ndarray, j: np.ndarray, act: str = "none",
                chunk: int = 8192, ulp_gate: float | None = 0.99, what: str = "") -> dict:
    """D at independent entries (i[p], j[p]) against the oracle's per-entry evaluators.

    kind "linear": ops A [M,K], B [N,K], optional bias [N], R [M,N];
    kind "ffn":    ops X, W1, W3;
    kind "dact":   ops dY [M,N'], W [N',K] (entry (m, k) uses column k of W), Z [M,K];
    kind "matmul": ops A [M,K], B [K,N] (entry (m, n) uses column n of B), optional bias, R.
    Operand rows are gathered on the device in chunks, so K may be large.  Checks the
    tolerance on every entry and, when ulp_gate is set, that at least that fraction of
    entries lies within one bf16 ulp of the float64 result.  Returns a small report."""
    got = _gather_pairs(D, i, j)
    P = i.size
    ref = np.empty(P, np.uint16)
    ref64 = np.empty(P, np.float64)
    for s in range(0, P, chunk):
        ii, jj = i[s:s + chunk], j[s:s + chunk]
        if kind == "linear":
            Ar, Br = _gather(ops["A"], ii), _gather(ops["B"], jj)
            bias = ops.get("bias")
            R = ops.get("R")
            bv = bits(bias)[jj] if bias is not None else None
            rv = _gather_pairs(R, ii, jj) if R is not None else None
            ref[s:s + ii.size] = oracle.linear_entries(Ar, Br, bv, rv, act)
            ref64[s:s + ii.size] = oracle.linear_entries(Ar, Br, bv, rv, act, f64=True)
        elif kind == "matmul":  # ops A [M,K], B [K,N] (entry (m, n) uses column n of B), bias, R
            Ar = _gather(ops["A"], ii)
            Bc = bits(ops["B"][:, torch.from_numpy(jj).to(ops["B"].device)].t().contiguous())
            bias = ops.get("bias")
            R = ops.get("R")
            bv = bits(bias)[jj] if bias is not None else None
            rv = _gather_pairs(R, ii, jj) if R is not None else None
            ref[s:s + ii.size] = oracle.linear_entries(Ar, Bc, bv, rv, act)
            ref64[s:s + ii.size] = oracle.linear_entries(Ar, Bc, bv, rv, act, f64=True)
        elif kind == "ffn":
            Xr, W1r, W3r = _gather(ops["X"], ii), _gather(ops["W1"], jj), _gather(ops["W3"], jj)
            ref[s:s + ii.size] = oracle.ffn_entries(Xr, W1r, W3r)
            ref64[s:s + ii.size] = oracle.ffn_entries(Xr, W1r, W3r, f64=True)
        elif kind == "dact":
            Yr = _gather(ops["dY"], ii)
            Wc = bits(ops["W"][:, torch.from_numpy(jj).to(ops["W"].device)].t().contiguous())
            zv = _gather_pairs(ops["Z"], ii, jj)
            ref[s:s + ii.size] = oracle.dact_entries(Yr, Wc, zv, act)
            ref64[s:s + ii.size] = oracle.dact_entries(Yr, Wc, zv, act, f64=True)
        else:
            raise ValueError(kind)
    err = assert_close(got, ref, what)
    frac = within_one_ulp_frac(got, ref64)
    if ulp_gate is not None:
        assert frac >= ulp_gate, f"{what}: {frac:.4f} of entries within 1 ulp of the float64 result"
    return {"max_abs_err": err, "within_1ulp": frac, "entries": int(P)}


def _gather_pairs(t: torch.Tensor, i: np.ndarray, j: np.ndarray) -> np.ndarray:
    ti = torch.from_numpy(i).to(t.device)
    tj = torch.from_numpy(j).to(t.device)
    return bits(t[ti, tj])
