"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method: it only draws random numbers,
rounds them to bf16 (the inputs *are* bf16), and picks sample indices.  Both the
CUDA path and the CPU oracle receive what it produces.

Recipes (the pages give no workload shapes or value distributions; these are the
synthetic stand-ins the library is measured and checked on):

* ``plain``      A[256,512], B[384,512] ~ N(0,1); D = A.B^T, no epilogue.
* ``mlp_gelu``   X[8192,4096] ~ N(0,1); W[14336,4096], bias[14336] ~ N(0, 0.02);
                 D = GELU_tanh(X.W^T + bias).
* ``llama_ffn``  X[8192,4096] ~ N(0,1); W1, W3[14336,4096] ~ N(0, 0.02);
                 D = silu(X.W1^T) * (X.W3^T).
* ``ragged``     M in {127,1000,3001,8191}, N in {96,4099,12288}, K in {64,4096,65536};
                 A ~ N(0,1), B ~ N(0,1)/sqrt(K), R ~ N(0,1); D = A.B^T + R.
                 (Reading: only B carries the 1/sqrt(K) so that A.B^T has unit
                 variance like R; scaling both would make the product ~1/sqrt(K),
                 smaller than the tolerance.)
* ``int64``      A[65536,65536] (2^32 elements), B[4096,65536] ~ U(-1,1)/256; D = A.B^T.
* ``mlp_dact``   the MLP layer's backward activation-gradient product: dY[8192,14336] ~ N(0,1)
                 (the gradient of the layer's output), W[14336,4096] ~ N(0, 0.02) (the MLP
                 weight, in the layout the forward pass reads), Z[8192,4096] ~ N(0,1) (the
                 stored pre-activation of the layer's input); D = (dY.W) * GELU_tanh'(Z).

N(mu, s) means standard deviation s.  Every tensor is drawn in fp32 from its own
``torch.Generator`` seeded with ``seed + offset`` (A/X: 0, B/W/W1: 1, bias/W3: 2,
R: 3) and rounded to bf16 with round-to-nearest-even by ``Tensor.to``.
"""
from __future__ import annotations

import math

import numpy as np
import torch

OFFSETS = {"A": 0, "B": 1, "bias": 2, "W3": 2, "R": 3}

RAGGED_M = (127, 1000, 3001, 8191)
RAGGED_N = (96, 4099, 12288)
RAGGED_K = (64, 4096, 65536)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, *, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    """i.i.d. N(0, std^2) drawn in fp32, rounded to bf16."""
    x = torch.randn(tuple(shape), generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def uniform_bf16(shape, *, seed: int, lo: float, hi: float, scale: float = 1.0,
                 device="cpu", chunk_rows: int | None = None) -> torch.Tensor:
    """i.i.d. U(lo, hi) * scale drawn in fp32, rounded to bf16.

    With ``chunk_rows`` the rows are drawn in chunks, chunk c from its own
    generator seeded ``seed * 2**32 + c`` (keeps the fp32 staging buffer small for
    multi-GiB operands)."""
    shape = tuple(shape)
    if chunk_rows is None:
        x = torch.rand(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
        x.mul_((hi - lo) * scale).add_(lo * scale)
        return x.to(torch.bfloat16)
    out = torch.empty(shape, device=device, dtype=torch.bfloat16)
    rows = shape[0]
    for c, r0 in enumerate(range(0, rows, chunk_rows)):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.rand((r1 - r0,) + shape[1:], generator=_gen(seed * 2**32 + c, device),
                       device=device, dtype=torch.float32)
        x.mul_((hi - lo) * scale).add_(lo * scale)
        out[r0:r1].copy_(x)
        del x
    return out


def randint_bf16(shape, *, seed: int, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """Integers uniform in [lo, hi] (inclusive), stored exactly as bf16."""
    x = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed, device), device=device)
    return x.to(torch.bfloat16)


# ---- the workloads --------------------------------------------------------------------------

def plain(device="cpu", seed: int = 0, M: int = 256, N: int = 384, K: int = 512) -> dict:
    return {"A": randn_bf16((M, K), seed=seed + OFFSETS["A"], device=device),
            "B": randn_bf16((N, K), seed=seed + OFFSETS["B"], device=device),
            "act": "none"}


def mlp_gelu(device="cpu", seed: int = 0, M: int = 8192, N: int = 14336, K: int = 4096) -> dict:
    return {"A": randn_bf16((M, K), seed=seed + OFFSETS["A"], device=device),
            "B": randn_bf16((N, K), seed=seed + OFFSETS["B"], std=0.02, device=device),
            "bias": randn_bf16((N,), seed=seed + OFFSETS["bias"], std=0.02, device=device),
            "act": "gelu_tanh"}


def llama_ffn(device="cpu", seed: int = 0, M: int = 8192, N: int = 14336, K: int = 4096) -> dict:
    return {"X": randn_bf16((M, K), seed=seed + OFFSETS["A"], device=device),
            "W1": randn_bf16((N, K), seed=seed + OFFSETS["B"], std=0.02, device=device),
            "W3": randn_bf16((N, K), seed=seed + OFFSETS["W3"], std=0.02, device=device)}


def ragged(M: int, N: int, K: int, device="cpu", seed: int = 0) -> dict:
    return {"A": randn_bf16((M, K), seed=seed + OFFSETS["A"], device=device),
            "B": randn_bf16((N, K), seed=seed + OFFSETS["B"], std=1.0 / math.sqrt(K), device=device),
            "R": randn_bf16((M, N), seed=seed + OFFSETS["R"], device=device),
            "act": "none"}


def int64_case(device="cpu", seed: int = 0, M: int = 65536, N: int = 4096, K: int = 65536) -> dict:
    chunk = 4096
    return {"A": uniform_bf16((M, K), seed=seed + OFFSETS["A"], lo=-1.0, hi=1.0, scale=1.0 / 256,
                              device=device, chunk_rows=chunk),
            "B": uniform_bf16((N, K), seed=seed + OFFSETS["B"], lo=-1.0, hi=1.0, scale=1.0 / 256,
                              device=device, chunk_rows=chunk),
            "act": "none"}


def mlp_dact(device="cpu", seed: int = 0, M: int = 8192, N: int = 14336, K: int = 4096) -> dict:
    return {"dY": randn_bf16((M, N), seed=seed + OFFSETS["A"], device=device),
            "W": randn_bf16((N, K), seed=seed + OFFSETS["B"], std=0.02, device=device),
            "Z": randn_bf16((M, K), seed=seed + OFFSETS["R"], device=device),
            "act": "gelu_tanh"}


def ragged_combos():
    return [(m, n, k) for m in RAGGED_M for n in RAGGED_N for k in RAGGED_K]


# ---- output sampling --------------------------------------------------------------------------

def sample_indices(M: int, N: int, *, seed: int = 1234, rows: int = 256, cols: int = 256,
                   tile_m: int = 128, tile_n: int = 256) -> tuple[np.ndarray, np.ndarray]:
    """Rows and columns of a sampled output grid (|rows| * |cols| entries, 65536 by default).

    The grid always holds the first and last row/column and both sides of up to
    rows/8 (cols/8) tile boundaries spread evenly over the range; the rest are drawn
    uniformly without replacement from ``numpy.random.default_rng(seed)``.  Sorted."""
    rng = np.random.default_rng(seed)

    def pick(extent: int, want: int, tile: int) -> np.ndarray:
        if extent <= want:
            return np.arange(extent, dtype=np.int64)
        # first/last index, plus both sides of tile boundaries spread evenly over the range
        bounds = np.arange(tile, extent, tile, dtype=np.int64)
        nb = min(bounds.size, want // 8)
        if nb:
            bounds = bounds[np.linspace(0, bounds.size - 1, nb).round().astype(np.int64)]
        special = np.unique(np.concatenate([[0, extent - 1], bounds - 1, bounds]))
        rest = np.setdiff1d(np.arange(extent, dtype=np.int64), special)
        extra = rng.choice(rest, size=want - special.size, replace=False)
        return np.sort(np.concatenate([special, extra]))

    return pick(M, rows, tile_m), pick(N, cols, tile_n)


def sample_pairs(M: int, N: int, *, n: int = 65536, seed: int = 4242) -> tuple[np.ndarray, np.ndarray]:
    """n independent output entries (i, j): the four corners, then i and j drawn
    independently and uniformly with replacement from ``numpy.random.default_rng(seed)``."""
    rng = np.random.default_rng(seed)
    i = rng.integers(0, M, size=n, dtype=np.int64)
    j = rng.integers(0, N, size=n, dtype=np.int64)
    corners = np.array([[0, 0], [0, N - 1], [M - 1, 0], [M - 1, N - 1]], dtype=np.int64)
    k = min(4, n)
    i[:k], j[:k] = corners[:k, 0], corners[:k, 1]
    return i, j


def to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (a reinterpretation, no arithmetic)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
