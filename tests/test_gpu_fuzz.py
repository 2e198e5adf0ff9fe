"""Seeded randomized parity: random shapes (tile multiples, odd sizes, single rows and
columns, K = 0), random epilogues (bias, activation, epilogue input, second output),
every entry point (linear, pre-activation, FFN, their split-K forms, MatmulOp with B in
its [K, N] layout, the activation gradient) and random
configuration overrides, each compared element by element with the CPU oracle.  Every
case draws from its own seed, so a failure reproduces from its test id alone."""
import os

import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu

DEV = "cuda"
N_CASES = int(os.environ.get("GB_FUZZ_CASES", "256"))
MAX_MACS = 1 << 27  # keeps every oracle call well under a second

CONFIG_ITEMS = ["pair=0", "pair=1", "epi=1", "epi=2", "pingpong=1", "pingpong=0", "boxes=2", "boxes=5",
                "boxes=8", "stages=2", "stages=4", "grid=3", "grid=7", "bn=128", "group=1", "group=3",
                "zigzag=1", "persistent=0", "mc=1", "prod=1", "prod=3", "issue=3", "wide=0", "r_async=1",
                "epi=4"]


def _dim(rng) -> int:
    kind = rng.integers(0, 4)
    if kind == 0:
        return int(rng.integers(1, 17))        # a handful of rows or columns
    if kind == 1:
        return int(rng.integers(1, 700))       # anything, mostly ragged
    if kind == 2:
        return int(rng.integers(1, 90)) * 8    # 16-byte aligned rows
    return int(rng.choice([128, 256, 384, 512, 1024]))


def _case(seed: int) -> dict:
    rng = np.random.default_rng(seed)
    M, N = _dim(rng), _dim(rng)
    K = int(rng.choice([0, 8, 64, 200, 520, 1024, 2048]))
    while M * N * max(K, 1) > MAX_MACS:
        if M >= N:
            M = max(1, M // 2)
        else:
            N = max(1, N // 2)
    entry = str(rng.choice(["linear", "linear", "preact", "ffn", "linear_split", "ffn_split", "matmul", "dact"]))
    if entry == "matmul" and K == 0:
        K = 64  # (K = 0 is covered by the other entry points)
    items = [str(x) for x in rng.choice(CONFIG_ITEMS, size=int(rng.integers(0, 3)), replace=False)]
    if "pingpong=1" in items and "epi=1" in items:
        items.remove("epi=1")
    return dict(M=M, N=N, K=K, entry=entry, config=",".join(items),
                bias=bool(rng.random() < 0.5), R=bool(rng.random() < 0.5),
                act=str(rng.choice(["none", "gelu_tanh", "silu", "relu"])),
                d_offset=bool(rng.random() < 0.25), splits=int(rng.choice([0, 2, 3, 5])))


@pytest.fixture(autouse=True)
def _reset():
    gb.set_config(None)
    yield
    gb.set_config(None)
    gb.device_status()


def _padded(rows, cols, seed, std=1.0):
    """A [rows, cols] view on the device whose rows start 16 bytes apart (leading dimension
    rounded up to 8), as an MN-major or K-major TMA operand needs."""
    full = inputs.randn_bf16((rows, max(8, (cols + 7) // 8 * 8)), seed=seed, std=std)
    return full.to(DEV)[:, :cols]


def _out(M, N, offset):
    """D, either contiguous or a view whose rows start 2 bytes past a 16-byte boundary."""
    if not offset:
        return torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV), None
    big = torch.zeros((M, N + 1), dtype=torch.bfloat16, device=DEV)
    return big[:, 1:], big


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed):
    c = _case(1000 + seed)
    M, N, K = c["M"], c["N"], c["K"]
    what = f"seed {1000 + seed}: {c}"
    gb.set_config(c["config"] or None)
    A = inputs.randn_bf16((M, K), seed=seed * 10 + 1)
    B = inputs.randn_bf16((N, K), seed=seed * 10 + 2, std=1.0 / np.sqrt(max(K, 1)))
    D, big = _out(M, N, c["d_offset"])
    if c["entry"] == "dact":
        # dY [M, N] . W [N, K], times act'(Z) with Z [M, K]: the contraction runs over N
        dY = _padded(M, N, seed * 10 + 6)
        W = inputs.randn_bf16((N, K), seed=seed * 10 + 7, std=1.0 / np.sqrt(max(N, 1)))
        Z = inputs.randn_bf16((M, K), seed=seed * 10 + 8)
        Dk, bigk = _out(M, K, c["d_offset"])
        gb.linear_dact(dY, W.to(DEV), Z.to(DEV), act=c["act"], out=Dk)
        gb.device_status()
        assert_close(bits(Dk), oracle.dact(bits(dY), bits(W), bits(Z), c["act"]), what + " " + gb.last_plan())
        if bigk is not None:
            assert torch.all(bigk[:, 0] == 0)
        return
    if c["entry"] == "matmul":
        Bk = _padded(K, N, seed * 10 + 2, std=1.0 / np.sqrt(max(K, 1)))
        bias = inputs.randn_bf16((N,), seed=seed * 10 + 4, std=0.1) if c["bias"] else None
        R = inputs.randn_bf16((M, N), seed=seed * 10 + 5) if c["R"] else None
        gb.matmul(A.to(DEV), Bk, None if bias is None else bias.to(DEV), None if R is None else R.to(DEV),
                  act=c["act"], out=D)
        gb.device_status()
        ref = oracle.matmul(bits(A), bits(Bk), None if bias is None else bits(bias), None if R is None else bits(R),
                            c["act"])
        assert_close(bits(D), ref, what + " " + gb.last_plan())
        if big is not None:
            assert torch.all(big[:, 0] == 0)
        return
    if c["entry"].startswith("ffn"):
        B3 = inputs.randn_bf16((N, K), seed=seed * 10 + 3, std=1.0 / np.sqrt(max(K, 1)))
        split = (c["splits"] or "auto") if c["entry"] == "ffn_split" else None
        gb.ffn_gated(A.to(DEV), B.to(DEV), B3.to(DEV), out=D, split_k=split)
        gb.device_status()
        assert_close(bits(D), oracle.ffn_gated(bits(A), bits(B), bits(B3)), what + " " + gb.last_plan())
    else:
        bias = inputs.randn_bf16((N,), seed=seed * 10 + 4, std=0.1) if c["bias"] else None
        R = inputs.randn_bf16((M, N), seed=seed * 10 + 5) if c["R"] else None
        args = (A.to(DEV), B.to(DEV), None if bias is None else bias.to(DEV), None if R is None else R.to(DEV))
        ref_args = (bits(A), bits(B), None if bias is None else bits(bias), None if R is None else bits(R), c["act"])
        if c["entry"] == "preact":
            Z = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
            gb.linear_preact(*args, act=c["act"], out=D, preact=Z)
            gb.device_status()
            refD, refZ = oracle.linear_preact(*ref_args)
            assert_close(bits(D), refD, what + " D " + gb.last_plan())
            assert_close(bits(Z), refZ, what + " Z " + gb.last_plan())
        else:
            split = (c["splits"] or "auto") if c["entry"] == "linear_split" else None
            gb.linear(*args, act=c["act"], out=D, split_k=split)
            gb.device_status()
            assert_close(bits(D), oracle.linear(*ref_args), what + " " + gb.last_plan())
    if big is not None:  # nothing written outside the view
        assert torch.all(big[:, 0] == 0)
