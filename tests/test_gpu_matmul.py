"""The MatmulOp form D = bf16(act(A.B + bias) + R) with B in its [K,N] layout (an MN-major
tensor-core operand, "Translate MmaOp patterns properly on Hopper", description), against
the oracle: random and integer-exact operands over multi-tile ragged shapes, every
epilogue form, views with padded leading dimensions, unaligned D/R rows, schedule
overrides (identical bits), and a full-size launch checked on 65536 sampled entries."""
import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_bitexact, assert_close, bits, check_pairs, int_tensor

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def _reset_config():
    gb.set_config(None)
    yield
    gb.set_config(None)
    gb.device_status()


def run(A, B, bias=None, R=None, act="none", **kw):
    d = gb.matmul(A.to(DEV), B.to(DEV), None if bias is None else bias.to(DEV), None if R is None else R.to(DEV),
                  act=act, **kw)
    gb.device_status()
    return bits(d)


def ref(A, B, bias=None, R=None, act="none"):
    return oracle.matmul(bits(A), bits(B), None if bias is None else bits(bias), None if R is None else bits(R), act)


@pytest.mark.parametrize("act", ["none", "gelu_tanh", "silu", "relu"])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (513, 1320, 64), (129, 264, 4096), (1, 8, 8), (700, 96, 520),
                                   (2100, 2048, 64)])
def test_matmul_random(M, N, K, act):
    A = inputs.randn_bf16((M, K), seed=M + 1)
    B = inputs.randn_bf16((K, N), seed=N + 2, std=1.0 / np.sqrt(K))
    bias = inputs.randn_bf16((N,), seed=3, std=0.1)
    R = inputs.randn_bf16((M, N), seed=4)
    got = run(A, B, bias, R, act)
    assert "kernel=matmul" in gb.last_plan(), gb.last_plan()
    assert_close(got, ref(A, B, bias, R, act), f"{M}x{N}x{K} {act}")
    assert_close(run(A, B), ref(A, B), f"{M}x{N}x{K} plain")


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 712, 520), (257, 136, 72), (64, 64, 4096)])
def test_matmul_integer_bit_exact(M, N, K, pair):
    gb.set_config(f"pair={pair}")
    A, B = int_tensor((M, K), 5), int_tensor((K, N), 6)
    bias, R = int_tensor((N,), 7, -4, 4), int_tensor((M, N), 8, -4, 4)
    assert_bitexact(run(A, B), ref(A, B), "no epilogue")
    assert_bitexact(run(A, B, bias, R, "relu"), ref(A, B, bias, R, "relu"), "bias+relu+R")
    # against the linear form on the transposed operand: the same sums
    d_lin = gb.linear(A.to(DEV), B.t().contiguous().to(DEV), bias.to(DEV), R.to(DEV), act="relu")
    gb.device_status()
    assert_bitexact(run(A, B, bias, R, "relu"), bits(d_lin), "matmul vs linear on B^T")


@pytest.mark.parametrize("spec", ["pair=0", "pair=1", "epi=1", "epi=2", "bn=128", "stages=2", "grid=3", "wide=0",
                                  "wide=1", "pingpong=1", "prod=1", "group=2,grid=5", "zigzag=1,grid=4"])
def test_matmul_schedules_identical_bits(spec):
    M, N, K = 700, 904, 320
    A = inputs.randn_bf16((M, K), seed=20)
    B = inputs.randn_bf16((K, N), seed=21, std=0.1)
    bias = inputs.randn_bf16((N,), seed=22, std=0.1)
    R = inputs.randn_bf16((M, N), seed=23)
    base = run(A, B, bias, R, "gelu_tanh")
    gb.set_config(spec)
    got = run(A, B, bias, R, "gelu_tanh")
    if "zigzag=1" in spec:  # reversed K order: a different fp32 sum order
        assert_close(got, ref(A, B, bias, R, "gelu_tanh"), spec)
    else:
        assert_bitexact(got, base, spec)


def test_matmul_views_unaligned_rows_and_padded_b():
    """B [K, 4099] as a view of a [K, 4104] buffer (ldb a multiple of 8, N not), R and D with
    rows 8198 bytes apart (the shared-memory transposes), A as a column slice."""
    M, N, K = 200, 4099, 136
    Abig = inputs.randn_bf16((M, K + 40), seed=30)
    A = Abig[:, 8:8 + K]
    Bbig = inputs.randn_bf16((K, 4104), seed=31, std=1.0 / np.sqrt(K))
    B = Bbig[:, :N]
    R = inputs.randn_bf16((M, N), seed=32)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    gb.matmul(Abig.to(DEV)[:, 8:8 + K], Bbig.to(DEV)[:, :N], None, R.to(DEV), act="silu", out=D)
    gb.device_status()
    plan = gb.last_plan()
    assert "d_store=st.transposed" in plan and "r_load=ld.transposed" in plan, plan
    assert_close(bits(D), ref(A.contiguous(), B.contiguous(), None, R, "silu"), "N=4099")


def test_matmul_k_zero_and_empty():
    M, N = 64, 40
    bias = inputs.randn_bf16((N,), seed=40, std=0.5)
    R = inputs.randn_bf16((M, N), seed=41)
    A = torch.empty((M, 0), dtype=torch.bfloat16, device=DEV)
    B = torch.empty((0, N), dtype=torch.bfloat16, device=DEV)
    d = gb.matmul(A, B, bias.to(DEV), R.to(DEV), act="relu")
    gb.device_status()
    assert_close(bits(d), ref(torch.empty((M, 0), dtype=torch.bfloat16), torch.empty((0, N), dtype=torch.bfloat16),
                              bias, R, "relu"), "K=0")
    e = gb.matmul(torch.empty((0, 8), dtype=torch.bfloat16, device=DEV),
                  torch.empty((8, 16), dtype=torch.bfloat16, device=DEV))
    gb.device_status()
    assert e.shape == (0, 16)


def test_matmul_mlp_shape_sampled():
    """X[8192,4096] . W[4096,14336] (the MLP weight stored [K,N]) + bias, GELU-tanh: 65536
    independent sampled entries against the oracle's per-entry evaluator, >= 99 % within
    one bf16 ulp of the float64 result."""
    M, N, K = 8192, 14336, 4096
    X = inputs.randn_bf16((M, K), seed=50, device=DEV)
    W = inputs.randn_bf16((K, N), seed=51, std=0.02, device=DEV)
    bias = inputs.randn_bf16((N,), seed=52, std=0.02, device=DEV)
    D = gb.matmul(X, W, bias, act="gelu_tanh")
    gb.device_status()
    assert "kernel=matmul pair=1" in gb.last_plan(), gb.last_plan()
    i, j = inputs.sample_pairs(M, N, n=65536, seed=53)
    check_pairs("matmul", D, {"A": X, "B": W, "bias": bias}, i, j, act="gelu_tanh", what="matmul MLP shape")
