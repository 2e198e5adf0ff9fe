"""Split-K (the schedule the pages' persistent Hopper scheduler lacks): the CUDA
path against the CPU oracle for skinny shapes, explicit split counts, CTA pairs,
the FFN fusion, workspace reuse across calls, repeat runs, and bit-exactness on
integer inputs."""
import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_bitexact, assert_close, bits, int_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset():
    gb.set_config(None)
    yield
    gb.set_config(None)
    gb.device_status()


def _lin(M, N, K, seed=0, bias=False, R=False, act="none"):
    A = inputs.randn_bf16((M, K), seed=seed)
    B = inputs.randn_bf16((N, K), seed=seed + 1, std=1.0 / np.sqrt(K))
    b = inputs.randn_bf16((N,), seed=seed + 2, std=0.1) if bias else None
    r = inputs.randn_bf16((M, N), seed=seed + 3) if R else None
    ref = oracle.linear(bits(A), bits(B), None if b is None else bits(b), None if r is None else bits(r), act)
    dev = [None if t is None else t.to(DEV) for t in (A, B, b, r)]
    return dev, ref


@pytest.mark.parametrize("M,N,K", [(127, 96, 65536), (1000, 96, 4096), (127, 4099, 4096), (3001, 96, 4096),
                                   (200, 300, 2000), (129, 257, 520)])
def test_auto_split_matches_oracle(M, N, K):
    (A, B, b, r), ref = _lin(M, N, K, bias=True, R=True, act="gelu_tanh")
    D = gb.linear(A, B, b, r, act="gelu_tanh", split_k="auto")
    gb.device_status()
    assert_close(bits(D), ref, f"{M}x{N}x{K} {gb.last_plan()}")


def test_auto_split_actually_splits_skinny_shapes():
    A = torch.zeros((127, 65536), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((96, 65536), dtype=torch.bfloat16, device=DEV)
    gb.linear(A, B, split_k="auto")
    gb.device_status()
    plan = gb.last_plan()
    splits = int(plan.split("splits=")[1].split()[0])
    assert splits > 16, plan


@pytest.mark.parametrize("epi", [1, 2])
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 1000])
@pytest.mark.parametrize("pair", [0, 1])
def test_explicit_splits(splits, pair, epi):
    gb.set_config(f"pair={pair},epi={epi}")
    M, N, K = 300, 520, 1000      # 16 k-blocks; 1000 is clamped to 16
    (A, B, b, r), ref = _lin(M, N, K, seed=10, bias=True, R=True, act="silu")
    D = gb.linear(A, B, b, r, act="silu", split_k=splits)
    gb.device_status()
    assert_close(bits(D), ref, f"splits={splits} {gb.last_plan()}")


@pytest.mark.parametrize("splits", [2, 5])
def test_integer_inputs_bit_exact(splits):
    M, N, K = 260, 300, 640
    A, B = int_tensor((M, K), 20), int_tensor((N, K), 21)
    R = int_tensor((M, N), 22, -3, 3)
    ref = oracle.linear(bits(A), bits(B), None, bits(R))
    D = gb.linear(A.to(DEV), B.to(DEV), None, R.to(DEV), split_k=splits)
    gb.device_status()
    assert_bitexact(bits(D), ref, f"splits={splits}")


def test_repeat_runs_agree():
    """The fp32 additions across K ranges happen in L2 in no fixed order: repeated
    calls agree within the tolerance, and bit for bit when every partial sum is exact."""
    (A, B, _, _), ref = _lin(127, 1000, 8192, seed=30)
    ws = torch.empty(gb.splitk_workspace_bytes(127, 1000, 8192, 0), dtype=torch.uint8, device=DEV)
    d1 = gb.linear(A, B, split_k="auto", workspace=ws)
    d2 = gb.linear(A, B, split_k="auto", workspace=ws)
    gb.device_status()
    assert_close(bits(d1), ref, "run 1")
    assert_close(bits(d2), bits(d1), "run 2 vs run 1")
    Ai, Bi = int_tensor((127, 8192), 31).to(DEV), int_tensor((1000, 8192), 32).to(DEV)
    e1 = gb.linear(Ai, Bi, split_k="auto", workspace=ws)
    e2 = gb.linear(Ai, Bi, split_k="auto", workspace=ws)
    gb.device_status()
    assert torch.equal(e1.view(torch.int16), e2.view(torch.int16))


def test_workspace_reuse_across_shapes():
    """One workspace for calls of different shapes in a row: the per-slab counters are
    cleared by every call, so each result is right."""
    cases = [(127, 96, 8192), (300, 200, 4096), (127, 96, 8192)]
    need = max(gb.splitk_workspace_bytes(M, N, K, 0) for M, N, K in cases)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    for i, (M, N, K) in enumerate(cases):
        (A, B, _, r), ref = _lin(M, N, K, seed=40 + i, R=True)
        D = gb.linear(A, B, None, r, split_k="auto", workspace=ws)
        gb.device_status()
        assert_close(bits(D), ref, f"case {i}")


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("splits", ["auto", 3])
def test_ffn_split(pair, splits):
    gb.set_config(f"pair={pair}")
    M, N, K = 300, 260, 2048
    X = inputs.randn_bf16((M, K), seed=50)
    W1 = inputs.randn_bf16((N, K), seed=51, std=1.0 / np.sqrt(K))
    W3 = inputs.randn_bf16((N, K), seed=52, std=1.0 / np.sqrt(K))
    D = gb.ffn_gated(X.to(DEV), W1.to(DEV), W3.to(DEV), split_k=splits)
    gb.device_status()
    assert_close(bits(D), oracle.ffn_gated(bits(X), bits(W1), bits(W3)), f"ffn {gb.last_plan()}")


def test_workspace_checks():
    A = torch.zeros((127, 4096), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((96, 4096), dtype=torch.bfloat16, device=DEV)
    D = torch.empty((127, 96), dtype=torch.bfloat16, device=DEV)
    need = gb.splitk_workspace_bytes(127, 96, 4096, 8)
    assert need > 0
    L = gb.lib()
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    st = L.gb_gemm_linear_splitk(A.data_ptr(), 4096, B.data_ptr(), 4096, None, None, 0, 0, D.data_ptr(), 96,
                                 127, 96, 4096, 8, small.data_ptr(), small.numel(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 1 and b"smaller" in L.gb_last_error()
    st = L.gb_gemm_linear_splitk(A.data_ptr(), 4096, B.data_ptr(), 4096, None, None, 0, 0, D.data_ptr(), 96,
                                 127, 96, 4096, 8, None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 1 and b"workspace" in L.gb_last_error()
    # no split needed -> no workspace needed
    assert gb.splitk_workspace_bytes(8192, 8192, 4096, 0) == 0


@pytest.mark.parametrize("splits", [0, 2, 3])
@pytest.mark.parametrize("form", ["plain", "bias_gelu", "residual", "residual_bias_silu", "unaligned_d"])
def test_queried_workspace_covers_every_epilogue(form, splits):
    """The size query knows only M, N, K and the split count, while a call may pick
    another epilogue layout (an epilogue input or unaligned rows take two epilogue
    warpgroups, no input one).  A workspace of exactly the queried size must do for
    every epilogue form.  80 tiles of 256 x 256 and K = 1280: without an epilogue input
    the plan takes one epilogue warpgroup, with one it takes two."""
    M, N, K = 1280, 4096, 1280
    A = inputs.randn_bf16((M, K), seed=200, device=DEV)
    B = inputs.randn_bf16((N, K), seed=201, std=1.0 / np.sqrt(K), device=DEV)
    bias = inputs.randn_bf16((N,), seed=202, std=0.1, device=DEV) if "bias" in form else None
    R = inputs.randn_bf16((M, N), seed=203, device=DEV) if "residual" in form else None
    act = {"bias_gelu": "gelu_tanh", "residual_bias_silu": "silu"}.get(form, "none")
    ws = torch.empty(gb.splitk_workspace_bytes(M, N, K, splits), dtype=torch.uint8, device=DEV)
    if form == "unaligned_d":
        Dbig = torch.zeros((M, N + 1), dtype=torch.bfloat16, device=DEV)
        D = Dbig[:, 1:]
        gb.linear(A, B, bias, R, act=act, out=D, split_k=splits or "auto", workspace=ws)
    else:
        D = gb.linear(A, B, bias, R, act=act, split_k=splits or "auto", workspace=ws)
    gb.device_status()
    plan = gb.last_plan()
    r, c = inputs.sample_indices(M, N, seed=204)
    rr, cc = torch.from_numpy(r).to(DEV), torch.from_numpy(c).to(DEV)
    ref = oracle.linear(bits(A[rr]), bits(B[cc]), None if bias is None else bits(bias)[c],
                        None if R is None else bits(R[rr][:, cc]), act)
    assert_close(bits(D[rr][:, cc]), ref, f"{form} {plan}")


@pytest.mark.parametrize("splits", [0, 3])
def test_split_k_with_d_aliasing_r(splits):
    """D == R through the split-K entry point: the last split of each slab reads R and
    writes D for the same elements, after every partial is in."""
    M, N, K = 127, 200, 8192
    A = inputs.randn_bf16((M, K), seed=210)
    B = inputs.randn_bf16((N, K), seed=211, std=1.0 / np.sqrt(K))
    bias = inputs.randn_bf16((N,), seed=212, std=0.1)
    R = inputs.randn_bf16((M, N), seed=213)
    ref = oracle.linear(bits(A), bits(B), bits(bias), bits(R), "silu")
    RD = R.to(DEV).clone()
    gb.linear(A.to(DEV), B.to(DEV), bias.to(DEV), RD, act="silu", out=RD, split_k=splits or "auto")
    gb.device_status()
    assert int(gb.last_plan().split("splits=")[1].split()[0]) > 1, gb.last_plan()
    assert_close(bits(RD), ref, f"split-K D == R, splits={splits}")


@pytest.mark.parametrize("M,N,K", [(1, 1, 65536), (1, 1, 8), (2, 3, 40000), (1, 200, 16384)])
def test_tiny_outputs_long_k(M, N, K):
    """One or a few output elements over a long K: a single tile split into many K ranges
    (the automatic count caps at 64), all reducing into the same slab; and integer inputs
    bit-exact."""
    (A, B, b, r), ref = _lin(M, N, K, seed=220, bias=True, R=True, act="relu")
    D = gb.linear(A, B, b, r, act="relu", split_k="auto")
    gb.device_status()
    assert_close(bits(D), ref, f"{M}x{N}x{K} {gb.last_plan()}")
    Ai, Bi = int_tensor((M, K), 221, -1, 1), int_tensor((N, K), 222, -1, 1)
    Di = gb.linear(Ai.to(DEV), Bi.to(DEV), split_k="auto")
    gb.device_status()
    assert_bitexact(bits(Di), oracle.linear(bits(Ai), bits(Bi)), f"int {M}x{N}x{K}")
