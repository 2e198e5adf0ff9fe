"""Full-size workloads on the GPU, in the launch configuration the benchmark times,
checked against the CPU oracle on two seeded samples of 65536 output entries each
-- a 256 x 256 grid of rows and columns that always includes the first/last row
and column and tile boundaries, and 65536 independent (i, j) pairs -- or on every
entry when the oracle can afford it.  On the sampled pairs at least 99 % of the
entries must also lie within one bf16 ulp of the float64 result.

Workloads (shapes and distributions as in ``dense_bf16_gemm_persistent_gb300.inputs``):
MLP linear + bias + GELU_tanh 8192x14336x4096; Llama-FFN 8192x14336x4096; the
ragged residual sweep (36 combos of M, N, K); the 2^32-element A of the 64-bit
indexing case."""
import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_bitexact, assert_close, bits, check_pairs, ulp_hist

pytestmark = pytest.mark.gpu

DEV = "cuda"
FULL_COMPARE_MACS = 2 ** 33


@pytest.fixture(autouse=True)
def _defaults():
    gb.set_config(None)
    yield
    gb.device_status()
    torch.cuda.empty_cache()


def sample(M, N, seed=1234):
    return inputs.sample_indices(M, N, seed=seed)


def rows_of(t: torch.Tensor, idx: np.ndarray) -> np.ndarray:
    return bits(t[torch.from_numpy(idx).to(t.device)])


def grid_of(t: torch.Tensor, r: np.ndarray, c: np.ndarray) -> np.ndarray:
    rr = torch.from_numpy(r).to(t.device)
    cc = torch.from_numpy(c).to(t.device)
    return bits(t[rr][:, cc])


def test_mlp_gelu_8192x14336x4096():
    w = inputs.mlp_gelu(device=DEV)
    D = gb.linear(w["A"], w["B"], w["bias"], None, act="gelu_tanh")
    gb.device_status()
    r, c = sample(8192, 14336)
    ref = oracle.linear(rows_of(w["A"], r), rows_of(w["B"], c), bits(w["bias"])[c], None, "gelu_tanh")
    got = grid_of(D, r, c)
    assert_close(got, ref, "mlp_gelu")
    ref64 = oracle.linear_f64(rows_of(w["A"], r), rows_of(w["B"], c), bits(w["bias"])[c], None, "gelu_tanh")
    h = ulp_hist(got, ref64)
    assert sum(v for k, v in h.items() if k <= 1) >= 0.99 * got.size, h
    i, j = inputs.sample_pairs(8192, 14336, seed=11)
    check_pairs("linear", D, w, i, j, act="gelu_tanh", what="mlp_gelu pairs")


def test_llama_ffn_8192x14336x4096():
    w = inputs.llama_ffn(device=DEV)
    D = gb.ffn_gated(w["X"], w["W1"], w["W3"])
    gb.device_status()
    r, c = sample(8192, 14336, seed=4321)
    ref = oracle.ffn_gated(rows_of(w["X"], r), rows_of(w["W1"], c), rows_of(w["W3"], c))
    assert_close(grid_of(D, r, c), ref, "llama_ffn")
    i, j = inputs.sample_pairs(8192, 14336, seed=12)
    check_pairs("ffn", D, w, i, j, what="llama_ffn pairs")


@pytest.mark.parametrize("split_k", [None, "auto"], ids=["nosplit", "autosplit"])
@pytest.mark.parametrize("M,N,K", inputs.ragged_combos(), ids=lambda v: str(v))
def test_ragged_residual(M, N, K, split_k):
    """D = A.B^T + R with every tile edge predicated (M, N not tile multiples); also
    through the split-K entry point with its automatic split count."""
    w = inputs.ragged(M, N, K, device=DEV)
    D = gb.linear(w["A"], w["B"], None, w["R"], split_k=split_k)
    gb.device_status()
    if M * N * K <= FULL_COMPARE_MACS:
        ref = oracle.linear(bits(w["A"]), bits(w["B"]), None, bits(w["R"]))
        assert_close(bits(D), ref, f"ragged {M}x{N}x{K}")
        if K == 65536:
            ref64 = oracle.linear_f64(bits(w["A"]), bits(w["B"]), None, bits(w["R"]))
            h = ulp_hist(bits(D), ref64)
            assert sum(v for k, v in h.items() if k <= 1) >= 0.99 * D.numel(), h
    else:
        r, c = sample(M, N, seed=M + N + K)
        ref = oracle.linear(rows_of(w["A"], r), rows_of(w["B"], c), None, grid_of(w["R"], r, c))
        assert_close(grid_of(D, r, c), ref, f"ragged {M}x{N}x{K}")
        i, j = inputs.sample_pairs(M, N, seed=M * 3 + N + K)
        check_pairs("linear", D, {"A": w["A"], "B": w["B"], "R": w["R"]}, i, j,
                    ulp_gate=0.99 if K == 65536 else None, what=f"ragged {M}x{N}x{K} pairs")
    if K == 4096 and split_k is None:
        # the product alone (R = 0), and the residual alone (A = 0: D must equal R exactly)
        Z = torch.zeros_like(w["R"])
        D0 = gb.linear(w["A"], w["B"], None, Z)
        gb.device_status()
        r, c = sample(M, N, seed=7)
        ref0 = oracle.linear(rows_of(w["A"], r), rows_of(w["B"], c))
        assert_close(grid_of(D0, r, c), ref0, "R=0")
        DA = gb.linear(torch.zeros_like(w["A"]), w["B"], None, w["R"])
        gb.device_status()
        assert torch.equal(DA.view(torch.int16), w["R"].view(torch.int16))


def test_int64_indexing_65536x4096x65536():
    """A has 2^32 elements (8 GiB): rows past 32768 sit beyond byte offset 2^32."""
    M, N, K = 65536, 4096, 65536
    w = inputs.int64_case(device=DEV)
    D = gb.linear(w["A"], w["B"])
    gb.device_status()
    r, c = sample(M, N, seed=99)
    assert (r >= 32768).sum() >= 100
    ref = oracle.linear(rows_of(w["A"], r), rows_of(w["B"], c))
    assert_close(grid_of(D, r, c), ref, "int64")
    i, j = inputs.sample_pairs(M, N, seed=13)
    assert (i >= 32768).sum() >= 30000
    check_pairs("linear", D, w, i, j, what="int64 pairs")
    # an index-revealing pattern: A[i, 0] = (i mod 7) - 3, B[n, 0] = 1, all else 0  ->  D[i, n] = (i mod 7) - 3
    A = w["A"]
    A.zero_()
    A[:, 0] = ((torch.arange(M, device=DEV) % 7) - 3).to(torch.bfloat16)
    B = w["B"]
    B.zero_()
    B[:, 0] = 1
    D = gb.linear(A, B, out=D)
    gb.device_status()
    want = ((torch.arange(M, device=DEV) % 7) - 3).to(torch.bfloat16)[:, None].expand(M, N)
    assert torch.equal(D.view(torch.int16), want.contiguous().view(torch.int16))
    del w, A, B, D


def test_bench_configuration_is_the_default():
    """The benchmark times the default plan; the sampled checks above run under it."""
    w = inputs.mlp_gelu(device=DEV, M=1024, N=2048, K=512)
    gb.linear(w["A"], w["B"], w["bias"], None, act="gelu_tanh")
    plan = gb.last_plan()
    assert "kernel=linear pair=1" in plan and "tile=256x256x64" in plan and "d_store=tma" in plan, plan


@pytest.mark.parametrize("spec", ["mc=1,issue=2", "issue=2", "prod=2", "prod=2,mc=1"])
def test_mlp_schedules_identical_bits_full_size(spec):
    """The whole 8192x14336 MLP output under the multicast and issue-loop schedules equals
    the default schedule's bit for bit (the per-element sum order is the same)."""
    w = inputs.mlp_gelu(device=DEV)
    D0 = gb.linear(w["A"], w["B"], w["bias"], None, act="gelu_tanh")
    gb.device_status()
    gb.set_config(spec)
    D1 = gb.linear(w["A"], w["B"], w["bias"], None, act="gelu_tanh")
    gb.device_status()
    gb.set_config(None)
    assert torch.equal(D0.view(torch.int16), D1.view(torch.int16)), spec
