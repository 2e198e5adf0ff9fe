"""gb_gemm_linear_splitk_noalloc: split-K whose scratch is the library's own static
device array, for callers that may not allocate device memory.  Called through
the C ABI and compared with gb_gemm_linear_splitk (caller workspace) on two calls
in a row: the static array keeps the first call's contents, so the second call
also checks that the counters are cleared before use.  Collected last on
purpose, and independent of every other test's state."""
import ctypes

import numpy as np
import pytest
import torch

import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu


def _call_noalloc(L, A, B, bias, R, act, D, splits):
    M, K = A.shape
    N = B.shape[0]
    return L.gb_gemm_linear_splitk_noalloc(
        A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), bias.data_ptr(), R.data_ptr(), R.stride(0),
        gb.ACT[act], D.data_ptr(), D.stride(0), M, N, K, splits, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_on_two_calls():
    gb.set_config(None)
    L = gb.lib()
    M, N, K = 127, 96, 16384          # one output tile, 256 k-blocks: split-K applies
    for call, seed in enumerate((101, 202)):
        A = inputs.randn_bf16((M, K), seed=seed, device="cuda")
        B = inputs.randn_bf16((N, K), seed=seed + 1, std=1.0 / np.sqrt(K), device="cuda")
        bias = inputs.randn_bf16((N,), seed=seed + 2, std=0.1, device="cuda")
        R = inputs.randn_bf16((M, N), seed=seed + 3, device="cuda")
        want = gb.linear(A, B, bias, R, act="gelu_tanh", split_k="auto")
        gb.device_status()
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = _call_noalloc(L, A, B, bias, R, "gelu_tanh", D, 0)
        assert st == 0, L.gb_last_error().decode()
        gb.device_status()
        plan = gb.last_plan()
        assert int(plan.split("splits=")[1].split()[0]) > 1, plan
        assert_close(bits(D), bits(want), f"call {call}")


def test_noalloc_rejects_more_than_the_static_scratch():
    L = gb.lib()
    n = ctypes.c_size_t(0)
    assert L.gb_static_scratch_bytes(ctypes.byref(n)) == 0
    M, N, K = 8192, 8192, 65536       # 4096 splits of this would need far more than the static scratch
    need = gb.splitk_workspace_bytes(M, N, K, 1024)
    assert need > n.value
    A = torch.empty((M, 64), dtype=torch.bfloat16, device="cuda")  # never read: the call is rejected first
    st = L.gb_gemm_linear_splitk_noalloc(A.data_ptr(), K, A.data_ptr(), K, None, None, 0, 0, A.data_ptr(), N,
                                         M, N, K, 1024, torch.cuda.current_stream().cuda_stream)
    assert st == 2
    assert b"static scratch" in L.gb_last_error()
