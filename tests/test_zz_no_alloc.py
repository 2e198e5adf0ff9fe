"""gb_gemm_linear_splitk_noalloc: split-K whose scratch is the library's own static
device array, for callers that may not allocate device memory (a framework whose
caching allocator must own every device allocation, a serving runtime that
reserves all memory at start-up).  Called through the C ABI and compared with the
CPU oracle on two calls in a row: the static array keeps the first call's
contents, so the second call also checks that the counters and partial sums are
cleared before use.  The second call must not change the device's free memory or
torch's allocator statistics.  Collected last on purpose, and independent of
every other test's state."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu


def _call_noalloc(L, A, B, bias, R, act, D, splits):
    M, K = A.shape
    N = B.shape[0]
    return L.gb_gemm_linear_splitk_noalloc(
        A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), None if bias is None else bias.data_ptr(),
        None if R is None else R.data_ptr(), 0 if R is None else R.stride(0), gb.ACT[act], D.data_ptr(),
        D.stride(0), M, N, K, splits, torch.cuda.current_stream().cuda_stream)


def _scratch_bytes(L) -> int:
    n = ctypes.c_size_t(0)
    assert L.gb_static_scratch_bytes(ctypes.byref(n)) == 0
    return int(n.value)


def test_noalloc_matches_the_oracle_on_two_calls():
    gb.set_config(None)
    L = gb.lib()
    M, N, K = 127, 96, 16384          # one output tile, 256 k-blocks: split-K applies
    for call, seed in enumerate((101, 202)):
        A = inputs.randn_bf16((M, K), seed=seed, device="cuda")
        B = inputs.randn_bf16((N, K), seed=seed + 1, std=1.0 / np.sqrt(K), device="cuda")
        bias = inputs.randn_bf16((N,), seed=seed + 2, std=0.1, device="cuda")
        R = inputs.randn_bf16((M, N), seed=seed + 3, device="cuda")
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        stats0 = torch.cuda.memory_stats()
        st = _call_noalloc(L, A, B, bias, R, "gelu_tanh", D, 0)
        assert st == 0, L.gb_last_error().decode()
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        stats1 = torch.cuda.memory_stats()
        gb.device_status()
        plan = gb.last_plan()
        assert int(plan.split("splits=")[1].split()[0]) > 1, plan
        if call == 1:  # the first call may load the kernel's code; the second allocates nothing
            assert free1 == free0, (free0, free1)
            for key in ("allocated_bytes.all.current", "reserved_bytes.all.current", "allocation.all.allocated"):
                assert stats1.get(key) == stats0.get(key), key
        want = oracle.linear(bits(A), bits(B), bits(bias), bits(R), "gelu_tanh")
        assert_close(bits(D), want, f"call {call}")


def test_noalloc_rejects_more_than_the_static_scratch():
    """An explicit split count whose partials exceed the static scratch is refused on
    the host.  The tensors really have the shapes passed, so nothing could go out of
    bounds even if the refusal regressed: 4096x4096 output in 256 tiles of 256x256
    fp32 partials is 64 MiB, more than the 32 MiB array."""
    L = gb.lib()
    M, N, K, splits = 4096, 4096, 256, 4
    cap = _scratch_bytes(L)
    need = gb.splitk_workspace_bytes(M, N, K, splits)
    assert need > cap
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = _call_noalloc(L, A, B, None, None, "none", D, splits)
    assert st == 2
    assert b"static scratch" in L.gb_last_error()
    # splits = 1 needs no scratch and runs
    st = _call_noalloc(L, A, B, None, None, "none", D, 1)
    assert st == 0, L.gb_last_error().decode()
    gb.device_status()
    assert "splits=1" in gb.last_plan()


@pytest.mark.parametrize("M,N,K", [(127, 96, 65536), (8191, 96, 65536), (127, 12288, 65536), (1000, 4099, 65536),
                                   (4096, 4096, 65536)])
def test_noalloc_automatic_plan_fits_the_static_scratch(M, N, K):
    """The automatic split count only splits tile sets that fill at most half of the
    units, so its partials stay well inside the static scratch."""
    assert gb.splitk_workspace_bytes(M, N, K, 0) <= _scratch_bytes(gb.lib())
