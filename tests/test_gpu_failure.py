"""Failure detection on the GPU without a GPU fault: the test hook makes the
producer never issue its first pipeline stage, so a bounded wait inside the
kernel runs out.  The kernel must drain what it has in flight, free TMEM,
return, and report GB_ERR_TIMEOUT through the device status word; the CUDA
context must stay usable (a normal call right after is correct)."""
import numpy as np
import pytest

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("extra", ["", "prod=2", "prod=3", "mc=1", "mc=1,prod=2"])
@pytest.mark.parametrize("epi", [1, 2])
@pytest.mark.parametrize("kind", ["linear", "ffn"])
@pytest.mark.parametrize("pair", [0, 1])
def test_wait_timeout_is_reported_and_context_survives(kind, pair, epi, extra):
    """Also with two producer threads (A and B loads from different warps) and with the
    A tile multicast between two CTA pairs: every role still drains and returns."""
    if "mc=1" in extra and not pair:
        pytest.skip("A multicast is a CTA-pair schedule")
    M, N, K = 512, 768, 1024
    A = inputs.randn_bf16((M, K), seed=1).cuda()
    B = inputs.randn_bf16((N, K), seed=2, std=1.0 / np.sqrt(K)).cuda()
    B3 = inputs.randn_bf16((N, K), seed=3, std=1.0 / np.sqrt(K)).cuda()
    gb.device_status()
    gb.set_config(f"pair={pair},epi={epi}" + (f",{extra}" if extra else ""))
    gb.set_wait_timeout_ns(100_000_000)  # 0.1 s
    gb.set_fault_injection(1)
    try:
        if kind == "linear":
            gb.linear(A, B)
        else:
            gb.ffn_gated(A, B, B3)
        with pytest.raises(gb.GBError) as ei:
            gb.device_status()
        assert ei.value.status == 4, str(ei.value)
        assert "timed out" in str(ei.value)
    finally:
        gb.set_fault_injection(0)
        gb.set_wait_timeout_ns(0)
    gb.device_status()  # the status word was cleared by the read above
    if kind == "linear":
        D = gb.linear(A, B)
        gb.device_status()
        assert_close(bits(D), oracle.linear(bits(A), bits(B)), "after timeout")
    else:
        D = gb.ffn_gated(A, B, B3)
        gb.device_status()
        assert_close(bits(D), oracle.ffn_gated(bits(A), bits(B), bits(B3)), "after timeout")
    gb.set_config(None)


@pytest.mark.parametrize("spec", ["epi=4", "epi=4,wide=0", "epi=4,wide=1", "epi=2,wide=1", "epi=2,wide=2",
                                  "epi=2,pingpong=1,wide=0"])
def test_wait_timeout_with_epilogue_input_queues(spec):
    """A residual launch whose R boxes are in flight when the waits run out (paired
    path, 32x32 and 32x64 boxes, two and four epilogue warpgroups): the epilogue drains
    its R loads before it returns and the context stays usable."""
    M, N, K = 600, 1024, 128
    A = inputs.randn_bf16((M, K), seed=4).cuda()
    B = inputs.randn_bf16((N, K), seed=5, std=1.0 / np.sqrt(K)).cuda()
    R = inputs.randn_bf16((M, N), seed=6).cuda()
    gb.device_status()
    gb.set_config(spec)
    gb.set_wait_timeout_ns(100_000_000)  # 0.1 s
    gb.set_fault_injection(1)
    try:
        gb.linear(A, B, None, R)
        with pytest.raises(gb.GBError) as ei:
            gb.device_status()
        assert ei.value.status == 4, str(ei.value)
    finally:
        gb.set_fault_injection(0)
        gb.set_wait_timeout_ns(0)
    gb.device_status()
    D = gb.linear(A, B, None, R)
    gb.device_status()
    plan = gb.last_plan()
    gb.set_config(None)
    assert f"epi={spec.split('epi=')[1][0]}" in plan, plan
    assert_close(bits(D), oracle.linear(bits(A), bits(B), None, bits(R)), f"after timeout {spec}")


@pytest.mark.parametrize("kind", ["matmul", "dact"])
@pytest.mark.parametrize("pair", [0, 1])
def test_wait_timeout_with_mn_major_b(kind, pair):
    """The MN-major B path (B stored [K, N]; two producer threads take the B boxes of
    alternate stages): a wait that runs out is reported and the context survives."""
    M, N, K = 512, 768, 1024
    A = inputs.randn_bf16((M, K), seed=11).cuda()
    B = inputs.randn_bf16((K, N), seed=12, std=1.0 / np.sqrt(K)).cuda()
    Z = inputs.randn_bf16((M, N), seed=13).cuda()
    gb.device_status()
    gb.set_config(f"pair={pair}")
    gb.set_wait_timeout_ns(100_000_000)  # 0.1 s
    gb.set_fault_injection(1)
    try:
        if kind == "matmul":
            gb.matmul(A, B)
        else:  # dY [M, K] . W [K, N] with the gradient of Z [M, N]
            gb.linear_dact(A, B, Z, act="gelu_tanh")
        with pytest.raises(gb.GBError) as ei:
            gb.device_status()
        assert ei.value.status == 4, str(ei.value)
    finally:
        gb.set_fault_injection(0)
        gb.set_wait_timeout_ns(0)
    gb.device_status()
    if kind == "matmul":
        D = gb.matmul(A, B)
        gb.device_status()
        assert_close(bits(D), oracle.matmul(bits(A), bits(B)), "after timeout")
    else:
        D = gb.linear_dact(A, B, Z, act="gelu_tanh")
        gb.device_status()
        assert_close(bits(D), oracle.dact(bits(A), bits(B), bits(Z), "gelu_tanh"), "after timeout")
    gb.set_config(None)
