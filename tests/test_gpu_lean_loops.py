"""The producer's and the MMA issuer's lean loops (one per operand form: K-major B,
MN-major B, A multicast between two pairs) against the general loops they replace in the
common case.  The loops only change when each box is issued, never what is computed, so
every schedule gives the same bits; the default one is also checked against the oracle.

prod=1 sends the loads through the general producer loop (one thread issues A and B),
issue=3 sends the MMAs through the general issue loop, mc=1 selects A multicast."""
import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_bitexact, assert_close, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"

SCHEDULES = ["prod=1", "issue=3", "prod=1,issue=3", "zigzag=1", "mc=1", "mc=1,prod=1", "mc=1,zigzag=1", "prod=3"]


@pytest.fixture(autouse=True)
def _reset_config():
    gb.set_config(None)
    yield
    gb.set_config(None)
    gb.device_status()


def _run(fn, spec):
    gb.set_config(spec)
    out = fn()
    gb.device_status()
    gb.set_config(None)
    return bits(out)


def test_linear_k_major_b():
    M, N, K = 700, 1000, 576  # 9 k-blocks, ragged tiles in M and N
    A = inputs.randn_bf16((M, K), seed=301)
    B = inputs.randn_bf16((N, K), seed=302, std=1.0 / np.sqrt(K))
    bias = inputs.randn_bf16((N,), seed=303, std=0.1)
    fn = lambda: gb.linear(A.to(DEV), B.to(DEV), bias.to(DEV), act="gelu_tanh")
    base = _run(fn, None)
    assert_close(base, oracle.linear(bits(A), bits(B), bits(bias), None, "gelu_tanh"), "default")
    for spec in SCHEDULES:
        assert_bitexact(_run(fn, spec), base, spec)


def test_linear_split_k_and_residual():
    """Split-K items start mid-K (kb0 > 0) and zig-zag reverses them."""
    M, N, K = 520, 768, 2048
    A = inputs.randn_bf16((M, K), seed=311)
    B = inputs.randn_bf16((N, K), seed=312, std=1.0 / np.sqrt(K))
    R = inputs.randn_bf16((M, N), seed=313)
    ref = oracle.linear(bits(A), bits(B), None, bits(R), "none")
    for split in (2, 3):
        fn = lambda: gb.linear(A.to(DEV), B.to(DEV), None, R.to(DEV), split_k=split)
        base = _run(fn, None)
        assert_close(base, ref, f"split {split}")
        for spec in ["prod=1", "issue=3", "zigzag=1", "mc=1", "prod=1,zigzag=1"]:
            assert_close(_run(fn, spec), ref, f"split {split} {spec}")


def test_ffn_two_b_operands():
    M, N, K = 600, 640, 512
    X = inputs.randn_bf16((M, K), seed=321)
    W1 = inputs.randn_bf16((N, K), seed=322, std=1.0 / np.sqrt(K))
    W3 = inputs.randn_bf16((N, K), seed=323, std=1.0 / np.sqrt(K))
    fn = lambda: gb.ffn_gated(X.to(DEV), W1.to(DEV), W3.to(DEV))
    base = _run(fn, None)
    assert_close(base, oracle.ffn_gated(bits(X), bits(W1), bits(W3)), "default")
    for spec in SCHEDULES:
        assert_bitexact(_run(fn, spec), base, spec)


def test_matmul_mn_major_b():
    M, N, K = 640, 896, 448  # N a multiple of 8: B's [K, N] rows are 16-byte aligned
    A = inputs.randn_bf16((M, K), seed=331)
    B = inputs.randn_bf16((K, N), seed=332, std=1.0 / np.sqrt(K))
    fn = lambda: gb.matmul(A.to(DEV), B.to(DEV), act="relu")
    base = _run(fn, None)
    assert_close(base, oracle.matmul(bits(A), bits(B), None, None, "relu"), "default")
    for spec in ["prod=1", "issue=3", "prod=1,issue=3", "zigzag=1", "mc=1", "prod=3"]:
        assert_bitexact(_run(fn, spec), base, spec)


def test_single_cta_tiles():
    """One-CTA tiles (no pair): the lean loops' non-pair branch, with one and two B operands."""
    M, N, K = 128, 1000, 384
    A = inputs.randn_bf16((M, K), seed=341)
    B = inputs.randn_bf16((N, K), seed=342, std=1.0 / np.sqrt(K))
    fn = lambda: gb.linear(A.to(DEV), B.to(DEV))
    base = _run(fn, "pair=0")
    assert_close(base, oracle.linear(bits(A), bits(B), None, None, "none"), "pair=0")
    for spec in ["pair=0,prod=1", "pair=0,issue=3", "pair=0,zigzag=1"]:
        assert_bitexact(_run(fn, spec), base, spec)
    W3 = inputs.randn_bf16((N, K), seed=343, std=1.0 / np.sqrt(K))
    fn2 = lambda: gb.ffn_gated(A.to(DEV), B.to(DEV), W3.to(DEV))
    base2 = _run(fn2, "pair=0")
    assert_close(base2, oracle.ffn_gated(bits(A), bits(B), bits(W3)), "ffn pair=0")
    for spec in ["pair=0,prod=1", "pair=0,issue=3"]:
        assert_bitexact(_run(fn2, spec), base2, spec)
