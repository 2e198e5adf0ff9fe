"""Pin checks for the CPU oracle, written against mathematics and library routines.

Each check takes an ``Oracle`` instance, so the same checks run on the real
oracle (``test_oracle_pins.py``) and on deliberately broken copies of it
(``test_oracle_mutants.py``, which asserts that each planted mistake fails at
least one check).  Nothing here re-types the oracle's formulas: the expected
values come from exact integer arithmetic, float64 numpy / torch routines,
closed forms, identities, or the Higham error bound of a recursive fp32 sum.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

U32 = 2.0 ** -24  # unit roundoff of binary32


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def f32_of(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rand_bf16(rng: np.random.Generator, shape, std=1.0) -> np.ndarray:
    x = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32))
    return bits(x.to(torch.bfloat16))


def int_bf16(rng: np.random.Generator, shape, lo=-2, hi=2) -> tuple[np.ndarray, np.ndarray]:
    v = rng.integers(lo, hi + 1, size=shape)
    return bits(torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)), v.astype(np.int64)


def lib_round_bf16(x_f32: np.ndarray) -> np.ndarray:
    """torch's float32 -> bfloat16 conversion (round to nearest even)."""
    return bits(torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16))


# ---- rounding ---------------------------------------------------------------------------------

def check_f32_to_bf16(o) -> None:
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(1e3),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-30),
        # exact ties: bf16 value + half an ulp (low 16 bits 0x8000), both parities
        ((rng.integers(0x3000, 0x5000, 4000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, np.inf, -np.inf], dtype=np.float32),
    ])
    np.testing.assert_array_equal(o.f32_to_bf16(x), lib_round_bf16(x))


def _bf16_value(b: int) -> Fraction:
    return Fraction(float(f32_of(np.array([b], dtype=np.uint16))[0]))


def check_f64_to_bf16(o) -> None:
    """Brute force: the nearest bf16 (ties to the even pattern) by exact rational distance."""
    rng = np.random.default_rng(8)
    xs = np.concatenate([rng.standard_normal(300) * 10.0,
                         rng.standard_normal(50) * 1e-3,
                         # values exactly halfway between two bf16 numbers, plus and minus a tiny bit
                         np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40,
                                   1.0 + 2.0 ** -8 - 2.0 ** -40, -(2.0 + 2.0 ** -7)])])
    got = o.f64_to_bf16(xs)
    for x, g in zip(xs, got):
        center = int(lib_round_bf16(np.array([x], dtype=np.float32))[0])
        best = None
        for cand in (center - 1, center, center + 1):
            if (cand ^ center) & 0x8000:  # stay on the same sign
                continue
            d = abs(_bf16_value(cand) - Fraction(float(x)))
            key = (d, cand & 1)
            if best is None or key < best[0]:
                best = (key, cand)
        assert int(g) == best[1], (x, hex(int(g)), hex(best[1]))


# ---- the sum ----------------------------------------------------------------------------------

def check_acc_error_bound(o) -> None:
    """|fl32(sum) - exact| <= gamma_K * sum |a b| for a recursive fp32 sum (Higham, Thm 3.1)."""
    rng = np.random.default_rng(11)
    for M, N, K in [(1, 1, 1), (3, 5, 7), (16, 16, 256), (9, 13, 100), (2, 3, 255)]:
        A = rand_bf16(rng, (M, K))
        B = rand_bf16(rng, (N, K))
        a, b = f32_of(A).astype(np.float64), f32_of(B).astype(np.float64)
        exact = a @ b.T                # products exact; float64 sum error << fp32 bound
        absum = np.abs(a) @ np.abs(b).T
        gamma = K * U32 / (1 - K * U32)
        acc = o.acc_f32(A, B).astype(np.float64)
        err = np.abs(acc - exact)
        assert np.all(err <= gamma * absum + 1e-30), (M, N, K, float(err.max()))
        # and the float64 twin agrees with numpy to float64 accuracy
        y = o.linear_f64(A, B)
        assert np.allclose(y, exact, rtol=1e-12, atol=1e-12 * absum.max())


def check_fp32_sequential_sum(o) -> None:
    """The sum is a recursive binary32 sum in ascending k, not a more exact or reordered
    one.  2^24 + 1 rounds back to 2^24 in binary32 (a tie, to even), so
    [2^24, 1, -2^24] . [1, 1, 1] is 0 summed in that order; the exact value is 1, and
    so is the descending-order sum (-2^24 + 1 = -16777215 exactly, + 2^24 = 1)."""
    A = lib_round_bf16(np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)], [1.0, 2.0 ** 24, -(2.0 ** 24)]], dtype=np.float32))
    B = lib_round_bf16(np.ones((1, 3), dtype=np.float32))
    acc = o.acc_f32(A, B)
    assert float(acc[0, 0]) == 0.0, float(acc[0, 0])   # the 1 is absorbed
    assert float(acc[1, 0]) == 0.0, float(acc[1, 0])   # 1 + 2^24 rounds to 2^24 as well
    np.testing.assert_array_equal(o.linear(A, B), lib_round_bf16(np.zeros((2, 1), dtype=np.float32)))
    # many small terms after a large one are each absorbed
    row = np.concatenate([[2.0 ** 24], np.ones(50), [-(2.0 ** 24)]]).astype(np.float32)[None, :]
    A2 = lib_round_bf16(row)
    B2 = lib_round_bf16(np.ones((1, row.shape[1]), dtype=np.float32))
    assert float(o.acc_f32(A2, B2)[0, 0]) == 0.0


def check_integer_exact(o) -> None:
    """Small-integer operands: every partial sum is an exact integer in fp32, so the
    result is the exact integer product rounded once to bf16 -- bit for bit."""
    rng = np.random.default_rng(12)
    for M, N, K in [(1, 1, 1), (5, 7, 64), (17, 9, 33), (32, 40, 64)]:
        A, a = int_bf16(rng, (M, K))
        B, b = int_bf16(rng, (N, K))
        bias, bv = int_bf16(rng, (N,), -3, 3)
        R, rv = int_bf16(rng, (M, N), -3, 3)
        exact = a @ b.T
        np.testing.assert_array_equal(o.linear(A, B), lib_round_bf16(exact.astype(np.float32)))
        np.testing.assert_array_equal(o.linear(A, B, bias=bias, R=R),
                                      lib_round_bf16((exact + bv[None, :] + rv).astype(np.float32)))
        relu = np.maximum(exact + bv[None, :], 0) + rv
        np.testing.assert_array_equal(o.linear(A, B, bias=bias, R=R, act="relu"),
                                      lib_round_bf16(relu.astype(np.float32)))


def check_transpose_and_index(o) -> None:
    """A row-index/column-index encoded pattern: D[m,n] = m + 16 n exactly, which a
    transposed operand or a wrong row/column index cannot reproduce."""
    M, N, K = 9, 7, 24
    a = np.zeros((M, K), np.float32)
    b = np.zeros((N, K), np.float32)
    a[:, 0] = np.arange(M)          # A[m,0] = m, A[m,1] = 1
    a[:, 1] = 1.0
    b[:, 0] = 1.0                   # B[n,0] = 1, B[n,1] = 16 n
    b[:, 1] = 16.0 * np.arange(N)
    A, B = lib_round_bf16(a), lib_round_bf16(b)
    want = np.arange(M)[:, None] + 16 * np.arange(N)[None, :]
    np.testing.assert_array_equal(o.linear(A, B), lib_round_bf16(want.astype(np.float32)))


def check_identity_b(o) -> None:
    rng = np.random.default_rng(13)
    M, K = 37, 48
    A = rand_bf16(rng, (M, K))
    B = lib_round_bf16(np.eye(K, dtype=np.float32))
    np.testing.assert_array_equal(o.linear(A, B), A)
    R = rand_bf16(rng, (M, K))
    # the one rounding after the fp32 add: torch computes the same pair of operations
    want = (from_bits(A).float() + from_bits(R).float()).to(torch.bfloat16)
    np.testing.assert_array_equal(o.linear(A, B, R=R), bits(want))


def check_zero_bias_and_linearity(o) -> None:
    rng = np.random.default_rng(14)
    M, N, K = 12, 10, 40
    A = rand_bf16(rng, (M, K))
    B = rand_bf16(rng, (N, K))
    zero = np.zeros(N, np.uint16)
    for act in ("none", "gelu_tanh", "silu", "relu"):
        np.testing.assert_array_equal(o.linear(A, B, bias=zero, act=act), o.linear(A, B, act=act))
    A1, a1 = int_bf16(rng, (M, K), -1, 1)
    A2, a2 = int_bf16(rng, (M, K), -1, 1)
    A12 = lib_round_bf16((a1 + a2).astype(np.float32))
    Bi, _ = int_bf16(rng, (N, K), -2, 2)
    s = f32_of(o.linear(A1, Bi)) + f32_of(o.linear(A2, Bi))
    np.testing.assert_array_equal(o.linear(A12, Bi), lib_round_bf16(s))


def check_bias_broadcast_and_residual(o) -> None:
    """Bias is added per column n (broadcast over rows); R is per element."""
    M, N, K = 4, 6, 8
    A = np.zeros((M, K), np.uint16)            # product is exactly zero
    B = np.zeros((N, K), np.uint16)
    bias = lib_round_bf16(np.arange(N, dtype=np.float32) + 1)
    R = lib_round_bf16(100.0 * np.arange(M, dtype=np.float32)[:, None] + np.zeros((M, N), np.float32))
    want = np.arange(N)[None, :] + 1 + 100 * np.arange(M)[:, None]
    np.testing.assert_array_equal(o.linear(A, B, bias=bias, R=R), lib_round_bf16(want.astype(np.float32)))


def check_k_zero(o) -> None:
    """K = 0: the empty sum is 0, so D = bf16(act(bias) + R)."""
    rng = np.random.default_rng(15)
    M, N = 5, 9
    A = np.zeros((M, 0), np.uint16)
    B = np.zeros((N, 0), np.uint16)
    bias = rand_bf16(rng, (N,))
    R = rand_bf16(rng, (M, N))
    t_bias = from_bits(bias).double()
    want = torch.nn.functional.gelu(t_bias, approximate="tanh")[None, :] + from_bits(R).double()
    got = f32_of(o.linear(A, B, bias=bias, R=R, act="gelu_tanh")).astype(np.float64)
    assert np.all(np.abs(got - want.numpy()) <= 2.0 ** -8 * np.abs(want.numpy()) + 1e-6)
    np.testing.assert_array_equal(o.linear(A, B), np.zeros((M, N), np.uint16))


# ---- activations ------------------------------------------------------------------------------

def check_activation_closed_forms(o) -> None:
    z = np.array([0.0], np.float32)
    for act in ("none", "gelu_tanh", "silu", "relu"):
        assert o.act_f32(act, z)[0] == 0.0
    big = np.array([12.0, 30.0, 80.0], np.float32)
    np.testing.assert_array_equal(o.act_f32("gelu_tanh", big), big)      # tanh saturates to 1
    np.testing.assert_array_equal(o.act_f32("relu", -big), np.zeros(3, np.float32))
    assert np.all(np.abs(o.act_f32("gelu_tanh", -big)) <= 1e-30)
    assert np.all(np.abs(o.act_f32("silu", np.array([-40.0, -80.0], np.float32))) < 1e-15)
    np.testing.assert_allclose(o.act_f32("silu", np.array([40.0], np.float32)), [40.0], rtol=1e-7)
    # silu(x) - silu(-x) = x (since sigma(x) + sigma(-x) = 1)
    x = np.linspace(-10, 10, 2001).astype(np.float32)
    d = o.act_f64("silu", x.astype(np.float64)) - o.act_f64("silu", -x.astype(np.float64))
    np.testing.assert_allclose(d, x.astype(np.float64), rtol=0, atol=1e-12)
    # gelu_tanh(x) - gelu_tanh(-x) = x as well (tanh is odd)
    d = o.act_f64("gelu_tanh", x.astype(np.float64)) - o.act_f64("gelu_tanh", -x.astype(np.float64))
    np.testing.assert_allclose(d, x.astype(np.float64), rtol=0, atol=1e-12)


def check_activation_vs_library(o) -> None:
    """fp32 activations against torch's float64 routines at 10^4 points, and the tanh
    form of GELU against the exact erf form (they differ by under 1e-3 everywhere)."""
    rng = np.random.default_rng(16)
    x = np.concatenate([rng.standard_normal(9000) * 4.0, np.linspace(-20, 20, 1000)]).astype(np.float32)
    t = torch.from_numpy(x.astype(np.float64))
    lib = {"gelu_tanh": torch.nn.functional.gelu(t, approximate="tanh").numpy(),
           "silu": torch.nn.functional.silu(t).numpy(),
           "relu": torch.relu(t).numpy(),
           "none": t.numpy()}
    for act, want in lib.items():
        got32 = o.act_f32(act, x).astype(np.float64)
        # a few fp32 roundings, plus the cancellation in 1 + tanh(.) near -1 (absolute ~|x| 2^-24)
        tol = 16 * U32 * np.abs(want) + 1e-7 * np.abs(x) + 1e-37
        assert np.all(np.abs(got32 - want) <= tol), act
        got64 = o.act_f64(act, x.astype(np.float64))
        np.testing.assert_allclose(got64, want, rtol=1e-13, atol=1e-13)
    erf_gelu = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x.astype(np.float64)])
    assert np.max(np.abs(o.act_f64("gelu_tanh", x.astype(np.float64)) - erf_gelu)) < 1e-3


def check_epilogue_order(o) -> None:
    """act is applied to acc + bias, and R is added after the activation."""
    M, N, K = 2, 3, 4
    a = np.zeros((M, K), np.float32)
    a[:, 0] = 1.0
    b = np.zeros((N, K), np.float32)
    b[:, 0] = -4.0                      # acc = -4 everywhere
    A, B = lib_round_bf16(a), lib_round_bf16(b)
    bias = lib_round_bf16(np.array([1.0, 2.0, 6.0], np.float32))   # acc + bias = -3, -2, 2
    R = lib_round_bf16(np.full((M, N), 0.5, np.float32))
    got = f32_of(o.linear(A, B, bias=bias, R=R, act="relu"))
    np.testing.assert_array_equal(got, np.tile(np.array([0.5, 0.5, 2.5], np.float32), (M, 1)))


# ---- Llama-FFN fusion -------------------------------------------------------------------------

def check_ffn(o) -> None:
    rng = np.random.default_rng(17)
    # (1) X.W3^T == 1 exactly, X.W1^T runs over small integers: D = bf16(silu(a1))
    M, N, K = 6, 17, 16
    x = np.zeros((M, K), np.float32)
    x[:, 0] = 1.0
    x[:, 1] = np.arange(M)
    w1 = np.zeros((N, K), np.float32)
    w1[:, 0] = np.arange(N) - 8.0       # a1[m,n] = (n - 8) + m * 0
    w3 = np.zeros((N, K), np.float32)
    w3[:, 0] = 1.0                      # a3 = 1
    X, W1, W3 = lib_round_bf16(x), lib_round_bf16(w1), lib_round_bf16(w3)
    a1 = np.tile(np.arange(N) - 8.0, (M, 1))
    silu = torch.nn.functional.silu(torch.from_numpy(a1)).numpy()
    got = f32_of(o.ffn_gated(X, W1, W3)).astype(np.float64)
    assert np.all(np.abs(got - silu) <= 2.0 ** -8 * np.abs(silu) + 1e-30)
    # (2) the gate multiplies the up-projection: a3 = 3 scales the result by 3
    W3b = lib_round_bf16(3.0 * w3)
    got3 = f32_of(o.ffn_gated(X, W1, W3b)).astype(np.float64)
    assert np.all(np.abs(got3 - 3.0 * silu) <= 2.0 ** -8 * np.abs(3.0 * silu) + 1e-30)
    # (3) random operands: fp32 result within one bf16 rounding of the float64 definition
    M, N, K = 9, 11, 64
    X = rand_bf16(rng, (M, K))
    W1 = rand_bf16(rng, (N, K), 0.2)
    W3 = rand_bf16(rng, (N, K), 0.2)
    xf, w1f, w3f = (f32_of(v).astype(np.float64) for v in (X, W1, W3))
    a1, a3 = xf @ w1f.T, xf @ w3f.T
    ref = torch.nn.functional.silu(torch.from_numpy(a1)).numpy() * a3
    np.testing.assert_allclose(o.ffn_gated_f64(X, W1, W3), ref, rtol=1e-12, atol=1e-14)
    got = f32_of(o.ffn_gated(X, W1, W3)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


def check_leading_dims(o) -> None:
    """Strided views (leading dimension > row length: A, B and the epilogue input R)
    give the same bits as packed copies."""
    rng = np.random.default_rng(18)
    Abig = rand_bf16(rng, (10, 70))
    Bbig = rand_bf16(rng, (6, 80))
    A, B = Abig[:, 3:53], Bbig[:, 10:60]
    np.testing.assert_array_equal(o.linear(A, B), o.linear(np.ascontiguousarray(A), np.ascontiguousarray(B)))
    Rbig = rand_bf16(rng, (10, 15))
    R = Rbig[:, 4:10]                                   # leading dimension 15 > N = 6
    bias = rand_bf16(rng, (6,), 0.1)
    np.testing.assert_array_equal(o.linear(A, B, bias=bias, R=R, act="silu"),
                                  o.linear(np.ascontiguousarray(A), np.ascontiguousarray(B), bias=bias,
                                           R=np.ascontiguousarray(R), act="silu"))


def check_preact_output(o) -> None:
    """The second output is the pre-activation bf16(acc + bias): exact on integer
    operands (so a ReLU that clips negatives shows whether it was taken before or
    after the activation), and D is unchanged by asking for it."""
    rng = np.random.default_rng(19)
    M, N, K = 9, 14, 32
    A, a = int_bf16(rng, (M, K))
    B, b = int_bf16(rng, (N, K))
    bias, bv = int_bf16(rng, (N,), -5, 5)
    R, rv = int_bf16(rng, (M, N), -2, 2)
    D, Z = o.linear_preact(A, B, bias=bias, R=R, act="relu")
    pre = a @ b.T + bv[None, :]
    assert (pre < 0).any()
    np.testing.assert_array_equal(Z, lib_round_bf16(pre.astype(np.float32)))
    np.testing.assert_array_equal(D, lib_round_bf16((np.maximum(pre, 0) + rv).astype(np.float32)))
    np.testing.assert_array_equal(D, o.linear(A, B, bias=bias, R=R, act="relu"))
    A2 = rand_bf16(rng, (M, K))
    B2 = rand_bf16(rng, (N, K), 0.3)
    D2, Z2 = o.linear_preact(A2, B2, act="none")
    np.testing.assert_array_equal(D2, Z2)


# ---- activation gradient (backward pass consumer of the pre-activation) --------------------

def check_dact_closed_forms(o) -> None:
    """act'(0) = 1/2 for GELU and SiLU; ReLU' is the step with 0 at 0; the identity's
    derivative is 1; GELU' and SiLU' tend to 1 for large x and to 0 for very negative x."""
    z = np.array([0.0], np.float32)
    assert o.dact_f32_values("gelu_tanh", z)[0] == 0.5
    assert o.dact_f32_values("silu", z)[0] == 0.5
    np.testing.assert_array_equal(o.dact_f32_values("relu", np.array([-2.0, -0.0, 0.0, 1e-30, 3.0], np.float32)),
                                  np.array([0, 0, 0, 1, 1], np.float32))
    np.testing.assert_array_equal(o.dact_f32_values("none", np.array([-5.0, 0.0, 7.0], np.float32)),
                                  np.ones(3, np.float32))
    big = np.array([12.0, 30.0, 80.0], np.float32)
    np.testing.assert_array_equal(o.dact_f32_values("gelu_tanh", big), np.ones(3, np.float32))
    np.testing.assert_array_equal(o.dact_f32_values("silu", np.array([40.0, 80.0], np.float32)),
                                  np.ones(2, np.float32))
    assert np.all(np.abs(o.dact_f32_values("gelu_tanh", -big)) <= 1e-30)
    assert np.all(np.abs(o.dact_f32_values("silu", np.array([-40.0, -80.0], np.float32))) < 1e-15)
    # silu'(x) + silu'(-x) = 1 and gelu'(x) + gelu'(-x) = 1 (derivatives of x - f(-x) = f(x))
    x = np.linspace(-10, 10, 2001)
    for act in ("silu", "gelu_tanh"):
        np.testing.assert_allclose(o.dact_f64_values(act, x) + o.dact_f64_values(act, -x), 1.0, rtol=0, atol=1e-12)


def check_dact_vs_autograd(o) -> None:
    """act' against torch autograd of torch's own float64 activations at 10^4 points,
    and against central finite differences of the oracle's float64 activations."""
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.standard_normal(9000) * 4.0, np.linspace(-20, 20, 1000)])
    x = x[np.abs(x) > 1e-3]  # keep ReLU's kink out of the finite differences
    fns = {"gelu_tanh": lambda t: torch.nn.functional.gelu(t, approximate="tanh"),
           "silu": torch.nn.functional.silu, "relu": torch.relu, "none": lambda t: t * 1.0}
    for act, fn in fns.items():
        t = torch.from_numpy(x.copy()).requires_grad_(True)
        fn(t).sum().backward()
        want = t.grad.numpy()
        np.testing.assert_allclose(o.dact_f64_values(act, x), want, rtol=1e-12, atol=1e-13)
        got32 = o.dact_f32_values(act, x.astype(np.float32)).astype(np.float64)
        want32 = o.dact_f64_values(act, x.astype(np.float32).astype(np.float64))
        assert np.all(np.abs(got32 - want32) <= 1e-6 + 16 * U32 * np.abs(want32)), act
        h = 1e-5
        fd = (o.act_f64(act, x + h) - o.act_f64(act, x - h)) / (2 * h)
        assert np.all(np.abs(o.dact_f64_values(act, x) - fd) <= 1e-8 * (1 + np.abs(x))), act


def check_dact_integer_exact(o) -> None:
    """Small-integer dY and W: the sum over n is an exact integer, so with the ReLU
    derivative (0 or 1, from the sign of integer Z, including Z = 0) or the identity's,
    D is that integer masked and rounded once -- bit for bit."""
    rng = np.random.default_rng(22)
    for M, N, K in [(1, 1, 1), (5, 64, 7), (17, 33, 9), (12, 40, 31)]:
        dY, dy = int_bf16(rng, (M, N))
        W, w = int_bf16(rng, (N, K))
        Z, zv = int_bf16(rng, (M, K), -3, 3)
        g = dy @ w
        np.testing.assert_array_equal(o.dact(dY, W, Z, "none"), lib_round_bf16(g.astype(np.float32)))
        # the mask multiplies: a negative sum times 0 is -0, as in IEEE arithmetic
        mask = (zv > 0).astype(np.float32)
        np.testing.assert_array_equal(o.dact(dY, W, Z, "relu"), lib_round_bf16(g.astype(np.float32) * mask))


def check_dact_index_and_transpose(o) -> None:
    """D[m,k] = m + 16 k exactly: dY[m,0] = m, dY[m,1] = 1, W[0,k] = 1, W[1,k] = 16 k;
    a W read as [K,N], or a swapped row/column index, cannot give it."""
    M, N, K = 9, 6, 7
    dy = np.zeros((M, N), np.float32)
    dy[:, 0] = np.arange(M)
    dy[:, 1] = 1.0
    w = np.zeros((N, K), np.float32)
    w[0, :] = 1.0
    w[1, :] = 16.0 * np.arange(K)
    Z = lib_round_bf16(np.ones((M, K), np.float32))
    want = np.arange(M)[:, None] + 16 * np.arange(K)[None, :]
    for act in ("relu", "none"):
        np.testing.assert_array_equal(o.dact(lib_round_bf16(dy), lib_round_bf16(w), Z, act),
                                      lib_round_bf16(want.astype(np.float32)))


def check_dact_identity_and_order(o) -> None:
    """W = I: D = bf16(dY * act'(Z)) within one rounding of the float64 product; and the
    sum over n is a binary32 sum in ascending n (2^24 + 1 is absorbed)."""
    rng = np.random.default_rng(23)
    M, K = 13, 24
    dY = rand_bf16(rng, (M, K))
    Z = rand_bf16(rng, (M, K), 2.0)
    W = lib_round_bf16(np.eye(K, dtype=np.float32))
    z = torch.from_numpy(f32_of(Z).astype(np.float64)).requires_grad_(True)
    torch.nn.functional.gelu(z, approximate="tanh").sum().backward()
    ref = f32_of(dY).astype(np.float64) * z.grad.numpy()
    got = f32_of(o.dact(dY, W, Z, "gelu_tanh")).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
    np.testing.assert_allclose(o.dact_f64(dY, W, Z, "gelu_tanh"), ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(o.dact(dY, W, Z, "relu"),
                                  lib_round_bf16(f32_of(dY) * (f32_of(Z) > 0).astype(np.float32)))
    dy = lib_round_bf16(np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)]], np.float32))
    ones = lib_round_bf16(np.ones((3, 1), np.float32))
    one = lib_round_bf16(np.ones((1, 1), np.float32))
    assert int(o.dact(dy, ones, one, "none")[0, 0]) == 0
    assert o.dact_f64(dy, ones, one, "none")[0, 0] == 1.0


# ---- single entries (sampled checks of large outputs) -----------------------------------------

def check_entries(o) -> None:
    """The per-entry evaluators against exact integer arithmetic at independent
    (i, j) pairs (linear with bias/ReLU/R, dact with ReLU), the FFN at integer silu
    points, and every float64 twin against numpy/torch float64."""
    rng = np.random.default_rng(24)
    M, N, K, P = 11, 13, 40, 300
    A, a = int_bf16(rng, (M, K))
    B, b = int_bf16(rng, (N, K))
    bias, bv = int_bf16(rng, (N,), -3, 3)
    R, rv = int_bf16(rng, (M, N), -3, 3)
    i = rng.integers(0, M, P)
    j = rng.integers(0, N, P)
    exact = (a @ b.T + bv[None, :])[i, j]
    np.testing.assert_array_equal(o.linear_entries(A[i], B[j], bias[j], R[i, j], "relu"),
                                  lib_round_bf16((np.maximum(exact, 0) + rv[i, j]).astype(np.float32)))
    np.testing.assert_array_equal(o.linear_entries(A[i], B[j]), lib_round_bf16((a @ b.T)[i, j].astype(np.float32)))
    # dact: row i of dY with column j of W
    Wt, w = int_bf16(rng, (K, N))           # W [K_contract=K, N_out=N]
    Z, zv = int_bf16(rng, (M, N), -3, 3)
    g = (a @ w)[i, j]
    np.testing.assert_array_equal(o.dact_entries(A[i], np.ascontiguousarray(Wt.T)[j], Z[i, j], "relu"),
                                  lib_round_bf16(g.astype(np.float32) * (zv[i, j] > 0).astype(np.float32)))
    # FFN: X.W3 = 1, X.W1 = integer n - 8
    x = np.zeros((M, K), np.float32)
    x[:, 0] = 1.0
    w1 = np.zeros((N, K), np.float32)
    w1[:, 0] = np.arange(N) - 8.0
    w3 = np.zeros((N, K), np.float32)
    w3[:, 0] = 1.0
    X, W1, W3 = lib_round_bf16(x), lib_round_bf16(w1), lib_round_bf16(w3)
    silu = torch.nn.functional.silu(torch.from_numpy((np.arange(N) - 8.0)[j])).numpy()
    got = f32_of(o.ffn_entries(X[i], W1[j], W3[j])).astype(np.float64)
    assert np.all(np.abs(got - silu) <= 2.0 ** -8 * np.abs(silu) + 1e-30)
    # float64 twins on random operands
    Ar, Br, Cr = rand_bf16(rng, (P, K)), rand_bf16(rng, (P, K), 0.2), rand_bf16(rng, (P, K), 0.2)
    af, bf, cf = (f32_of(v).astype(np.float64) for v in (Ar, Br, Cr))
    dot_ab, dot_ac = (af * bf).sum(1), (af * cf).sum(1)
    bz = rand_bf16(rng, (P,))
    t = torch.from_numpy(dot_ab + f32_of(bz).astype(np.float64))
    np.testing.assert_allclose(o.linear_entries(Ar, Br, bz, None, "gelu_tanh", f64=True),
                               torch.nn.functional.gelu(t, approximate="tanh").numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o.ffn_entries(Ar, Br, Cr, f64=True),
                               torch.nn.functional.silu(torch.from_numpy(dot_ab)).numpy() * dot_ac,
                               rtol=1e-12, atol=1e-13)
    zt = torch.from_numpy(f32_of(bz).astype(np.float64)).requires_grad_(True)
    torch.nn.functional.silu(zt).sum().backward()
    np.testing.assert_allclose(o.dact_entries(Ar, Br, bz, "silu", f64=True), dot_ab * zt.grad.numpy(),
                               rtol=1e-12, atol=1e-13)


def check_matmul_form(o) -> None:
    """The MatmulOp form (B given as [K,N]): integer operands against numpy's exact integer
    product, an index pattern that a transposed or misread B cannot reproduce (D[m,n] =
    m + 16 n with B[0,n] = 1, B[1,n] = 16 n), and the identity B = I_K returning A."""
    rng = np.random.default_rng(31)
    for M, N, K in [(1, 1, 1), (6, 9, 40), (13, 5, 64)]:
        A, a = int_bf16(rng, (M, K))
        B, b = int_bf16(rng, (K, N))
        bias, bv = int_bf16(rng, (N,), -3, 3)
        R, rv = int_bf16(rng, (M, N), -3, 3)
        exact = a @ b
        np.testing.assert_array_equal(o.matmul(A, B), lib_round_bf16(exact.astype(np.float32)))
        relu = np.maximum(exact + bv[None, :], 0) + rv
        np.testing.assert_array_equal(o.matmul(A, B, bias=bias, R=R, act="relu"), lib_round_bf16(relu.astype(np.float32)))
    M, N, K = 9, 7, 24
    a = np.zeros((M, K), np.float32)
    b = np.zeros((K, N), np.float32)
    a[:, 0] = np.arange(M)
    a[:, 1] = 1.0
    b[0, :] = 1.0
    b[1, :] = 16.0 * np.arange(N)
    want = np.arange(M)[:, None] + 16 * np.arange(N)[None, :]
    np.testing.assert_array_equal(o.matmul(lib_round_bf16(a), lib_round_bf16(b)), lib_round_bf16(want.astype(np.float32)))
    A = rand_bf16(rng, (11, 16))
    np.testing.assert_array_equal(o.matmul(A, lib_round_bf16(np.eye(16, dtype=np.float32))), A)


ALL_CHECKS = [check_f32_to_bf16, check_f64_to_bf16, check_acc_error_bound, check_fp32_sequential_sum,
              check_integer_exact,
              check_transpose_and_index, check_identity_b, check_zero_bias_and_linearity,
              check_bias_broadcast_and_residual, check_k_zero, check_activation_closed_forms,
              check_activation_vs_library, check_epilogue_order, check_ffn, check_leading_dims,
              check_preact_output, check_dact_closed_forms, check_dact_vs_autograd, check_dact_integer_exact,
              check_dact_index_and_transpose, check_dact_identity_and_order, check_entries, check_matmul_form]
