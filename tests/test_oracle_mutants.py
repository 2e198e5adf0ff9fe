"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU) and
check that at least one pin in ``oracle_pins`` rejects it.  This is what makes
the pins meaningful: a dropped term, a wrong sign, a transposed operand or a
wrong constant anywhere in the oracle must fail one of them."""
import os
import shutil

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text to find, replacement, which occurrence (0-based)) -- every mutant keeps all
# memory accesses in bounds, so a mutant can only compute a wrong value, never crash.
MUTANTS = [
    ("drop_first_term", "for (int64_t k = 0; k < K; ++k) {\n        float p", "for (int64_t k = 1; k < K; ++k) {\n        float p", 0),
    ("drop_last_term", "for (int64_t k = 0; k < K; ++k) {\n        float p", "for (int64_t k = 0; k + 1 < K; ++k) {\n        float p", 0),
    ("sum_sign", "acc = acc + p;", "acc = acc - p;", 0),
    ("transposed_operands", "float v = dot_f32(A + m * lda, B + n * ldb, K);", "float v = dot_f32(A + (n % M) * lda, B + (m % N) * ldb, K);", 0),
    ("acc_index", "C[m * ldc + n] = dot_f32(A + m * lda, B + n * ldb, K);", "C[m * ldc + n] = dot_f32(A + m * lda, B + m % N * ldb, K);", 0),
    ("bias_dropped", "if (bias) v = v + bf16_to_f32(bias[n]);", "if (0) v = v + bf16_to_f32(bias[n]);", 0),
    ("bias_index", "if (bias) v = v + bf16_to_f32(bias[n]);", "if (bias) v = v + bf16_to_f32(bias[0]);", 0),
    ("bias_sign", "if (bias) v = v + bf16_to_f32(bias[n]);", "if (bias) v = v - bf16_to_f32(bias[n]);", 0),
    ("residual_index", "if (R) v = v + bf16_to_f32(R[m * ldr + n]);", "if (R) v = v + bf16_to_f32(R[m * ldr]);", 0),
    ("residual_before_act", "            v = act_f32(act, v);\n            if (R) v = v + bf16_to_f32(R[m * ldr + n]);",
     "            if (R) v = v + bf16_to_f32(R[m * ldr + n]);\n            v = act_f32(act, v);", 0),
    ("gelu_cubic_coeff", "const float a = 0.044715f;", "const float a = 0.04715f;", 0),
    ("gelu_sqrt2pi", "const float c = 0.7978845608028654f;", "const float c = 0.7978845608028654f * 1.01f;", 0),
    ("gelu_half", "return 0.5f * x * (1.0f + tanhf(inner));", "return x * (1.0f + tanhf(inner));", 0),
    ("silu_sign", "case ORACLE_ACT_SILU: return x / (1.0f + expf(-x));", "case ORACLE_ACT_SILU: return x / (1.0f + expf(x));", 0),
    ("relu_leaky", "case ORACLE_ACT_RELU: return x > 0.0f ? x : 0.0f;", "case ORACLE_ACT_RELU: return x > 0.0f ? x : 0.01f * x;", 0),
    ("round_truncate", "u += 0x7fffu + lsb;", "u += 0u * lsb;", 0),
    ("round_ties_away", "u += 0x7fffu + lsb;", "u += 0x8000u + 0u * lsb;", 0),
    ("f64_round_precision", "int qexp = e - 8;", "int qexp = e - 9;", 0),
    ("ffn_swap_gate", "float v = act_f32(ORACLE_ACT_SILU, a1) * a3;", "float v = act_f32(ORACLE_ACT_SILU, a3) * a1;", 0),
    ("ffn_same_weight", "float a3 = dot_f32(X + m * ldx, W3 + n * ldw3, K);", "float a3 = dot_f32(X + m * ldx, W1 + n * ldw1, K);", 0),
    ("ffn_f64_swap", "Y[m * ldy + n] = act_f64(ORACLE_ACT_SILU, a1) * a3;", "Y[m * ldy + n] = act_f64(ORACLE_ACT_SILU, a3) * a1;", 0),
    ("preact_after_act", "            Z[m * ldz + n] = f32_to_bf16(v);\n            v = act_f32(act, v);",
     "            v = act_f32(act, v);\n            Z[m * ldz + n] = f32_to_bf16(v);", 0),
    ("preact_no_bias", "            if (bias) v = v + bf16_to_f32(bias[n]);\n            Z[m * ldz + n] = f32_to_bf16(v);",
     "            Z[m * ldz + n] = f32_to_bf16(v);\n            if (bias) v = v + bf16_to_f32(bias[n]);", 0),
    ("f64_dot_drop", "for (int64_t k = 0; k < K; ++k) {\n        double p", "for (int64_t k = 1; k < K; ++k) {\n        double p", 0),
    ("acc_in_double", "    float acc = 0.0f;\n    for (int64_t k = 0; k < K; ++k) {\n        float p",
     "    double acc = 0.0;\n    for (int64_t k = 0; k < K; ++k) {\n        float p", 0),
    ("sum_descending", "for (int64_t k = 0; k < K; ++k) {\n        float p", "for (int64_t k = K - 1; k >= 0; --k) {\n        float p", 0),
    ("lda_ignored", "float v = dot_f32(A + m * lda, B + n * ldb, K);", "float v = dot_f32(A + m * K, B + n * ldb, K);", 0),
    ("ldr_ignored", "if (R) v = v + bf16_to_f32(R[m * ldr + n]);", "if (R) v = v + bf16_to_f32(R[m * N + n]);", 0),
    # activation gradient
    ("dact_w_row_not_column", "float g = dot_f32_strided(dY + m * lddy, W + k, ldw, N);",
     "float g = dot_f32_strided(dY + m * lddy, W + (k % N) * ldw, 1, N < K ? N : K);", 0),
    ("dact_dy_row", "float g = dot_f32_strided(dY + m * lddy, W + k, ldw, N);",
     "float g = dot_f32_strided(dY + (m / 2) * lddy, W + k, ldw, N);", 0),
    ("dact_z_index", "float v = g * dact_f32(act, bf16_to_f32(Z[m * ldz + k]));",
     "float v = g * dact_f32(act, bf16_to_f32(Z[m * ldz]));", 0),
    ("dact_no_derivative", "float v = g * dact_f32(act, bf16_to_f32(Z[m * ldz + k]));",
     "float v = g * act_f32(act, bf16_to_f32(Z[m * ldz + k]));", 0),
    ("dact_strided_drop_last", "for (int64_t k = 0; k < K; ++k) {\n        float p = bf16_to_f32(a[k]) * bf16_to_f32(b[k * stride]);",
     "for (int64_t k = 0; k + 1 < K; ++k) {\n        float p = bf16_to_f32(a[k]) * bf16_to_f32(b[k * stride]);", 0),
    ("dact_sum_in_double", "    float acc = 0.0f;\n    for (int64_t k = 0; k < K; ++k) {\n        float p = bf16_to_f32(a[k]) * bf16_to_f32(b[k * stride]);",
     "    double acc = 0.0;\n    for (int64_t k = 0; k < K; ++k) {\n        float p = bf16_to_f32(a[k]) * bf16_to_f32(b[k * stride]);", 0),
    ("dgelu_half", "return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t)", "return (1.0f + t) + 0.5f * x * (1.0f - t * t)", 0),
    ("dgelu_sech2_sign", "0.5f * x * (1.0f - t * t)", "0.5f * x * (1.0f + t * t)", 0),
    ("dgelu_cubic_factor", "c * (1.0f + 3.0f * a * x * x)", "c * (1.0f + a * x * x)", 0),
    ("dgelu_f64_cubic_factor", "c * (1.0 + 3.0 * a * x * x)", "c * (1.0 + a * x * x)", 0),
    ("dsilu_form", "return sg * (1.0f + x * (1.0f - sg));", "return sg * (1.0f + x * sg);", 0),
    ("dsilu_f64_form", "return sg * (1.0 + x * (1.0 - sg));", "return sg * (1.0 + x * sg);", 0),
    ("drelu_at_zero", "case ORACLE_ACT_RELU: return x > 0.0f ? 1.0f : 0.0f;", "case ORACLE_ACT_RELU: return x >= 0.0f ? 1.0f : 0.0f;", 0),
    ("dnone_zero", "case ORACLE_ACT_NONE: return 1.0f;", "case ORACLE_ACT_NONE: return 0.0f;", 0),
    ("dact_f64_no_derivative", "Y[m * ldy + k] = g * dact_f64(act, (double)bf16_to_f32(Z[m * ldz + k]));",
     "Y[m * ldy + k] = g;", 0),
    # per-entry evaluators
    ("entries_bias_dropped", "if (bias) v = v + bf16_to_f32(bias[p]);", "if (0) v = v + bf16_to_f32(bias[p]);", 0),
    ("entries_residual_before_act", "        v = act_f32(act, v);\n        if (R) v = v + bf16_to_f32(R[p]);",
     "        if (R) v = v + bf16_to_f32(R[p]);\n        v = act_f32(act, v);", 0),
    ("entries_b_row", "float v = dot_f32(A + p * K, B + p * K, K);", "float v = dot_f32(A + p * K, B + (p / 2) * K, K);", 0),
    ("entries_f64_act_dropped", "        v = act_f64(act, v);\n        if (R) v = v + (double)bf16_to_f32(R[p]);",
     "        if (R) v = v + (double)bf16_to_f32(R[p]);", 0),
    ("ffn_entries_swap", "out[p] = f32_to_bf16(act_f32(ORACLE_ACT_SILU, a1) * a3);",
     "out[p] = f32_to_bf16(act_f32(ORACLE_ACT_SILU, a3) * a1);", 0),
    ("ffn_entries_f64_swap", "out[p] = act_f64(ORACLE_ACT_SILU, a1) * a3;", "out[p] = act_f64(ORACLE_ACT_SILU, a3) * a1;", 0),
    ("dact_entries_z_ignored", "out[p] = f32_to_bf16(g * dact_f32(act, bf16_to_f32(Z[p])));", "out[p] = f32_to_bf16(g);", 0),
    ("dact_entries_f64_z_ignored", "out[p] = g * dact_f64(act, (double)bf16_to_f32(Z[p]));", "out[p] = g;", 0),
]


def _replace_nth(text: str, old: str, new: str, n: int) -> str:
    idx = -1
    for _ in range(n + 1):
        idx = text.index(old, idx + 1)
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, nth):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} no longer matches oracle.c"
    mutant_src = tmp_path / f"oracle_{name}.c"
    mutant_src.write_text(_replace_nth(src, old, new, nth))
    so = oracle.build_library(str(mutant_src), str(tmp_path / f"liboracle_{name}.so"), force=True)
    mut = oracle.Oracle(so)
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mut)
        except AssertionError:
            failures.append(check.__name__)
    assert failures, f"planted mistake {name!r} passed every oracle pin"


def test_unmutated_copy_passes(tmp_path):
    """The harness itself: an unmodified copy builds and passes every pin."""
    dst = tmp_path / "oracle_copy.c"
    shutil.copy(SRC, dst)
    mut = oracle.Oracle(oracle.build_library(str(dst), str(tmp_path / "liboracle_copy.so"), force=True))
    for check in oracle_pins.ALL_CHECKS:
        check(mut)
