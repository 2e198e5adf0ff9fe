"""Write the small golden fixtures under tests/golden/ (inputs and expected outputs).

The pages this library follows print no worked example and no numeric output, so
every stored expected value here is written by this script, which calls only the
CPU oracle (``oracle/``).  The fixtures freeze the oracle's results on small
seeded inputs: a later change to the oracle's arithmetic shows up as a diff of
these files, and the GPU tests compare the CUDA path against the same values.

Usage:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def _bf16(rng, shape, std):
    return oracle.f32_to_bf16((rng.standard_normal(shape) * std).astype(np.float32))


def _write(path, header, arrays):
    with open(path, "w") as f:
        for line in header:
            f.write(f"# {line}\n")
        for name, a in arrays:
            a = np.atleast_2d(a) if a.ndim == 1 else a
            f.write(f"{name} {a.shape[0]} {a.shape[1]}\n")
            for row in a:
                f.write(" ".join(f"{int(v):04x}" for v in row) + "\n")


def main():
    common = ["bf16 values as 16-bit hex patterns, row-major",
              "expected D written by tests/golden/make_golden.py from the CPU oracle (oracle/oracle.c);",
              "the source pages print no numbers for this operation"]
    rng = np.random.default_rng(2024)
    # linear + bias + GELU-tanh, ragged sizes
    M, N, K = 5, 7, 40
    A, B, bias = _bf16(rng, (M, K), 1.0), _bf16(rng, (N, K), 0.2), _bf16(rng, (N,), 0.2)
    D = oracle.linear(A, B, bias=bias, act="gelu_tanh")
    _write(os.path.join(HERE, "linear_bias_gelu_5x7x40.txt"),
           ["D = bf16(gelu_tanh(A.B^T + bias)), fp32 accumulate"] + common,
           [("A", A), ("B", B), ("bias", bias), ("D", D)])
    # linear + residual (epilogue input), no activation
    M, N, K = 3, 9, 24
    A, B, R = _bf16(rng, (M, K), 1.0), _bf16(rng, (N, K), 0.2), _bf16(rng, (M, N), 1.0)
    D = oracle.linear(A, B, R=R)
    _write(os.path.join(HERE, "linear_residual_3x9x24.txt"),
           ["D = bf16(A.B^T + R), fp32 accumulate"] + common,
           [("A", A), ("B", B), ("R", R), ("D", D)])
    # bias + SiLU + residual
    M, N, K = 4, 5, 16
    A, B = _bf16(rng, (M, K), 1.0), _bf16(rng, (N, K), 0.3)
    bias, R = _bf16(rng, (N,), 0.3), _bf16(rng, (M, N), 1.0)
    D = oracle.linear(A, B, bias=bias, R=R, act="silu")
    _write(os.path.join(HERE, "linear_bias_silu_residual_4x5x16.txt"),
           ["D = bf16(silu(A.B^T + bias) + R), fp32 accumulate"] + common,
           [("A", A), ("B", B), ("bias", bias), ("R", R), ("D", D)])
    # Llama-FFN horizontal fusion
    M, N, K = 4, 6, 32
    X, W1, W3 = _bf16(rng, (M, K), 1.0), _bf16(rng, (N, K), 0.2), _bf16(rng, (N, K), 0.2)
    D = oracle.ffn_gated(X, W1, W3)
    _write(os.path.join(HERE, "ffn_gated_4x6x32.txt"),
           ["D = bf16(silu(X.W1^T) * (X.W3^T)), both products fp32-accumulated"] + common,
           [("X", X), ("W1", W1), ("W3", W3), ("D", D)])


if __name__ == "__main__":
    main()
