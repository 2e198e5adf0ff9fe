"""Golden fixtures: small inputs and expected outputs as text (see make_golden.py)."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name: str) -> dict:
    """Parse one fixture file into {array name: uint16 numpy array}."""
    out = {}
    with open(os.path.join(HERE, name)) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    i = 0
    while i < len(lines):
        key, r, c = lines[i].split()
        r, c = int(r), int(c)
        rows = [[int(v, 16) for v in lines[i + 1 + j].split()] for j in range(r)]
        out[key] = np.array(rows, dtype=np.uint16).reshape(r, c)
        i += 1 + r
    if "bias" in out:
        out["bias"] = out["bias"].reshape(-1)
    return out


FIXTURES = ["linear_bias_gelu_5x7x40.txt", "linear_residual_3x9x24.txt",
            "linear_bias_silu_residual_4x5x16.txt", "ffn_gated_4x6x32.txt"]
