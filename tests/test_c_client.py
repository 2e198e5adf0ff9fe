"""The C ABI from plain C: tests/c_client/gemm_client.c compiles against
include/gbgemm.h as C99 and links against libgbgemm.so and the CUDA runtime (CPU);
on a GPU it runs one linear call (bias, GELU-tanh, epilogue input) whose output
matches the oracle, and a call the library rejects."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "gemm_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir) -> str:
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    from dense_bf16_gemm_persistent_gb300 import _build
    lib = _build.build()
    lib_dir = os.path.dirname(lib)
    exe = os.path.join(str(out_dir), "gemm_client")
    cmd = [gcc, "-std=c99", "-Wall", "-Werror", "-O2", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-L", lib_dir, "-lgbgemm", "-L", os.path.join(CUDA, "lib64"),
           "-lcudart", f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_c_client_runs(tmp_path):
    import oracle
    from dense_bf16_gemm_persistent_gb300 import inputs
    exe = _compile(tmp_path)
    M, N, K = 300, 520, 256
    t = {"A": inputs.randn_bf16((M, K), seed=190), "B": inputs.randn_bf16((N, K), seed=191, std=1.0 / 16),
         "bias": inputs.randn_bf16((N,), seed=192, std=0.1), "R": inputs.randn_bf16((M, N), seed=193)}
    bits = {k: inputs.to_bits(v) for k, v in t.items()}
    for k, v in bits.items():
        np.ascontiguousarray(v).tofile(os.path.join(str(tmp_path), f"{k}.bin"))
    r = subprocess.run([exe, str(tmp_path), str(M), str(N), str(K)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr + r.stdout
    D = np.fromfile(os.path.join(str(tmp_path), "D.bin"), dtype=np.uint16).reshape(M, N)
    from tests.gpu_util import assert_close
    assert_close(D, oracle.linear(bits["A"], bits["B"], bits["bias"], bits["R"], "gelu_tanh"), "C client")
