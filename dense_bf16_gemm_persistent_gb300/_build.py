"""Compile the CUDA library (libgbgemm.so) in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libgbgemm.so")
LOG_DIR = os.path.join(PKG, "_build")
SOURCES = ["gbgemm.cu"]
HEADERS = ["gemm_kernel.cuh", "ptx.cuh", "probe.cuh"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-Xptxas", "-v",
              "--diag-suppress", "177"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "gbgemm.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def _check_register_budgets(log: str) -> None:
    """Refuse a build whose kernels could block forever in setmaxnreg.inc: for every
    kernel with two epilogue warpgroups (384 threads), the launch register count
    times the threads must cover the budgets the warpgroups lower and raise to
    (constants of WarpLayout in gemm_kernel.cuh)."""
    import re
    src = open(os.path.join(CSRC, "gemm_kernel.cuh")).read()

    def const(name):
        return int(re.search(rf"static constexpr int {name} = (\d+);", src).group(1))

    control, epilogue = const("kRegsControl"), const("kRegsEpilogue")
    entries = re.findall(r"Compiling entry function '(\w+)'.*?Used (\d+) registers", log, flags=re.S)
    if not entries:
        raise RuntimeError("no kernels in the ptxas report")
    for name, regs in entries:
        if "gemm_persistent_kernel" not in name:
            continue
        m = re.search(r"Li(\d+)EEEv", name)  # the last template argument: epilogue warpgroups
        epi = int(m.group(1)) if m else 1
        if epi != 2:
            continue
        threads, need = 384, 128 * control + 256 * epilogue
        if int(regs) * threads < need:
            raise RuntimeError(f"{name} launches with {regs} registers/thread x {threads} threads, less than "
                               f"the {need} its warpgroup register budgets need")


TRACE_LIB = os.path.join(PKG, "libgbgemm_trace.so")


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Build libgbgemm.so next to this file; the -Xptxas -v report goes to _build/ptxas.log.
    trace=True builds the instrumented libgbgemm_trace.so instead (-DGB_TRACE: the kernels
    record where each role waited; see gb_set_trace_buffer)."""
    out = TRACE_LIB if trace else LIB
    if not force and not _stale(out):
        return out
    os.makedirs(LOG_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *NVCC_FLAGS, *(["-DGB_TRACE"] if trace else []), "-shared", "-o", tmp,
           *[os.path.join(CSRC, s) for s in SOURCES]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(LOG_DIR, "ptxas_trace.log" if trace else "ptxas.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stderr[-4000:]}")
    _check_register_budgets(res.stdout + res.stderr)
    if verbose:
        print(res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
