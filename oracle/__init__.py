"""CPU oracle for the bf16 GEMM + fused epilogue (ctypes wrapper over ``oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` are the only callers.  The package
``dense_bf16_gemm_persistent_gb300`` never imports this module, and this module
never imports the package: the two share no code.

Arrays cross this boundary as numpy ``uint16`` bf16 bit patterns, row-major,
last dimension contiguous.  See ``oracle.c`` for the definitions (plain fp32
sum in ascending k with no FMA, fp32 epilogue, one round-to-nearest-even to
bf16) and the readings taken where the source pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ACT = {"none": 0, "gelu_tanh": 1, "silu": 2, "relu": 3}

_lock = threading.Lock()
_default = None


def build_library(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile an oracle C source with gcc (-O2, OpenMP, no FP contraction)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _mat(x, name: str) -> tuple[int, int]:
    """Return (pointer, leading dimension in elements) of a bf16 bit-pattern matrix."""
    if x is None:
        return 0, 0
    if x.dtype != np.uint16:
        raise TypeError(f"{name}: expected uint16 bf16 bit patterns, got {x.dtype}")
    if x.size == 0:
        return x.ctypes.data, x.shape[-1]
    if x.ndim == 1:
        if x.strides[0] != 2:
            raise ValueError(f"{name}: vector must be contiguous")
        return x.ctypes.data, x.shape[0]
    if x.ndim != 2 or x.strides[1] != 2 or x.strides[0] % 2:
        raise ValueError(f"{name}: expected a 2-D row-major matrix with a contiguous last dim")
    return x.ctypes.data, max(x.strides[0] // 2, x.shape[1])


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test's mutant)."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_linear_f32.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, i64, i64, i64]
        lib.oracle_linear_f64.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, i64, i64, i64]
        lib.oracle_linear_preact_f32.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, p, i64,
                                                 i64, i64, i64]
        lib.oracle_ffn_f32.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64]
        lib.oracle_ffn_f64.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64]
        lib.oracle_acc_f32.argtypes = [p, i64, p, i64, p, i64, i64, i64, i64]
        lib.oracle_act_f32_array.argtypes = [ctypes.c_int, p, p, i64]
        lib.oracle_act_f64_array.argtypes = [ctypes.c_int, p, p, i64]
        lib.oracle_f32_to_bf16_array.argtypes = [p, p, i64]
        lib.oracle_f64_to_bf16_array.argtypes = [p, p, i64]
        lib.oracle_dact_f32.argtypes = [p, i64, p, i64, p, i64, ctypes.c_int, p, i64, i64, i64, i64]
        lib.oracle_dact_f64.argtypes = [p, i64, p, i64, p, i64, ctypes.c_int, p, i64, i64, i64, i64]
        lib.oracle_dact_f32_array.argtypes = [ctypes.c_int, p, p, i64]
        lib.oracle_dact_f64_array.argtypes = [ctypes.c_int, p, p, i64]
        lib.oracle_linear_entries_f32.argtypes = [p, p, i64, p, p, ctypes.c_int, p, i64]
        lib.oracle_linear_entries_f64.argtypes = [p, p, i64, p, p, ctypes.c_int, p, i64]
        lib.oracle_ffn_entries_f32.argtypes = [p, p, p, i64, p, i64]
        lib.oracle_ffn_entries_f64.argtypes = [p, p, p, i64, p, i64]
        lib.oracle_dact_entries_f32.argtypes = [p, p, i64, p, ctypes.c_int, p, i64]
        lib.oracle_dact_entries_f64.argtypes = [p, p, i64, p, ctypes.c_int, p, i64]
        lib.oracle_num_threads.restype = ctypes.c_int
        for name in ("oracle_linear_f32", "oracle_linear_f64", "oracle_linear_preact_f32", "oracle_ffn_f32",
                     "oracle_ffn_f64", "oracle_dact_f32", "oracle_dact_f64",
                     "oracle_acc_f32", "oracle_act_f32_array", "oracle_act_f64_array",
                     "oracle_dact_f32_array", "oracle_dact_f64_array",
                     "oracle_linear_entries_f32", "oracle_linear_entries_f64", "oracle_ffn_entries_f32",
                     "oracle_ffn_entries_f64", "oracle_dact_entries_f32", "oracle_dact_entries_f64",
                     "oracle_f32_to_bf16_array", "oracle_f64_to_bf16_array"):
            getattr(lib, name).restype = None
        self.lib = lib
        self.path = so_path

    @staticmethod
    def _dims(A, B):
        M, K = A.shape
        N = B.shape[0]
        if B.ndim != 2 or B.shape[1] != K:
            raise ValueError("inner dimensions differ")
        return M, N, K

    def linear(self, A, B, bias=None, R=None, act: str = "none"):
        """D[M,N] = bf16( act(A.B^T + bias) + R ), fp32 arithmetic; bf16 bits out."""
        M, N, K = self._dims(A, B)
        if bias is not None and bias.shape != (N,):
            raise ValueError("bias must have shape (N,)")
        if R is not None and R.shape != (M, N):
            raise ValueError("R must have shape (M, N)")
        D = np.empty((M, N), dtype=np.uint16)
        pa, lda = _mat(A, "A")
        pb, ldb = _mat(B, "B")
        pbias, _ = _mat(bias, "bias")
        pr, ldr = _mat(R, "R")
        self.lib.oracle_linear_f32(pa, lda, pb, ldb, pbias, pr, ldr, ACT[act], D.ctypes.data, N, M, N, K)
        return D

    def matmul(self, A, B, bias=None, R=None, act: str = "none"):
        """D[M,N] = bf16( act(A.B + bias) + R ) with B given as [K,N] (the MatmulOp form of
        "Translate MmaOp patterns properly on Hopper", description).  By definition A.B =
        A.(B^T)^T: the same sum over k in the same order as linear() on B^T, so B is
        transposed (a copy) and linear() evaluates it."""
        Bt = np.ascontiguousarray(np.asarray(B).T)
        return self.linear(A, Bt, bias, R, act)

    def linear_preact(self, A, B, bias=None, R=None, act: str = "none"):
        """(D, Z): D as in linear(), Z[M,N] = bf16(A.B^T + bias), the pre-activation."""
        M, N, K = self._dims(A, B)
        D = np.empty((M, N), dtype=np.uint16)
        Z = np.empty((M, N), dtype=np.uint16)
        pa, lda = _mat(A, "A")
        pb, ldb = _mat(B, "B")
        pbias, _ = _mat(bias, "bias")
        pr, ldr = _mat(R, "R")
        self.lib.oracle_linear_preact_f32(pa, lda, pb, ldb, pbias, pr, ldr, ACT[act], D.ctypes.data, N,
                                          Z.ctypes.data, N, M, N, K)
        return D, Z

    def linear_f64(self, A, B, bias=None, R=None, act: str = "none"):
        """The same expression in float64, unrounded (diagnostic / error bounds)."""
        M, N, K = self._dims(A, B)
        Y = np.empty((M, N), dtype=np.float64)
        pa, lda = _mat(A, "A")
        pb, ldb = _mat(B, "B")
        pbias, _ = _mat(bias, "bias")
        pr, ldr = _mat(R, "R")
        self.lib.oracle_linear_f64(pa, lda, pb, ldb, pbias, pr, ldr, ACT[act], Y.ctypes.data, N, M, N, K)
        return Y

    def ffn_gated(self, X, W1, W3):
        """D[M,N] = bf16( silu(X.W1^T) * (X.W3^T) ), fp32 arithmetic; bf16 bits out."""
        M, N, K = self._dims(X, W1)
        if W3.shape != W1.shape:
            raise ValueError("W1 and W3 must have the same shape")
        D = np.empty((M, N), dtype=np.uint16)
        px, ldx = _mat(X, "X")
        p1, ld1 = _mat(W1, "W1")
        p3, ld3 = _mat(W3, "W3")
        self.lib.oracle_ffn_f32(px, ldx, p1, ld1, p3, ld3, D.ctypes.data, N, M, N, K)
        return D

    def ffn_gated_f64(self, X, W1, W3):
        M, N, K = self._dims(X, W1)
        Y = np.empty((M, N), dtype=np.float64)
        px, ldx = _mat(X, "X")
        p1, ld1 = _mat(W1, "W1")
        p3, ld3 = _mat(W3, "W3")
        self.lib.oracle_ffn_f64(px, ldx, p1, ld1, p3, ld3, Y.ctypes.data, N, M, N, K)
        return Y

    def dact(self, dY, W, Z, act: str = "none"):
        """D[M,K] = bf16( (dY.W) * act'(Z) ): dY [M,N], W [N,K] (the forward weight), Z [M,K];
        the fp32 sum runs over n in ascending order; bf16 bits out."""
        M, N = dY.shape
        if W.ndim != 2 or W.shape[0] != N:
            raise ValueError("W must have shape (N, K)")
        K = W.shape[1]
        if Z.shape != (M, K):
            raise ValueError("Z must have shape (M, K)")
        D = np.empty((M, K), dtype=np.uint16)
        py, ldy = _mat(dY, "dY")
        pw, ldw = _mat(W, "W")
        pz, ldz = _mat(Z, "Z")
        self.lib.oracle_dact_f32(py, ldy, pw, ldw, pz, ldz, ACT[act], D.ctypes.data, K, M, N, K)
        return D

    def dact_f64(self, dY, W, Z, act: str = "none"):
        M, N = dY.shape
        K = W.shape[1]
        if W.shape[0] != N or Z.shape != (M, K):
            raise ValueError("shapes: dY (M,N), W (N,K), Z (M,K)")
        Y = np.empty((M, K), dtype=np.float64)
        py, ldy = _mat(dY, "dY")
        pw, ldw = _mat(W, "W")
        pz, ldz = _mat(Z, "Z")
        self.lib.oracle_dact_f64(py, ldy, pw, ldw, pz, ldz, ACT[act], Y.ctypes.data, K, M, N, K)
        return Y

    @staticmethod
    def _rows(x, name, P=None, K=None):
        x = np.ascontiguousarray(x, dtype=np.uint16)
        if x.ndim != 2 or (P is not None and x.shape[0] != P) or (K is not None and x.shape[1] != K):
            raise ValueError(f"{name}: expected shape ({P}, {K}), got {x.shape}")
        return x

    @staticmethod
    def _vals(x, name, P):
        if x is None:
            return None, 0
        x = np.ascontiguousarray(x, dtype=np.uint16)
        if x.shape != (P,):
            raise ValueError(f"{name}: expected shape ({P},)")
        return x, x.ctypes.data

    def linear_entries(self, Arows, Brows, bias=None, R=None, act: str = "none", f64: bool = False):
        """Single entries of linear(): entry p = row p of Arows with row p of Brows, plus the
        entry's bias and R values (each of shape (P,), or None)."""
        A = self._rows(Arows, "Arows")
        P, K = A.shape
        B = self._rows(Brows, "Brows", P, K)
        bias, pbias = self._vals(bias, "bias", P)
        R, pr = self._vals(R, "R", P)
        out = np.empty(P, dtype=np.float64 if f64 else np.uint16)
        fn = self.lib.oracle_linear_entries_f64 if f64 else self.lib.oracle_linear_entries_f32
        fn(A.ctypes.data, B.ctypes.data, K, pbias, pr, ACT[act], out.ctypes.data, P)
        return out

    def ffn_entries(self, Xrows, W1rows, W3rows, f64: bool = False):
        X = self._rows(Xrows, "Xrows")
        P, K = X.shape
        W1 = self._rows(W1rows, "W1rows", P, K)
        W3 = self._rows(W3rows, "W3rows", P, K)
        out = np.empty(P, dtype=np.float64 if f64 else np.uint16)
        fn = self.lib.oracle_ffn_entries_f64 if f64 else self.lib.oracle_ffn_entries_f32
        fn(X.ctypes.data, W1.ctypes.data, W3.ctypes.data, K, out.ctypes.data, P)
        return out

    def dact_entries(self, dYrows, Wcols, Z, act: str = "none", f64: bool = False):
        """Single entries of dact(): entry p = row p of dYrows with column p of W gathered as
        row p of Wcols (both length N), times act' of the entry's Z value (shape (P,))."""
        Y = self._rows(dYrows, "dYrows")
        P, N = Y.shape
        W = self._rows(Wcols, "Wcols", P, N)
        Z, pz = self._vals(Z, "Z", P)
        if Z is None:
            raise ValueError("Z is required")
        out = np.empty(P, dtype=np.float64 if f64 else np.uint16)
        fn = self.lib.oracle_dact_entries_f64 if f64 else self.lib.oracle_dact_entries_f32
        fn(Y.ctypes.data, W.ctypes.data, N, pz, ACT[act], out.ctypes.data, P)
        return out

    def acc_f32(self, A, B):
        """Raw fp32 accumulator A.B^T (ascending k, no FMA), no epilogue."""
        M, N, K = self._dims(A, B)
        C = np.empty((M, N), dtype=np.float32)
        pa, lda = _mat(A, "A")
        pb, ldb = _mat(B, "B")
        self.lib.oracle_acc_f32(pa, lda, pb, ldb, C.ctypes.data, N, M, N, K)
        return C

    def act_f32(self, act: str, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty_like(x)
        self.lib.oracle_act_f32_array(ACT[act], x.ctypes.data, y.ctypes.data, x.size)
        return y

    def act_f64(self, act: str, x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.empty_like(x)
        self.lib.oracle_act_f64_array(ACT[act], x.ctypes.data, y.ctypes.data, x.size)
        return y

    def dact_f32_values(self, act: str, x):
        """act'(x) in fp32 (the derivative the dact epilogue multiplies by)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty_like(x)
        self.lib.oracle_dact_f32_array(ACT[act], x.ctypes.data, y.ctypes.data, x.size)
        return y

    def dact_f64_values(self, act: str, x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.empty_like(x)
        self.lib.oracle_dact_f64_array(ACT[act], x.ctypes.data, y.ctypes.data, x.size)
        return y

    def f32_to_bf16(self, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f32_to_bf16_array(x.ctypes.data, y.ctypes.data, x.size)
        return y

    def f64_to_bf16(self, x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f64_to_bf16_array(x.ctypes.data, y.ctypes.data, x.size)
        return y

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())


def default() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build_library())
        return _default


def linear(A, B, bias=None, R=None, act: str = "none"):
    return default().linear(A, B, bias, R, act)


def matmul(A, B, bias=None, R=None, act: str = "none"):
    return default().matmul(A, B, bias, R, act)


def linear_f64(A, B, bias=None, R=None, act: str = "none"):
    return default().linear_f64(A, B, bias, R, act)


def linear_preact(A, B, bias=None, R=None, act: str = "none"):
    return default().linear_preact(A, B, bias, R, act)


def ffn_gated(X, W1, W3):
    return default().ffn_gated(X, W1, W3)


def ffn_gated_f64(X, W1, W3):
    return default().ffn_gated_f64(X, W1, W3)


def dact(dY, W, Z, act: str = "none"):
    return default().dact(dY, W, Z, act)


def dact_f64(dY, W, Z, act: str = "none"):
    return default().dact_f64(dY, W, Z, act)


def linear_entries(Arows, Brows, bias=None, R=None, act: str = "none", f64: bool = False):
    return default().linear_entries(Arows, Brows, bias, R, act, f64)


def ffn_entries(Xrows, W1rows, W3rows, f64: bool = False):
    return default().ffn_entries(Xrows, W1rows, W3rows, f64)


def dact_entries(dYrows, Wcols, Z, act: str = "none", f64: bool = False):
    return default().dact_entries(dYrows, Wcols, Z, act, f64)


def acc_f32(A, B):
    return default().acc_f32(A, B)


def act_f32(act: str, x):
    return default().act_f32(act, x)


def act_f64(act: str, x):
    return default().act_f64(act, x)


def f32_to_bf16(x):
    return default().f32_to_bf16(x)


def f64_to_bf16(x):
    return default().f64_to_bf16(x)


def num_threads() -> int:
    return default().num_threads()


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a bit shift, no arithmetic)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    return (x.astype(np.uint32) << 16).view(np.float32)

