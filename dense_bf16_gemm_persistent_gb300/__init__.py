"""Python binding of gbgemm: persistent tcgen05 bf16 GEMM with a fused epilogue (GB300, sm_103a).

Argument marshalling only.  Every step of the computation runs in the CUDA
library ``libgbgemm.so`` through its C ABI (``include/gbgemm.h``); there is no
fallback of any kind, and every call raises if the library is missing.

    linear(A, B, bias=None, R=None, act="none")  ->  bf16(act(A @ B.T + bias) + R)
    ffn_gated(X, W1, W3)                         ->  bf16(silu(X @ W1.T) * (X @ W3.T))
    linear_dact(dY, W, Z, act="none")            ->  bf16((dY @ W) * act'(Z))

Tensors are torch CUDA bf16 tensors, 2-D with a contiguous last dimension
(bias: contiguous 1-D).  Work is enqueued on ``torch.cuda.current_stream()``
unless a stream is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# GBGEMM_TRACE=1 loads the instrumented build (libgbgemm_trace.so, see gb_set_trace_buffer)
LIB_PATH = os.path.join(_PKG, "libgbgemm_trace.so" if os.environ.get("GBGEMM_TRACE") == "1" else "libgbgemm.so")

ACT = {"none": 0, "gelu_tanh": 1, "silu": 2, "relu": 3}
STATUS = {0: "GB_OK", 1: "GB_ERR_INVALID_ARG", 2: "GB_ERR_UNSUPPORTED", 3: "GB_ERR_CUDA", 4: "GB_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class GBError(RuntimeError):
    """A non-OK gb_status_t, with the library's message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libgbgemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"the CUDA library {LIB_PATH} is not built; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(LIB_PATH)
        i64, p, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.gb_gemm_linear.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, i64, i64, i64, p]
        L.gb_gemm_ffn_gated.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64, p]
        L.gb_gemm_linear_preact.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, p, i64, i64, i64, i64,
                                            p]
        L.gb_gemm_linear_dact.argtypes = [p, i64, p, i64, p, i64, ctypes.c_int, p, i64, i64, i64, i64, p]
        L.gb_gemm_matmul.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, i64, i64, i64, p]
        L.gb_gemm_linear_splitk.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, i64, i64, i64,
                                             ctypes.c_int, p, ctypes.c_size_t, p]
        L.gb_gemm_ffn_gated_splitk.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64, i64, ctypes.c_int, p,
                                               ctypes.c_size_t, p]
        L.gb_splitk_workspace_bytes.argtypes = [ctypes.c_int, i64, i64, i64, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_size_t)]
        L.gb_gemm_linear_splitk_noalloc.argtypes = [p, i64, p, i64, p, p, i64, ctypes.c_int, p, i64, i64, i64,
                                                     i64, ctypes.c_int, p]
        L.gb_static_scratch_bytes.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
        L.gb_get_device_status.argtypes = [p]
        L.gb_last_error.argtypes = []
        L.gb_last_error.restype = ctypes.c_char_p
        L.gb_set_config.argtypes = [ctypes.c_char_p]
        L.gb_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        L.gb_set_fault_injection.argtypes = [ctypes.c_int]
        L.gb_last_plan.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
        L.gb_set_trace_buffer.argtypes = [p, ctypes.c_size_t]
        L.gb_measure_mma_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        L.gb_probe_mma_issue.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_double)]
        L.gb_version.argtypes = []
        L.gb_version.restype = ctypes.c_char_p
        for name in ("gb_gemm_linear", "gb_gemm_ffn_gated", "gb_gemm_linear_preact", "gb_gemm_linear_dact",
                     "gb_gemm_matmul",
                     "gb_gemm_linear_splitk",
                     "gb_gemm_ffn_gated_splitk",
                     "gb_splitk_workspace_bytes", "gb_gemm_linear_splitk_noalloc", "gb_static_scratch_bytes",
                     "gb_get_device_status", "gb_set_config",
                     "gb_set_wait_timeout_ns", "gb_set_fault_injection", "gb_last_plan", "gb_set_trace_buffer",
                     "gb_measure_mma_rate", "gb_probe_mma_issue"):
            getattr(L, name).restype = st
        _lib = L
        return L


def _check(status: int) -> None:
    if status != 0:
        raise GBError(status, lib().gb_last_error().decode(errors="replace"))


def _mat(t: torch.Tensor | None, name: str, rows: int | None = None, cols: int | None = None):
    """(pointer, leading dimension in elements) of a 2-D bf16 CUDA tensor."""
    if t is None:
        return None, 0
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA bfloat16 tensor, got {t.dtype} on {t.device}")
    shape, stride = t.shape, t.stride()  # (each attribute read costs host time on small calls)
    if len(shape) != 2 or (shape[1] > 1 and stride[1] != 1):
        raise ValueError(f"{name}: expected a 2-D tensor with a contiguous last dimension")
    r, c = shape
    if rows is not None and r != rows or cols is not None and c != cols:
        raise ValueError(f"{name}: shape {tuple(shape)} does not match ({rows}, {cols})")
    # one row: its stride is arbitrary; keep a real row pitch (e.g. of a padded buffer's
    # view) when there is one, else the width
    ld = stride[0] if r > 1 or stride[0] >= c else max(c, 1)
    return t.data_ptr(), max(ld, 1)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def splitk_workspace_bytes(M: int, N: int, K: int, splits: int = 0, ffn: bool = False) -> int:
    """Bytes of workspace the split-K call needs on the current device (0: no split)."""
    n = ctypes.c_size_t(0)
    _check(lib().gb_splitk_workspace_bytes(1 if ffn else 0, M, N, K, int(splits), ctypes.byref(n)))
    return int(n.value)


def _workspace(split_k, workspace, M, N, K, ffn, device):
    splits = 0 if split_k == "auto" else int(split_k)
    need = splitk_workspace_bytes(M, N, K, splits, ffn)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, {need} needed")
    return splits, workspace


def linear(A: torch.Tensor, B: torch.Tensor, bias: torch.Tensor | None = None, R: torch.Tensor | None = None,
           act: str = "none", out: torch.Tensor | None = None, stream=None, split_k=None,
           workspace: torch.Tensor | None = None) -> torch.Tensor:
    """D = bf16(act(A @ B.T + bias) + R) on the GPU (A [M,K], B [N,K], bias [N], R [M,N]).

    split_k: None (never split), "auto", or a number of K ranges; the fp32 partials
    go to `workspace` (a CUDA tensor, allocated here when not given)."""
    M, K = A.shape
    N = B.shape[0]
    if act not in ACT:
        raise ValueError(f"act must be one of {sorted(ACT)}")
    pa, lda = _mat(A, "A", M, K)
    pb, ldb = _mat(B, "B", N, K)
    pr, ldr = _mat(R, "R", M, N)
    if bias is not None:
        if bias.dtype != torch.bfloat16 or not bias.is_cuda or bias.shape != (N,) or (N > 1 and bias.stride(0) != 1):
            raise ValueError("bias: expected a contiguous CUDA bfloat16 tensor of shape (N,)")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    pd, ldd = _mat(out, "out", M, N)
    pbias = bias.data_ptr() if bias is not None else None
    if split_k is None:
        _check(lib().gb_gemm_linear(pa, lda, pb, ldb, pbias, pr, ldr, ACT[act], pd, ldd, M, N, K, _stream(stream)))
    else:
        splits, ws = _workspace(split_k, workspace, M, N, K, False, A.device)
        _check(lib().gb_gemm_linear_splitk(pa, lda, pb, ldb, pbias, pr, ldr, ACT[act], pd, ldd, M, N, K, splits,
                                           ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)))
    return out


def linear_preact(A: torch.Tensor, B: torch.Tensor, bias: torch.Tensor | None = None, R: torch.Tensor | None = None,
                  act: str = "none", out: torch.Tensor | None = None, preact: torch.Tensor | None = None,
                  stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """(D, Z): D as linear(), Z = bf16(A @ B.T + bias), the pre-activation, from the same pass."""
    M, K = A.shape
    N = B.shape[0]
    if act not in ACT:
        raise ValueError(f"act must be one of {sorted(ACT)}")
    pa, lda = _mat(A, "A", M, K)
    pb, ldb = _mat(B, "B", N, K)
    pr, ldr = _mat(R, "R", M, N)
    if bias is not None:
        if bias.dtype != torch.bfloat16 or not bias.is_cuda or bias.shape != (N,) or (N > 1 and bias.stride(0) != 1):
            raise ValueError("bias: expected a contiguous CUDA bfloat16 tensor of shape (N,)")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if preact is None:
        preact = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    pd, ldd = _mat(out, "out", M, N)
    pz, ldz = _mat(preact, "preact", M, N)
    _check(lib().gb_gemm_linear_preact(pa, lda, pb, ldb, bias.data_ptr() if bias is not None else None, pr, ldr,
                                       ACT[act], pd, ldd, pz, ldz, M, N, K, _stream(stream)))
    return out, preact


def matmul(A: torch.Tensor, B: torch.Tensor, bias: torch.Tensor | None = None, R: torch.Tensor | None = None,
           act: str = "none", out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D = bf16(act(A @ B + bias) + R) on the GPU with B in its [K,N] layout (A [M,K], B [K,N],
    bias [N], R [M,N])."""
    M, K = A.shape
    N = B.shape[1]
    if act not in ACT:
        raise ValueError(f"act must be one of {sorted(ACT)}")
    pa, lda = _mat(A, "A", M, K)
    pb, ldb = _mat(B, "B", K, N)
    pr, ldr = _mat(R, "R", M, N)
    if bias is not None:
        if bias.dtype != torch.bfloat16 or not bias.is_cuda or bias.shape != (N,) or (N > 1 and bias.stride(0) != 1):
            raise ValueError("bias: expected a contiguous CUDA bfloat16 tensor of shape (N,)")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    pd, ldd = _mat(out, "out", M, N)
    _check(lib().gb_gemm_matmul(pa, lda, pb, ldb, bias.data_ptr() if bias is not None else None, pr, ldr, ACT[act],
                                pd, ldd, M, N, K, _stream(stream)))
    return out


def linear_dact(dY: torch.Tensor, W: torch.Tensor, Z: torch.Tensor, act: str = "none",
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D = bf16((dY @ W) * act'(Z)) on the GPU: dY [M,N], W [N,K] (the layer's weight as linear()
    takes it), Z [M,K] (the stored pre-activation); D [M,K]."""
    M, N = dY.shape
    K = W.shape[1]
    if act not in ACT:
        raise ValueError(f"act must be one of {sorted(ACT)}")
    py, ldy = _mat(dY, "dY", M, N)
    pw, ldw = _mat(W, "W", N, K)
    pz, ldz = _mat(Z, "Z", M, K)
    if out is None:
        out = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device)
    pd, ldd = _mat(out, "out", M, K)
    _check(lib().gb_gemm_linear_dact(py, ldy, pw, ldw, pz, ldz, ACT[act], pd, ldd, M, N, K, _stream(stream)))
    return out


def ffn_gated(X: torch.Tensor, W1: torch.Tensor, W3: torch.Tensor, out: torch.Tensor | None = None,
              stream=None, split_k=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """D = bf16(silu(X @ W1.T) * (X @ W3.T)) on the GPU (X [M,K], W1/W3 [N,K]); split_k as in linear()."""
    M, K = X.shape
    N = W1.shape[0]
    px, ldx = _mat(X, "X", M, K)
    p1, ld1 = _mat(W1, "W1", N, K)
    p3, ld3 = _mat(W3, "W3", N, K)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    pd, ldd = _mat(out, "out", M, N)
    if split_k is None:
        _check(lib().gb_gemm_ffn_gated(px, ldx, p1, ld1, p3, ld3, pd, ldd, M, N, K, _stream(stream)))
    else:
        splits, ws = _workspace(split_k, workspace, M, N, K, True, X.device)
        _check(lib().gb_gemm_ffn_gated_splitk(px, ldx, p1, ld1, p3, ld3, pd, ldd, M, N, K, splits, ws.data_ptr(),
                                              ws.numel() * ws.element_size(), _stream(stream)))
    return out


def device_status(stream=None) -> None:
    """Synchronise the stream and raise GBError if a kernel recorded a device-side fault."""
    _check(lib().gb_get_device_status(_stream(stream)))


def set_config(spec: str | None = None) -> None:
    """Override the tile heuristic ("bn=128,grid=8,persistent=0,group=4,zigzag=1"); None restores it."""
    _check(lib().gb_set_config(spec.encode() if spec else None))


def set_wait_timeout_ns(ns: int) -> None:
    _check(lib().gb_set_wait_timeout_ns(int(ns)))


def set_fault_injection(mode: int) -> None:
    _check(lib().gb_set_fault_injection(int(mode)))


def measure_mma_rate(cta_group: int = 2, n: int = 256, alternate: bool = False, num_mma: int = 8192,
                     units: int = 1) -> tuple[float, float]:
    """(dense bf16 FLOP per SM per clock, cycles per MMA) of back-to-back tcgen05.mma (see the header)."""
    rate, cyc = ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().gb_measure_mma_rate(int(cta_group), int(n), 1 if alternate else 0, int(num_mma), int(units),
                                     ctypes.byref(rate), ctypes.byref(cyc)))
    return rate.value, cyc.value


def probe_mma_issue(cta_group: int = 2, n: int = 256, mode: int = 0, alu: int = 0, num_mma: int = 8192,
                    units: int = 1) -> tuple[float, float]:
    """(cycles per MMA, TMEM loads per MMA) with the steps of `mode` around or beside the MMAs
    (see the header)."""
    cyc, lds = ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().gb_probe_mma_issue(int(cta_group), int(n), int(mode), int(alu), int(num_mma), int(units),
                                    ctypes.byref(cyc), ctypes.byref(lds)))
    return cyc.value, lds.value


def set_trace_buffer(buf: torch.Tensor | None) -> None:
    """Trace records go to `buf` (a CUDA tensor) in a GB_TRACE build; None turns tracing off."""
    if buf is None:
        _check(lib().gb_set_trace_buffer(None, 0))
    else:
        _check(lib().gb_set_trace_buffer(buf.data_ptr(), buf.numel() * buf.element_size()))


def last_plan() -> str:
    buf = ctypes.create_string_buffer(512)
    _check(lib().gb_last_plan(buf, len(buf)))
    return buf.value.decode()


def version() -> str:
    return lib().gb_version().decode()
