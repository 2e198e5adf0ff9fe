"""The C-ABI library on the CPU: it loads, exports every symbol the header
declares, and rejects invalid arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbgemm.h")

GB_OK, GB_ERR_INVALID_ARG, GB_ERR_UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    from dense_bf16_gemm_persistent_gb300 import _build
    _build.build()
    import dense_bf16_gemm_persistent_gb300 as gb
    return gb.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gb_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gb_gemm_linear", "gb_gemm_ffn_gated", "gb_get_device_status", "gb_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in gbgemm.h but not exported"


def test_version(L):
    assert re.fullmatch(r"\d+\.\d+\.\d+", L.gb_version().decode())


# Fake, never-dereferenced device addresses: validation rejects the call first.
P16 = 0x10000      # 16-byte aligned
P2 = 0x10002       # 2-byte aligned only
P1 = 0x10001       # odd


def lin(L, A=P16, lda=64, B=P16, ldb=64, bias=None, R=None, ldr=0, act=0, D=P16, ldd=32, M=16, N=32, K=64):
    return L.gb_gemm_linear(A, lda, B, ldb, bias, R, ldr, act, D, ldd, M, N, K, None)


@pytest.mark.parametrize("kwargs,status,needle", [
    (dict(A=None), GB_ERR_INVALID_ARG, "A is null"),
    (dict(B=None), GB_ERR_INVALID_ARG, "B is null"),
    (dict(D=None), GB_ERR_INVALID_ARG, "D is null"),
    (dict(M=-1), GB_ERR_INVALID_ARG, "negative"),
    (dict(K=-5), GB_ERR_INVALID_ARG, "negative"),
    (dict(lda=32), GB_ERR_INVALID_ARG, "lda"),
    (dict(ldb=8), GB_ERR_INVALID_ARG, "ldb"),
    (dict(ldd=31), GB_ERR_INVALID_ARG, "ldd"),
    (dict(R=P16, ldr=16), GB_ERR_INVALID_ARG, "ldr"),
    (dict(act=7), GB_ERR_INVALID_ARG, "activation"),
    (dict(act=-1), GB_ERR_INVALID_ARG, "activation"),
    (dict(A=P2), GB_ERR_UNSUPPORTED, "16-byte"),
    (dict(B=P2), GB_ERR_UNSUPPORTED, "16-byte"),
    (dict(lda=68, K=60), GB_ERR_UNSUPPORTED, "multiples of 8"),
    (dict(D=P1), GB_ERR_UNSUPPORTED, "2-byte"),
    (dict(bias=P1), GB_ERR_UNSUPPORTED, "2-byte"),
    (dict(M=1 << 31), GB_ERR_UNSUPPORTED, "2^31"),
    (dict(K=1 << 31, lda=1 << 31, ldb=1 << 31), GB_ERR_UNSUPPORTED, "2^31"),
])
def test_linear_rejects(L, kwargs, status, needle):
    assert lin(L, **kwargs) == status
    assert needle in L.gb_last_error().decode()


def test_empty_problem_is_a_noop(L):
    # M == 0 or N == 0: nothing to compute, no device call, GB_OK even with null pointers
    assert L.gb_gemm_linear(None, 0, None, 0, None, None, 0, 0, None, 0, 0, 5, 7, None) == GB_OK
    assert L.gb_gemm_linear(None, 0, None, 0, None, None, 0, 0, None, 0, 5, 0, 7, None) == GB_OK
    assert L.gb_gemm_ffn_gated(None, 0, None, 0, None, 0, None, 0, 0, 4, 4, None) == GB_OK


@pytest.mark.parametrize("args,needle", [
    ((None, 64, P16, 64, P16, 64, P16, 32, 16, 32, 64), "X is null"),
    ((P16, 64, None, 64, P16, 64, P16, 32, 16, 32, 64), "W1 is null"),
    ((P16, 64, P16, 64, None, 64, P16, 32, 16, 32, 64), "W3 is null"),
    ((P16, 64, P16, 64, P16, 32, P16, 32, 16, 32, 64), "ldw3"),
    ((P16, 64, P16, 64, P2, 64, P16, 32, 16, 32, 64), "16-byte"),
])
def test_ffn_rejects(L, args, needle):
    assert L.gb_gemm_ffn_gated(*args, None) != GB_OK
    assert needle in L.gb_last_error().decode()


def test_config_parser(L):
    assert L.gb_set_config(b"bn=128,grid=4,persistent=0,group=8,zigzag=1,pair=1,stages=3,boxes=4,pingpong=1") == GB_OK
    assert L.gb_set_config(b"r_async=0,r_boxes=5") == GB_OK
    assert L.gb_set_config(None) == GB_OK
    assert L.gb_set_config(b"") == GB_OK
    for bad in (b"bn=96", b"nope=1", b"grid", b"group=0", b"zigzag=2", b"bn=12x", b"pair=2", b"stages=-1", b"boxes=1",
                b"boxes=9", b"pingpong=2", b"pingpong=-2", b"r_async=2", b"r_boxes=1", b"r_boxes=9"):
        assert L.gb_set_config(bad) == GB_ERR_INVALID_ARG, bad
    assert L.gb_set_config(None) == GB_OK


def test_every_config_key_is_documented_and_accepted(L):
    """Each key gb_set_config takes is described in the header, and accepted alone."""
    header = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                               "gbgemm.h")).read()
    decl = header.index("gb_status_t gb_set_config(")
    doc = header[header.rindex("/*", 0, decl):decl]  # the comment block above the declaration
    keys = {"bn": 256, "grid": 8, "persistent": 1, "group": 16, "zigzag": 0, "pair": 0, "stages": 4, "epi": 2,
            "boxes": 2, "r_boxes": 3, "pingpong": 0, "hint_a": 2, "hint_b": 1, "hint_r": 0, "hint_d": 1, "mc": 1,
            "issue": 3, "prod": 1, "r_async": 1, "wide": 2}
    for k, v in keys.items():
        assert re.search(r"\b" + k + r"\b", doc), f"{k} is not described in gbgemm.h"
        assert L.gb_set_config(f"{k}={v}".encode()) == GB_OK, k
    assert L.gb_set_config(b"tmem_ld=64") == GB_ERR_INVALID_ARG  # (a key the planner never read; removed)
    assert L.gb_set_config(None) == GB_OK


def test_misc_entry_points(L):
    assert L.gb_set_wait_timeout_ns(1000) == GB_OK
    assert L.gb_set_wait_timeout_ns(0) == GB_OK
    assert L.gb_set_fault_injection(9) == GB_ERR_INVALID_ARG
    assert L.gb_set_fault_injection(0) == GB_OK
    assert L.gb_last_plan(None, 10) == GB_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(64)
    assert L.gb_last_plan(buf, 64) == GB_OK


def test_kernels_have_no_stack_frame_or_spills(L):
    """Every kernel compiles with 0 bytes of stack frame and no spills (ptxas -v)."""
    from dense_bf16_gemm_persistent_gb300 import _build
    log = open(os.path.join(_build.LOG_DIR, "ptxas.log")).read()
    entries = re.findall(r"Compiling entry function '(\w+)'", log)
    props = re.findall(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", log)
    assert entries and len(props) >= len(entries)
    for e, (stack, st, ld) in zip(entries, props):
        assert (int(stack), int(st), int(ld)) == (0, 0, 0), e


def test_splitk_entry_points_validate_first(L):
    assert L.gb_splitk_workspace_bytes(0, 16, 16, 16, 0, None) == GB_ERR_INVALID_ARG
    n = ctypes.c_size_t(7)
    assert L.gb_splitk_workspace_bytes(0, -1, 16, 16, 0, ctypes.byref(n)) == GB_ERR_INVALID_ARG
    assert L.gb_gemm_linear_splitk(None, 64, P16, 64, None, None, 0, 0, P16, 32, 16, 32, 64, 4, P16, 1 << 20,
                                   None) == GB_ERR_INVALID_ARG
    assert b"A is null" in L.gb_last_error()
    assert L.gb_gemm_ffn_gated_splitk(P16, 64, P16, 64, None, 64, P16, 32, 16, 32, 64, 4, P16, 1 << 20,
                                      None) == GB_ERR_INVALID_ARG
    # empty problems need no workspace and no device
    assert L.gb_gemm_linear_splitk(None, 0, None, 0, None, None, 0, 0, None, 0, 0, 5, 7, 0, None, 0,
                                   None) == GB_OK


def test_preact_entry_point_validates_first(L):
    args = dict(A=P16, lda=64, B=P16, ldb=64, bias=None, R=None, ldr=0, act=0, D=P16, ldd=32, M=16, N=32, K=64)

    def call(**kw):
        a = dict(args, **kw)
        return L.gb_gemm_linear_preact(a["A"], a["lda"], a["B"], a["ldb"], a["bias"], a["R"], a["ldr"], a["act"],
                                       a["D"], a["ldd"], kw.get("Z", P16), kw.get("ldz", 32), a["M"], a["N"], a["K"],
                                       None)
    assert call(Z=None) == GB_ERR_INVALID_ARG and b"Z is null" in L.gb_last_error()
    assert call(ldz=16) == GB_ERR_INVALID_ARG and b"ldz" in L.gb_last_error()
    assert call(Z=P1) == GB_ERR_UNSUPPORTED
    assert L.gb_gemm_linear_preact(None, 0, None, 0, None, None, 0, 0, None, 0, None, 0, 0, 4, 4, None) == GB_OK


def dact(L, dY=P16, lddy=64, W=P16, ldw=32, Z=P16, ldz=32, act=1, D=P16, ldd=32, M=16, N=64, K=32):
    return L.gb_gemm_linear_dact(dY, lddy, W, ldw, Z, ldz, act, D, ldd, M, N, K, None)


@pytest.mark.parametrize("kwargs,status,needle", [
    (dict(Z=None), GB_ERR_INVALID_ARG, "Z is null"),
    (dict(dY=None), GB_ERR_INVALID_ARG, "dY is null"),
    (dict(W=None), GB_ERR_INVALID_ARG, "W is null"),
    (dict(lddy=32), GB_ERR_INVALID_ARG, "lddy"),
    (dict(ldw=16), GB_ERR_INVALID_ARG, "ldw"),
    (dict(ldz=16), GB_ERR_INVALID_ARG, "ldz"),
    (dict(ldd=16), GB_ERR_INVALID_ARG, "ldd"),
    (dict(act=9), GB_ERR_INVALID_ARG, "activation"),
    (dict(W=P2), GB_ERR_UNSUPPORTED, "16-byte"),
    (dict(ldw=36), GB_ERR_UNSUPPORTED, "multiples of 8"),
    (dict(Z=P1), GB_ERR_UNSUPPORTED, "2-byte"),
])
def test_dact_rejects(L, kwargs, status, needle):
    assert dact(L, **kwargs) == status
    assert needle in L.gb_last_error().decode()


def matmul(L, A=P16, lda=64, B=P16, ldb=32, bias=None, R=None, ldr=0, act=1, D=P16, ldd=32, M=16, N=32, K=64):
    return L.gb_gemm_matmul(A, lda, B, ldb, bias, R, ldr, act, D, ldd, M, N, K, None)


@pytest.mark.parametrize("kwargs,status,needle", [
    (dict(A=None), GB_ERR_INVALID_ARG, "A is null"),
    (dict(B=None), GB_ERR_INVALID_ARG, "B is null"),
    (dict(lda=32), GB_ERR_INVALID_ARG, "lda"),
    (dict(ldb=16), GB_ERR_INVALID_ARG, "ldb"),
    (dict(ldd=16), GB_ERR_INVALID_ARG, "ldd"),
    (dict(R=P16, ldr=16), GB_ERR_INVALID_ARG, "ldr"),
    (dict(act=9), GB_ERR_INVALID_ARG, "activation"),
    (dict(B=P2), GB_ERR_UNSUPPORTED, "16-byte"),
    (dict(ldb=36), GB_ERR_UNSUPPORTED, "multiples of 8"),
    (dict(D=P1), GB_ERR_UNSUPPORTED, "2-byte"),
])
def test_matmul_rejects(L, kwargs, status, needle):
    """The MatmulOp entry point (B given as [K,N]): ldb is checked against N, not K."""
    assert matmul(L, **kwargs) == status
    assert needle in L.gb_last_error().decode()
    # M = 0 or N = 0: nothing to do, no pointer is needed
    assert L.gb_gemm_matmul(None, 0, None, 0, None, None, 0, 0, None, 0, 0, 4, 4, None) == GB_OK


def test_probe_rejects_bad_arguments(L):
    import ctypes
    r, c = ctypes.c_double(0), ctypes.c_double(0)
    assert L.gb_measure_mma_rate(3, 256, 0, 1024, 1, ctypes.byref(r), ctypes.byref(c)) == GB_ERR_INVALID_ARG
    assert L.gb_measure_mma_rate(2, 64, 0, 1024, 1, ctypes.byref(r), ctypes.byref(c)) == GB_ERR_INVALID_ARG
    assert L.gb_measure_mma_rate(2, 256, 0, 4, 1, ctypes.byref(r), ctypes.byref(c)) == GB_ERR_INVALID_ARG
