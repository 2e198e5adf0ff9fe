"""CUDA path vs the CPU oracle on sizes the oracle finishes in seconds: every
output element is compared.  Shapes span several tiles and ragged tails; the
epilogue variants, store paths, the configuration overrides and the edge cases
(K = 0, M or N = 0, one row, D aliasing R) are all covered."""
import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_bitexact, assert_close, bits, int_tensor

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset_config():
    gb.set_config(None)
    yield
    gb.set_config(None)
    gb.device_status()


def run_linear(A, B, bias=None, R=None, act="none", **kw):
    d = gb.linear(A.to(DEV), B.to(DEV), None if bias is None else bias.to(DEV),
                  None if R is None else R.to(DEV), act=act, **kw)
    gb.device_status()
    return bits(d)


def ref_linear(A, B, bias=None, R=None, act="none"):
    return oracle.linear(bits(A), bits(B), None if bias is None else bits(bias),
                         None if R is None else bits(R), act)


def test_plain_256x384x512():
    """The plain-matmul workload: A[256,512], B[384,512] ~ N(0,1), seed 0, no epilogue."""
    w = inputs.plain()
    assert_close(run_linear(w["A"], w["B"]), ref_linear(w["A"], w["B"]), "plain")


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 128), (300, 700, 520), (1, 1, 8), (129, 257, 72),
                                   (127, 255, 4096), (513, 96, 1000)])
def test_integer_inputs_bit_exact(M, N, K, pair):
    """Small-integer operands: every partial sum is exact in fp32 in any order, so the
    GPU must reproduce the oracle bit for bit."""
    gb.set_config(f"pair={pair}")
    A = int_tensor((M, K), 1)
    B = int_tensor((N, K), 2)
    bias = int_tensor((N,), 3, -4, 4)
    R = int_tensor((M, N), 4, -4, 4)
    assert_bitexact(run_linear(A, B), ref_linear(A, B), "no epilogue")
    assert_bitexact(run_linear(A, B, bias, R, "relu"), ref_linear(A, B, bias, R, "relu"), "bias+relu+R")


def test_index_pattern_exact():
    """D[m,n] = m + 16 n (exact): catches swapped rows/columns and tile-placement errors."""
    M, N, K = 300, 260, 64
    a = torch.zeros(M, K)
    a[:, 0] = torch.arange(M) % 128
    a[:, 1] = 1
    b = torch.zeros(N, K)
    b[:, 0] = 1
    b[:, 1] = 16 * (torch.arange(N) % 16)
    A, B = a.to(torch.bfloat16), b.to(torch.bfloat16)
    want = ((torch.arange(M) % 128)[:, None] + 16 * (torch.arange(N) % 16)[None, :]).float().to(torch.bfloat16)
    assert_bitexact(run_linear(A, B), bits(want), "index pattern")


@pytest.mark.parametrize("M", [1, 127, 128, 129, 255, 257, 513])
@pytest.mark.parametrize("N", [1, 96, 128, 129, 256, 257, 520])
@pytest.mark.parametrize("K", [8, 64, 200])
def test_tile_edges(M, N, K):
    A = inputs.randn_bf16((M, K), seed=M * 7 + N)
    B = inputs.randn_bf16((N, K), seed=N * 11 + K, std=1.0 / np.sqrt(K))
    assert_close(run_linear(A, B), ref_linear(A, B), f"{M}x{N}x{K}")


@pytest.mark.parametrize("act", ["none", "gelu_tanh", "silu", "relu"])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("with_r", [False, True])
def test_epilogue_variants(act, with_bias, with_r):
    M, N, K = 333, 777, 320
    A = inputs.randn_bf16((M, K), seed=20)
    B = inputs.randn_bf16((N, K), seed=21, std=0.1)
    bias = inputs.randn_bf16((N,), seed=22, std=0.5) if with_bias else None
    R = inputs.randn_bf16((M, N), seed=23) if with_r else None
    assert_close(run_linear(A, B, bias, R, act), ref_linear(A, B, bias, R, act), f"{act} {with_bias} {with_r}")


@pytest.mark.parametrize("r_async", [0, 1])
def test_unaligned_d_and_r_use_plain_loads_and_stores(r_async):
    """N = 4099: rows of D and R are 8198 bytes apart (not a multiple of 16), so the
    kernel stores D through its shared-memory transpose with plain stores, and reads R
    either the same way at use (r_async=0) or by cp.async words into a prefetch queue."""
    gb.set_config(f"r_async={r_async}")
    M, N, K = 200, 4099, 128
    A = inputs.randn_bf16((M, K), seed=30)
    B = inputs.randn_bf16((N, K), seed=31, std=1.0 / np.sqrt(K))
    R = inputs.randn_bf16((M, N), seed=32)
    got = run_linear(A, B, None, R)
    plan = gb.last_plan()
    assert "d_store=st.transposed" in plan, plan
    assert ("r_load=cp.async" if r_async else "r_load=ld.transposed") in plan, plan
    assert_close(got, ref_linear(A, B, None, R), "N=4099")


def _unaligned_r(M, N, ldr, off, seed):
    """R[M, N] as a view with leading dimension `ldr` starting `off` elements into its
    buffer: the host copy (contiguous) and the device view."""
    big = inputs.randn_bf16((M * ldr + off + 8,), seed=seed)
    host = big[off:off + M * ldr].view(M, ldr)[:, :N]
    dev = big.to(DEV)[off:off + M * ldr].view(M, ldr)[:, :N]
    return host.contiguous(), dev


@pytest.mark.parametrize("spec", ["", "epi=1", "epi=2", "pair=0,grid=3", "pingpong=1", "r_boxes=2", "r_boxes=8",
                                  "r_boxes=8,stages=2", "grid=1", "bn=128,grid=5", "boxes=8,r_boxes=3"])
@pytest.mark.parametrize("M,N,K,ldr,off", [
    (300, 4099, 520, 4099, 0),   # odd row stride: segments alternate between word and half-word starts
    (130, 520, 192, 522, 2),     # 4-byte (not 16-byte) aligned base, even stride: every segment word-aligned
    (77, 516, 64, 519, 2),       # 4-byte aligned base, odd stride, ragged M
    (45, 13, 72, 13, 0),         # N < 32: every segment shorter than a chunk
    (129, 33, 0, 35, 4),         # K = 0: D = R; a 1-column tail chunk
    (257, 1001, 4096, 1001, 0),  # long K, ragged in every dimension
])
def test_unaligned_r_cp_async_queue(spec, M, N, K, ldr, off):
    """R rows not 16-byte aligned but the base 4-byte aligned: the cp.async prefetch queue.
    Bit-identical to the synchronous loads at use (the same bf16 values are combined in
    the same order) and within tolerance of the oracle; the elements outside the view
    (the stride's padding, the element before an odd segment) do not leak in."""
    A = inputs.randn_bf16((M, K), seed=M + K)
    B = inputs.randn_bf16((N, K), seed=N + 1, std=1.0 / np.sqrt(max(K, 1)))
    bias = inputs.randn_bf16((N,), seed=5, std=0.1)
    R_host, R_dev = _unaligned_r(M, N, ldr, off, seed=ldr + off)
    assert R_dev.data_ptr() % 4 == 0 and (R_dev.data_ptr() % 16 != 0 or ldr % 8 != 0)
    outs = {}
    for ra in (0, 1):
        gb.set_config(",".join(x for x in (spec, f"r_async={ra}") if x))
        d = gb.linear(A.to(DEV), B.to(DEV), bias.to(DEV), R_dev, act="gelu_tanh")
        gb.device_status()
        plan = gb.last_plan()
        assert ("r_load=cp.async" if ra else "r_load=ld.transposed") in plan, plan
        outs[ra] = bits(d)
    assert_bitexact(outs[1], outs[0], f"{spec} {M}x{N}x{K} ldr={ldr} off={off}")
    assert_close(outs[1], ref_linear(A, B, bias, R_host, "gelu_tanh"), f"{spec} {M}x{N}x{K}")


def test_unaligned_r_2_byte_base_stays_synchronous():
    """A base only 2-byte aligned cannot be copied in aligned words without reading the
    element before the tensor: the synchronous loads serve it."""
    M, N, K = 64, 300, 64
    A = inputs.randn_bf16((M, K), seed=7)
    B = inputs.randn_bf16((N, K), seed=8, std=0.1)
    R_host, R_dev = _unaligned_r(M, N, 301, 1, seed=9)
    assert R_dev.data_ptr() % 4 == 2
    d = gb.linear(A.to(DEV), B.to(DEV), None, R_dev)
    gb.device_status()
    assert "r_load=ld.transposed" in gb.last_plan(), gb.last_plan()
    assert_close(bits(d), ref_linear(A, B, None, R_host), "2-byte base")


def test_strided_views_and_offset_d():
    """Operands with leading dimension > K, and D / R as column slices of bigger buffers."""
    M, N, K = 190, 300, 136
    Abig = inputs.randn_bf16((M, K + 40), seed=40)
    Bbig = inputs.randn_bf16((N, K + 24), seed=41, std=0.1)
    A, B = Abig[:, 8:8 + K], Bbig[:, 16:16 + K]
    Rbig = inputs.randn_bf16((M, N + 13), seed=42)
    R = Rbig[:, 5:5 + N]
    Dbig = torch.zeros((M, N + 9), dtype=torch.bfloat16, device=DEV)
    D = Dbig[:, 3:3 + N]
    gb.linear(A.to(DEV), B.to(DEV), None, R.to(DEV), act="silu", out=D)
    gb.device_status()
    assert_close(bits(D), oracle.linear(bits(A.contiguous()), bits(B.contiguous()), None, bits(R.contiguous()),
                                        "silu"), "strided")
    # columns outside the view are untouched
    assert torch.all(Dbig[:, :3] == 0) and torch.all(Dbig[:, 3 + N:] == 0)


@pytest.mark.parametrize("spec", ["", "epi=1", "epi=2", "pair=0,grid=3", "pingpong=1"])
@pytest.mark.parametrize("with_r", [False, True])
def test_bias_only_2_byte_aligned(spec, with_r):
    """A bias that starts 2 bytes past a 16-byte boundary takes the scalar bias loads
    (the vector loads need 16-byte alignment): express, paired and general epilogues."""
    gb.set_config(spec or None)
    M, N, K = 300, 520, 192
    A = inputs.randn_bf16((M, K), seed=195)
    B = inputs.randn_bf16((N, K), seed=196, std=1.0 / np.sqrt(K))
    bias_big = inputs.randn_bf16((N + 1,), seed=197, std=0.1)
    bias = bias_big[1:]
    R = inputs.randn_bf16((M, N), seed=198) if with_r else None
    bias_dev = bias_big.to(DEV)[1:]
    assert bias_dev.data_ptr() % 16 == 2
    D = gb.linear(A.to(DEV), B.to(DEV), bias_dev, None if R is None else R.to(DEV), act="gelu_tanh")
    gb.device_status()
    assert_close(bits(D), ref_linear(A, B, bias.contiguous(), R, "gelu_tanh"), f"{spec} R={with_r}")


@pytest.mark.parametrize("spec", ["", "epi=1", "pair=0,grid=3", "pingpong=1", "boxes=8"])
@pytest.mark.parametrize("K", [64, 520])
def test_unaligned_r_with_aligned_d(spec, K):
    """R rows only 2-byte aligned (R read through the shared-memory transpose) while D
    rows are 16-byte aligned (D stored by TMA), and the reverse."""
    gb.set_config(spec or None)
    M, N = 300, 520
    A = inputs.randn_bf16((M, K), seed=200)
    B = inputs.randn_bf16((N, K), seed=201, std=1.0 / np.sqrt(K))
    Rbig = inputs.randn_bf16((M, N + 1), seed=202)
    R = Rbig[:, 1:]
    Rd = Rbig.to(DEV)[:, 1:]
    D = gb.linear(A.to(DEV), B.to(DEV), None, Rd, act="relu")
    gb.device_status()
    plan = gb.last_plan()
    assert "r_load=ld.transposed" in plan and "d_store=tma" in plan, plan
    ref = ref_linear(A, B, None, R.contiguous(), "relu")
    assert_close(bits(D), ref, f"{spec} {plan}")
    Dbig = torch.zeros((M, N + 1), dtype=torch.bfloat16, device=DEV)
    gb.linear(A.to(DEV), B.to(DEV), None, R.contiguous().to(DEV), act="relu", out=Dbig[:, 1:])
    gb.device_status()
    plan = gb.last_plan()
    assert "r_load=tma" in plan and "d_store=st.transposed" in plan, plan
    assert_close(bits(Dbig[:, 1:]), ref, f"{spec} {plan}")


def test_d_aliases_r():
    M, N, K = 260, 384, 96
    A = inputs.randn_bf16((M, K), seed=50)
    B = inputs.randn_bf16((N, K), seed=51, std=0.1)
    R = inputs.randn_bf16((M, N), seed=52)
    ref = ref_linear(A, B, None, R, "gelu_tanh")
    RD = R.to(DEV).clone()
    gb.linear(A.to(DEV), B.to(DEV), None, RD, act="gelu_tanh", out=RD)
    gb.device_status()
    assert_close(bits(RD), ref, "D == R")


def test_k_zero_gives_epilogue_of_zero():
    M, N = 150, 270
    A = torch.zeros((M, 0), dtype=torch.bfloat16)
    B = torch.zeros((N, 0), dtype=torch.bfloat16)
    bias = inputs.randn_bf16((N,), seed=60)
    R = inputs.randn_bf16((M, N), seed=61)
    d = gb.linear(torch.empty((M, 0), dtype=torch.bfloat16, device=DEV),
                  torch.empty((N, 0), dtype=torch.bfloat16, device=DEV), bias.to(DEV), R.to(DEV), act="gelu_tanh")
    gb.device_status()
    assert_close(bits(d), oracle.linear(bits(A), bits(B), bits(bias), bits(R), "gelu_tanh"), "K=0")


def test_empty_outputs():
    A = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.empty((32, 64), dtype=torch.bfloat16, device=DEV)
    assert gb.linear(A, B).shape == (0, 32)
    assert gb.linear(B, A).shape == (32, 0)


@pytest.mark.parametrize("epi", [1, 2])
@pytest.mark.parametrize("pair", [-1, 0, 1])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 500, 200), (1, 7, 8), (257, 129, 1000)])
def test_ffn_gated(M, N, K, pair, epi):
    gb.set_config(f"pair={pair},epi={epi}")
    X = inputs.randn_bf16((M, K), seed=70)
    W1 = inputs.randn_bf16((N, K), seed=71, std=1.0 / np.sqrt(K))
    W3 = inputs.randn_bf16((N, K), seed=72, std=1.0 / np.sqrt(K))
    d = gb.ffn_gated(X.to(DEV), W1.to(DEV), W3.to(DEV))
    gb.device_status()
    assert_close(bits(d), oracle.ffn_gated(bits(X), bits(W1), bits(W3)), f"ffn {M}x{N}x{K}")


def test_ffn_integer_bit_exact_when_gate_is_relu_like():
    """With W1 chosen so that X.W1^T is a large positive or zero integer, silu is x or 0
    exactly in fp32, and the product with an integer X.W3^T is exact."""
    M, N, K = 130, 140, 64
    X = int_tensor((M, K), 80, 0, 1)
    W1 = torch.zeros((N, K))
    W1[:, 0] = 200.0
    W1[::3, 0] = 0.0                 # every third column: X.W1^T = 0 -> silu = 0
    X[:, 0] = 1                      # so X.W1^T = 200 (silu(200) == 200 in fp32) or 0
    W3 = int_tensor((N, K), 81, -2, 2)
    W1b = W1.to(torch.bfloat16)
    d = gb.ffn_gated(X.to(DEV), W1b.to(DEV), W3.to(DEV))
    gb.device_status()
    assert_bitexact(bits(d), oracle.ffn_gated(bits(X), bits(W1b), bits(W3)), "ffn exact")


@pytest.mark.parametrize("spec", ["bn=128", "bn=256", "persistent=0", "grid=3", "grid=1", "group=1",
                                  "group=3,grid=5", "bn=128,grid=7,group=2", "pair=0", "pair=1",
                                  "pair=1,grid=2", "pair=1,persistent=0", "pair=0,grid=5,group=2",
                                  "pair=1,group=1,grid=6", "stages=2", "stages=3,pair=1,grid=3",
                                  "stages=4,pair=0", "stages=16", "epi=1", "epi=2", "epi=1,pair=0,grid=3",
                                  "epi=2,pair=1,grid=2,stages=3", "boxes=2", "boxes=8,grid=3",
                                  "boxes=5,stages=6", "boxes=3,epi=1,pair=0", "pingpong=1", "pingpong=1,grid=3",
                                  "pingpong=1,pair=0,grid=2", "issue=1", "issue=2", "issue=2,pair=0",
                                  "issue=2,stages=2", "issue=1,zigzag=1", "mc=1", "mc=1,issue=2",
                                  "mc=1,grid=4", "mc=1,epi=2,issue=1", "hint_a=2,hint_b=1,hint_d=1,hint_r=1",
                                  "prod=2", "prod=2,pair=0", "prod=2,epi=2,stages=2", "prod=2,mc=1",
                                  "prod=2,issue=2,grid=3", "prod=3", "prod=3,pair=0", "prod=3,epi=2",
                                  "issue=3"])
def test_config_overrides_give_identical_bits(spec):
    """Tile size, grid, swizzle and persistence change which CTA computes a tile but not
    the per-element accumulation order within the tile: identical bits."""
    M, N, K = 700, 900, 256
    A = inputs.randn_bf16((M, K), seed=90)
    B = inputs.randn_bf16((N, K), seed=91, std=0.1)
    bias = inputs.randn_bf16((N,), seed=92, std=0.1)
    base = run_linear(A, B, bias, None, "gelu_tanh")
    gb.set_config(spec)
    got = run_linear(A, B, bias, None, "gelu_tanh")
    assert_bitexact(got, base, spec)
    assert_close(got, ref_linear(A, B, bias, None, "gelu_tanh"), spec)


@pytest.mark.parametrize("spec", ["zigzag=1,grid=4", "zigzag=1,grid=1", "zigzag=0,grid=4"])
def test_zigzag(spec):
    """Reversing K changes the accumulation order: within tolerance on random inputs,
    bit-exact on integer inputs."""
    M, N, K = 520, 600, 640
    gb.set_config(spec)
    A = inputs.randn_bf16((M, K), seed=93)
    B = inputs.randn_bf16((N, K), seed=94, std=1.0 / np.sqrt(K))
    assert_close(run_linear(A, B), ref_linear(A, B), spec)
    Ai, Bi = int_tensor((M, K), 95), int_tensor((N, K), 96)
    assert_bitexact(run_linear(Ai, Bi), ref_linear(Ai, Bi), spec)


def test_golden_fixtures():
    from tests import golden
    for name in golden.FIXTURES:
        g = golden.load(name)
        t = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(DEV) for k, v in g.items()}
        if "X" in g:
            d = gb.ffn_gated(t["X"], t["W1"], t["W3"])
        else:
            act = "gelu_tanh" if "gelu" in name else ("silu" if "silu" in name else "none")
            d = gb.linear(t["A"], t["B"], t.get("bias"), t.get("R"), act=act)
        gb.device_status()
        assert_close(bits(d), g["D"], name)


def test_repeated_calls_and_streams():
    """Back-to-back launches on a side stream reuse cached descriptors and stay correct."""
    M, N, K = 384, 512, 192
    A = inputs.randn_bf16((M, K), seed=100)
    B = inputs.randn_bf16((N, K), seed=101, std=0.1)
    ref = ref_linear(A, B, None, None, "relu")
    s = torch.cuda.Stream()
    Ad, Bd = A.to(DEV), B.to(DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        outs = [gb.linear(Ad, Bd, act="relu") for _ in range(5)]
    gb.device_status(s)
    for o in outs:
        assert_close(bits(o), ref, "repeat")


@pytest.mark.parametrize("spec", ["", "grid=1", "grid=3", "pair=0,grid=2", "pair=1,grid=2", "bn=128,grid=3",
                                  "persistent=0", "epi=1,grid=2", "epi=2,grid=2", "epi=1,pair=0"])
@pytest.mark.parametrize("M,N", [(700, 904), (129, 264), (1, 8), (520, 1000)])
def test_residual_by_tma(spec, M, N):
    """R with 16-byte aligned rows is prefetched by TMA; a small grid makes each
    epilogue warp's prefetch run across many tiles."""
    gb.set_config(spec or None)
    K = 192
    A = inputs.randn_bf16((M, K), seed=110)
    B = inputs.randn_bf16((N, K), seed=111, std=0.1)
    bias = inputs.randn_bf16((N,), seed=112, std=0.1)
    R = inputs.randn_bf16((M, N), seed=113)
    got = run_linear(A, B, bias, R, "gelu_tanh")
    assert "r_load=tma" in gb.last_plan(), gb.last_plan()
    assert_close(got, ref_linear(A, B, bias, R, "gelu_tanh"), f"{spec} {M}x{N}")


@pytest.mark.parametrize("spec", ["boxes=2", "boxes=3", "boxes=8", "boxes=8,stages=2", "boxes=5,grid=3",
                                  "boxes=8,epi=1", "boxes=4,epi=2,pair=0,grid=2", "boxes=7,pair=1,grid=2"])
@pytest.mark.parametrize("K", [64, 1024])
def test_box_queue_depths(spec, K):
    """Per-warp queues of D staging boxes and TMA-loaded R boxes, 2 to 8 deep, with
    the ring shortened to make room: a small grid makes every warp's queues wrap
    many times across tiles.  The queue depth changes no arithmetic: identical bits
    to the default plan, and the oracle's result within tolerance."""
    M, N = 700, 1160
    A = inputs.randn_bf16((M, K), seed=140)
    B = inputs.randn_bf16((N, K), seed=141, std=1.0 / np.sqrt(K))
    bias = inputs.randn_bf16((N,), seed=142, std=0.1)
    R = inputs.randn_bf16((M, N), seed=143)
    base = run_linear(A, B, bias, R, "gelu_tanh")
    gb.set_config(spec)
    got = run_linear(A, B, bias, R, "gelu_tanh")
    plan = gb.last_plan()
    d_boxes, r_boxes = (int(v) for v in plan.split("boxes=")[1].split()[0].split("/"))
    want = int(spec.split("boxes=")[1].split(",")[0])
    assert "r_load=tma" in plan and d_boxes == r_boxes and 2 <= d_boxes <= want, plan
    assert_bitexact(got, base, plan)
    assert_close(got, ref_linear(A, B, bias, R, "gelu_tanh"), plan)
    # second output and no epilogue input: D and Z share the D queue
    D, Z = gb.linear_preact(A.to(DEV), B.to(DEV), bias.to(DEV), None, act="relu")
    gb.device_status()
    assert_close(bits(D), ref_linear(A, B, bias, None, "relu"), "D " + gb.last_plan())
    assert_close(bits(Z), ref_linear(A, B, bias, None, "none"), "Z " + gb.last_plan())


@pytest.mark.parametrize("spec", ["pingpong=1", "pingpong=1,grid=3", "pingpong=1,pair=0,grid=5", "pingpong=1,boxes=8",
                                  "pingpong=1,pair=1,grid=2,stages=2", "pingpong=0,epi=2", "pingpong=0,grid=3"])
@pytest.mark.parametrize("K", [64, 640])
def test_pingpong_all_epilogues(spec, K):
    """Ping-pong on and off: the two epilogue warpgroups alternate whole tiles (each owns
    one TMEM buffer) or share every tile's chunks.  Same per-element arithmetic either
    way, so identical bits to the default plan for bias+GELU+R (R by TMA), unaligned
    rows (transposes), the second output Z and the FFN; and the oracle's result within
    tolerance."""
    M, N = 520, 776
    A = inputs.randn_bf16((M, K), seed=160)
    B = inputs.randn_bf16((N, K), seed=161, std=1.0 / np.sqrt(K))
    B3 = inputs.randn_bf16((N, K), seed=162, std=1.0 / np.sqrt(K))
    bias = inputs.randn_bf16((N,), seed=163, std=0.1)
    R = inputs.randn_bf16((M, N), seed=164)
    Ad, Bd, B3d, biasd, Rd = (t.to(DEV) for t in (A, B, B3, bias, R))

    def all_outputs():
        out = {"lin": bits(gb.linear(Ad, Bd, biasd, Rd, act="gelu_tanh"))}
        Dodd = torch.zeros((M, N + 1), dtype=torch.bfloat16, device=DEV)[:, 1:]  # rows not 16-byte aligned
        Rodd = torch.zeros((M, N + 1), dtype=torch.bfloat16, device=DEV)[:, 1:]
        Rodd.copy_(Rd)
        gb.linear(Ad, Bd, biasd, Rodd, act="silu", out=Dodd)
        out["odd"] = bits(Dodd)
        D, Z = gb.linear_preact(Ad, Bd, biasd, None, act="relu")
        out["D"], out["Z"] = bits(D), bits(Z)
        out["ffn"] = bits(gb.ffn_gated(Ad, Bd, B3d))
        gb.device_status()
        return out

    base = all_outputs()
    gb.set_config(spec)
    got = all_outputs()
    plan = gb.last_plan()
    assert f"pingpong={spec[9]}" in plan and "epi=2" in plan, plan
    for k in base:
        assert_bitexact(got[k], base[k], f"{spec} {k}")
    assert_close(got["lin"], ref_linear(A, B, bias, R, "gelu_tanh"), spec)
    assert_close(got["odd"], ref_linear(A, B, bias, R, "silu"), spec)
    assert_close(got["Z"], ref_linear(A, B, bias, None, "none"), spec)
    assert_close(got["ffn"], oracle.ffn_gated(bits(A), bits(B), bits(B3)), spec)


def test_pingpong_is_ignored_by_split_k_and_refused_with_one_warpgroup():
    M, N, K = 127, 96, 4096
    A = inputs.randn_bf16((M, K), seed=170)
    B = inputs.randn_bf16((N, K), seed=171, std=1.0 / 64)
    R = inputs.randn_bf16((M, N), seed=172)
    gb.set_config("pingpong=1")
    got = run_linear(A, B, None, R, split_k="auto")
    plan = gb.last_plan()
    assert "pingpong=0" in plan and int(plan.split("splits=")[1].split()[0]) > 1, plan
    assert_close(got, ref_linear(A, B, None, R), plan)
    gb.set_config("pingpong=1,epi=1")
    with pytest.raises(gb.GBError):
        run_linear(A, B)


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("rem", [1, 8, 17, 100, 128, 129, 240, 255])
def test_ragged_last_tile_column(pair, rem):
    """A ragged last tile column at every width boundary (one column, a box, half a pair's
    B rows, one past half, all but one): bit-exact on integer inputs and against the oracle
    on random ones, with full tile columns before it on the same accumulator buffers."""
    gb.set_config(f"pair={pair},grid=2")
    M, N, K = 300, 512 + rem, 200
    Ai, Bi = int_tensor((M, K), 180), int_tensor((N, K), 181)
    Ri = int_tensor((M, N), 182, -4, 4)
    assert_bitexact(run_linear(Ai, Bi, None, Ri), ref_linear(Ai, Bi, None, Ri), f"int rem={rem}")
    A = inputs.randn_bf16((M, K), seed=183)
    B = inputs.randn_bf16((N, K), seed=184, std=1.0 / np.sqrt(K))
    bias = inputs.randn_bf16((N,), seed=185, std=0.1)
    assert_close(run_linear(A, B, bias, None, "gelu_tanh"), ref_linear(A, B, bias, None, "gelu_tanh"), f"rem={rem}")


def test_short_k_plan_takes_deep_queues():
    """Work items of at most 4 k-blocks get a short ring and deep queues -- with wide
    32x64 boxes a 2-stage ring, two D boxes and the deepest R queue that fits; with 32x32
    boxes a 3-stage ring and the deepest D and R queues -- and, with at least 4 work items
    per unit, the ping-pong schedule; long-K items keep the deepest ring, two boxes per
    warp and the shared schedule."""
    A = inputs.randn_bf16((512, 4096), seed=150)
    B = inputs.randn_bf16((512, 4096), seed=151, std=1.0 / 64)
    R = inputs.randn_bf16((512, 512), seed=152)
    run_linear(A[:, :64].contiguous(), B[:, :64].contiguous(), None, R)
    short = gb.last_plan()
    assert "stages=2" in short and "boxes=2/" in short and "boxes=2/2" not in short, short
    assert "pingpong=0" in short and "tma.64x32" in short, short  # 4 tiles only
    gb.set_config("wide=0")
    run_linear(A[:, :64].contiguous(), B[:, :64].contiguous(), None, R)
    short = gb.last_plan()
    gb.set_config(None)
    assert "stages=3" in short and "boxes=2/" not in short and "pingpong=0" in short, short
    run_linear(A, B, None, R)
    long = gb.last_plan()
    assert "boxes=2/2" in long and "stages=3 " not in long and "pingpong=0" in long, long
    # 16 x 20 tiles of 256 x 256 on at most 76 CTA pairs: ping-pong (plan only)
    Ab = torch.zeros((4096, 64), dtype=torch.bfloat16, device=DEV)
    Bb = torch.zeros((5120, 64), dtype=torch.bfloat16, device=DEV)
    Rb = torch.zeros((4096, 5120), dtype=torch.bfloat16, device=DEV)
    D = gb.linear(Ab, Bb, None, Rb)
    gb.device_status()
    big = gb.last_plan()
    # ... on the lean kernel: four epilogue warpgroups, one 32x64 D box and three 32x32 R
    # boxes per warp, a 2-stage ring
    assert "pingpong=1" in big and "epi=4" in big and "stages=2" in big and "boxes=1/3" in big, big
    assert "d_store=tma.64x32" in big and "r_load=tma " in big + " ", big
    assert torch.equal(D.view(torch.int16), Rb.view(torch.int16))


def test_residual_by_tma_aliasing_d():
    M, N, K = 600, 520, 128
    A = inputs.randn_bf16((M, K), seed=120)
    B = inputs.randn_bf16((N, K), seed=121, std=0.1)
    R = inputs.randn_bf16((M, N), seed=122)
    ref = ref_linear(A, B, None, R, "relu")
    gb.set_config("grid=2")
    RD = R.to(DEV).clone()
    gb.linear(A.to(DEV), B.to(DEV), None, RD, act="relu", out=RD)
    gb.device_status()
    assert "r_load=tma" in gb.last_plan()
    assert_close(bits(RD), ref, "D == R by TMA")


@pytest.mark.parametrize("spec", ["", "pair=0", "grid=3", "epi=1", "epi=1,pair=0,grid=2"])
@pytest.mark.parametrize("M,N", [(300, 4099), (33, 1001), (129, 17), (257, 263)])
def test_unaligned_rows_all_epilogues(spec, M, N):
    """Odd N (rows only 2-byte aligned): D and R through the transpose, every row and
    column tail, with bias and activation, and D written into a strided view."""
    gb.set_config(spec or None)
    K = 136
    A = inputs.randn_bf16((M, K), seed=130)
    B = inputs.randn_bf16((N, K), seed=131, std=0.1)
    bias = inputs.randn_bf16((N,), seed=132, std=0.1)
    R = inputs.randn_bf16((M, N), seed=133)
    Dbig = torch.zeros((M, N + 3), dtype=torch.bfloat16, device=DEV)
    D = Dbig[:, 1:1 + N]
    gb.linear(A.to(DEV), B.to(DEV), bias.to(DEV), R.to(DEV), act="silu", out=D)
    gb.device_status()
    assert "st.transposed" in gb.last_plan()
    assert_close(bits(D), ref_linear(A, B, bias, R, "silu"), f"{spec} {M}x{N}")
    assert torch.all(Dbig[:, 0] == 0) and torch.all(Dbig[:, 1 + N:] == 0)


@pytest.mark.parametrize("spec", ["", "epi=1", "epi=2", "pair=0,grid=3", "pair=1,grid=2,epi=1"])
@pytest.mark.parametrize("act", ["gelu_tanh", "relu"])
@pytest.mark.parametrize("d_off,z_off", [(0, 0), (0, 1), (1, 0), (1, 1)], ids=["dz_tma", "z_transp", "d_transp",
                                                                               "both_transp"])
def test_preact_second_output(spec, act, d_off, z_off):
    """Z = bf16(A.B^T + bias) next to D = bf16(act(.) + R); outputs offset by one element
    (rows no longer 16-byte aligned) take the shared-memory transpose path."""
    gb.set_config(spec or None)
    M, N, K = 333, 520, 200
    A = inputs.randn_bf16((M, K), seed=140)
    B = inputs.randn_bf16((N, K), seed=141, std=0.1)
    bias = inputs.randn_bf16((N,), seed=142, std=0.5)
    R = inputs.randn_bf16((M, N), seed=143)
    Dbuf = torch.zeros((M, N + 8), dtype=torch.bfloat16, device=DEV)
    Zbuf = torch.zeros((M, N + 8), dtype=torch.bfloat16, device=DEV)
    D, Z = Dbuf[:, d_off:d_off + N], Zbuf[:, z_off:z_off + N]
    gb.linear_preact(A.to(DEV), B.to(DEV), bias.to(DEV), R.to(DEV), act=act, out=D, preact=Z)
    gb.device_status()
    plan = gb.last_plan()
    assert ("z_store=tma" in plan) == (z_off == 0) and ("d_store=tma" in plan) == (d_off == 0), plan
    ref_d, ref_z = oracle.linear_preact(bits(A), bits(B), bits(bias), bits(R), act)
    assert_close(bits(D), ref_d, f"D {spec}")
    assert_close(bits(Z), ref_z, f"Z {spec}")


def test_preact_integer_exact_and_k_zero():
    M, N, K = 200, 300, 64
    A, B = int_tensor((M, K), 150), int_tensor((N, K), 151)
    bias = int_tensor((N,), 152, -5, 5)
    D, Z = gb.linear_preact(A.to(DEV), B.to(DEV), bias.to(DEV), act="relu")
    gb.device_status()
    ref_d, ref_z = oracle.linear_preact(bits(A), bits(B), bits(bias), None, "relu")
    assert_bitexact(bits(D), ref_d, "D")
    assert_bitexact(bits(Z), ref_z, "Z")
    # K = 0: Z is the bias broadcast over rows
    D0, Z0 = gb.linear_preact(torch.empty((M, 0), dtype=torch.bfloat16, device=DEV),
                              torch.empty((N, 0), dtype=torch.bfloat16, device=DEV), bias.to(DEV), act="gelu_tanh")
    gb.device_status()
    assert torch.equal(Z0.view(torch.int16), bias.to(DEV).view(torch.int16)[None, :].expand(M, N))


@pytest.mark.parametrize("spec", ["mc=1", "mc=1,issue=2", "issue=2", "prod=2", "prod=2,mc=1", "prod=3"])
def test_schedules_identical_bits_on_ragged_shapes(spec):
    """A multicast between CTA pairs and the issue loops on shapes with an odd number of
    tile-columns (a multicast partner tile past N), ragged M, an epilogue input and the FFN."""
    for M, N, K in [(700, 900, 520), (513, 1300, 200), (300, 257, 64)]:
        A = inputs.randn_bf16((M, K), seed=M + 1)
        B = inputs.randn_bf16((N, K), seed=N + 2, std=0.1)
        bias = inputs.randn_bf16((N,), seed=3, std=0.1)
        R = inputs.randn_bf16((M, N), seed=4)
        base = run_linear(A, B, bias, R, "silu")
        gb.set_config(spec)
        got = run_linear(A, B, bias, R, "silu")
        assert ("mc=1" in gb.last_plan()) == ("mc=1" in spec), gb.last_plan()
        gb.set_config(None)
        assert_bitexact(got, base, f"{spec} {M}x{N}x{K}")
        X, W1, W3 = A, B, inputs.randn_bf16((N, K), seed=N + 5, std=0.1)
        d0 = bits(gb.ffn_gated(X.to(DEV), W1.to(DEV), W3.to(DEV)))
        gb.set_config(spec)
        d1 = bits(gb.ffn_gated(X.to(DEV), W1.to(DEV), W3.to(DEV)))
        gb.device_status()
        gb.set_config(None)
        assert_bitexact(d1, d0, f"ffn {spec} {M}x{N}x{K}")


@pytest.mark.parametrize("spec", ["", "wide=1", "wide=1,pingpong=1", "wide=1,pingpong=0", "wide=1,epi=1",
                                  "wide=1,bn=128", "wide=1,bn=128,epi=2,pingpong=0", "wide=1,boxes=8",
                                  "wide=1,pair=0,grid=3", "wide=1,stages=2,grid=2", "wide=1,r_boxes=2,boxes=2"])
def test_wide_boxes_identical_bits(spec):
    """32x64 R and D boxes (128-byte swizzle) on the paired epilogue path: the same values
    combined in the same order as with 32x32 boxes, so identical bits -- on shapes whose
    last 64-column step is partial (N = 904, 264, 96: one chunk, 8 or 32 columns, the box's
    other half zero-filled on load and clipped by the store; N = 1320: a full chunk and an
    8-column one), ragged M, short and long K, with bias, activation and the residual."""
    for M, N, K in [(700, 904, 64), (513, 1320, 200), (300, 264, 64), (129, 96, 128), (64, 2048, 64)]:
        A = inputs.randn_bf16((M, K), seed=M + 11)
        B = inputs.randn_bf16((N, K), seed=N + 12, std=0.1)
        bias = inputs.randn_bf16((N,), seed=13, std=0.1)
        R = inputs.randn_bf16((M, N), seed=14)
        gb.set_config("wide=0")
        base = run_linear(A, B, bias, R, "gelu_tanh")
        assert "r_load=tma " in gb.last_plan() + " ", gb.last_plan()
        gb.set_config(spec or None)
        got = run_linear(A, B, bias, R, "gelu_tanh")
        plan = gb.last_plan()
        gb.set_config(None)
        assert "d_store=tma.64x32" in plan and "r_load=tma.64x32" in plan, plan
        assert_bitexact(got, base, f"{spec} {M}x{N}x{K}")
        if (M, N, K) == (700, 904, 64):
            assert_close(got, ref_linear(A, B, bias, R, "gelu_tanh"), spec)


@pytest.mark.parametrize("spec", ["epi=4", "epi=4,wide=0", "epi=4,wide=1", "epi=4,wide=2,r_boxes=2", "epi=4,grid=4",
                                  "epi=4,stages=2,r_boxes=4", "epi=4,boxes=2", "epi=4,r_boxes=2,grid=2",
                                  "epi=4,hint_r=1,hint_d=1", "epi=4,stages=1", "epi=2,wide=2", "epi=2,wide=2,pingpong=0",
                                  "epi=1,wide=2"])
def test_four_epilogue_warpgroups_identical_bits(spec):
    """The lean kernel (four epilogue warpgroups, paired path only; warpgroups 2h, 2h + 1
    serve the tiles of parity h): identical bits to the two-warpgroup kernel on ragged
    residual shapes with bias and activation, short and long K."""
    for M, N, K in [(700, 904, 64), (513, 1320, 200), (300, 264, 64), (2100, 2048, 64), (64, 512, 1000)]:
        A = inputs.randn_bf16((M, K), seed=M + 21)
        B = inputs.randn_bf16((N, K), seed=N + 22, std=0.1)
        bias = inputs.randn_bf16((N,), seed=23, std=0.1)
        R = inputs.randn_bf16((M, N), seed=24)
        gb.set_config("epi=2")
        base = run_linear(A, B, bias, R, "silu")
        gb.set_config(spec)
        got = run_linear(A, B, bias, R, "silu")
        plan = gb.last_plan()
        gb.set_config(None)
        if M > 128 and "epi=4" in spec:
            assert "epi=4" in plan and "pingpong=1" in plan, plan
        if "wide=0" not in spec:  # 32x64 D boxes; 32x64 R boxes on request, or by default off the lean kernel
            r_wide = "wide=1" in spec or ("wide=" not in spec and "epi=4" not in plan)
            assert "d_store=tma.64x32" in plan and ("r_load=tma.64x32" in plan) == r_wide, plan
        assert_bitexact(got, base, f"{spec} {M}x{N}x{K}")
        if (M, N, K) == (700, 904, 64):
            assert_close(got, ref_linear(A, B, bias, R, "silu"), spec)


def test_four_epilogue_warpgroups_fall_back():
    """epi=4 where the lean kernel does not apply runs the two-warpgroup kernel: no
    epilogue input, an unaligned R, a split-K plan, single CTAs, the FFN."""
    M, N, K = 300, 512, 512
    A = inputs.randn_bf16((M, K), seed=31)
    B = inputs.randn_bf16((N, K), seed=32, std=0.05)
    R = inputs.randn_bf16((M, N), seed=33)
    gb.set_config("epi=4")
    d = run_linear(A, B)
    assert "epi=2" in gb.last_plan(), gb.last_plan()
    assert_close(d, ref_linear(A, B), "no R")
    Rbig = inputs.randn_bf16((M, N + 1), seed=34)
    d = gb.linear(A.to(DEV), B.to(DEV), None, Rbig.to(DEV)[:, 1:])
    gb.device_status()
    assert "epi=2" in gb.last_plan(), gb.last_plan()
    assert_close(bits(d), ref_linear(A, B, None, Rbig[:, 1:].contiguous()), "unaligned R")
    d = gb.linear(A.to(DEV), B.to(DEV), None, R.to(DEV), split_k=4)
    gb.device_status()
    assert "epi=2" in gb.last_plan() and "splits=4" in gb.last_plan(), gb.last_plan()
    assert_close(bits(d), ref_linear(A, B, None, R), "split")
    gb.set_config("epi=4,pair=0")
    d = run_linear(A, B, None, R)
    assert "epi=2" in gb.last_plan() and "pair=0" in gb.last_plan(), gb.last_plan()
    assert_close(d, ref_linear(A, B, None, R), "single CTAs")
