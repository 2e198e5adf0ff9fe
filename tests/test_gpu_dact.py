"""The activation-gradient entry point, D = bf16((dY.W) * act'(Z)), against the CPU
oracle: every element on shapes that span several tiles with ragged tails in all
three dimensions, for every activation's derivative, both tile shapes, TMA and
plain-load paths for Z and D, aliasing and the empty contraction; bit for bit on
integer operands; and the full-size MLP backward shape on sampled entries."""
import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_bitexact, assert_close, bits, check_pairs, int_tensor, ulp_hist

pytestmark = pytest.mark.gpu

DEV = "cuda"
ACTS = ["none", "gelu_tanh", "silu", "relu"]


@pytest.fixture(autouse=True)
def _reset_config():
    gb.set_config(None)
    yield
    gb.set_config(None)
    gb.device_status()


def ld8(n: int) -> int:
    return max(8, (n + 7) // 8 * 8)


def operands(M, N, K, seed, w_std=None, z_std=1.0):
    """dY [M,N], W [N,K], Z [M,K] on the device.  dY and W are views into buffers whose rows
    are padded to a multiple of 8 elements (the TMA row rule), so N and K can be ragged."""
    dY = inputs.randn_bf16((M, ld8(N)), seed=seed, device=DEV)[:, :N]
    W = inputs.randn_bf16((N, ld8(K)), seed=seed + 1, std=w_std or 1.0 / np.sqrt(max(N, 1)), device=DEV)[:, :K]
    Z = inputs.randn_bf16((M, K), seed=seed + 2, std=z_std, device=DEV)
    return dY, W, Z


def run(dY, W, Z, act, **kw):
    d = gb.linear_dact(dY, W, Z, act=act, **kw)
    gb.device_status()
    return bits(d)


def ref(dY, W, Z, act):
    return oracle.dact(bits(dY), bits(W), bits(Z), act)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M,N,K", [(128, 64, 256), (256, 512, 256), (300, 700, 520), (1, 8, 1), (129, 72, 257),
                                   (513, 1000, 96), (127, 4096, 255), (1000, 200, 1500)])
def test_dact_random(M, N, K, act):
    dY, W, Z = operands(M, N, K, seed=M + 3 * N + 5 * K, z_std=2.0)
    assert_close(run(dY, W, Z, act), ref(dY, W, Z, act), f"{M}x{N}x{K} {act}")
    assert "kernel=linear_dact" in gb.last_plan()


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("M,N,K", [(128, 64, 256), (300, 200, 520), (257, 129, 130), (64, 640, 384)])
def test_dact_integer_bit_exact(M, N, K, pair):
    """Integer dY and W (exact sums), integer Z (ReLU' exactly 0 or 1; the identity's 1):
    the GPU reproduces the oracle bit for bit, signed zeros included."""
    gb.set_config(f"pair={pair}")
    dY = int_tensor((M, ld8(N)), 1).to(DEV)[:, :N]
    W = int_tensor((N, ld8(K)), 2).to(DEV)[:, :K]
    Z = int_tensor((M, K), 3, -3, 3).to(DEV)
    for act in ("relu", "none"):
        assert_bitexact(run(dY, W, Z, act), ref(dY, W, Z, act), f"{act} pair={pair}")


def test_dact_index_pattern():
    """D[m,k] = m + 16 k exactly: catches a W read as [K,N] or swapped indices."""
    M, N, K = 300, 64, 264
    dy = torch.zeros(M, N)
    dy[:, 0] = torch.arange(M) % 128
    dy[:, 1] = 1
    w = torch.zeros(N, K)
    w[0, :] = 1
    w[1, :] = 16 * (torch.arange(K) % 16)
    Z = torch.ones(M, K).to(torch.bfloat16).to(DEV)
    want = ((torch.arange(M) % 128)[:, None] + 16 * (torch.arange(K) % 16)[None, :]).float().to(torch.bfloat16)
    for act in ("relu", "none"):
        assert_bitexact(run(dy.to(torch.bfloat16).to(DEV), w.to(torch.bfloat16).to(DEV), Z, act), bits(want), act)


@pytest.mark.parametrize("cfg", ["pair=0", "pair=1", "epi=1", "epi=2", "stages=3", "boxes=4", "bn=128",
                                 "pingpong=1", "grid=8", "persistent=0", "wide=1", "wide=1,pingpong=1",
                                 "wide=1,epi=1,bn=128"])
def test_dact_configs_identical_bits(cfg):
    """Every schedule gives the same bits (the per-element sum order inside a tile is fixed)."""
    M, N, K = 400, 320, 600
    dY, W, Z = operands(M, N, K, seed=41, w_std=0.05)
    base = run(dY, W, Z, "silu")
    assert_close(base, ref(dY, W, Z, "silu"), "default")
    gb.set_config(cfg)
    got = run(dY, W, Z, "silu")
    assert_bitexact(got, base, cfg)
    assert_close(got, ref(dY, W, Z, "silu"), cfg)


@pytest.mark.parametrize("act", ["gelu_tanh", "relu"])
def test_dact_unaligned_z_and_d(act):
    """K = 4099: rows of Z and D are 8198 bytes apart, so both go through the
    shared-memory transposes with plain loads and stores."""
    M, N, K = 200, 128, 4099
    dY, W, Z = operands(M, N, K, seed=50)
    got = run(dY, W, Z, act)
    plan = gb.last_plan()
    assert "d_store=st.transposed" in plan and "r_load=ld.transposed" in plan, plan
    assert_close(got, ref(dY, W, Z, act), f"K=4099 {act}")
    gb.set_config("r_async=1")
    pre = run(dY, W, Z, act)
    assert "r_load=cp.async" in gb.last_plan(), gb.last_plan()
    assert_bitexact(pre, got, f"K=4099 {act} cp.async queue vs loads at use")


def test_dact_strided_views_and_vector_loads():
    """dY and W as views (leading dimension > row), Z with aligned rows read by vector
    loads after a split is ruled out, D as a column slice of a bigger buffer."""
    M, N, K = 190, 136, 300
    dYbig = inputs.randn_bf16((M, N + 40), seed=60, device=DEV)
    Wbig = inputs.randn_bf16((N, K + 28), seed=61, std=0.1, device=DEV)  # leading dimension 328
    dY, W = dYbig[:, 8:8 + N], Wbig[:, 16:16 + K]
    Zbig = inputs.randn_bf16((M, K + 13), seed=62, device=DEV)
    Z = Zbig[:, 5:5 + K]
    Dbig = torch.zeros((M, K + 9), dtype=torch.bfloat16, device=DEV)
    D = Dbig[:, 3:3 + K]
    gb.linear_dact(dY, W, Z, act="gelu_tanh", out=D)
    gb.device_status()
    want = oracle.dact(bits(dY.contiguous()), bits(W.contiguous()), bits(Z.contiguous()), "gelu_tanh")
    assert_close(bits(D), want, "strided")


def test_dact_d_aliases_z():
    M, N, K = 256, 192, 512
    dY, W, Z = operands(M, N, K, seed=70, w_std=0.1)
    want = ref(dY, W, Z, "silu")
    Zd = Z.clone()
    gb.linear_dact(dY, W, Zd, act="silu", out=Zd)
    gb.device_status()
    assert_close(bits(Zd), want, "D == Z")


def test_dact_empty_contraction_and_outputs():
    """N = 0: D = 0 * act'(Z).  For ReLU and the identity act' is exactly 0 or 1, so the
    signed zeros match the oracle bit for bit; for GELU and SiLU, act' of very negative z
    is a tiny negative number that each side rounds in its own way (possibly to +0), so
    only the value 0 is checked, not the sign of the zero.  M or K = 0: no-op."""
    M, K = 130, 300
    dY = torch.zeros((M, 0), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((0, K), dtype=torch.bfloat16, device=DEV)
    Z = inputs.randn_bf16((M, K), seed=80, std=3.0, device=DEV)
    for act in ACTS:
        D = gb.linear_dact(dY, W, Z, act=act)
        gb.device_status()
        want = oracle.dact(bits(dY), bits(W), bits(Z), act)
        if act in ("relu", "none"):
            assert_bitexact(bits(D), want, act)
        else:
            assert torch.all(D.float() == 0), act
            assert_close(bits(D), want, act)
    out = gb.linear_dact(torch.zeros((0, 8), dtype=torch.bfloat16, device=DEV),
                         torch.zeros((8, 16), dtype=torch.bfloat16, device=DEV),
                         torch.zeros((0, 16), dtype=torch.bfloat16, device=DEV), act="relu")
    assert out.shape == (0, 16)


def test_dact_mlp_backward_8192x14336x4096():
    """The full-size MLP backward product in the benchmark's launch configuration:
    sampled on a 256 x 256 grid and on 65536 independent entries (>= 99 % within one
    bf16 ulp of the float64 result)."""
    w = inputs.mlp_dact(device=DEV)
    D = gb.linear_dact(w["dY"], w["W"], w["Z"], act="gelu_tanh")
    gb.device_status()
    M, N, K = 8192, 14336, 4096
    r, c = inputs.sample_indices(M, K, seed=31)
    rr, cc = torch.from_numpy(r).to(DEV), torch.from_numpy(c).to(DEV)
    got = bits(D[rr][:, cc])
    dYs, Ws, Zs = bits(w["dY"][rr]), bits(w["W"][:, cc]), bits(w["Z"][rr][:, cc])
    assert_close(got, oracle.dact(dYs, Ws, Zs, "gelu_tanh"), "mlp_dact grid")
    h = ulp_hist(got, oracle.dact_f64(dYs, Ws, Zs, "gelu_tanh"))
    assert sum(v for k, v in h.items() if k <= 1) >= 0.99 * got.size, h
    i, j = inputs.sample_pairs(M, K, seed=32)
    check_pairs("dact", D, w, i, j, act="gelu_tanh", what="mlp_dact pairs")


@pytest.mark.parametrize("cg,n", [(2, 256), (2, 128), (1, 256), (1, 128)])
def test_mma_rate_probe(cg, n):
    """The tensor-core rate probe returns a positive rate no larger than the dense bf16
    rate per SM and clock can be (8192 FLOP; 5 % slack for the timing's edges)."""
    rate, cyc = gb.measure_mma_rate(cta_group=cg, n=n, num_mma=4096, units=1)
    assert cyc > 0 and 0 < rate <= 8192 * 1.05, (rate, cyc)
