"""The calls under CUDA-graph capture: each call enqueues only stream work (a workspace
clear and one kernel launch) once the per-device setup has run, so a captured graph
replays the same computation on whatever the captured buffers hold at replay time."""
import numpy as np
import pytest
import torch

import oracle
import dense_bf16_gemm_persistent_gb300 as gb
from dense_bf16_gemm_persistent_gb300 import inputs
from tests.gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset():
    gb.set_config(None)
    yield
    gb.set_config(None)
    gb.device_status()


def _fill(t: torch.Tensor, seed: int, std: float = 1.0) -> None:
    t.copy_(inputs.randn_bf16(tuple(t.shape), seed=seed, std=std))


def test_graph_capture_and_replay():
    M, N, K = 520, 776, 640
    A = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    B = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    B3 = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    bias = torch.empty((N,), dtype=torch.bfloat16, device=DEV)
    R = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    Ms, Ns, Ks = 127, 96, 16384                      # skinny: the split-K call clears its workspace
    As = torch.empty((Ms, Ks), dtype=torch.bfloat16, device=DEV)
    Bs = torch.empty((Ns, Ks), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(gb.splitk_workspace_bytes(Ms, Ns, Ks, 0), dtype=torch.uint8, device=DEV)
    D1 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    D2 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    D3 = torch.empty((Ms, Ns), dtype=torch.bfloat16, device=DEV)

    def calls(stream):
        gb.linear(A, B, bias, R, act="gelu_tanh", out=D1, stream=stream)
        gb.ffn_gated(A, B, B3, out=D2, stream=stream)
        gb.linear(As, Bs, out=D3, split_k="auto", workspace=ws, stream=stream)

    def fill_all(seed):
        _fill(A, seed)
        _fill(B, seed + 1, 1.0 / np.sqrt(K))
        _fill(B3, seed + 2, 1.0 / np.sqrt(K))
        _fill(bias, seed + 3, 0.1)
        _fill(R, seed + 4)
        _fill(As, seed + 5)
        _fill(Bs, seed + 6, 1.0 / np.sqrt(Ks))

    def check(what):
        assert_close(bits(D1), oracle.linear(bits(A), bits(B), bits(bias), bits(R), "gelu_tanh"), what + " linear")
        assert_close(bits(D2), oracle.ffn_gated(bits(A), bits(B), bits(B3)), what + " ffn")
        assert_close(bits(D3), oracle.linear(bits(As), bits(Bs)), what + " split-K")

    fill_all(300)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                    # per-device setup happens outside the capture
        calls(side)
    torch.cuda.current_stream().wait_stream(side)
    gb.device_status()
    check("eager")

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls(torch.cuda.current_stream())
    for seed in (400, 500):                          # new contents in the captured buffers
        fill_all(seed)
        for D in (D1, D2, D3):
            D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        gb.device_status()
        check(f"replay {seed}")
