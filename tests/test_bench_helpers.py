"""bench.py helpers that need no GPU: the device-code hash and launch plan that keep
recorded ncu traffic attached to the launch it was measured on."""
import os
import shutil

import bench


def test_code_tokens_drop_comments_and_layout_only():
    src = 'int a = 1;  // one\n/* block\n comment */ char q = \'/\';\nconst char* s = "x // y /* z */";\n'
    assert bench.code_tokens(src) == 'int a = 1; char q = \'/\'; const char* s = "x // y /* z */";'
    assert bench.code_tokens("a  =\n\tb; // c") == bench.code_tokens("a = b;")
    assert bench.code_tokens("a = b;") != bench.code_tokens("a = c;")


def test_recorded_traffic_follows_the_code(tmp_path, monkeypatch):
    csrc = tmp_path / "dense_bf16_gemm_persistent_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cuh").write_text("__global__ void k() { int x = 1; }\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "traffic_w.txt").write_text(
        f"# note\ndram_bytes_per_launch: 1234\nsource_sha256: {h}\n")
    assert bench.recorded_traffic("w") == 1234.0
    (csrc / "k.cuh").write_text("// a new comment\n__global__ void k() {\n  int x = 1;\n}\n")
    assert bench.recorded_traffic("w") == 1234.0          # comments and layout: same code
    (csrc / "host.cu").write_text("int host_side_planner = 1;\n")
    assert bench.recorded_traffic("w") == 1234.0          # host code is pinned by the plan instead
    (tmp_path / "profiles" / "traffic_w.txt").write_text(
        f"dram_bytes_per_launch: 1234\nsource_sha256: {h}\nplan: tile=256x256x64 stages=6\n")
    assert bench.recorded_traffic("w", "tile=256x256x64 stages=6") == 1234.0
    assert bench.recorded_traffic("w", "tile=256x256x64 stages=5") is None   # another launch
    (csrc / "k.cuh").write_text("__global__ void k() { int x = 2; }\n")
    assert bench.recorded_traffic("w", "tile=256x256x64 stages=6") is None   # changed device code
