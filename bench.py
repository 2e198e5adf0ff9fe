"""Benchmark: bf16 GEMM + fused epilogue throughput (TFLOP/s) on GB300.

One step = one call of the hot path on one batch of synthetic input: by default
the MLP-forward linear layer D = GELU_tanh(X W^T + bias) with X[8192,4096],
W[14336,4096], bias[14336] (X ~ N(0,1), W and bias ~ N(0,0.02), bf16, fp32
accumulation).  `--workload llama_ffn` times the Llama-FFN fusion instead.

After the timed steps, the same run times every configuration once more (the
plain matmul as a latency, the MLP linear, the Llama FFN, the 64-bit-indexing
case, the stored pre-activation, the backward activation-gradient product and
the skinny, short-K and unaligned ragged rows) and reports each under
`per_shape`, with its median and minimum launch time, its roofline fraction,
plan and sampled SM clock, and -- from the CPU-oracle leg -- its error on
sampled entries.  `nominal_peak` is the tensor cores' dense bf16 rate per SM and
clock measured by a tcgen05 probe, times SMs and clock.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  `value` is the device-timed throughput of the
whole job (all ranks; inputs resident in HBM); `e2e` is the same metric with the
host->device copy of the inputs from pinned memory and the device->host copy of
D inside the timed region; `roofline` relates the kernel's achieved TFLOP/s to
the measured dense bf16 peak; `cpu_baseline` is the CPU oracle timed on a
bounded sample of the same workload.  `--impl reference` times that oracle as
the reference arm.  Under torchrun each rank runs its own replica (the workload
has no exchange step): weak scaling, no data-path collective.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "bf16 GEMM+epilogue TFLOP/s and % of GB300 dense bf16 peak, per shape"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1000 * 1000

WORKLOADS = {
    "mlp_gelu": dict(M=8192, N=14336, K=4096, kind="linear", act="gelu_tanh", bias=True, residual=False,
                     name="mlp_gelu_8192x14336x4096"),
    "llama_ffn": dict(M=8192, N=14336, K=4096, kind="ffn", act="none", bias=False, residual=False,
                      name="llama_ffn_8192x14336x4096"),
    "plain": dict(M=256, N=384, K=512, kind="linear", act="none", bias=False, residual=False,
                  name="plain_256x384x512"),
    "mlp_noepi": dict(M=8192, N=14336, K=4096, kind="linear", act="none", bias=False, residual=False,
                      name="linear_noepi_8192x14336x4096"),
    # the MLP linear storing also its pre-activation Z = bf16(X.W^T + bias) (second output)
    "mlp_preact": dict(M=8192, N=14336, K=4096, kind="linear", act="gelu_tanh", bias=True, residual=False,
                       preact=True, name="mlp_preact_8192x14336x4096"),
    "int64": dict(M=65536, N=4096, K=65536, kind="linear", act="none", bias=False, residual=False,
                  name="int64_65536x4096x65536"),
    # the MLP layer's backward activation-gradient product D[M,K] = (dY[M,N] . W[N,K]) * gelu'(Z[M,K])
    "mlp_dact": dict(M=8192, N=14336, K=4096, kind="dact", act="gelu_tanh", bias=False, residual=False,
                     name="mlp_dact_8192x14336x4096"),
    # the MLP linear in the MatmulOp form: X[8192,4096] . W[4096,14336] (the weight stored [K,N])
    "mlp_matmul": dict(M=8192, N=14336, K=4096, kind="matmul", act="gelu_tanh", bias=True, residual=False,
                       name="mlp_matmul_8192x14336x4096"),
}

# Every configuration, timed after the main workload: plain matmul (latency), MLP linear,
# Llama FFN, 64-bit indexing, the MLP with its stored pre-activation, the backward
# activation-gradient product, and ragged rows (skinny and long K, short K, unaligned N).
PER_SHAPE = ["plain", "mlp_gelu", "llama_ffn", "int64", "mlp_preact", "mlp_dact", "mlp_matmul",
             "ragged:127,96,65536", "ragged:8191,96,65536", "ragged:8191,12288,64",
             "ragged:1000,4099,4096", "ragged:3001,4099,4096", "ragged:8191,4099,4096"]


def workload(spec: str) -> dict:
    """A named workload, or "ragged:M,N,K" (D = A.B^T + R through the split-K entry point)."""
    if spec in WORKLOADS:
        return dict(WORKLOADS[spec])
    if spec.startswith("ragged:"):
        M, N, K = (int(v) for v in spec.split(":", 1)[1].split(","))
        return dict(M=M, N=N, K=K, kind="linear", act="none", bias=False, residual=True, split_k="auto",
                    name=f"ragged_residual_{M}x{N}x{K}")
    raise SystemExit(f"unknown workload {spec!r}")


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(dist, x: float, device=None) -> float:
    """Max of a float over ranks (identity on one rank)."""
    if dist is None:
        return x
    import torch
    dev = device if (device is not None and dist.get_backend() == "nccl") else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_replicas(per_rank_units: float, local_seconds: float, dist, device=None):
    """Whole-job throughput of N independent replicas: all units / the slowest rank's time."""
    world = dist.get_world_size() if dist is not None else 1
    slowest = reduce_max(dist, local_seconds, device)
    return per_rank_units * world / slowest, slowest


# ------------------------------------------------------------------ peaks, clocks, traffic

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background (read-only queries)."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t_marks = []
        self.out_path = os.path.join("/tmp", f"gbgemm_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.out_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self):
        self.t_marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.out_path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[4], parts[6:10]))
                except Exception:
                    continue
        os.unlink(self.out_path)
        if not rows:
            return None
        t0, t1 = (self.t_marks[0], self.t_marks[-1]) if len(self.t_marks) >= 2 else (0, 1e30)
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0] or rows
        sm = sorted(r[1] for r in inside)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[4]) if v.lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": "timed region (+-1 s) at 100 ms sampling"}


def code_tokens(text: str) -> str:
    """C++/CUDA source with comments removed and whitespace collapsed (string and
    character literals kept verbatim): what the compiler sees, not how it is annotated."""
    out, i, n, quote = [], 0, len(text), None
    while i < n:
        c = text[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 2
                continue
            if c == quote:
                quote = None
            i += 1
        elif c in "\"'":
            quote = c
            out.append(c)
            i += 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the device code (the kernel headers, comments and layout ignored). Recorded
    counters stay attached to the code they were taken on; together with the launch plan
    (recorded beside them) this pins the launch they describe."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_bf16_gemm_persistent_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith(".cuh"):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, plan: str | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current device code and (when the record names one) the same launch plan; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != kernel_source_hash():
            return None
        if "plan" in kv and plan is not None and kv["plan"] != plan.strip():
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ workloads

def out_shape(wl: dict) -> tuple[int, int]:
    """D is [M, N]; for the activation gradient the contraction runs over N and D is [M, K]."""
    return (wl["M"], wl["K"]) if wl["kind"] == "dact" else (wl["M"], wl["N"])


def make_inputs(wl: dict, device):
    from dense_bf16_gemm_persistent_gb300 import inputs
    M, N, K = wl["M"], wl["N"], wl["K"]
    if wl["kind"] == "ffn":
        return inputs.llama_ffn(device=device, M=M, N=N, K=K)
    if wl["kind"] == "dact":
        return inputs.mlp_dact(device=device, M=M, N=N, K=K)
    if wl["kind"] == "matmul":  # the MLP recipe with W laid out [K, N]
        t = inputs.mlp_gelu(device=device, M=M, N=N, K=K)
        t["B"] = t["B"].t().contiguous()
        t.setdefault("R", None)
        return t
    if wl["name"].startswith("ragged"):
        t = inputs.ragged(M, N, K, device=device)
    elif wl["name"].startswith("int64"):
        t = inputs.int64_case(device=device, M=M, N=N, K=K)
    elif wl["name"].startswith("plain") or wl["name"].startswith("linear_noepi"):
        t = inputs.plain(device=device, M=M, N=N, K=K)
    else:
        return inputs.mlp_gelu(device=device, M=M, N=N, K=K)
    t.setdefault("bias", None)
    t.setdefault("R", None)
    return t


def algorithmic_bytes(wl: dict) -> float:
    """One read of every input and one write of D (and of Z, the pre-activation, when
    the workload stores it), all bf16."""
    M, N, K = wl["M"], wl["N"], wl["K"]
    if wl["kind"] == "dact":  # dY, W and Z read once, D written once
        return 2.0 * (M * N + N * K + 2 * M * K)
    b = M * K + N * K * (2 if wl["kind"] == "ffn" else 1) + M * N * (2 if wl.get("preact") else 1)
    if wl.get("bias"):
        b += N
    if wl.get("residual"):
        b += M * N
    return 2.0 * b


def flops_per_step(wl: dict) -> float:
    per = 2.0 * wl["M"] * wl["N"] * wl["K"]
    return 2 * per if wl["kind"] == "ffn" else per


def step_fn(wl: dict, t: dict, out, workspace=None, stream=None):
    import dense_bf16_gemm_persistent_gb300 as gb
    if wl["kind"] == "ffn":
        return lambda: gb.ffn_gated(t["X"], t["W1"], t["W3"], out=out, stream=stream)
    if wl["kind"] == "dact":
        return lambda: gb.linear_dact(t["dY"], t["W"], t["Z"], act=t["act"], out=out, stream=stream)
    if wl.get("preact"):
        import torch
        z = torch.empty_like(out)
        return lambda: gb.linear_preact(t["A"], t["B"], t.get("bias"), t.get("R"), act=t["act"], out=out,
                                        preact=z, stream=stream)
    if wl["kind"] == "matmul":
        return lambda: gb.matmul(t["A"], t["B"], t.get("bias"), t.get("R"), act=t["act"], out=out, stream=stream)
    split = wl.get("split_k")
    return lambda: gb.linear(t["A"], t["B"], t.get("bias"), t.get("R"), act=t["act"], out=out, split_k=split,
                             workspace=workspace, stream=stream)


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)

def oracle_sample_inputs(wl: dict, rows: int) -> dict:
    """CPU-generated inputs of the workload's recipe for its first `rows` output rows."""
    from dense_bf16_gemm_persistent_gb300 import inputs
    small = dict(wl, M=rows)
    t = make_inputs(small, "cpu")
    return {k: (inputs.to_bits(v) if hasattr(v, "dtype") else v) for k, v in t.items() if v is not None}


def oracle_sample_run(wl: dict, h: dict, rows: int):
    """Run the CPU oracle on the first `rows` output rows.  Returns (seconds, flops, threads)."""
    import oracle
    K, N = wl["K"], wl["N"]
    if wl["kind"] == "ffn":
        t0 = time.perf_counter()
        oracle.ffn_gated(h["X"][:rows], h["W1"], h["W3"])
        return time.perf_counter() - t0, 4.0 * rows * N * K, oracle.num_threads()
    if wl["kind"] == "dact":
        t0 = time.perf_counter()
        oracle.dact(h["dY"][:rows], h["W"], h["Z"][:rows], h["act"])
        return time.perf_counter() - t0, 2.0 * rows * N * K, oracle.num_threads()
    R = h.get("R")
    t0 = time.perf_counter()
    run = oracle.linear_preact if wl.get("preact") else oracle.matmul if wl["kind"] == "matmul" else oracle.linear
    run(h["A"][:rows], h["B"], h.get("bias"), None if R is None else R[:rows], h["act"])
    return time.perf_counter() - t0, 2.0 * rows * N * K, oracle.num_threads()


def calibrate_rows(wl: dict, target_s: float) -> tuple[int, dict]:
    """Rows of output the oracle computes in about target_s seconds, and their inputs.  The
    timing probe has two rows per host thread, so the estimate sees the oracle's parallel
    rate (it parallelises over rows)."""
    import oracle
    probe = min(max(4, 2 * oracle.num_threads()), wl["M"])
    h = oracle_sample_inputs(wl, probe)
    dt, _, _ = oracle_sample_run(wl, h, probe)
    rows = min(max(probe, int(probe * target_s / max(dt, 1e-3))), wl["M"])
    return rows, oracle_sample_inputs(wl, rows)


def cpu_baseline(wl: dict, target_s: float = 12.0) -> dict:
    rows, h = calibrate_rows(wl, target_s)
    dt, fl, threads = oracle_sample_run(wl, h, rows)
    cols = out_shape(wl)[1]
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows} full output rows ({rows}x{cols} entries) of {wl['name']}, "
                      f"{dt:.1f} s on {threads} host threads"}


def run_reference(args, wl: dict):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    rows, h = calibrate_rows(wl, args.ref_step_s)
    for _ in range(args.warmup):
        oracle_sample_run(wl, h, rows)
    total_s, total_fl, threads = 0.0, 0.0, 1
    for _ in range(args.steps):
        dt, fl, threads = oracle_sample_run(wl, h, rows)
        total_s += dt
        total_fl += fl
    value = total_fl / total_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"each step: {rows} full output rows ({rows}x{wl['N']}, K={wl['K']}) "
                                       f"of {wl['name']} on {threads} host threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def needs_l2_flush(wl: dict) -> bool:
    return algorithmic_bytes(wl) < 2 * L2_BYTES


def config_of(wl: dict) -> dict:
    ws = algorithmic_bytes(wl)
    if wl["kind"] == "ffn":
        epi = "silu(acc1) * acc3"
    elif wl["kind"] == "dact":
        epi = f"(dY.W) * {wl['act']}'(Z)"
    elif wl.get("residual"):
        epi = "acc + R"
    elif wl.get("bias"):
        epi = f"{wl['act']}(acc + bias)" + (", and Z = acc + bias" if wl.get("preact") else "")
    else:
        epi = "none"
    cfg = {"workload": wl["name"], "M": wl["M"], "N": wl["N"], "K": wl["K"], "epilogue": epi,
           "l2": (f"flushed between timed steps (256 MB write; inputs+output {ws / 1e6:.1f} MB)"
                  if needs_l2_flush(wl) else f"no flush: inputs+output {ws / 1e6:.0f} MB > 2x 129 MB L2")}
    if wl.get("split_k"):
        cfg["split_k"] = wl["split_k"]
    return cfg


# ------------------------------------------------------------------ our arm

def launch_stats(launch_ms: list[float]) -> dict:
    ms = sorted(launch_ms)
    return {"mean": sum(ms) / len(ms), "median": ms[len(ms) // 2], "min": ms[0], "max": ms[-1], "n": len(ms)}


def roofline_of(wl: dict, launch_ms: float, peaks: dict, peak_src: str, traffic=None) -> dict:
    """Achieved vs the measured peak of the kernel's bound (tensor or HBM), from the
    arithmetic intensity of the workload against the ridge of the measured peaks."""
    fl = flops_per_step(wl)
    alg_bytes = algorithmic_bytes(wl)
    achieved = fl / (launch_ms / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    if fl / alg_bytes >= peak * 1e12 / (hbm * 1e9):
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                "traffic": traffic, "peak_source": f"{peak_src} bf16_tflops (burst, cuBLAS 8192^3)",
                "frac_of_sustained": achieved / peak_sustained}
    gbs = alg_bytes / (launch_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": traffic,
            "peak_source": f"{peak_src} hbm_gbs (copy)", "tflops": achieved}


def _bits(t):
    from dense_bf16_gemm_persistent_gb300 import inputs
    return inputs.to_bits(t)


def sampled_accuracy(wl: dict, t: dict, out, n: int, seed: int) -> dict:
    """The CPU oracle at n independent output entries of this run's D (outside every timed
    region): max |err|, the library's tolerance |err| <= 2^-7 (|ref| + 1), and the bf16-ULP
    histogram of D against the float64 result rounded once to bf16."""
    import numpy as np
    import torch
    import oracle
    from dense_bf16_gemm_persistent_gb300 import inputs
    Mo, No = out_shape(wl)
    i, j = inputs.sample_pairs(Mo, No, n=n, seed=seed)
    dev = out.device
    ti, tj = torch.from_numpy(i).to(dev), torch.from_numpy(j).to(dev)
    got = _bits(out[ti, tj])
    ref = np.empty(n, np.uint16)
    ref64 = np.empty(n, np.float64)
    chunk = 4096
    for s0 in range(0, n, chunk):
        ci, cj = ti[s0:s0 + chunk], tj[s0:s0 + chunk]
        sl = slice(s0, s0 + ci.numel())
        if wl["kind"] == "ffn":
            args = (_bits(t["X"][ci]), _bits(t["W1"][cj]), _bits(t["W3"][cj]))
            ref[sl] = oracle.ffn_entries(*args)
            ref64[sl] = oracle.ffn_entries(*args, f64=True)
        elif wl["kind"] == "dact":
            args = (_bits(t["dY"][ci]), _bits(t["W"][:, cj].t().contiguous()), _bits(t["Z"][ci, cj]))
            ref[sl] = oracle.dact_entries(*args, act=t["act"])
            ref64[sl] = oracle.dact_entries(*args, act=t["act"], f64=True)
        else:
            bias = _bits(t["bias"][cj]) if t.get("bias") is not None else None
            R = _bits(t["R"][ci, cj]) if t.get("R") is not None else None
            # B rows [N, K]; for the matmul form, columns of B [K, N]
            B = _bits(t["B"][:, cj].t().contiguous()) if wl["kind"] == "matmul" else _bits(t["B"][cj])
            A = _bits(t["A"][ci])
            ref[sl] = oracle.linear_entries(A, B, bias, R, t["act"])
            ref64[sl] = oracle.linear_entries(A, B, bias, R, t["act"], f64=True)
    g = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (ref.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.abs(g - r)

    def key(x):  # bf16 patterns in numeric order
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7fff), x & 0x7fff)
    d = np.abs(key(got) - key(oracle.f64_to_bf16(ref64)))
    hist = {str(k): int((d == k).sum()) for k in range(3)}
    hist[">=3"] = int((d >= 3).sum())
    return {"entries": int(n), "max_abs_err": float(np.nanmax(err)) if n else 0.0,
            "tolerance_ok": bool(np.all(err <= 2.0 ** -7 * (np.abs(r) + 1.0))),
            "within_1ulp_of_f64": float((d <= 1).mean()), "ulp_hist_vs_f64": hist,
            "sample": f"{n} independent (i, j) entries, numpy default_rng({seed})"}


def time_steps(step, steps: int, warmup: int, prewarm_s: float, flush, stream, local: int, dist=None, device=None):
    """Pre-warm, W untimed steps, then K steps with an event pair around each launch on
    the launching stream (an L2 flush between the pairs when the working set fits in L2),
    with the SM clock sampled during the timed region."""
    import torch
    import dense_bf16_gemm_persistent_gb300 as gb
    sampler = ClockSampler(local)
    t_end = time.time() + prewarm_s
    step()
    torch.cuda.synchronize()
    while time.time() < t_end:
        for _ in range(10):
            step()
        torch.cuda.synchronize()
    for _ in range(warmup):
        step()
    gb.device_status()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(dist, device)
    torch.cuda.synchronize()
    sampler.mark()
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    barrier(dist, device)
    gb.device_status()
    return [ev0[i].elapsed_time(ev1[i]) for i in range(steps)], sampler.stop()


def measure_shape(spec: str, args, device, local: int, peaks: dict, peak_src: str) -> dict:
    """One per_shape entry: the workload's own inputs, timed like the main step."""
    import torch
    import dense_bf16_gemm_persistent_gb300 as gb
    wl = workload(spec)
    t = make_inputs(wl, device)
    out = torch.empty(out_shape(wl), dtype=torch.bfloat16, device=device)
    ws = None
    if wl.get("split_k"):
        ws = torch.empty(max(1, gb.splitk_workspace_bytes(wl["M"], wl["N"], wl["K"], 0)), dtype=torch.uint8,
                         device=device)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device) if needs_l2_flush(wl) else None
    steps = args.shape_steps if flops_per_step(wl) < 1e13 else max(3, args.shape_steps // 4)
    launch_ms, clocks = time_steps(step_fn(wl, t, out, ws), steps, max(3, args.warmup), args.shape_prewarm_s, flush,
                                   torch.cuda.current_stream(device), local)
    st = launch_stats(launch_ms)
    plan = gb.last_plan()
    entry = {"workload": wl["name"], "M": wl["M"], "N": wl["N"], "K": wl["K"],
             "epilogue": config_of(wl)["epilogue"], "ms_median": st["median"], "ms_min": st["min"],
             "ms_mean": st["mean"], "launches": st["n"],
             "tflops": flops_per_step(wl) / (st["median"] / 1e3) / 1e12,
             "roofline": roofline_of(wl, st["median"], peaks, peak_src),
             "plan": plan, "clocks": clocks, "l2": config_of(wl)["l2"]}
    if wl.get("split_k"):
        entry["entry_point"] = "gb_gemm_linear_splitk (automatic split count, caller workspace)"
    if spec == "plain":
        entry["latency_us"] = {"median": st["median"] * 1e3, "min": st["min"] * 1e3}
    if not args.skip_cpu:
        n = 16384 if wl["K"] <= 16384 else 4096
        entry["accuracy"] = sampled_accuracy(wl, t, out, n, seed=7)
    del t, out, ws, flush
    torch.cuda.empty_cache()
    return entry


def nominal_peak(sms: int, sm_max_mhz: float, sm_load_mhz: float | None) -> dict:
    """SMs x clock x the dense bf16 rate per SM and clock of the kernels' MMA shape,
    pinned by the tcgen05 probe (one CTA pair alone, and every SM pair at once)."""
    import dense_bf16_gemm_persistent_gb300 as gb
    r1, c1 = gb.measure_mma_rate(cta_group=2, n=256, num_mma=16384, units=1)
    ra, ca = gb.measure_mma_rate(cta_group=2, n=256, num_mma=16384, units=sms // 2)
    d = {"probe": "tcgen05.mma.cta_group::2.kind::f16, M=256 N=256 K=16 bf16 -> fp32, back to back from shared "
                  "memory (no loads, no epilogue), clock64 cycles",
         "flops_per_clk_per_sm": r1, "cycles_per_mma": c1,
         "flops_per_clk_per_sm_all_sms": ra, "cycles_per_mma_all_sms": ca,
         "sms": sms, "sm_max_mhz": sm_max_mhz, "tflops_at_max_clock": r1 * sms * sm_max_mhz * 1e6 / 1e12}
    if sm_load_mhz:
        d["sm_mhz_under_load"] = sm_load_mhz
        d["tflops_at_clock_under_load"] = r1 * sms * sm_load_mhz * 1e6 / 1e12
    return d


def run_ours(args, wl: dict):
    import torch
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")
    import dense_bf16_gemm_persistent_gb300 as gb
    gb.lib()
    gb.set_config(args.config)

    t = make_inputs(wl, device)
    out = torch.empty(out_shape(wl), dtype=torch.bfloat16, device=device)
    ws = None
    if wl.get("split_k"):
        ws = torch.empty(max(1, gb.splitk_workspace_bytes(wl["M"], wl["N"], wl["K"], 0)), dtype=torch.uint8,
                         device=device)
    step = step_fn(wl, t, out, ws)
    stream = torch.cuda.current_stream(device)
    fl = flops_per_step(wl)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device) if needs_l2_flush(wl) else None

    # timed region: K steps, an event pair around each launch on the launching stream
    launch_ms, clocks = time_steps(step, args.steps, args.warmup, args.prewarm_s, flush, stream, local, dist, device)
    local_ms = sum(launch_ms)
    value, slowest_s = aggregate_replicas(fl * args.steps / 1e12, local_ms / 1e3, dist, device)
    plan = gb.last_plan()

    # End to end through the public API: every step copies its inputs from pinned
    # host memory to the device, runs the call, and copies D back to pinned host
    # memory.  Steps are pipelined the way a host-fed user would run them: three
    # streams (copy in, compute, copy out) and two device buffers for inputs and
    # outputs, so step i+1's inputs move while step i computes and step i-1's
    # result drains.  Every step's copies are inside the timed region.
    e2e = None
    if not args.skip_e2e:
        if wl["kind"] == "ffn":
            names = ["X", "W1", "W3"]
        elif wl["kind"] == "dact":
            names = ["dY", "W", "Z"]
        else:
            names = [k for k in ("A", "B", "bias", "R") if t.get(k) is not None]
        host = {k: t[k].cpu().pin_memory() for k in names}
        s_in, s_comp, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
        dev_in = [{k: torch.empty_like(t[k]) for k in names} for _ in range(2)]
        dev_out = [torch.empty(out_shape(wl), dtype=torch.bfloat16, device=device) for _ in range(2)]
        host_out = [torch.empty(out_shape(wl), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        steps_b = []
        for bi in range(2):
            tin = dict(dev_in[bi])
            tin["act"] = t.get("act")
            steps_b.append(step_fn(wl, tin, dev_out[bi], ws, stream=s_comp))
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = host_out[0].numel() * host_out[0].element_size()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def run_pipeline(n: int, compute: bool = True):
            for i in range(n):
                bi = i % 2
                if i >= 2:
                    s_in.wait_event(ev_done[bi])      # compute i-2 has read dev_in[bi]
                with torch.cuda.stream(s_in):
                    for k in names:
                        dev_in[bi][k].copy_(host[k], non_blocking=True)
                ev_in[bi].record(s_in)
                s_comp.wait_event(ev_in[bi])
                if i >= 2:
                    s_comp.wait_event(ev_out[bi])     # copy-out i-2 has read dev_out[bi]
                if compute:
                    steps_b[bi]()
                ev_done[bi].record(s_comp)
                s_out.wait_event(ev_done[bi])
                with torch.cuda.stream(s_out):
                    host_out[bi].copy_(dev_out[bi], non_blocking=True)
                ev_out[bi].record(s_out)
            return ev_out[(n - 1) % 2]

        run_pipeline(max(2, args.warmup))
        torch.cuda.synchronize()
        n_e2e = max(3, args.steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist, device)
        torch.cuda.synchronize()
        e0.record(s_in)
        last = run_pipeline(n_e2e)
        s_in.wait_event(last)
        s_in.wait_event(ev_out[n_e2e % 2])
        e1.record(s_in)
        torch.cuda.synchronize()
        barrier(dist, device)
        gb.device_status()
        e2e_ms = e0.elapsed_time(e1)
        e2e_val, _ = aggregate_replicas(fl * n_e2e / 1e12, e2e_ms / 1e3, dist, device)
        # The same pipeline with the copies alone (a separate, reported measurement, not
        # part of the e2e number): the host link's ceiling for this step's bytes.
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        c0.record(s_in)
        last = run_pipeline(n_e2e, compute=False)
        s_in.wait_event(last)
        s_in.wait_event(ev_out[n_e2e % 2])
        c1.record(s_in)
        torch.cuda.synchronize()
        copy_ms = c0.elapsed_time(c1) / n_e2e
        e2e = {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e2e, "pipelined": "3 streams, double-buffered device inputs and outputs",
               "ms_per_step": e2e_ms / n_e2e,
               "copies_only_ms_per_step": copy_ms,
               "link_gbs_copies_only": (h2d + d2h) / (copy_ms / 1e3) / 1e9,
               "note": "copies_only: the same pipeline without the GEMM call, timed separately"}
        del host, dev_in, dev_out, host_out, steps_b

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    st = launch_stats(launch_ms)
    traffic = recorded_traffic(wl["name"], plan)
    roofline = roofline_of(wl, st["mean"], peaks, peak_src, traffic)
    roofline.update({"kernel": "gb::gemm_persistent_kernel", "avg_launch_ms": st["mean"],
                     "flops_per_launch": fl, "algorithmic_bytes_per_launch": algorithmic_bytes(wl),
                     "clock_note": "timed after a pre-warm, so under the power cap (see clocks)"})
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": slowest_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(wl),
        "launch_ms": st,
        "roofline": roofline,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "plan": plan,
    }
    if not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_s)
        line["accuracy"] = sampled_accuracy(wl, t, out, 65536, seed=3)
    del t, out, ws, flush
    torch.cuda.empty_cache()
    if world == 1 and args.per_shape != "none":
        specs = PER_SHAPE if args.per_shape == "all" else [x for x in args.per_shape.split(";") if x]
        line["per_shape"] = [measure_shape(sp, args, device, local, peaks, peak_src) for sp in specs]
        gb.set_config(args.config)
    if world == 1 and not args.skip_nominal:
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        sm_max = (clocks or {}).get("sm_max_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
        line["nominal_peak"] = nominal_peak(sms, sm_max, (clocks or {}).get("sm_mhz"))
        npk = line["nominal_peak"]
        if "tflops_at_clock_under_load" in npk:
            line["roofline"]["frac_of_nominal_at_clock"] = roofline["achieved"] / npk["tflops_at_clock_under_load"] \
                if roofline["bound"] == "tensor" else None
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mlp_gelu",
                    help=f"one of {sorted(WORKLOADS)} or ragged:M,N,K (epilogue input, split-K entry point)")
    ap.add_argument("--prewarm-s", type=float, default=1.0, help="untimed seconds of steps before warm-up")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-s", type=float, default=12.0, help="target seconds of CPU-oracle work")
    ap.add_argument("--ref-step-s", type=float, default=4.0, help="reference arm: seconds per step")
    ap.add_argument("--config", default=None, help="tile-configuration override (gb_set_config syntax)")
    ap.add_argument("--per-shape", default="all",
                    help="'all' (every configuration, see PER_SHAPE), 'none', or workloads separated by ';'")
    ap.add_argument("--shape-steps", type=int, default=20, help="timed launches per per_shape workload")
    ap.add_argument("--shape-prewarm-s", type=float, default=0.3)
    ap.add_argument("--skip-nominal", action="store_true", help="skip the tcgen05 rate probe")
    args = ap.parse_args(argv)
    if args.warmup < 0 or args.steps < 1:
        ap.error("--steps >= 1 and --warmup >= 0")
    wl = workload(args.workload)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
