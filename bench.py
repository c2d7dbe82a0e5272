"""Throughput benchmark of the grouped MX GEMM hot path on GB300.

Default workload (one GPU): the a8w4 grouped forward -- G = 8 experts, 4096
tokens routed top-2 with Dirichlet(0.5)-skewed expert probabilities (S = 8192
rows), hidden K = 4096, expert FFN N = 14336; activations MXFP8 E4M3, weights
MXFP4 E2M1.  One step = every row of the hot path over one batch:
    quantize X (BF16 -> MXFP8, row-wise), quantize W (BF16 -> MXFP4, row-wise),
    grouped_gemm_fwd (split validation, scale packing, tcgen05 GEMM, BF16 out).
Metric: TFLOPS = 2 * sum(m_g) * N * K / step time.

`--workload mxfp4_moe_train` times the MXFP4 MoE training step (G = 32,
16384 tokens top-8 Zipf(1.1), K = 7168, N = 2048): all quantizers plus fwd,
dgrad and the variable-K wgrad with in-place fp32 accumulation; TFLOPS counts
the three GEMMs.

Timing: W warm-up steps, then K steps between CUDA events on the launching
stream, barrier + synchronize on both sides, max over ranks.  Inputs are
larger than L2 (129 MB), so no flush is needed.  Multi-GPU (torchrun): every
rank runs an independent replica of the workload (weak scaling; the path has
no exchange step).  `--impl reference` times the CPU oracle instead on a
bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

PEAK_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0     # nominal dense ratios (4.5 / 2.25 and 13.5 / 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0


# --------------------------------------------------------------------------- helpers
def peaks():
    try:
        with open(PEAK_FILE) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx = [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 6:
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for n, v in zip(names, p[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float (elapsed time) over all ranks."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- workloads
class A8W4Forward:
    name = "a8w4_fwd"

    def __init__(self, dev):
        import torch
        import fp8_bf16_mxfp4_gb300 as mxg
        self.mxg = mxg
        w = synth.WORKLOADS["a8w4_fwd"]
        self.w = w
        self.splits = w.splits()
        self.G, self.N, self.K = w.G, w.N, w.K
        self.S = int(self.splits.sum())
        x = synth.normal_bf16(w.act_rng(), (self.S, self.K), outlier_frac=w.outlier_frac)
        wt = synth.normal_bf16(w.weight_rng(), (self.G * self.N, self.K), outlier_frac=w.outlier_frac)
        to = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
        self.x_host = to(x).pin_memory()
        self.x = self.x_host.to(dev)
        self.wt = to(wt).to(dev)
        del x, wt
        self.splits_host = torch.from_numpy(self.splits).pin_memory()
        self.d_splits = self.splits_host.to(dev)
        S, N, K, G = self.S, self.N, self.K, self.G
        self.qx = torch.empty((S, K), dtype=torch.uint8, device=dev)
        self.sx = torch.empty((S, K // 32), dtype=torch.uint8, device=dev)
        self.qw = torch.empty((G * N, K // 2), dtype=torch.uint8, device=dev)
        self.sw = torch.empty((G * N, K // 32), dtype=torch.uint8, device=dev)
        self.y = torch.empty((S, N), dtype=torch.bfloat16, device=dev)
        self.y_host = torch.empty((S, N), dtype=torch.bfloat16).pin_memory()
        self.ws = torch.empty(mxg.gemm_workspace_size("fwd", G, S, N, K), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.flops = 2.0 * S * N * K
        self.launches_per_step = 2 + 3   # two quantizers; plan + scale pack + GEMM
        self.gemm_events = []

    def step(self, time_gemm=False):
        import torch
        mxg = self.mxg
        A = mxg.mx_quantize_rowwise(self.x, "e4m3", q=self.qx, s=self.sx)
        W = mxg.mx_quantize_rowwise(self.wt, "e2m1", q=self.qw, s=self.sw)
        if time_gemm:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
        mxg.grouped_gemm_fwd(A, W, self.d_splits, self.N, out=self.y, workspace=self.ws,
                             status=self.status)
        if time_gemm:
            e1.record()
            self.gemm_events.append((e0, e1))

    def e2e_step(self):
        self.x.copy_(self.x_host, non_blocking=True)
        self.d_splits.copy_(self.splits_host, non_blocking=True)
        self.step()
        self.y_host.copy_(self.y, non_blocking=True)

    def h2d_bytes(self):
        return self.x_host.numel() * 2 + self.splits_host.numel() * 4

    def d2h_bytes(self):
        return self.y_host.numel() * 2

    def gemm_algorithmic(self):
        return self.flops, "tensor", "TFLOP/s"

    def gemm_peak(self, pk):
        return pk["bf16_tflops_sustained"] * FP8_OVER_BF16, "bf16_tflops_sustained x 2 (fp8/bf16 nominal)"

    def config(self):
        return {"workload": "a8w4 grouped forward: G=8, 4096 tokens top-2 Dirichlet(0.5) -> S=8192, "
                            "K=4096, N=14336; X MXFP8 E4M3, W MXFP4 E2M1 (UE8M0 / 32), BF16 out",
                "G": self.G, "S": self.S, "N": self.N, "K": self.K, "m_splits": self.splits.tolist(),
                "step": "quantize X + quantize W + grouped_gemm_fwd",
                "l2": "inputs larger than L2 (X 67 MB + W 940 MB BF16), no flush"}

    def check(self):
        self.mxg.check_status(self.status)


def build_workload(name, dev):
    if name == "a8w4_fwd":
        return A8W4Forward(dev)
    raise SystemExit(f"unknown workload {name}")


# --------------------------------------------------------------------------- CPU oracle arm
def oracle_sample(seconds_hint=False):
    """Bounded oracle sample of the a8w4 step: 2048 activation rows and 2048
    weight rows of one expert at K = 4096 (about the flop-per-quantized-element
    ratio of the full step): oracle quantize both, dequantize, fp64 matmul."""
    import oracle
    w = synth.WORKLOADS["a8w4_fwd"]
    rng = np.random.default_rng(12345)
    rows = 1024 if seconds_hint else 2048
    x = synth.normal_bf16(rng, (rows, w.K), outlier_frac=w.outlier_frac)
    wt = synth.normal_bf16(rng, (rows, w.K), outlier_frac=w.outlier_frac)
    t0 = time.perf_counter()
    xd, xs = oracle.quantize_mx_rowwise(x, "e4m3")
    wd, ws = oracle.quantize_mx_rowwise(wt, "e2m1")
    A = oracle.dequantize_mx(xd, xs, "e4m3")
    W = oracle.dequantize_mx(oracle.unpack_e2m1(wd), ws, "e2m1")
    oracle.grouped_fwd(A, W, [rows], rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * rows * w.K
    return flops, dt, f"{rows} X rows x {rows} W rows of one expert, K={w.K}: oracle quantize both + fp64 matmul"


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    c = cores()
    os.environ.setdefault("OMP_NUM_THREADS", str(c))
    for _ in range(args.warmup):
        oracle_sample(seconds_hint=True)
    tot_f, tot_t = 0.0, 0.0
    sample = ""
    for _ in range(args.steps):
        f, t, sample = oracle_sample(seconds_hint=True)
        tot_f += f
        tot_t += t
    v = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": "grouped MXFP4/a8w4 GEMM TFLOPS (fwd/dgrad/wgrad) and % of GB300 FP4/FP8 peak",
            "value": v, "unit": "TFLOPS", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / max(args.steps, 1) * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "a8w4 grouped forward (bounded oracle sample)"},
            "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": c, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch
    rank, world, local = dist_setup(args.gpus)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = build_workload(args.workload, dev)

    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    wl.check()

    # ---- device-resident timed region
    barrier(world)
    torch.cuda.synchronize()
    wl.gemm_events = []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local) as clk:
        ev0.record()
        for _ in range(args.steps):
            wl.step(time_gemm=True)
        ev1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world, dev)
    gemm_ms = statistics.mean(a.elapsed_time(b) for a, b in wl.gemm_events)
    wl.check()

    # ---- end to end: pinned host input -> device -> result back to host
    for _ in range(max(1, args.warmup // 2)):
        wl.e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        wl.e2e_step()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    wl.check()

    if rank != 0:
        return
    steps = args.steps
    value = world * wl.flops * steps / (ms_max * 1e-3) / 1e12
    e2e_value = world * wl.flops * steps / (e2e_ms * 1e-3) / 1e12
    pk, src = peaks()
    alg, bound, unit = wl.gemm_algorithmic()
    achieved = alg / (gemm_ms * 1e-3) / 1e12
    peak, peak_note = wl.gemm_peak(pk)
    cpu_f, cpu_t, sample = oracle_sample()
    line = {
        "metric": "grouped MXFP4/a8w4 GEMM TFLOPS (fwd/dgrad/wgrad) and % of GB300 FP4/FP8 peak",
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms_max / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxf8f6f4 (e4m3 x e2m1, fp32 accumulate)", "data": "synthetic",
        "config": wl.config(),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "grouped_gemm_fwd call (plan + scale pack + tcgen05 GEMM)",
                     "peak_source": f"{src}: {peak_note}", "gemm_ms": gemm_ms},
        "cpu_baseline": {"value": cpu_f / cpu_t / 1e12, "unit": "TFLOPS", "cores": cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": wl.h2d_bytes(),
                "d2h_bytes_per_step": wl.d2h_bytes(), "ms_per_step": e2e_ms / steps},
        "gpu_launches": wl.launches_per_step * steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="a8w4_fwd")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
