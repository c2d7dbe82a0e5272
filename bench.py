"""Throughput benchmark of the grouped MX GEMM hot path on GB300.

Default workload (one GPU): the a8w4 grouped forward -- G = 8 experts, 4096
tokens routed top-2 with Dirichlet(0.5)-skewed expert probabilities (S = 8192
rows), hidden K = 4096, expert FFN N = 14336; activations MXFP8 E4M3, weights
MXFP4 E2M1.  One step = every row of the hot path over one batch:
    quantize X (BF16 -> MXFP8, row-wise), quantize W (BF16 -> MXFP4, row-wise),
    with the scales written straight into the tensor cores' staging order, then
    grouped_gemm_fwd (split validation, tcgen05 GEMM, BF16 out).
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
    """nvidia-smi sampling of SM clocks and throttle reasons; only samples that
    arrive inside the marked region are summarised (the nearest one after its
    start when the region is shorter than the sampling interval)."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []          # (host time, line)
        self.t_start = None
        self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def wait_first_sample(self, timeout=10.0):
        t0 = time.monotonic()
        while self.proc is not None and not self.lines and time.monotonic() - t0 < timeout:
            time.sleep(0.01)
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()
        time.sleep(0.12)       # let the sample in flight arrive

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        t0 = self.t_start or 0.0
        t1 = self.t_end or float("inf")
        inside = [ln for t, ln in self.lines if t0 <= t <= t1]
        note = "in region"
        if not inside:
            after = [ln for t, ln in self.lines if t >= t0][:1]
            inside, note = after, "nearest after region start"
        sm, mx = [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
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
                "samples": len(sm), "window": note}


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
def _to_bf16(bits):
    import torch
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


# algorithmic bytes per element of a quantized operand (codes + scales)
OPERAND_BYTES = {"e2m1": 0.5 + 1 / 32, "e4m3": 1 + 1 / 32, "bw_act": 1 + 4 / 128, "bw_w": 1 + 4 / 16384,
                 "bw_pow2": 1 + 1 / 32}


def padded_total(splits, pad):
    return int(sum(-(-int(m) // pad) * pad for m in splits))


def gemm_bytes(a_elems, a_fmt, b_elems, b_fmt, out_elems, out_bytes, accumulate=False):
    """Algorithmic HBM bytes of one GEMM call: both operands read once (codes
    and scales), the output written once (read and written when added in
    place)."""
    return (a_elems * OPERAND_BYTES[a_fmt] + b_elems * OPERAND_BYTES[b_fmt]
            + out_elems * out_bytes * (2 if accumulate else 1))


class _Timed:
    """Per-call CUDA events around the GEMM launches of the timed steps."""

    def __init__(self):
        self.events = {}

    def run(self, name, fn, enabled):
        import torch
        if not enabled:
            return fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        r = fn()
        e1.record()
        self.events.setdefault(name, []).append((e0, e1))
        return r

    def mean_ms(self):
        return {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in self.events.items()}


class A8W4Forward:
    """a8w4 grouped forward (the default)."""
    name = "a8w4_fwd"
    call_kernels = "plan + tcgen05 GEMM; scales arrive packed"

    def __init__(self, dev):
        import torch
        import fp8_bf16_mxfp4_gb300 as mxg
        self.mxg = mxg
        w = synth.WORKLOADS["a8w4_fwd"]
        self.splits = w.splits()
        self.G, self.N, self.K = w.G, w.N, w.K
        self.S = int(self.splits.sum())
        x = synth.normal_bf16(w.act_rng(), (self.S, self.K), outlier_frac=w.outlier_frac)
        wt = synth.normal_bf16(w.weight_rng(), (self.G * self.N, self.K), outlier_frac=w.outlier_frac)
        self.x_host = _to_bf16(x).pin_memory()
        self.x = self.x_host.to(dev)
        self.wt = _to_bf16(wt).to(dev)
        del x, wt
        self.splits_host = torch.from_numpy(self.splits).pin_memory()
        self.d_splits = self.splits_host.to(dev)
        S, N, K, G = self.S, self.N, self.K, self.G
        self.y = torch.empty((S, N), dtype=torch.bfloat16, device=dev)
        self.y_host = torch.empty((S, N), dtype=torch.bfloat16).pin_memory()
        self.ws = torch.empty(mxg.gemm_workspace_size("fwd", G, S, N, K), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.flops = 2.0 * S * N * K
        self.launches_per_step = 2 + 2   # two quantizers (scales written packed); plan + GEMM
        self.timed = _Timed()
        self.gemm_info = {"fwd": (self.flops, FP8_OVER_BF16, "mxf8f6f4 (a8w4)")}
        self.pass_bytes = {"fwd": gemm_bytes(S * K, "e4m3", G * N * K, "e2m1", S * N, 2)}

    def step(self, time_gemm=False):
        mxg = self.mxg
        A = mxg.mx_quantize_rowwise_packed(self.x, "e4m3", m_splits=self.d_splits, status=self.status)
        W = mxg.mx_quantize_rowwise_packed(self.wt, "e2m1", groups=self.G)
        self.timed.run("fwd", lambda: mxg.grouped_gemm_fwd(A, W, self.d_splits, self.N, out=self.y,
                                                           workspace=self.ws, status=self.status),
                       time_gemm)

    # end-to-end tensors: device attribute -> pinned host attribute
    e2e_in = (("x", "x_host"), ("d_splits", "splits_host"))
    e2e_out = (("y", "y_host"),)

    def h2d_bytes(self):
        return self.x_host.numel() * 2 + self.splits_host.numel() * 4

    def d2h_bytes(self):
        return self.y_host.numel() * 2

    def config(self):
        return {"workload": "a8w4 grouped forward: G=8, 4096 tokens top-2 Dirichlet(0.5) -> S=8192, "
                            "K=4096, N=14336; X MXFP8 E4M3, W MXFP4 E2M1 (UE8M0 / 32), BF16 out",
                "G": self.G, "S": self.S, "N": self.N, "K": self.K, "m_splits": self.splits.tolist(),
                "step": "quantize X + quantize W (scales in the MMA staging order) + grouped_gemm_fwd",
                "l2": "inputs larger than L2 (X 67 MB + W 940 MB BF16), no flush"}

    dtype = "mxf8f6f4 (e4m3 x e2m1, fp32 accumulate)"
    # DRAM bytes (read + write) of one GEMM call per pass, counted by ncu on
    # GB300 for the current kernels (dram__bytes_read.sum + dram__bytes_write.sum).
    traffic_bytes = {"fwd": 284407296 + 212500736}

    def check(self):
        self.mxg.check_status(self.status)


class MXFP4Train:
    """MXFP4 MoE training step of one expert layer: fwd, dgrad, variable-K wgrad."""
    name = "mxfp4_moe_train"
    call_kernels = "plan + tcgen05 GEMM; scales arrive packed"
    elem = "e2m1"
    # DRAM bytes (read + write) of one GEMM call per pass, counted by ncu on
    # GB300 for the current kernels (dram__bytes_read.sum + dram__bytes_write.sum).
    traffic_bytes = {"fwd": 768069888 + 508036352, "dgrad": 396351232 + 1817983232,
                     "wgrad": 2797496064 + 1840005888}

    def __init__(self, dev):
        import torch
        import fp8_bf16_mxfp4_gb300 as mxg
        self.mxg = mxg
        w = synth.WORKLOADS["mxfp4_moe_train"]
        self.splits = w.splits()
        self.G, self.N, self.K, self.pad = w.G, w.N, w.K, w.pad
        self.S = int(self.splits.sum())
        G, N, K, S = self.G, self.N, self.K, self.S
        self.x_host = _to_bf16(synth.normal_bf16(w.act_rng(0), (S, K))).pin_memory()
        self.dy_host = _to_bf16(synth.normal_bf16(w.act_rng(1), (S, N))).pin_memory()
        self.x = self.x_host.to(dev)
        self.dy = self.dy_host.to(dev)
        self.w = _to_bf16(synth.normal_bf16(w.weight_rng(), (G * N, K))).to(dev)
        self.splits_host = torch.from_numpy(self.splits).pin_memory()
        self.d_splits = self.splits_host.to(dev)
        self.w_splits = torch.full((G,), N, dtype=torch.int32, device=dev)
        self.cap = mxg.mx_padded_rows_capacity(S, G, self.pad)
        self.main_grad = (torch.randn((G, N, K), device=dev, dtype=torch.float32) * 1e-3)
        self.y = torch.empty((S, N), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((S, K), dtype=torch.bfloat16, device=dev)
        self.y_host = torch.empty((S, N), dtype=torch.bfloat16).pin_memory()
        self.dx_host = torch.empty((S, K), dtype=torch.bfloat16).pin_memory()
        ws = max(mxg.gemm_workspace_size("fwd", G, S, N, K), mxg.gemm_workspace_size("dgrad", G, S, N, K),
                 mxg.gemm_workspace_size("wgrad", G, self.cap, N, K, self.pad))
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        f = 2.0 * S * N * K
        self.flops = 3 * f
        # six quantizers, all writing staging-order scales; three GEMM calls of plan + GEMM
        self.launches_per_step = 6 + 3 * 2
        self.timed = _Timed()
        self.gemm_info = {p: (f, FP4_OVER_BF16, "mxf4") for p in ("fwd", "dgrad", "wgrad")}
        self.pass_bytes = self._pass_bytes(self.elem)

    def _pass_bytes(self, e):
        G, N, K, S = self.G, self.N, self.K, self.S
        sp = padded_total(self.splits, self.pad)
        return {"fwd": gemm_bytes(S * K, e, G * N * K, e, S * N, 2),
                "dgrad": gemm_bytes(S * N, e, K * G * N, e, S * K, 2),
                "wgrad": gemm_bytes(N * sp, e, K * sp, e, G * N * K, 4, accumulate=True)}

    def step(self, time_gemm=False):
        mxg, G, N, K, pad = self.mxg, self.G, self.N, self.K, self.pad
        Xq = mxg.mx_quantize_rowwise_packed(self.x, self.elem, m_splits=self.d_splits, status=self.status)
        Wq = mxg.mx_quantize_rowwise_packed(self.w, self.elem, groups=G)
        self.timed.run("fwd", lambda: mxg.grouped_gemm_fwd(Xq, Wq, self.d_splits, N, out=self.y,
                                                           workspace=self.ws, status=self.status), time_gemm)
        dYq = mxg.mx_quantize_rowwise_packed(self.dy, self.elem, m_splits=self.d_splits, status=self.status)
        Wt, _ = mxg.mx_quantize_colwise_segment_padded(self.w, self.w_splits, 32, self.elem,
                                                       capacity=G * N, status=self.status, packed=True)
        self.timed.run("dgrad", lambda: mxg.grouped_gemm_dgrad(dYq, Wt, self.d_splits, out=self.dx,
                                                               workspace=self.ws, status=self.status), time_gemm)
        dYt, _ = mxg.mx_quantize_colwise_segment_padded(self.dy, self.d_splits, pad, self.elem,
                                                        capacity=self.cap, status=self.status, packed=True)
        Xt, _ = mxg.mx_quantize_colwise_segment_padded(self.x, self.d_splits, pad, self.elem,
                                                       capacity=self.cap, status=self.status, packed=True)
        self.timed.run("wgrad", lambda: mxg.grouped_gemm_wgrad(dYt, Xt, self.d_splits, self.S, pad,
                                                               out=self.main_grad, accumulate=True,
                                                               workspace=self.ws, status=self.status), time_gemm)

    e2e_in = (("x", "x_host"), ("dy", "dy_host"), ("d_splits", "splits_host"))
    e2e_out = (("y", "y_host"), ("dx", "dx_host"))

    def h2d_bytes(self):
        return (self.x_host.numel() + self.dy_host.numel()) * 2 + self.splits_host.numel() * 4

    def d2h_bytes(self):
        return (self.y_host.numel() + self.dx_host.numel()) * 2

    def config(self):
        return {"workload": "MXFP4 MoE training step: G=32, 16384 tokens top-8 Zipf(1.1) -> S=131072, "
                            "hidden K=7168, FFN N=2048; fwd TN, dgrad NN, wgrad NT (pad 32, fp32 "
                            "accumulate into main_grad), BF16 in/out",
                "G": self.G, "S": self.S, "N": self.N, "K": self.K, "pad": self.pad,
                "step": "6 quantizers + grouped fwd + dgrad + wgrad",
                "l2": "inputs larger than L2 (X 1.9 GB, W 0.94 GB BF16), no flush"}

    dtype = "mxf4 (e2m1 x e2m1, fp32 accumulate)"

    def check(self):
        self.mxg.check_status(self.status)


class DenseMXFP4:
    """Dense MXFP4 per-pass GEMMs (G = 1) of the sweep "seqlen 2048 x mbs
    {1, 2, 4}" (M = 2048, 4096, 8192 tokens), hidden 8192, FFN 28672: fwd TN,
    dgrad NN and wgrad NT, each with BF16 and with FP32 output (six GEMM
    calls per step, after the six quantizers)."""
    M = 8192
    name = "dense_mxfp4_m8192"
    call_kernels = "plan + tcgen05 GEMM; scales arrive packed"
    # DRAM bytes (read + write) of one GEMM call per pass, counted by ncu on
    # GB300 for the current kernels (dram__bytes_read.sum + dram__bytes_write.sum).
    traffic_bytes = {"fwd_bf16": 225919488 + 440607744, "fwd_f32": 434404096 + 896570112,
                     "dgrad_bf16": 1032064768 + 120869120, "dgrad_f32": 1069566976 + 244512768,
                     "wgrad_bf16": 330752000 + 430036480, "wgrad_f32": 461681920 + 888530176}

    def __init__(self, dev):
        import torch
        import fp8_bf16_mxfp4_gb300 as mxg
        self.mxg = mxg
        w = synth.WORKLOADS[self.name]
        self.splits = w.splits()
        self.G, self.N, self.K, self.pad = w.G, w.N, w.K, w.pad
        self.S = int(self.splits.sum())
        G, N, K, S = self.G, self.N, self.K, self.S
        self.x_host = _to_bf16(synth.normal_bf16(w.act_rng(0), (S, K), std=w.std)).pin_memory()
        self.dy_host = _to_bf16(synth.normal_bf16(w.act_rng(1), (S, N), std=w.std)).pin_memory()
        self.x = self.x_host.to(dev)
        self.dy = self.dy_host.to(dev)
        self.w = _to_bf16(synth.normal_bf16(w.weight_rng(), (N, K), std=w.std)).to(dev)
        self.splits_host = torch.from_numpy(self.splits).pin_memory()
        self.d_splits = self.splits_host.to(dev)
        self.w_splits = torch.full((1,), N, dtype=torch.int32, device=dev)
        self.cap = mxg.mx_padded_rows_capacity(S, G, self.pad)
        self.dw = torch.empty((G, N, K), device=dev, dtype=torch.float32)
        self.dw16 = torch.empty((G, N, K), device=dev, dtype=torch.bfloat16)
        self.y = torch.empty((S, N), dtype=torch.bfloat16, device=dev)
        self.y32 = torch.empty((S, N), dtype=torch.float32, device=dev)
        self.dx = torch.empty((S, K), dtype=torch.bfloat16, device=dev)
        self.dx32 = torch.empty((S, K), dtype=torch.float32, device=dev)
        self.y_host = torch.empty((S, N), dtype=torch.bfloat16).pin_memory()
        self.dx_host = torch.empty((S, K), dtype=torch.bfloat16).pin_memory()
        ws = max(mxg.gemm_workspace_size("fwd", G, S, N, K), mxg.gemm_workspace_size("dgrad", G, S, N, K),
                 mxg.gemm_workspace_size("wgrad", G, self.cap, N, K, self.pad))
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        f = 2.0 * S * N * K
        self.flops = 6 * f
        # six quantizers, all writing staging-order scales; six GEMM calls of plan + GEMM
        self.launches_per_step = 6 + 6 * 2
        self.timed = _Timed()
        self.gemm_info = {f"{p}_{o}": (f, FP4_OVER_BF16, "mxf4")
                          for p in ("fwd", "dgrad", "wgrad") for o in ("bf16", "f32")}
        sp = padded_total(self.splits, self.pad)
        self.pass_bytes = {}
        for o, ob in (("bf16", 2), ("f32", 4)):
            self.pass_bytes[f"fwd_{o}"] = gemm_bytes(S * K, "e2m1", N * K, "e2m1", S * N, ob)
            self.pass_bytes[f"dgrad_{o}"] = gemm_bytes(S * N, "e2m1", K * N, "e2m1", S * K, ob)
            self.pass_bytes[f"wgrad_{o}"] = gemm_bytes(N * sp, "e2m1", K * sp, "e2m1", N * K, ob)

    def step(self, time_gemm=False):
        import torch
        mxg, N, pad, ws, st, T = self.mxg, self.N, self.pad, self.ws, self.status, self.timed
        Xq = mxg.mx_quantize_rowwise_packed(self.x, "e2m1", m_splits=self.d_splits, status=st)
        Wq = mxg.mx_quantize_rowwise_packed(self.w, "e2m1", groups=1)
        T.run("fwd_bf16", lambda: mxg.grouped_gemm_fwd(Xq, Wq, self.d_splits, N, out=self.y, workspace=ws,
                                                        status=st), time_gemm)
        T.run("fwd_f32", lambda: mxg.grouped_gemm_fwd(Xq, Wq, self.d_splits, N, out=self.y32,
                                                       out_dtype=torch.float32, workspace=ws, status=st),
              time_gemm)
        dYq = mxg.mx_quantize_rowwise_packed(self.dy, "e2m1", m_splits=self.d_splits, status=st)
        Wt, _ = mxg.mx_quantize_colwise_segment_padded(self.w, self.w_splits, 32, "e2m1",
                                                       capacity=N, status=st, packed=True)
        T.run("dgrad_bf16", lambda: mxg.grouped_gemm_dgrad(dYq, Wt, self.d_splits, out=self.dx, workspace=ws,
                                                            status=st), time_gemm)
        T.run("dgrad_f32", lambda: mxg.grouped_gemm_dgrad(dYq, Wt, self.d_splits, out=self.dx32,
                                                           out_dtype=torch.float32, workspace=ws, status=st),
              time_gemm)
        dYt, _ = mxg.mx_quantize_colwise_segment_padded(self.dy, self.d_splits, pad, "e2m1",
                                                        capacity=self.cap, status=st, packed=True)
        Xt, _ = mxg.mx_quantize_colwise_segment_padded(self.x, self.d_splits, pad, "e2m1",
                                                       capacity=self.cap, status=st, packed=True)
        T.run("wgrad_bf16", lambda: mxg.grouped_gemm_wgrad(dYt, Xt, self.d_splits, self.S, pad, out=self.dw16,
                                                            out_dtype=torch.bfloat16, workspace=ws, status=st),
              time_gemm)
        T.run("wgrad_f32", lambda: mxg.grouped_gemm_wgrad(dYt, Xt, self.d_splits, self.S, pad, out=self.dw,
                                                           accumulate=False, workspace=ws, status=st), time_gemm)

    e2e_in = (("x", "x_host"), ("dy", "dy_host"), ("d_splits", "splits_host"))
    e2e_out = (("y", "y_host"), ("dx", "dx_host"))

    def h2d_bytes(self):
        return (self.x_host.numel() + self.dy_host.numel()) * 2 + self.splits_host.numel() * 4

    def d2h_bytes(self):
        return (self.y_host.numel() + self.dx_host.numel()) * 2

    def config(self):
        return {"workload": f"dense MXFP4 per-pass GEMMs (G=1): M={self.S} tokens (seqlen 2048 x mbs "
                            f"{self.S // 2048}), hidden K=8192, FFN N=28672, inputs ~N(0,0.02); fwd TN, "
                            "dgrad NN, wgrad NT, each with BF16 and with FP32 output",
                "G": 1, "S": self.S, "N": self.N, "K": self.K,
                "step": "6 quantizers + fwd, dgrad, wgrad x {BF16, FP32} out",
                "l2": "W 470 MB BF16 and every step's operands together exceed L2, no flush"}

    dtype = "mxf4 (e2m1 x e2m1, fp32 accumulate)"

    def check(self):
        self.mxg.check_status(self.status)


class DenseMXFP4M2048(DenseMXFP4):
    M = 2048
    name = "dense_mxfp4_m2048"
    traffic_bytes = {"fwd_bf16": 133795840 + 84969216, "fwd_f32": 134309888 + 183715328,
                     "dgrad_bf16": 220680192 + 20125184, "dgrad_f32": 235941376 + 41113344,
                     "wgrad_bf16": 120382976 + 416103168, "wgrad_f32": 268303616 + 879753728}


class DenseMXFP4M4096(DenseMXFP4):
    M = 4096
    name = "dense_mxfp4_m4096"
    traffic_bytes = {"fwd_bf16": 143735040 + 198029824, "fwd_f32": 153152256 + 418276864,
                     "dgrad_bf16": 484013568 + 54761216, "dgrad_f32": 504029696 + 112482560,
                     "wgrad_bf16": 143730432 + 420033536, "wgrad_f32": 320843776 + 885835520}


class MXFP8Train(MXFP4Train):
    """The MXFP4 training step's shapes with MXFP8 (E4M3) operands in all
    three passes (kind::mxf8f6f4)."""
    name = "mxfp8_moe_train"
    elem = "e4m3"
    traffic_bytes = {"fwd": 2330992384 + 522683648, "dgrad": 821914112 + 1831402496,
                     "wgrad": 3288205056 + 1853214464}

    def __init__(self, dev):
        super().__init__(dev)
        f = 2.0 * self.S * self.N * self.K
        self.gemm_info = {p: (f, FP8_OVER_BF16, "mxf8f6f4 (mxfp8)") for p in ("fwd", "dgrad", "wgrad")}
        self.pass_bytes = self._pass_bytes("e4m3")

    def config(self):
        c = super().config()
        c["workload"] = ("MXFP8 MoE training step: G=32, 16384 tokens top-8 Zipf(1.1) -> S=131072, "
                         "hidden K=7168, FFN N=2048; fwd TN, dgrad NN, wgrad NT (pad 32, fp32 accumulate "
                         "into main_grad), E4M3 with UE8M0 per 32, BF16 in/out")
        return c

    dtype = "mxf8f6f4 (e4m3 x e4m3, fp32 accumulate)"


class BlockwiseFP8:
    """Blockwise-FP8 grouped training step: fwd, dgrad, variable-K wgrad."""
    call_kernels = "plan + 2-SM tcgen05 GEMM with CUDA-core promotion"
    name = "blockwise_fp8"
    # DRAM bytes (read + write) of one GEMM call per pass, counted by ncu on
    # GB300 for the current kernels (dram__bytes_read.sum + dram__bytes_write.sum).
    traffic_bytes = {"fwd": 714261504 + 250356992, "dgrad": 608493568 + 436344320,
                     "wgrad": 405923584 + 885403648}

    def __init__(self, dev):
        import torch
        import fp8_bf16_mxfp4_gb300 as mxg
        self.mxg = mxg
        w = synth.WORKLOADS["blockwise_fp8"]
        self.splits = w.splits()
        self.G, self.N, self.K = w.G, w.N, w.K
        self.S = int(self.splits.sum())
        G, N, K, S = self.G, self.N, self.K, self.S
        self.x_host = _to_bf16(synth.normal_bf16(w.act_rng(0), (S, K))).pin_memory()
        self.dy_host = _to_bf16(synth.normal_bf16(w.act_rng(1), (S, N))).pin_memory()
        self.x = self.x_host.to(dev)
        self.dy = self.dy_host.to(dev)
        self.w = _to_bf16(synth.normal_bf16(w.weight_rng(), (G * N, K))).to(dev)
        self.splits_host = torch.from_numpy(self.splits).pin_memory()
        self.d_splits = self.splits_host.to(dev)
        self.cap = mxg.mx_padded_rows_capacity(S, G, 128)
        self.y = torch.empty((S, N), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((S, K), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
        self.y_host = torch.empty((S, N), dtype=torch.bfloat16).pin_memory()
        self.dx_host = torch.empty((S, K), dtype=torch.bfloat16).pin_memory()
        self.ws = torch.empty(4096, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        f = 2.0 * S * N * K
        self.flops = 3 * f
        self.launches_per_step = 5 + 3 * 2   # five quantizers; three GEMM calls of two kernels
        self.timed = _Timed()
        self.gemm_info = {p: (f, FP8_OVER_BF16, "f8f6f4 + fp32 promotion") for p in ("fwd", "dgrad", "wgrad")}
        sp = padded_total(self.splits, 128)
        self.pass_bytes = {"fwd": gemm_bytes(S * K, "bw_act", G * N * K, "bw_w", S * N, 2),
                           "dgrad": gemm_bytes(S * N, "bw_act", K * G * N, "bw_w", S * K, 2),
                           "wgrad": gemm_bytes(N * sp, "bw_act", K * sp, "bw_act", G * N * K, 2)}

    def step(self, time_gemm=False):
        mxg, N = self.mxg, self.N
        Xq = mxg.bw_quantize_1x128(self.x)
        Wq, Wt = mxg.bw_quantize_128x128(self.w)
        self.timed.run("fwd", lambda: mxg.bw_grouped_gemm_fwd(Xq, Wq, self.d_splits, N, out=self.y,
                                                              workspace=self.ws, status=self.status), time_gemm)
        dYq = mxg.bw_quantize_1x128(self.dy)
        self.timed.run("dgrad", lambda: mxg.bw_grouped_gemm_dgrad(dYq, Wt, self.d_splits, out=self.dx,
                                                                  workspace=self.ws, status=self.status), time_gemm)
        dYt, _ = mxg.bw_quantize_colwise_padded(self.dy, self.d_splits, capacity=self.cap, status=self.status)
        Xt, _ = mxg.bw_quantize_colwise_padded(self.x, self.d_splits, capacity=self.cap, status=self.status)
        self.timed.run("wgrad", lambda: mxg.bw_grouped_gemm_wgrad(dYt, Xt, self.d_splits, self.S, out=self.dw,
                                                                  workspace=self.ws, status=self.status), time_gemm)

    e2e_in = MXFP4Train.e2e_in
    e2e_out = MXFP4Train.e2e_out
    h2d_bytes = MXFP4Train.h2d_bytes
    d2h_bytes = MXFP4Train.d2h_bytes

    def config(self):
        return {"workload": "blockwise FP8 grouped step: G=16, 32768 rows uniform routing, K=7168, "
                            "N=4096; E4M3 with 1x128 activation / 128x128 weight fp32 scales; fwd, "
                            "dgrad, variable-K wgrad (pad 128), BF16 out",
                "G": self.G, "S": self.S, "N": self.N, "K": self.K,
                "step": "5 quantizers + grouped fwd + dgrad + wgrad",
                "l2": "inputs larger than L2 (X 0.47 GB, W 0.94 GB BF16), no flush"}

    dtype = "f8f6f4 (e4m3 x e4m3, fp32 accumulate + fp32 block promotion)"

    def check(self):
        self.mxg.check_status(self.status)


class BlockwiseFP8Pow2(BlockwiseFP8):
    """The blockwise-FP8 step with power-of-two scales: the quantizers write
    MXFP8 operands (UE8M0 bytes repeated over each 128-block) and the three
    passes run on the block-scaled MX GEMMs, with no promotion."""
    call_kernels = "plan + scale pack + tcgen05 GEMM"
    name = "blockwise_fp8_pow2"
    traffic_bytes = {"fwd": 756197632 + 252655872, "dgrad": 628492544 + 437733376,
                     "wgrad": 403800576 + 883552000}

    def __init__(self, dev):
        import torch
        super().__init__(dev)
        mxg, G, N, K, S = self.mxg, self.G, self.N, self.K, self.S
        ws = max(mxg.gemm_workspace_size("fwd", G, S, N, K), mxg.gemm_workspace_size("dgrad", G, S, N, K),
                 mxg.gemm_workspace_size("wgrad", G, self.cap, N, K, 128))
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.launches_per_step = 5 + 3 * 3   # five quantizers; three GEMM calls of three kernels
        f = 2.0 * S * N * K
        self.gemm_info = {p: (f, FP8_OVER_BF16, "mxf8f6f4 (pow2 blockwise)") for p in ("fwd", "dgrad", "wgrad")}
        sp = padded_total(self.splits, 128)
        self.pass_bytes = {"fwd": gemm_bytes(S * K, "bw_pow2", G * N * K, "bw_pow2", S * N, 2),
                           "dgrad": gemm_bytes(S * N, "bw_pow2", K * G * N, "bw_pow2", S * K, 2),
                           "wgrad": gemm_bytes(N * sp, "bw_pow2", K * sp, "bw_pow2", G * N * K, 2)}

    def step(self, time_gemm=False):
        mxg, N = self.mxg, self.N
        Xq = mxg.bw_quantize_1x128_pow2(self.x)
        Wq, Wt = mxg.bw_quantize_128x128_pow2(self.w)
        self.timed.run("fwd", lambda: mxg.grouped_gemm_fwd(Xq, Wq, self.d_splits, N, out=self.y,
                                                           workspace=self.ws, status=self.status), time_gemm)
        dYq = mxg.bw_quantize_1x128_pow2(self.dy)
        self.timed.run("dgrad", lambda: mxg.grouped_gemm_dgrad(dYq, Wt, self.d_splits, out=self.dx,
                                                               workspace=self.ws, status=self.status), time_gemm)
        dYt, _ = mxg.bw_quantize_colwise_padded_pow2(self.dy, self.d_splits, capacity=self.cap, status=self.status)
        Xt, _ = mxg.bw_quantize_colwise_padded_pow2(self.x, self.d_splits, capacity=self.cap, status=self.status)
        self.timed.run("wgrad", lambda: mxg.grouped_gemm_wgrad(dYt, Xt, self.d_splits, self.S, 128, out=self.dw,
                                                               out_dtype=torch_bf16(), workspace=self.ws,
                                                               status=self.status), time_gemm)

    def config(self):
        c = super().config()
        c["workload"] = ("blockwise FP8 grouped step, power-of-two scales: G=16, 32768 rows uniform "
                         "routing, K=7168, N=4096; E4M3 with 1x128 activation / 128x128 weight pow2 scales "
                         "as UE8M0 per 32; fwd, dgrad, variable-K wgrad (pad 128) on the MXFP8 GEMMs, BF16 out")
        return c

    dtype = "mxf8f6f4 (e4m3 x e4m3, pow2 block scales, fp32 accumulate)"


def torch_bf16():
    import torch
    return torch.bfloat16


WORKLOAD_CLASSES = {c.name: c for c in (A8W4Forward, MXFP4Train, MXFP8Train, BlockwiseFP8, DenseMXFP4,
                                        DenseMXFP4M2048, DenseMXFP4M4096, BlockwiseFP8Pow2)}


def build_workload(name, dev):
    if name not in WORKLOAD_CLASSES:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(WORKLOAD_CLASSES)}")
    return WORKLOAD_CLASSES[name](dev)


class E2EPipeline:
    """End-to-end steps through the library with host buffers: each step's
    inputs go host->device on one copy stream, the step runs on the compute
    stream, and its outputs go device->host on another copy stream.  Device
    inputs/outputs and pinned host outputs have two slots, so step i's copies
    overlap steps i-1 and i+1; events keep a slot from being overwritten while
    it is still read.  Every step moves its full inputs and outputs."""

    def __init__(self, wl, lanes=1):
        import torch
        self.wl = wl
        # each copy may be split by rows over `lanes` streams per direction (two
        # streams measured no faster than one on GB300: the host link is the limit)
        self.h2d = [torch.cuda.Stream() for _ in range(lanes)]
        self.d2h = [torch.cuda.Stream() for _ in range(lanes)]
        self.dev_in = [{a: getattr(wl, a) if k == 0 else torch.empty_like(getattr(wl, a)) for a, _ in wl.e2e_in}
                       for k in range(2)]
        self.dev_out = [{a: getattr(wl, a) if k == 0 else torch.empty_like(getattr(wl, a)) for a, _ in wl.e2e_out}
                        for k in range(2)]
        self.host_out = [{h: getattr(wl, h) if k == 0 else torch.empty_like(getattr(wl, h)).pin_memory()
                          for _, h in wl.e2e_out} for k in range(2)]
        self.in_free = [None, None]
        self.out_free = [[], []]
        self.i = 0

    @staticmethod
    def _part(t, c, n):
        r = t.shape[0]
        lo, hi = r * c // n, r * (c + 1) // n
        return t[lo:hi]

    def step(self):
        import torch
        wl, k = self.wl, self.i % 2
        comp = torch.cuda.current_stream()
        n = len(self.h2d)
        in_ready = []
        for c, st in enumerate(self.h2d):
            with torch.cuda.stream(st):
                if self.in_free[k] is not None:
                    st.wait_event(self.in_free[k])
                for a, h in wl.e2e_in:
                    dst, src = self.dev_in[k][a], getattr(wl, h)
                    if dst.shape[0] >= n:
                        self._part(dst, c, n).copy_(self._part(src, c, n), non_blocking=True)
                    elif c == 0:
                        dst.copy_(src, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(st)
                in_ready.append(ev)
        for ev in in_ready:
            comp.wait_event(ev)
        for ev in self.out_free[k]:
            comp.wait_event(ev)
        for a, _ in wl.e2e_in:
            setattr(wl, a, self.dev_in[k][a])
        for a, _ in wl.e2e_out:
            setattr(wl, a, self.dev_out[k][a])
        wl.step()
        done = torch.cuda.Event()
        done.record(comp)
        self.in_free[k] = done
        outs = []
        for c, st in enumerate(self.d2h):
            with torch.cuda.stream(st):
                st.wait_event(done)
                for a, h in wl.e2e_out:
                    self._part(self.host_out[k][h], c, n).copy_(self._part(self.dev_out[k][a], c, n),
                                                                non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(st)
                outs.append(ev)
        self.out_free[k] = outs
        self.i += 1

    def join(self):
        """Make the compute stream wait for every copy issued so far."""
        import torch
        comp = torch.cuda.current_stream()
        for evs in self.out_free:
            for ev in evs:
                comp.wait_event(ev)

    def start_on(self, ev):
        """Copies issued after this wait for `ev` (the timed region's start)."""
        for st in self.h2d + self.d2h:
            st.wait_event(ev)


# --------------------------------------------------------------------------- CPU oracle arm
ORACLE_SAMPLES = {
    # workload: (rows of A and of W sampled, K, A format, W format)
    "a8w4_fwd": (2048, 4096, "e4m3", "e2m1"),
    "mxfp4_moe_train": (1024, 7168, "e2m1", "e2m1"),
    "mxfp8_moe_train": (1024, 7168, "e4m3", "e4m3"),
    "blockwise_fp8": (1024, 7168, "bw", "bw"),
    "blockwise_fp8_pow2": (1024, 7168, "bw_pow2", "bw_pow2"),
    "dense_mxfp4_m8192": (1024, 8192, "e2m1", "e2m1"),
    "dense_mxfp4_m4096": (1024, 8192, "e2m1", "e2m1"),
    "dense_mxfp4_m2048": (1024, 8192, "e2m1", "e2m1"),
}


def oracle_sample(workload="a8w4_fwd", rows=None):
    """Bounded oracle sample of one GEMM of the workload: `rows` activation
    rows against `rows` weight rows of one expert at the workload's K --
    oracle quantization of both operands, dequantization and the fp64 matmul
    (about the step's flop per quantized element for the a8w4 forward)."""
    import oracle
    default_rows, K, ea, eb = ORACLE_SAMPLES[workload]
    rows = rows or default_rows
    rng = np.random.default_rng(12345)
    x = synth.normal_bf16(rng, (rows, K), outlier_frac=0.01)
    wt = synth.normal_bf16(rng, (rows, K), outlier_frac=0.01)
    t0 = time.perf_counter()
    if ea in ("bw", "bw_pow2"):
        p2 = ea == "bw_pow2"
        xc, xs = oracle.quantize_bw_1x128(x, pow2=p2)
        wc, ws = oracle.quantize_bw_128x128(wt.reshape(1, rows, K), pow2=p2)
        A = oracle.dequantize_bw_1x128(xc, xs)
        W = oracle.dequantize_bw_128x128(wc, ws)[0]
    else:
        xd, xs = oracle.quantize_mx_rowwise(x, ea)
        wd, ws = oracle.quantize_mx_rowwise(wt, eb)
        A = oracle.dequantize_mx(oracle.unpack_e2m1(xd) if ea == "e2m1" else xd, xs, ea)
        W = oracle.dequantize_mx(oracle.unpack_e2m1(wd) if eb == "e2m1" else wd, ws, eb)
    oracle.grouped_fwd(A, W, [rows], rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * rows * K
    return flops, dt, (f"{rows} A rows x {rows} W rows of one expert, K={K}: oracle quantize both "
                       f"+ dequantize + fp64 matmul")


def oracle_quantize_sample(workload="mxfp4_moe_train", rows=4096):
    """Bounded oracle sample of the row-wise quantizer of the workload's
    activation format: `rows` rows at the workload's K, timed in full, as
    algorithmic GB/s (BF16 read + codes + scales written)."""
    import oracle
    _, K, ea, _ = ORACLE_SAMPLES[workload]
    x = synth.normal_bf16(np.random.default_rng(54321), (rows, K))
    t0 = time.perf_counter()
    if ea in ("bw", "bw_pow2"):
        oracle.quantize_bw_1x128(x, pow2=ea == "bw_pow2")
        per_elt = 2 + 1 + 4 / 128
    else:
        oracle.quantize_mx_rowwise(x, ea)
        per_elt = 2 + (0.5 if ea == "e2m1" else 1.0) + 1 / 32
    dt = time.perf_counter() - t0
    fmt = {"e2m1": "MXFP4", "e4m3": "MXFP8", "bw": "1x128 FP8", "bw_pow2": "1x128 FP8 pow2"}[ea]
    return rows * K * per_elt / dt / 1e9, (f"oracle row-wise {fmt} quantize of {rows} x {K} BF16, "
                                           f"{per_elt:g} algorithmic bytes per element")


# Dense MMA instruction rates per SM and clock, measured on GB300 with
# back-to-back 128x256 block-scaled MMAs from resident shared memory: one
# 128x256x32 FP8 (or 128x256x64 FP4) MMA per 128 clocks.
RAW_MMA_FLOP_PER_CLK = {"fp8": 2 * 128 * 256 * 32 / 128, "fp4": 2 * 128 * 256 * 64 / 128}


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


SYNTH_OF = {"a8w4_fwd": "a8w4_fwd", "mxfp4_moe_train": "mxfp4_moe_train", "mxfp8_moe_train": "mxfp4_moe_train",
            "dense_mxfp4_m8192": "dense_mxfp4_m8192", "dense_mxfp4_m4096": "dense_mxfp4_m4096",
            "dense_mxfp4_m2048": "dense_mxfp4_m2048", "blockwise_fp8": "blockwise_fp8",
            "blockwise_fp8_pow2": "blockwise_fp8"}


def workload_config(name):
    """The GPU arm's `config` for a workload, built from its seeded synthetic
    description alone (no device memory): both arms print the same dict."""
    cls = WORKLOAD_CLASSES[name]
    w = synth.WORKLOADS[SYNTH_OF[name]]
    obj = cls.__new__(cls)
    obj.splits = w.splits()
    obj.G, obj.N, obj.K = w.G, w.N, w.K
    obj.pad = getattr(w, "pad", None)
    obj.S = int(obj.splits.sum())
    return obj.config()


def run_reference(args):
    """The oracle as the reference arm, timed on the host cores.  Each step is
    one bounded sample of the workload, sized so that warm-up plus timed steps
    stay within about two minutes whatever --steps is."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    c = cores()
    _, t_probe, _ = oracle_sample(args.workload, rows=256)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    default_rows = ORACLE_SAMPLES[args.workload][0]
    rows = int(256 * per_step / max(t_probe, 1e-3)) // 64 * 64
    rows = max(64, min(default_rows, rows))
    for _ in range(args.warmup):
        oracle_sample(args.workload, rows=rows)
    tot_f, tot_t = 0.0, 0.0
    sample = ""
    for _ in range(args.steps):
        f, t, sample = oracle_sample(args.workload, rows=rows)
        tot_f += f
        tot_t += t
    v = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": "grouped MXFP4/a8w4 GEMM TFLOPS (fwd/dgrad/wgrad) and % of GB300 FP4/FP8 peak",
            "value": v, "unit": "TFLOPS", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / max(args.steps, 1) * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload),
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
    import fp8_bf16_mxfp4_gb300 as mxg
    mxg.set_gemm_cta_group(args.cta_group)
    wl = build_workload(args.workload, dev)

    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    wl.check()

    # ---- device-resident timed region
    barrier(world)
    torch.cuda.synchronize()
    wl.timed.events = {}
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    smi_index = local
    with ClockSampler(smi_index) as clk:
        clk.wait_first_sample()
        ev0.record()
        for _ in range(args.steps):
            wl.step(time_gemm=True)
        ev1.record()
        torch.cuda.synchronize()
        clk.mark_end()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world, dev)
    gemm_ms = wl.timed.mean_ms()
    wl.check()

    # ---- end to end: pinned host inputs -> device -> results back to host
    e2e_ms = None
    if not args.skip_e2e:
        pipe = E2EPipeline(wl)
        for _ in range(max(2, args.warmup // 2)):
            pipe.step()
        pipe.join()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        pipe.start_on(e0)
        for _ in range(args.steps):
            pipe.step()
        pipe.join()
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        wl.check()

    if rank != 0:
        return
    steps = args.steps
    value = world * wl.flops * steps / (ms_max * 1e-3) / 1e12
    pk, src = peaks()
    clocks = clk.summary()
    # the burst bf16 figure for kernels timed in a region shorter than the
    # sustained measurement's seconds-long loop, the sustained one otherwise
    basis = "sustained" if ms_max >= 2000.0 else "burst"
    bf16_peak = pk["bf16_tflops_sustained" if basis == "sustained" else "bf16_tflops"]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or pk.get("sm_max_mhz", 2070.0)
    hbm = pk["hbm_gbs"]
    passes = {}
    for name, (f, ratio, kind) in wl.gemm_info.items():
        t = gemm_ms[name]
        peak = bf16_peak * ratio
        tf = f / (t * 1e-3) / 1e12
        raw = RAW_MMA_FLOP_PER_CLK["fp4" if kind.startswith("mxf4") else "fp8"] * sms * mhz * 1e6 / 1e12
        nbytes = wl.pass_bytes[name]
        t_tensor, t_hbm = f / (peak * 1e12), nbytes / (hbm * 1e9)     # seconds at each roof
        passes[name] = {"ms": t, "tflops": tf, "peak": peak, "frac": tf / peak, "mma": kind,
                        "raw_mma_tflops": raw, "frac_of_raw_mma": tf / raw,
                        "bytes": nbytes, "gbs": nbytes / (t * 1e-3) / 1e9,
                        "bound": "hbm" if t_hbm > t_tensor else "tensor",
                        "roofline_frac": max(t_tensor, t_hbm) / (t * 1e-3)}
    dom = max(passes, key=lambda k: passes[k]["ms"])
    d = passes[dom]
    if args.skip_cpu_baseline:
        cpu_f, cpu_t, sample, q_gbs, q_sample = 0.0, 1.0, "skipped", None, "skipped"
    else:
        cpu_f, cpu_t, sample = oracle_sample(args.workload)
        q_gbs, q_sample = oracle_quantize_sample(args.workload)
    line = {
        "metric": "grouped MXFP4/a8w4 GEMM TFLOPS (fwd/dgrad/wgrad) and % of GB300 FP4/FP8 peak",
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms_max / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": dict(wl.config(), gemm_cta_group=args.cta_group),
        "roofline": dict(
            ({"bound": "hbm", "achieved": d["gbs"], "peak": hbm, "unit": "GB/s", "frac": d["gbs"] / hbm,
              "peak_source": f"{src}: hbm_gbs (copy); of measured",
              "tensor_frac": d["frac"]} if d["bound"] == "hbm" else
             {"bound": "tensor", "achieved": d["tflops"], "peak": d["peak"], "unit": "TFLOP/s", "frac": d["frac"],
              "peak_source": f"{src}: bf16_tflops ({basis}) x {wl.gemm_info[dom][1]:g} "
                             f"(nominal {wl.gemm_info[dom][2]}/bf16 dense ratio); of measured",
              "hbm_frac": d["gbs"] / hbm}),
            traffic=getattr(wl, "traffic_bytes", {}).get(dom) if isinstance(getattr(wl, "traffic_bytes", None), dict)
            else None,
            algorithmic_bytes=d["bytes"], flops=wl.gemm_info[dom][0],
            kernel=f"grouped GEMM {dom} call ({getattr(wl, 'call_kernels', 'plan + scale pack + tcgen05 GEMM')})",
            gemm_ms=d["ms"], frac_of_raw_mma=d["frac_of_raw_mma"]),
        "passes": passes,
        "cpu_baseline": {"value": cpu_f / cpu_t / 1e12, "unit": "TFLOPS", "cores": cores(),
                         "kind": "oracle", "sample": sample},
        "cpu_baseline_quantize": {"value": q_gbs, "unit": "GB/s", "cores": cores(), "kind": "oracle",
                                  "sample": q_sample},
        "gpu_launches": wl.launches_per_step * steps,
        "clocks": clocks,
    }
    if e2e_ms is not None:
        line["e2e"] = {"value": world * wl.flops * steps / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                       "h2d_bytes_per_step": wl.h2d_bytes(), "d2h_bytes_per_step": wl.d2h_bytes(),
                       "ms_per_step": e2e_ms / steps}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mxfp4_moe_train", choices=sorted(WORKLOAD_CLASSES))
    ap.add_argument("--skip-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--skip-cpu-baseline", action="store_true",
                    help="omit the oracle legs (profiling runs of the GPU kernels)")
    ap.add_argument("--cta-group", type=int, default=2, choices=[1, 2],
                    help="MX GEMM kernel: 2 = CTA pairs sharing 256x256 tiles (default), 1 = one-SM kernel")
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
