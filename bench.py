"""Benchmark: conv GFLOP/s and fraction of the GB300 roofline, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extra]

A step is one forward convolution over the whole batch of the headline
workload (Conv3d, x [16,3,64,64,64], kernel (3,5,7), 64 output channels,
bias), through the C ABI (conv_fwd_nd), with inputs already resident in HBM.
L2 is flushed (a 2x-L2 buffer is written) before every step, outside the
per-step CUDA events.  The line also carries:
  e2e          the same metric with the step's inputs copied host->device from
               pinned memory and the output copied back, inside the timing;
  roofline     the dominant kernel's achieved rate against its pipe's peak,
               measured in the same run by the library's microbenchmarks
               (tcgen05.mma TF32 / BF16, FP32 FMA; scaled to the SM's maximum
               clock) or, for HBM-bound kernels, the measured copy bandwidth;
  pipe_peaks   those measured peaks, with the clock of each measurement;
  cpu_baseline the fp64 oracle timed on a bounded sample on the host cores;
  per_config   the other workloads (fused conv3d+min+softmax, long Conv1d,
               the two sweep shapes, the tiny Conv1d), each timed the same way,
               each with its own oracle timing on a smaller bounded sample.
With --impl reference the oracle itself is the measured implementation.
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the problem shards by batch with no exchange); value sums all ranks' work
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

HEADLINE = "conv3d_asym"
EXTRA = ["conv3d_min_softmax", "conv1d_long", "conv3d_sweep_a", "conv3d_sweep_b", "conv1d_tiny"]
METRIC = "conv GFLOP/s and % of GB300 roofline (fp32/TF32 or HBM) per config, 1 GPU"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
SM_MAX_MHZ_NOMINAL = 2070.0
BF16_TO_TF32 = 1.1 / 2.25  # nominal dense tensor-core ratio TF32 : BF16 (for the secondary, derived figure)
CPU_BASELINE_MACS = 8e9     # ~10-20 s of the oracle on the host cores
CONFIG_ORACLE_MACS = 2e9    # ~1-3 s of the oracle per extra config
REFERENCE_STEP_MACS = 1e9   # one reference-arm step: a ~1-2 s slab of the workload


def env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": SM_MAX_MHZ_NOMINAL}, "fallback"


def measure_pipe_peaks(cf, sm_max_mhz):
    """Peak rates of the pipes the kernels use, measured here by the library's microbenchmarks
    (conv_peak_mma, conv_peak_ffma), each scaled from the SM clock of its own run to the SM's
    maximum clock: the conservative denominator for a kernel timed at any clock up to it."""
    out = {}
    runs = {
        "tf32": [cf.peak_mma("tf32", 256, iss, True, 4000) for iss in (2, 4)],
        "bf16": [cf.peak_mma("bf16", 256, iss, True, 4000) for iss in (2, 4)],
        "ffma": [cf.peak_ffma(packed, 3000) for packed in (False, True)],
    }
    for name, rs in runs.items():
        r = max(rs, key=lambda d: d["tflops"])
        scale = sm_max_mhz / r["sm_mhz"] if r["sm_mhz"] > 0 else 1.0
        out[name] = {"tflops": r["tflops"] * scale, "measured_tflops": r["tflops"], "measured_mhz": r["sm_mhz"],
                     "scaled_to_mhz": sm_max_mhz, "cycles_per_op": r["cycles_per_op"]}
    out["tf32x3"] = {"tflops": out["tf32"]["tflops"] / 3.0, "note": "three TF32 products per fp32 multiply-add"}
    out["source"] = "microbenchmark"
    return out


def problem_counts(wl, out_dims, esize=4):
    """Algorithmic FLOPs (2 per MAC, padded taps included) and compulsory bytes (esize bytes per element)."""
    out_sp = int(np.prod(out_dims))
    k_sp = int(np.prod(wl.k_dims))
    flops = 2.0 * wl.N * wl.C_out * out_sp * wl.C_in * k_sp
    x_b = float(esize) * wl.N * wl.C_in * int(np.prod(wl.in_dims))
    w_b = float(esize) * wl.C_out * wl.C_in * k_sp
    b_b = float(esize) * wl.C_out if wl.bias else 0.0
    if wl.kind == "fused":
        y_b = float(esize) * wl.N * wl.C_out * out_dims[1] * out_dims[2]
    else:
        y_b = float(esize) * wl.N * wl.C_out * out_sp
    return flops, x_b + w_b + b_b + y_b, x_b + w_b + b_b, y_b


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background during the timed region.

    The sampler is started, and its first sample awaited (at most a few seconds),
    before the timed region begins; mark(start, end) records the region's host
    times, and summary() takes the median SM clock over the samples stamped
    inside it (the nearest sample after the region when it was too short to
    hold one) and every throttle reason seen in or next to it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 10

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.region = None
        self.path = os.path.join("/tmp", f"convfwd_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        deadline = time.time() + 5.0
        while time.time() < deadline and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)
        return self

    def mark(self, t_start, t_end):
        self.region = (t_start, t_end)

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(3 * self.PERIOD_MS / 1000.0)  # one more sample after the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    @staticmethod
    def parse(lines):
        """Rows (host time or None, SM MHz, max SM MHz, [reason fields]) of nvidia-smi's CSV."""
        import datetime
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            try:
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except ValueError:
                continue
        return rows

    @staticmethod
    def summarize(rows, region=None):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        use = rows
        in_region = None
        if region is not None and all(r[0] is not None for r in rows):
            t0, t1 = region
            inside = [r for r in rows if t0 <= r[0] <= t1]
            in_region = len(inside)
            if inside:
                use = inside
            else:
                after = [r for r in rows if r[0] > t1]
                use = after[:1] or rows[-1:]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, _, r in use:
            for nm, v in zip(names, r[1:5]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        mhz = [r[1] for r in use]
        loaded = [m for m in mhz if m > 0.5 * max(mhz)] or mhz
        out = {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[2] for r in use),
               "reasons": sorted(reasons), "samples": len(use)}
        if in_region is not None:
            out["samples_in_timed_region"] = in_region
            out["period_ms"] = ClockSampler.PERIOD_MS
        return out

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        with open(self.path) as f:
            return self.summarize(self.parse(f), self.region)


# --------------------------------------------------------------- our arm

class OurRunner:
    def __init__(self, wl, device, fused_algo="auto"):
        import torch
        import implicit_gemm_convolution_fwd_gb300 as cf
        self.torch, self.cf, self.wl, self.dev = torch, cf, wl, device
        # the fused op's kernel family: the planner (the library's own query says which
        # family it takes), or one family forced
        self.fused_code = {"auto": cf.CONV_ALGO_AUTO, "ffma": cf.CONV_ALGO_DIRECT_FFMA,
                           "tc": cf.CONV_ALGO_IGEMM_3XTF32}[fused_algo]
        x, w, b = wl.make_inputs(seed=0)
        self.host = {"x": x, "w": w, "b": b}
        self.x = torch.from_numpy(x).to(device)
        self.w = torch.from_numpy(w).to(device)
        self.b = None if b is None else torch.from_numpy(b).to(device)
        if wl.kind == "fused":
            self.out_dims = cf.out_dims(wl.in_dims, wl.k_dims, 1, 0, 1)
            self.y = torch.empty((wl.N, wl.C_out, self.out_dims[1], self.out_dims[2]), device=device)
            fam = self.fused_code
            if fam == cf.CONV_ALGO_AUTO:
                fam = cf.fused_select_algo((wl.N, wl.C_in) + tuple(wl.in_dims), (wl.C_out, wl.C_in) + tuple(wl.k_dims),
                                           wl.min_dim)
            self.algo = "fused_igemm_3xtf32" if fam == cf.CONV_ALGO_IGEMM_3XTF32 else "fused_ffma"
        else:
            self.out_dims = cf.out_dims(wl.in_dims, wl.k_dims, wl.stride, wl.pad, wl.dilation)
            self.y = torch.empty((wl.N, wl.C_out) + tuple(self.out_dims), device=device)
            self.algo = cf.ALGO_NAMES[cf.select_algo(wl.N, wl.C_in, wl.C_out, wl.in_dims, wl.k_dims, wl.stride,
                                                     wl.pad, wl.dilation)]
        self.stream = torch.cuda.current_stream(device)
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.flush_buf = torch.empty(int(2 * l2 // 4) + 1024, dtype=torch.float32, device=device)

    def launches_per_step(self):
        return 1

    def step(self):
        if self.wl.kind == "fused":
            self.cf.conv3d_min_softmax(self.x, self.w, self.b, self.wl.min_dim, out=self.y, stream=self.stream,
                                       algo=self.fused_code)
        else:
            self.cf.conv_fwd_nd(self.x, self.w, self.b, self.wl.stride, self.wl.pad, self.wl.dilation, out=self.y,
                                stream=self.stream)

    def flush(self):
        self.flush_buf.fill_(1.0)

    def timed(self, steps, warmup, flush=True):
        """Per-step device times (ms) with CUDA events on the launching stream."""
        torch = self.torch
        for _ in range(warmup):
            if flush:
                self.flush()
            self.step()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for s, e in evs:
            if flush:
                self.flush()
            s.record(self.stream)
            self.step()
            e.record(self.stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in evs]

    def timed_e2e(self, steps, warmup):
        """Same call with H2D of the step's inputs (pinned) and D2H of its output inside the timing.
        A plain fp32 conv goes through conv_fwd_nd_host (host buffers in and out, the batch in chunks whose
        copies overlap the convolution); other entry points copy around the device call."""
        torch = self.torch
        if self.wl.kind == "conv" and type(self) is OurRunner:
            return self.timed_e2e_host(steps, warmup)
        # host copies in the device tensors' dtype (the call's own input type)
        hx = torch.from_numpy(self.host["x"]).to(self.x.dtype).pin_memory()
        hw = torch.from_numpy(self.host["w"]).to(self.w.dtype).pin_memory()
        hb = None if self.host["b"] is None else torch.from_numpy(self.host["b"]).to(self.b.dtype).pin_memory()
        hy = torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory()

        def one():
            self.x.copy_(hx, non_blocking=True)
            self.w.copy_(hw, non_blocking=True)
            if hb is not None:
                self.b.copy_(hb, non_blocking=True)
            self.step()
            hy.copy_(self.y, non_blocking=True)

        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(self.stream)
        for _ in range(steps):
            one()
        e.record(self.stream)
        torch.cuda.synchronize()
        nbytes = lambda t: 0 if t is None else t.numel() * t.element_size()
        return s.elapsed_time(e) / steps, nbytes(hx) + nbytes(hw) + nbytes(hb), nbytes(hy)


    def timed_e2e_host(self, steps, warmup):
        torch, wl = self.torch, self.wl
        hx = torch.from_numpy(self.host["x"]).pin_memory()
        hw = torch.from_numpy(self.host["w"]).pin_memory()
        hb = None if self.host["b"] is None else torch.from_numpy(self.host["b"]).pin_memory()
        hy = torch.empty(self.y.shape, dtype=torch.float32).pin_memory()
        chunk = max(1, wl.N // 8)  # about eight chunks: the first copy-in and last copy-out are short
        ws = torch.empty(self.cf.host_workspace_bytes(wl.N, wl.C_in, wl.C_out, wl.in_dims, wl.k_dims, wl.stride,
                                                      wl.pad, wl.dilation, 1, chunk),
                         dtype=torch.uint8, device=self.dev)

        def one():
            self.cf.conv_fwd_nd_host(hx, hw, hb, wl.stride, wl.pad, wl.dilation, chunk=chunk, workspace=ws, out=hy,
                                     stream=self.stream)

        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(self.stream)
        for _ in range(steps):
            one()
        e.record(self.stream)
        torch.cuda.synchronize()
        nbytes = lambda t: 0 if t is None else t.numel() * t.element_size()
        del ws
        return s.elapsed_time(e) / steps, nbytes(hx) + nbytes(hw) + nbytes(hb), nbytes(hy)


class VariantRunner(OurRunner):
    """A benchmark workload run through one of the library's other entry points:
    16-bit tensors, the min over another dim, channels-last tensors or groups."""

    def __init__(self, wl, device, dtype=None, min_dim=None, channels_last=False, groups=1, workspace=False,
                 fused_algo="auto"):
        super().__init__(wl, device, fused_algo)
        torch = self.torch
        self.dtype, self.channels_last, self.groups = dtype, channels_last, groups
        self.ws = None
        self.ws_stream = 0  # workspace bytes for streamed weights
        if workspace:
            self.ws_stream = self.cf.workspace_bytes(wl.N, wl.C_in, wl.C_out, wl.in_dims, wl.k_dims, wl.stride,
                                                     wl.pad, wl.dilation)
            self.ws = torch.empty(max(self.ws_stream, 1), dtype=torch.uint8, device=device)
        self.min_dim = wl.min_dim if min_dim is None else min_dim
        if groups > 1:
            self.w = self.w[:, :wl.C_in // groups].contiguous()
        if dtype is not None:
            self.x, self.w = self.x.to(dtype), self.w.to(dtype)
            self.b = None if self.b is None else self.b.to(dtype)
            self.y = self.y.to(dtype)
        if channels_last:
            fmt = {3: torch.channels_last, 5: torch.channels_last_3d}[self.x.dim()]
            self.x, self.w = self.x.to(memory_format=fmt), self.w.to(memory_format=fmt)
            self.y = self.y.to(memory_format=fmt)
        if wl.kind == "fused":
            od = self.out_dims
            keep = [od[i] for i in range(3) if i != self.min_dim - 2]
            self.y = torch.empty((wl.N, wl.C_out, keep[0], keep[1]), device=device)
            fam = self.fused_code
            if fam == self.cf.CONV_ALGO_AUTO:
                fam = self.cf.fused_select_algo((wl.N, wl.C_in) + tuple(wl.in_dims),
                                                (wl.C_out, wl.C_in) + tuple(wl.k_dims), self.min_dim)
            self.algo = "fused_igemm_3xtf32" if fam == self.cf.CONV_ALGO_IGEMM_3XTF32 else "fused_ffma"

    def launches_per_step(self):
        # streamed weights: the weight split runs before the conv kernel
        return 1 + (self.ws is not None and self.ws_stream > 0)

    def step(self):
        if self.wl.kind == "fused":
            self.cf.conv3d_min_softmax(self.x, self.w, self.b, self.min_dim, out=self.y, stream=self.stream,
                                       algo=self.fused_code)
        elif self.ws is not None:
            self.cf.conv_fwd_nd_ws(self.x, self.w, self.b, self.wl.stride, self.wl.pad, self.wl.dilation,
                                   workspace=self.ws, out=self.y, stream=self.stream)
        else:
            self.cf.conv_fwd_nd(self.x, self.w, self.b, self.wl.stride, self.wl.pad, self.wl.dilation, out=self.y,
                                stream=self.stream, groups=self.groups, channels_last=self.channels_last)


# (name, workload, options): the other entry points on the benchmark workloads
VARIANTS = [
    ("conv3d_asym[bf16]", "conv3d_asym", {"dtype": "bfloat16"}),
    ("conv3d_asym[fp16]", "conv3d_asym", {"dtype": "float16"}),
    ("conv1d_long[bf16]", "conv1d_long", {"dtype": "bfloat16"}),
    ("conv3d_sweep_b[bf16]", "conv3d_sweep_b", {"dtype": "bfloat16"}),
    ("conv3d_min_softmax[min_dim=3]", "conv3d_min_softmax", {"min_dim": 3}),
    ("conv3d_min_softmax[min_dim=4]", "conv3d_min_softmax", {"min_dim": 4}),
    ("conv3d_min_softmax[ffma]", "conv3d_min_softmax", {"fused_algo": "ffma"}),
    ("conv3d_sweep_b[channels_last]", "conv3d_sweep_b", {"channels_last": True}),
    ("conv3d_sweep_b[groups=2]", "conv3d_sweep_b", {"groups": 2}),
    ("conv3d_wide_k[workspace]", "conv3d_wide_k", {"workspace": True}),
    ("conv3d_wide_k[no workspace]", "conv3d_wide_k", {}),
]


def run_variants(dev, peaks, pipes, steps):
    """ms and throughput of each VARIANTS entry (CUDA events, L2 flushed, median)."""
    import torch
    out = {}
    for name, wname, opts in VARIANTS:
        o = dict(opts)
        if "dtype" in o:
            o["dtype"] = getattr(torch, o["dtype"])
        r = VariantRunner(synth.WORKLOADS[wname], dev, **o)
        times = r.timed(steps, 3)
        m = statistics.median(times)
        flops, _, _, _ = problem_counts(r.wl, r.out_dims)
        flops /= r.groups  # each output channel sums over C_in / groups input channels
        entry = {"ms": m, "ms_min": min(times), "tflops": flops / (m * 1e-3) / 1e12}
        if r.dtype is None and r.wl.kind == "conv":
            entry["frac_of_3xtf32_peak"] = entry["tflops"] / pipes["tf32x3"]["tflops"]
        if r.dtype is not None:
            entry["frac_of_bf16_peak"] = entry["tflops"] / pipes["bf16"]["tflops"]
            entry["frac_of_cublas_bf16"] = entry["tflops"] / peaks["bf16_tflops"]
        if r.dtype is None and r.wl.kind == "fused":
            entry["kernel"] = r.algo
            if r.algo == "fused_igemm_3xtf32":
                entry["frac_of_3xtf32_peak"] = entry["tflops"] / pipes["tf32x3"]["tflops"]
            else:
                entry["frac_of_ffma_peak"] = entry["tflops"] / pipes["ffma"]["tflops"]
        out[name] = entry
        del r
    return out


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from one
# ncu capture, keyed by (kernel family, workload).  Each entry records the
# SHA-256 of the kernel's source file at capture time; when the source has
# changed since, the figure no longer describes the kernel and is reported as
# null.  "batch" is the batch of the captured case: traffic is scaled by
# N / batch when the capture used a smaller batch (traffic grows in proportion).
KERNEL_SOURCE = {"igemm_3xtf32": "igemm_tcgen05.cu", "igemm_3xtf32_streamed": "igemm_tcgen05.cu",
                 "fused_igemm_3xtf32": "igemm_tcgen05.cu",
                 "igemm_bf16": "igemm_bf16.cuh", "igemm_fp16": "igemm_bf16.cuh", "direct_ffma": "direct.cu",
                 "fused_ffma": "fused.cu"}
NCU_TRAFFIC = {
    ("igemm_3xtf32", "conv3d_asym"): {"bytes": 50.508800e6 + 824.164352e6, "batch": 16,
        "sha256": "6d0fc6e91eb83035c65561193ddc8ac9195b5fc0f6e0b6d1024af98b60a754d1"},
    ("igemm_3xtf32", "conv1d_long"): {"bytes": 537.356800e6 + 307.589120e6, "batch": 4,
        "sha256": "6d0fc6e91eb83035c65561193ddc8ac9195b5fc0f6e0b6d1024af98b60a754d1"},
    ("igemm_3xtf32", "conv3d_sweep_a"): {"bytes": 28.486400e6 + 0.137216e6, "batch": 8,
        "sha256": "6d0fc6e91eb83035c65561193ddc8ac9195b5fc0f6e0b6d1024af98b60a754d1"},
    ("igemm_3xtf32", "conv3d_sweep_b"): {"bytes": 113.426944e6 + 70.425600e6, "batch": 8,
        "sha256": "6d0fc6e91eb83035c65561193ddc8ac9195b5fc0f6e0b6d1024af98b60a754d1"},
    ("igemm_3xtf32_streamed", "conv3d_wide_k"): {"bytes": 35.390720e6 + 8.529920e6, "batch": 4,
        "sha256": "6d0fc6e91eb83035c65561193ddc8ac9195b5fc0f6e0b6d1024af98b60a754d1"},
    ("fused_igemm_3xtf32", "conv3d_min_softmax"): {"bytes": 37.828352e6 + 0.004352e6, "batch": 128,
        "sha256": "6d0fc6e91eb83035c65561193ddc8ac9195b5fc0f6e0b6d1024af98b60a754d1"},
    ("igemm_bf16", "conv3d_asym"): {"bytes": 25.302272e6 + 386.399744e6, "batch": 16,
        "sha256": "f3b938ade490fd2bf7935b687e4595f796a923254b86fe6c215db4fb9b533691"},
    ("fused_ffma", "conv3d_min_softmax"): {"bytes": 37.822976e6 + 0.001536e6, "batch": 128,
        "sha256": "d7b3eb929d7b9c18018afbc7d515d7c578250c6c7bcdeecece2e78aeb73812eb"},
    ("direct_ffma", "conv1d_tiny"): {"bytes": 0.051968e6, "batch": 2,
        "sha256": "c89212c4b2a3b47cebf81b80fa94530bb29ddb0f5ed58ae23df0585b90d2ac41"},
}


def source_sha(algo):
    import hashlib
    f = KERNEL_SOURCE.get(algo)
    if f is None:
        return None
    path = os.path.join(ROOT, "implicit_gemm_convolution_fwd_gb300", "csrc", f)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


def traffic_for(algo, wl):
    e = NCU_TRAFFIC.get((algo, wl.name.split("[")[0]))
    if e is None or e["sha256"] != source_sha(algo):
        return None
    return e["bytes"] * wl.N / e["batch"]


def roofline_for(runner, peaks, pipes, ms):
    """Roofline entry for the one kernel a step launches.  Compute peaks are the measured pipe peaks
    (`pipes`, see measure_pipe_peaks); HBM is MEASURED_PEAKS.json's copy bandwidth."""
    wl = runner.wl
    flops, bytes_alg, _, _ = problem_counts(wl, runner.out_dims, runner.y.element_size())
    t = ms * 1e-3
    hbm_peak = peaks["hbm_gbs"]
    if runner.algo in ("igemm_3xtf32", "igemm_3xtf32_streamed", "fused_igemm_3xtf32"):
        compute = {"bound": "tensor", "peak": pipes["tf32x3"]["tflops"],
                   "peak_note": "measured TF32 tcgen05.mma rate / 3 products (3xTF32)",
                   "derived_peak": peaks["bf16_tflops"] * BF16_TO_TF32 / 3.0}
    elif runner.algo in ("igemm_bf16", "igemm_fp16"):
        compute = {"bound": "tensor", "peak": pipes["bf16"]["tflops"],
                   "peak_note": "measured BF16 tcgen05.mma rate (FP16 the same)", "derived_peak": peaks["bf16_tflops"]}
    else:
        compute = {"bound": "alu", "peak": pipes["ffma"]["tflops"], "peak_note": "measured FP32 FMA rate",
                   "derived_peak": None}
    t_compute = flops / (compute["peak"] * 1e12)
    t_mem = bytes_alg / (hbm_peak * 1e9)
    # the fraction against the faster of the two fp32-accurate pipes, whichever
    # the kernel uses, so that the choice of path cannot flatter the number
    best = max(pipes["ffma"]["tflops"], pipes["tf32x3"]["tflops"])
    t_best = max(flops / (best * 1e12), t_mem)
    frac_best = t_best / t
    # the table's captures are of N C D H W launches; a channels-last run has none
    traffic = None if getattr(runner, "channels_last", False) else traffic_for(runner.algo, wl)
    common = {"traffic": traffic, "algorithmic_bytes": bytes_alg, "frac_best_path": frac_best,
              "peak_source": pipes["source"], "peak_mhz": pipes["tf32"]["scaled_to_mhz"]}
    if t_mem > t_compute:
        return dict(common, bound="hbm", achieved=bytes_alg / t / 1e9, peak=hbm_peak, unit="GB/s",
                    frac=(bytes_alg / t / 1e9) / hbm_peak, compute_frac=(flops / t / 1e12) / compute["peak"],
                    peak_note="measured copy bandwidth (MEASURED_PEAKS.json)")
    ach = flops / t / 1e12
    out = dict(common, bound=compute["bound"], achieved=ach, peak=compute["peak"], unit="TFLOP/s",
               frac=ach / compute["peak"], peak_note=compute["peak_note"], hbm_frac=(bytes_alg / t / 1e9) / hbm_peak)
    if compute["derived_peak"]:
        out["derived_peak"] = compute["derived_peak"]
        out["frac_of_derived_peak"] = ach / compute["derived_peak"]
    return out


# ----------------------------------------------------------- oracle legs

def oracle_sample(wl, target_macs):
    """A bounded sample of workload `wl` for the oracle: the leading batch items
    and, for long inputs, a leading slab of the outermost spatial dim of x,
    sized to about `target_macs` multiply-adds."""
    k_sp = int(np.prod(wl.k_dims))
    if wl.kind == "fused":
        od = [wl.in_dims[i] - wl.k_dims[i] + 1 for i in range(3)]
    else:
        import oracle
        od = list(oracle.out_dims(wl.in_dims, wl.k_dims, wl.stride, wl.pad, wl.dilation))
    per_item = wl.C_out * int(np.prod(od)) * wl.C_in * k_sp
    n = int(min(wl.N, max(1, target_macs // per_item)))
    x, w, b = wl.with_batch(n).make_inputs(seed=0)
    if n == 1 and per_item > 2 * target_macs:
        # keep enough of the outermost spatial dim for ~target_macs
        frac = target_macs / per_item
        keep_out = max(1, int(od[0] * frac))
        s0, d0, k0 = wl.stride[0], wl.dilation[0], wl.k_dims[0]
        keep_in = min(wl.in_dims[0], (keep_out - 1) * s0 + (k0 - 1) * d0 + 1)
        x = np.ascontiguousarray(x[:, :, :keep_in])
    return x, w, b


def time_oracle(wl, target_macs):
    import oracle
    x, w, b = oracle_sample(wl, target_macs)
    threads = oracle.threads()
    t0 = time.perf_counter()
    if wl.kind == "fused":
        y = oracle.conv3d_min_softmax(x, w, b, nthreads=threads)
        od = (x.shape[2] - w.shape[2] + 1,) + tuple(y.shape[2:])
    else:
        y = oracle.conv_nd(x, w, b, wl.stride, wl.pad, wl.dilation, nthreads=threads)
        od = y.shape[2:]
    dt = time.perf_counter() - t0
    macs = float(x.shape[0]) * wl.C_out * int(np.prod(od)) * wl.C_in * int(np.prod(wl.k_dims))
    sample = (f"{wl.name}: first {x.shape[0]} of {wl.N} batch items, x spatial {list(x.shape[2:])} "
              f"({macs:.3g} MACs, fp64 accumulation, {threads} threads)")
    return 2.0 * macs / dt / 1e9, dt, threads, sample


# ------------------------------------------------------------------ ranks

def slowest_rank_ms(ms, world, device=None):
    """Max over ranks of a per-rank step time (ms); identity for one rank.

    Every rank runs an independent replica (the batch shards with no data
    exchange), so the job's throughput is all ranks' work over the slowest
    rank's time."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step, ms, world):
    """Whole-job GFLOP/s: the work of all `world` replicas over the slowest step time."""
    return world * flops_per_rank_step / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-extra", action="store_true", help="skip the per-config table")
    ap.add_argument("--no-variants", action="store_true", help="skip the other entry points' table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small cases for profiler captures)")
    ap.add_argument("--dtype", choices=["f32", "bf16", "fp16"], default="f32",
                    help="run the workload on 16-bit tensors (the 16-bit tensor-core entry points)")
    ap.add_argument("--fused-algo", choices=["auto", "ffma", "tc"], default="auto",
                    help="kernel family of a fused workload (auto: the library's planner)")
    ap.add_argument("--channels-last", action="store_true",
                    help="x, w and y stored channels last (conv_fwd_nd_channels_last); a profiling aid")
    ap.add_argument("--workspace", action="store_true",
                    help="run the workload through conv_fwd_nd_ws (streamed weights when they exceed shared memory)")
    args = ap.parse_args()
    rank, world, local = env_rank()
    wl = synth.WORKLOADS[args.workload]
    if args.batch is not None:
        wl = wl.with_batch(args.batch)

    if args.impl == "reference":
        return main_reference(args, wl, rank, world)

    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()
    import implicit_gemm_convolution_fwd_gb300 as cf
    peaks, peaks_src = load_peaks()
    sm_max_mhz = float(peaks.get("sm_max_mhz") or SM_MAX_MHZ_NOMINAL)
    pipes = measure_pipe_peaks(cf, sm_max_mhz)  # before the timed region

    if args.dtype != "f32" or args.workspace or args.channels_last:
        dt = {"f32": None, "bf16": torch.bfloat16, "fp16": torch.float16}[args.dtype]
        runner = VariantRunner(wl, dev, dtype=dt, workspace=args.workspace, channels_last=args.channels_last)
        if dt is not None:
            runner.algo = "igemm_" + args.dtype
        elif runner.ws is not None and runner.ws_stream > 0:
            runner.algo = "igemm_3xtf32_streamed"
    else:
        runner = OurRunner(wl, dev, args.fused_algo)
    flops, bytes_alg, in_b, out_b = problem_counts(wl, runner.out_dims, runner.y.element_size())
    # warm-up, then EXACTLY K timed steps bracketed by barrier + synchronize
    with ClockSampler(local) as clk:  # live before the warm-up starts
        runner.timed(0, args.warmup)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        h0 = time.time()
        per_step = runner.timed(args.steps, 0)
        torch.cuda.synchronize()
        clk.mark(h0, time.time())
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    ms = slowest_rank_ms(sum(per_step) / len(per_step), world, dev)
    value = job_throughput(flops, ms, world)

    # the same step with L2 left warm (no flush): inputs that fit in L2 stay there
    warm = runner.timed(max(5, args.steps // 4), 2, flush=False)
    ms_warm = statistics.median(warm)

    e2e_ms, h2d, d2h = runner.timed_e2e(max(3, args.steps // 4), 2)
    e2e_ms = slowest_rank_ms(e2e_ms, world, dev)
    roof = roofline_for(runner, peaks, pipes, ms)
    roof["hbm_peak_source"] = peaks_src
    roof["kernel"] = runner.algo
    clocks = clk.summary()

    per_config = {}
    if not args.no_extra and rank == 0:
        del runner.flush_buf
        for name in EXTRA:
            if name == wl.name:
                continue
            r = OurRunner(synth.WORKLOADS[name], dev)
            times = r.timed(max(5, args.steps // 2), 3)
            m = statistics.median(times)
            m_warm = statistics.median(r.timed(max(5, args.steps // 4), 2, flush=False))
            f, bts, _, _ = problem_counts(r.wl, r.out_dims)
            rf = roofline_for(r, peaks, pipes, m)
            per_config[name] = {"algo": r.algo, "ms": m, "ms_min": min(times), "gflops": f / (m * 1e-3) / 1e9,
                                "gbs": bts / (m * 1e-3) / 1e9, "roofline_bound": rf["bound"],
                                "roofline_frac": rf["frac"], "roofline_peak": rf["peak"], "unit": rf["unit"],
                                "roofline_frac_best_path": rf["frac_best_path"], "ms_l2_warm": m_warm}
            if "frac_of_derived_peak" in rf:
                per_config[name]["roofline_frac_of_derived_peak"] = rf["frac_of_derived_peak"]
            del r
            torch.cuda.empty_cache()
    variants = {}
    if not args.no_extra and not args.no_variants and rank == 0:
        variants = run_variants(dev, peaks, pipes, max(5, args.steps // 4))
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, threads, sample = time_oracle(wl, CPU_BASELINE_MACS)
        cpu = {"value": v, "unit": "GFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
               "seconds": dt}
        # the oracle beside every other config too, on a smaller bounded sample each
        for name, entry in per_config.items():
            cv, cdt, cthreads, csample = time_oracle(synth.WORKLOADS[name], CONFIG_ORACLE_MACS)
            entry["cpu_baseline"] = {"value": cv, "unit": "GFLOP/s", "cores": cthreads, "kind": "oracle",
                                     "sample": csample, "seconds": cdt, "gpu_over_cpu": entry["gflops"] / cv}

    if world > 1:
        dist.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": args.dtype, "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": wl.name, "description": wl.description, "global_batch": wl.N * world,
                       "in_dims": list(wl.in_dims), "k_dims": list(wl.k_dims), "C_in": wl.C_in, "C_out": wl.C_out,
                       "stride": list(wl.stride), "pad": list(wl.pad), "dilation": list(wl.dilation),
                       "bias": wl.bias, "parallelism": f"replicas{world}",
                       "layout": "channels last" if args.channels_last else "N C (D) (H) W",
                       "l2": "flushed before every step (2x L2 write, outside the per-step events)",
                       "kernel": runner.algo, "gflop_per_step": flops / 1e9, "bytes_per_step": bytes_alg,
                       "gbs": bytes_alg / (ms * 1e-3) / 1e9, "ms_min": min(per_step),
                       "ms_median": statistics.median(per_step), "ms_l2_warm": ms_warm, "wall_s": wall},
            "e2e": {"value": job_throughput(flops, e2e_ms, world), "unit": "GFLOP/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "call": ("conv_fwd_nd_host (pinned host buffers, batch in chunks of max(1, N/8))"
                             if runner.wl.kind == "conv" and type(runner) is OurRunner
                             else "pinned host copies around the device call")},
            "gpu_launches": runner.launches_per_step() * args.steps,
            "roofline": roof, "clocks": clocks, "cpu_baseline": cpu, "per_config": per_config, "other_entry_points": variants,
            "pipe_peaks": pipes,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main_reference(args, wl, rank, world):
    """The oracle as the measured implementation, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        time_oracle(wl, REFERENCE_STEP_MACS)
    t0 = time.perf_counter()
    runs = [time_oracle(wl, REFERENCE_STEP_MACS) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    mean_dt = sum(r[1] for r in runs) / len(runs)
    v = statistics.mean(r[0] for r in runs)
    threads, sample = runs[0][2], runs[0][3]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": wl.name, "description": wl.description, "global_batch": wl.N,
                   "parallelism": "host cores", "wall_s": wall, "step": sample},
        "cpu_baseline": {"value": v, "unit": "GFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
