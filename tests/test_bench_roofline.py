"""The benchmark's roofline arithmetic, on the host: algorithmic FLOPs and bytes
of the workloads, the choice of bound, the fractions, and the ncu traffic
entry (scaled from the captured batch to the full one, dropped once the
kernel source no longer matches the capture).  Nothing here runs on a GPU."""
import os
import sys
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

PIPES = {"tf32": {"tflops": 1200.0, "scaled_to_mhz": 2070.0}, "bf16": {"tflops": 2400.0},
         "ffma": {"tflops": 80.0}, "tf32x3": {"tflops": 400.0}, "source": "microbenchmark"}
PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def _runner(name, algo, out_dims, dtype=torch.float32):
    wl = synth.WORKLOADS[name]
    return types.SimpleNamespace(wl=wl, algo=algo, out_dims=out_dims, y=torch.empty(1, dtype=dtype))


def test_headline_counts_match_the_worked_figures():
    # Conv3d x[16,3,64,64,64], kernel (3,5,7), C_out 64: output 62 x 60 x 58
    wl = synth.WORKLOADS["conv3d_asym"]
    flops, bytes_alg, in_b, out_b = bench.problem_counts(wl, (62, 60, 58))
    assert flops == 2.0 * 16 * 64 * 62 * 60 * 58 * 3 * 105
    assert out_b == 4.0 * 16 * 64 * 62 * 60 * 58
    assert in_b == 4.0 * (16 * 3 * 64 ** 3 + 64 * 3 * 105 + 64)
    assert bytes_alg == pytest.approx(934.17e6, rel=1e-4)


def test_tensor_bound_entry(monkeypatch):
    monkeypatch.setattr(bench, "traffic_for", lambda algo, wl: None)
    r = _runner("conv3d_asym", "igemm_3xtf32", (62, 60, 58))
    flops, bytes_alg, _, _ = bench.problem_counts(r.wl, r.out_dims)
    e = bench.roofline_for(r, PEAKS, PIPES, 0.5)
    assert e["bound"] == "tensor" and e["unit"] == "TFLOP/s" and e["peak"] == 400.0
    assert e["achieved"] == pytest.approx(flops / 0.5e-3 / 1e12)
    assert e["frac"] == pytest.approx(e["achieved"] / 400.0)
    # the best fp32-accurate pipe is the 3xTF32 one here, so both fractions agree
    assert e["frac_best_path"] == pytest.approx(e["frac"])
    assert e["hbm_frac"] == pytest.approx(bytes_alg / 0.5e-3 / 1e9 / 6800.0)


def test_hbm_bound_entry(monkeypatch):
    monkeypatch.setattr(bench, "traffic_for", lambda algo, wl: None)
    # long Conv1d: 2 FLOPs per MAC over 3 taps and 64 channels, 14.3 GB moved
    r = _runner("conv1d_long", "igemm_3xtf32", (174758,))
    _, bytes_alg, _, _ = bench.problem_counts(r.wl, r.out_dims)
    e = bench.roofline_for(r, PEAKS, PIPES, 2.3)
    assert e["bound"] == "hbm" and e["unit"] == "GB/s" and e["peak"] == 6800.0
    assert e["achieved"] == pytest.approx(bytes_alg / 2.3e-3 / 1e9)
    assert 0.0 < e["compute_frac"] < e["frac"]


def test_ffma_kernel_reports_the_best_path_too(monkeypatch):
    monkeypatch.setattr(bench, "traffic_for", lambda algo, wl: None)
    r = _runner("conv3d_min_softmax", "fused_ffma", (22, 30, 30))
    e = bench.roofline_for(r, PEAKS, PIPES, 0.2)
    assert e["bound"] == "alu" and e["peak"] == 80.0
    # against the faster 3xTF32 pipe the same time is a 5x smaller fraction
    assert e["frac_best_path"] == pytest.approx(e["frac"] * 80.0 / 400.0)


def test_traffic_scales_with_batch_and_drops_when_the_source_changed(monkeypatch):
    wl = synth.WORKLOADS["conv1d_long"]
    key = ("igemm_3xtf32", "conv1d_long")
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, {"bytes": 1.0e9, "batch": 4, "sha256": "abc"})
    monkeypatch.setattr(bench, "source_sha", lambda algo: "abc")
    assert bench.traffic_for("igemm_3xtf32", wl) == pytest.approx(1.0e9 * wl.N / 4)
    monkeypatch.setattr(bench, "source_sha", lambda algo: "changed")
    assert bench.traffic_for("igemm_3xtf32", wl) is None
    assert bench.traffic_for("no_such_kernel", wl) is None


def test_every_traffic_entry_names_a_known_kernel_source():
    for (algo, name), e in bench.NCU_TRAFFIC.items():
        assert algo in bench.KERNEL_SOURCE and name in synth.WORKLOADS
        assert e["batch"] >= 1 and e["bytes"] > 0 and len(e["sha256"]) == 64
        assert os.path.exists(os.path.join(ROOT, "implicit_gemm_convolution_fwd_gb300", "csrc",
                                           bench.KERNEL_SOURCE[algo]))
