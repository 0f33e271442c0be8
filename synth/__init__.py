"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's callers.

This package holds no convolution arithmetic.  It fills buffers with
counter-based pseudo-random numbers (SplitMix64 finaliser, see ``synth.c``) and
describes the benchmark workloads: tensor shapes, value distributions and conv
hyper-parameters.  Both the CUDA path and the oracle consume exactly the same
host buffers produced here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None

TENSOR_X, TENSOR_W, TENSOR_B = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` beside it (plain gcc, no -march)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        i64, u64, f64, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_int
        vp = ctypes.c_void_p
        lib.synth_uniform_f32.argtypes = [vp, i64, u64, u64, f64, f64, i32]
        lib.synth_normal_f32.argtypes = [vp, i64, u64, u64, i32]
        lib.synth_uniform_at.argtypes = [vp, vp, i64, u64, u64, f64, f64]
        lib.synth_hash.argtypes = [u64, u64, u64]
        lib.synth_hash.restype = u64
        for f in (lib.synth_uniform_f32, lib.synth_normal_f32, lib.synth_uniform_at):
            f.restype = i32
        _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def uniform(shape, lo: float, hi: float, seed: int, tensor: int, out: np.ndarray | None = None) -> np.ndarray:
    """float32 array of ``shape`` with elements lo + (hi-lo)*U[0,1) (24-bit uniforms)."""
    shape = tuple(int(s) for s in shape)
    a = np.empty(shape, np.float32) if out is None else out
    assert a.dtype == np.float32 and a.flags.c_contiguous and a.shape == shape
    rc = _load().synth_uniform_f32(a.ctypes.data, a.size, seed, tensor, float(lo), float(hi), _threads())
    assert rc == 0
    return a


def normal(shape, seed: int, tensor: int, out: np.ndarray | None = None) -> np.ndarray:
    """float32 array of ``shape`` with N(0,1) elements (Box-Muller in double)."""
    shape = tuple(int(s) for s in shape)
    a = np.empty(shape, np.float32) if out is None else out
    assert a.dtype == np.float32 and a.flags.c_contiguous and a.shape == shape
    rc = _load().synth_normal_f32(a.ctypes.data, a.size, seed, tensor, _threads())
    assert rc == 0
    return a


def hash3(seed: int, tensor: int, i: int) -> int:
    return int(_load().synth_hash(seed, tensor, i))


@dataclass(frozen=True)
class Workload:
    """One benchmark / parity configuration: shapes, hyper-parameters, input recipe."""
    name: str
    kind: str                 # "conv" (y = conv(x, w) + b) or "fused" (conv3d -> min(depth) -> softmax(channels))
    N: int
    C_in: int
    C_out: int
    in_dims: tuple
    k_dims: tuple
    stride: tuple
    pad: tuple
    dilation: tuple
    bias: bool
    x_dist: str               # "uniform01" or "normal"
    description: str = ""
    min_dim: int = 2
    extra: dict = field(default_factory=dict)

    @property
    def ndim(self) -> int:
        return len(self.in_dims)

    @property
    def fan_in(self) -> int:
        return self.C_in * int(np.prod(self.k_dims))

    @property
    def kaiming_bound(self) -> float:
        # kaiming_uniform_(a=sqrt(5)): gain = sqrt(2/(1+5)); bound = gain*sqrt(3/fan_in) = 1/sqrt(fan_in)
        return 1.0 / np.sqrt(self.fan_in)

    def x_shape(self):
        return (self.N, self.C_in) + tuple(self.in_dims)

    def w_shape(self):
        return (self.C_out, self.C_in) + tuple(self.k_dims)

    def make_inputs(self, seed: int = 0):
        """Host float32 (x, w, b_or_None) for this workload; b is None when bias is off."""
        if self.x_dist == "uniform01":
            x = uniform(self.x_shape(), 0.0, 1.0, seed, TENSOR_X)
        elif self.x_dist == "normal":
            x = normal(self.x_shape(), seed, TENSOR_X)
        else:
            raise ValueError(self.x_dist)
        bd = self.kaiming_bound
        w = uniform(self.w_shape(), -bd, bd, seed, TENSOR_W)
        b = uniform((self.C_out,), -bd, bd, seed, TENSOR_B) if self.bias else None
        return x, w, b

    def with_batch(self, N: int) -> "Workload":
        d = dict(self.__dict__)
        d["N"] = N
        d["name"] = f"{self.name}[N={N}]"
        return Workload(**d)


WORKLOADS = {
    "conv1d_tiny": Workload(
        "conv1d_tiny", "conv", 2, 4, 8, (1024,), (3,), (3,), (0,), (4,), False, "uniform01",
        "Conv1d tiny: x[2,4,1024] U[0,1), C_out=8, k=3, stride 3, dilation 4, no bias"),
    "conv3d_asym": Workload(
        "conv3d_asym", "conv", 16, 3, 64, (64, 64, 64), (3, 5, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1), True,
        "uniform01", "Conv3d asymmetric: x[16,3,64,64,64] U[0,1), C_out=64, kernel (3,5,7), bias"),
    "conv3d_min_softmax": Workload(
        "conv3d_min_softmax", "fused", 128, 3, 24, (24, 32, 32), (3, 3, 3), (1, 1, 1), (0, 0, 0), (1, 1, 1), True,
        "uniform01", "Fused Conv3d+min(depth)+softmax(channels): x[128,3,24,32,32] U[0,1), C_out=24, k=3^3"),
    "conv1d_long": Workload(
        "conv1d_long", "conv", 64, 64, 128, (524280,), (3,), (3,), (0,), (4,), False, "uniform01",
        "Conv1d long: x[64,64,524280] U[0,1), C_out=128, k=3, stride 3, dilation 4, no bias"),
    "conv3d_sweep_a": Workload(
        "conv3d_sweep_a", "conv", 8, 8, 32, (48, 48, 48), (3, 5, 7), (1, 2, 2), (1, 2, 3), (2, 1, 1), True,
        "normal", "Conv3d sweep: x[8,8,48^3] N(0,1), C_out=32, k (3,5,7), s (1,2,2), p (1,2,3), d (2,1,1)"),
    "conv3d_sweep_b": Workload(
        "conv3d_sweep_b", "conv", 8, 32, 32, (48, 48, 48), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), True,
        "normal", "Conv3d sweep, large K: x[8,32,48^3] N(0,1), C_out=32, k 3^3, s 1, p 1"),
    "conv3d_sweep_b_dil": Workload(
        "conv3d_sweep_b_dil", "conv", 8, 32, 32, (48, 48, 48), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 1, 1), True,
        "normal", "Conv3d sweep, large K, alternative reading with dilation (2,1,1)"),
    # not one of the pages' shapes: a layer whose weights (K = 1728 x 128) exceed
    # shared memory, for the streamed-weights entry point
    "conv3d_wide_k": Workload(
        "conv3d_wide_k", "conv", 4, 64, 128, (32, 32, 32), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), True,
        "normal", "Conv3d 64 -> 128 channels, k=3^3, pad 1: x[4,64,32,32,32] N(0,1) (weights exceed shared memory)"),
}
