"""ORACLE -- test infrastructure, not part of the product.

Plain fp64 CPU reference for the forward N-D convolution and the fused
Conv3d -> min(depth) -> softmax(channels), written in C (``oracle.c``) from the
POPCORNBENCH pages' definitions.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference legs may import this package.  It
shares no code with the CUDA library and never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc -O2 into ``liboracle.so`` (no -march, no fast-math)."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        # ORACLE_SO lets the mutation test load a deliberately broken copy in a
        # child process; normal use always builds and loads liboracle.so.
        so = os.environ.get("ORACLE_SO") or build()
        lib = ctypes.CDLL(so)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_out_dims.argtypes = [i32, vp, vp, vp, vp, vp, vp]
        lib.oracle_conv_nd.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, vp, vp, i32]
        lib.oracle_conv_nd_at.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, vp, vp, vp, vp, vp, i64, vp, i32]
        lib.oracle_conv_nd_grouped.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, vp, vp, vp, vp, vp, i32]
        lib.oracle_conv_nd_grouped_at.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, i64,
                                                  vp, i32]
        lib.oracle_input_read_counts.argtypes = [i32, vp, vp, vp, vp, vp, vp]
        lib.oracle_conv3d_min_softmax.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, i32, i32]
        lib.oracle_conv3d_min_softmax_at.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, i32, vp, i64, vp, i32]
        for f in (lib.oracle_out_dims, lib.oracle_conv_nd, lib.oracle_conv_nd_at, lib.oracle_input_read_counts,
                  lib.oracle_conv_nd_grouped, lib.oracle_conv_nd_grouped_at,
                  lib.oracle_conv3d_min_softmax, lib.oracle_conv3d_min_softmax_at):
            f.restype = i32
        _lib = lib
    return _lib


def threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _i64(seq):
    return np.ascontiguousarray(np.asarray(seq, dtype=np.int64))


def _per_dim(v, nd):
    """A hyper-parameter as nd int64 values: an int applies to every dim; a sequence must have nd entries
    (the C routines read exactly nd)."""
    a = np.atleast_1d(np.asarray(v, dtype=np.int64))
    if a.ndim != 1:
        raise OracleError("hyper-parameters must be an int or a flat sequence")
    if a.size == 1 and nd > 1:
        a = np.repeat(a, nd)
    if a.size != nd:
        raise OracleError(f"expected {nd} values per hyper-parameter, got {a.size}")
    return np.ascontiguousarray(a)


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


class OracleError(ValueError):
    pass


def out_dims(in_dims, k, stride, pad, dilation):
    """Output size per dim: floor((L + 2p - d(k-1) - 1)/s) + 1 (may be <= 0)."""
    nd = len(in_dims)
    arrs = [_per_dim(v, nd) for v in (in_dims, k, stride, pad, dilation)]
    out = np.zeros(nd, np.int64)
    if _load().oracle_out_dims(nd, *[_ptr(a) for a in arrs], _ptr(out)):
        raise OracleError("bad conv hyper-parameters")
    return tuple(int(v) for v in out)


def conv_nd(x, w, bias, stride, pad, dilation, nthreads=None, groups=1):
    """y = conv(x, w) + bias as float64, x [N,C_in,*in], w [C_out,C_in/groups,*k]."""
    x, w = _f32(x), _f32(w)
    b = None if bias is None else _f32(bias)
    nd = x.ndim - 2
    N, C_in = x.shape[:2]
    C_out = w.shape[0]
    if groups < 1 or C_in % groups or C_out % groups or w.shape[1] * groups != C_in or w.ndim != x.ndim:
        raise OracleError("weight shape mismatch")
    ins, ks = _i64(x.shape[2:]), _i64(w.shape[2:])
    s, p, d = _per_dim(stride, nd), _per_dim(pad, nd), _per_dim(dilation, nd)
    od = out_dims(x.shape[2:], w.shape[2:], stride, pad, dilation)
    if min(od) <= 0:
        raise OracleError("non-positive output size")
    y = np.empty((N, C_out) + od, np.float64)
    rc = _load().oracle_conv_nd_grouped(_ptr(x), _ptr(w), _ptr(b), _ptr(y), nd, N, C_in, C_out, groups, _ptr(ins),
                                        _ptr(ks), _ptr(s), _ptr(p), _ptr(d), nthreads or threads())
    if rc:
        raise OracleError("oracle_conv_nd_grouped rejected its arguments")
    return y


def conv_nd_at(x, w, bias, stride, pad, dilation, flat_idx, nthreads=None, groups=1):
    """y.flat[flat_idx] (float64) for the conv above, each output computed on its own."""
    x, w = _f32(x), _f32(w)
    b = None if bias is None else _f32(bias)
    nd = x.ndim - 2
    N, C_in = x.shape[:2]
    C_out = w.shape[0]
    ins, ks = _i64(x.shape[2:]), _i64(w.shape[2:])
    s, p, d = _per_dim(stride, nd), _per_dim(pad, nd), _per_dim(dilation, nd)
    idx = _i64(flat_idx)
    out = np.empty(idx.shape, np.float64)
    rc = _load().oracle_conv_nd_grouped_at(_ptr(x), _ptr(w), _ptr(b), nd, N, C_in, C_out, groups, _ptr(ins),
                                           _ptr(ks), _ptr(s), _ptr(p), _ptr(d), _ptr(idx), idx.size, _ptr(out),
                                           nthreads or threads())
    if rc:
        raise OracleError("oracle_conv_nd_grouped_at rejected its arguments")
    return out


def input_read_counts(in_dims, k, stride, pad, dilation):
    """int64 array over the input positions of one channel: how many (output, tap) pairs read each."""
    nd = len(in_dims)
    counts = np.zeros(tuple(int(v) for v in in_dims), np.int64)
    arrs = [_per_dim(v, nd) for v in (in_dims, k, stride, pad, dilation)]
    if _load().oracle_input_read_counts(nd, *[_ptr(a) for a in arrs], _ptr(counts)):
        raise OracleError("bad conv hyper-parameters")
    return counts


def _kept_axes(min_dim):
    """The two spatial output axes (0 = D, 1 = H, 2 = W) left after the min over tensor dim min_dim."""
    if min_dim not in (2, 3, 4):
        raise OracleError("min_dim must be 2, 3 or 4")
    return [a for a in range(3) if a != min_dim - 2]


def conv3d_min_softmax(x, w, bias, min_dim=2, nthreads=None):
    """float64 softmax_o(min over tensor dim min_dim of conv3d(x, w) + b), stride 1, pad 0, dilation 1.
    Shape [N, C_out, OH, OW] (min_dim 2), [N, C_out, OD, OW] (3) or [N, C_out, OD, OH] (4)."""
    x, w = _f32(x), _f32(w)
    b = None if bias is None else _f32(bias)
    N, C_in = x.shape[:2]
    C_out = w.shape[0]
    ins, ks = _i64(x.shape[2:]), _i64(w.shape[2:])
    od = out_dims(x.shape[2:], w.shape[2:], (1, 1, 1), (0, 0, 0), (1, 1, 1))
    if min(od) <= 0:
        raise OracleError("non-positive output size")
    ka, kb = _kept_axes(min_dim)
    y = np.empty((N, C_out, od[ka], od[kb]), np.float64)
    rc = _load().oracle_conv3d_min_softmax(_ptr(x), _ptr(w), _ptr(b), _ptr(y), N, C_in, C_out, _ptr(ins),
                                           _ptr(ks), min_dim, nthreads or threads())
    if rc:
        raise OracleError("oracle_conv3d_min_softmax rejected its arguments")
    return y


def conv3d_min_softmax_at(x, w, bias, cols, min_dim=2, nthreads=None):
    """float64 [len(cols), C_out]; cols are flat (n, a, b) indices of the [N, OA, OB] output grid
    (a, b: the two spatial axes kept after the min over tensor dim min_dim)."""
    x, w = _f32(x), _f32(w)
    b = None if bias is None else _f32(bias)
    N, C_in = x.shape[:2]
    C_out = w.shape[0]
    ins, ks = _i64(x.shape[2:]), _i64(w.shape[2:])
    _kept_axes(min_dim)
    cols = _i64(cols)
    out = np.empty((cols.size, C_out), np.float64)
    rc = _load().oracle_conv3d_min_softmax_at(_ptr(x), _ptr(w), _ptr(b), N, C_in, C_out, _ptr(ins), _ptr(ks),
                                              min_dim, _ptr(cols), cols.size, _ptr(out), nthreads or threads())
    if rc:
        raise OracleError("oracle_conv3d_min_softmax_at rejected its arguments")
    return out
