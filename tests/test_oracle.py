"""Pins for the oracle against what the pages and the mathematics fix.

Each test pins the oracle to something other than itself: the pages' worked
shape values (tests/golden/page_shapes.json), brute-force counting on tiny
inputs, closed forms (delta kernel, identity kernel, all-ones counts),
linearity, library routines in float64 (torch.nn.functional.conv*d, scipy's
softmax) and the read-once structure of the Conv1d long geometry.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import softmax as scipy_softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_shapes.json")
TORCH_CONV = {1: F.conv1d, 2: F.conv2d, 3: F.conv3d}


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- shapes

def test_page_worked_shapes():
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        got = oracle.out_dims(c["in"], c["k"], c["stride"], c["pad"], c["dilation"])
        assert list(got) == c["out"], c["cite"]


def test_out_dims_closed_forms_for_all_workloads():
    # conv1d tiny: (1024 - 8 - 1)//3 + 1 = 339; sweep a: D (48+2-4-1)+1, H,W (48+4-4-1)//2+1, (48+6-6-1)//2+1
    assert oracle.out_dims((1024,), (3,), (3,), (0,), (4,)) == (339,)
    assert oracle.out_dims((48, 48, 48), (3, 5, 7), (1, 2, 2), (1, 2, 3), (2, 1, 1)) == (46, 24, 24)
    assert oracle.out_dims((48, 48, 48), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1)) == (48, 48, 48)
    assert oracle.out_dims((48, 48, 48), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 1, 1)) == (46, 48, 48)


def test_out_dims_brute_force_count():
    # The output size is the number of start positions j >= 0 whose whole
    # dilated window stays inside the padded input: j*s + (k-1)*d <= L + 2p - 1.
    for L, k, s, p, d in itertools.product(range(1, 14), range(1, 5), range(1, 4), range(0, 3), range(1, 4)):
        brute = 0
        while brute * s + (k - 1) * d <= L + 2 * p - 1:
            brute += 1
        (got,) = oracle.out_dims((L,), (k,), (s,), (p,), (d,))
        if brute == 0:
            assert got <= 0, (L, k, s, p, d, got)
        else:
            assert got == brute, (L, k, s, p, d, got, brute)


# ------------------------------------------------- library cross-checks

@pytest.mark.parametrize("seed", range(12))
def test_matches_torch_float64(seed):
    rng = _rng(seed)
    nd = [1, 2, 3][seed % 3]
    N, C_in, C_out = int(rng.integers(1, 3)), int(rng.integers(1, 5)), int(rng.integers(1, 6))
    k = tuple(int(v) for v in rng.integers(1, 4, nd))
    s = tuple(int(v) for v in rng.integers(1, 4, nd))
    p = tuple(int(v) for v in rng.integers(0, 3, nd))
    d = tuple(int(v) for v in rng.integers(1, 3, nd))
    ins = tuple(int(v) for v in rng.integers(max(k) * max(d) + 1, 12, nd))
    x = rng.standard_normal((N, C_in) + ins).astype(np.float32)
    w = rng.standard_normal((C_out, C_in) + k).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32) if seed % 2 else None
    y = oracle.conv_nd(x, w, b, s, p, d, nthreads=2)
    ref = TORCH_CONV[nd](torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                         None if b is None else torch.from_numpy(b).double(),
                         stride=s, padding=p, dilation=d).numpy()
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- closed forms

@pytest.mark.parametrize("nd", [1, 2, 3])
def test_delta_kernel_selects_one_input(nd):
    rng = _rng(100 + nd)
    N, C_in, C_out = 2, 3, 4
    k = (3, 2, 4)[:nd]
    s = (2, 1, 3)[:nd]
    p = (1, 2, 0)[:nd]
    d = (2, 3, 1)[:nd]
    ins = (11, 9, 10)[:nd]
    x = rng.standard_normal((N, C_in) + ins).astype(np.float32)
    c0, o0 = 1, 2
    kp0 = (2, 1, 3)[:nd]
    w = np.zeros((C_out, C_in) + k, np.float32)
    w[(o0, c0) + kp0] = 1.0
    y = oracle.conv_nd(x, w, None, s, p, d, nthreads=2)
    od = y.shape[2:]
    expect = np.zeros_like(y)
    for n in range(N):
        for op in itertools.product(*[range(v) for v in od]):
            q = tuple(op[i] * s[i] + kp0[i] * d[i] - p[i] for i in range(nd))
            if all(0 <= q[i] < ins[i] for i in range(nd)):
                expect[(n, o0) + op] = x[(n, c0) + q]
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_identity_kernel_is_strided_copy(nd):
    rng = _rng(200 + nd)
    C = 3
    s = (3, 2, 1)[:nd]
    ins = (10, 7, 5)[:nd]
    x = rng.standard_normal((2, C) + ins).astype(np.float32)
    w = np.zeros((C, C) + (1,) * nd, np.float32)
    for c in range(C):
        w[(c, c) + (0,) * nd] = 1.0
    y = oracle.conv_nd(x, w, None, s, (0,) * nd, (1,) * nd, nthreads=2)
    sl = (slice(None), slice(None)) + tuple(slice(None, None, v) for v in s)
    assert np.array_equal(y, x[sl].astype(np.float64))


@pytest.mark.parametrize("nd", [1, 2, 3])
def test_all_ones_counts_in_bounds_taps(nd):
    C_in = 3
    k = (3, 4, 2)[:nd]
    s = (2, 1, 3)[:nd]
    p = (2, 1, 1)[:nd]
    d = (1, 2, 3)[:nd]
    ins = (9, 8, 10)[:nd]
    x = np.ones((1, C_in) + ins, np.float32)
    w = np.ones((2, C_in) + k, np.float32)
    y = oracle.conv_nd(x, w, None, s, p, d, nthreads=2)
    od = y.shape[2:]
    # per-dim count of in-bounds taps; the total is their product times C_in
    per_dim = [np.array([sum(1 for kk in range(k[i]) if 0 <= o * s[i] + kk * d[i] - p[i] < ins[i])
                         for o in range(od[i])]) for i in range(nd)]
    cnt = per_dim[0]
    for i in range(1, nd):
        cnt = np.multiply.outer(cnt, per_dim[i])
    assert np.array_equal(y[0, 0], C_in * cnt.astype(np.float64))
    assert np.array_equal(y[0, 1], C_in * cnt.astype(np.float64))


def test_linearity_and_bias():
    rng = _rng(7)
    x1 = rng.standard_normal((2, 3, 7, 6, 9)).astype(np.float32)
    x2 = rng.standard_normal((2, 3, 7, 6, 9)).astype(np.float32)
    w = rng.standard_normal((4, 3, 2, 3, 3)).astype(np.float32)
    b = rng.standard_normal(4).astype(np.float32)
    hp = ((1, 2, 1), (1, 0, 2), (2, 1, 1))
    a, bb = 0.5, -2.0  # exact in float32: a*x1 + bb*x2 rounds once
    xs = (a * x1.astype(np.float64) + bb * x2.astype(np.float64)).astype(np.float32)
    y1 = oracle.conv_nd(x1, w, None, *hp)
    y2 = oracle.conv_nd(x2, w, None, *hp)
    ys = oracle.conv_nd(xs, w, None, *hp)
    lin = a * y1 + bb * y2
    # xs differs from a*x1+bb*x2 only by one float32 rounding per element
    err_bound = np.abs(oracle.conv_nd(np.abs(xs), np.abs(w), None, *hp)).max() * 2.0 ** -23 + 1e-12
    assert np.abs(ys - lin).max() <= err_bound
    yb = oracle.conv_nd(x1, w, b, *hp)
    np.testing.assert_allclose(yb - y1, np.broadcast_to(b.astype(np.float64)[None, :, None, None, None], y1.shape),
                               rtol=0, atol=1e-12)


def test_sampled_points_equal_full():
    rng = _rng(11)
    x = rng.standard_normal((2, 3, 9, 8, 10)).astype(np.float32)
    w = rng.standard_normal((5, 3, 3, 2, 3)).astype(np.float32)
    b = rng.standard_normal(5).astype(np.float32)
    hp = ((2, 1, 1), (1, 1, 0), (1, 2, 3))
    y = oracle.conv_nd(x, w, b, *hp)
    idx = rng.integers(0, y.size, 300)
    got = oracle.conv_nd_at(x, w, b, *hp, idx)
    assert np.array_equal(got, y.reshape(-1)[idx])


def test_rejects_non_positive_output():
    with pytest.raises(oracle.OracleError):
        oracle.conv_nd(np.zeros((1, 1, 4), np.float32), np.zeros((1, 1, 3), np.float32), None, (1,), (0,), (3,))


# -------------------------------------------------- read-once structure

def test_read_once_conv1d_long_geometry():
    ro = json.load(open(GOLDEN))["read_once"]
    counts = oracle.input_read_counts(ro["in"], ro["k"], ro["stride"], ro["pad"], ro["dilation"])
    assert counts.max() == 1
    unread = np.flatnonzero(counts == 0).tolist()
    assert unread == ro["unread"], ro["cite"]


def test_read_counts_brute_force_small():
    # 2-D case with padding: count by enumerating every (output, tap) pair here.
    ins, k, s, p, d = (6, 7), (3, 2), (2, 1), (1, 2), (1, 3)
    counts = oracle.input_read_counts(ins, k, s, p, d)
    od = oracle.out_dims(ins, k, s, p, d)
    ref = np.zeros(ins, np.int64)
    for o0, o1, k0, k1 in itertools.product(range(od[0]), range(od[1]), range(k[0]), range(k[1])):
        q0, q1 = o0 * s[0] + k0 * d[0] - p[0], o1 * s[1] + k1 * d[1] - p[1]
        if 0 <= q0 < ins[0] and 0 <= q1 < ins[1]:
            ref[q0, q1] += 1
    assert np.array_equal(counts, ref)


# ---------------------------------------------------------------- fused

def _fused_inputs(seed, N=2, C_in=3, C_out=5, ins=(6, 7, 8), k=(3, 2, 3)):
    rng = _rng(seed)
    x = rng.random((N, C_in) + ins).astype(np.float32)
    w = (rng.random((C_out, C_in) + k).astype(np.float32) - 0.5)
    b = (rng.random(C_out).astype(np.float32) - 0.5)
    return x, w, b


def test_fused_rows_sum_to_one_and_open_interval():
    x, w, b = _fused_inputs(1)
    y = oracle.conv3d_min_softmax(x, w, b)
    assert np.abs(y.sum(axis=1) - 1.0).max() < 1e-12
    assert (y > 0).all() and (y < 1).all()


def test_fused_equals_softmax_of_min_of_conv():
    x, w, b = _fused_inputs(2)
    y = oracle.conv3d_min_softmax(x, w, b)
    z = oracle.conv_nd(x, w, b, (1, 1, 1), (0, 0, 0), (1, 1, 1))
    ref = scipy_softmax(z.min(axis=2), axis=1)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)


def test_fused_matches_torch_float64():
    x, w, b = _fused_inputs(3, N=2, C_in=3, C_out=24, ins=(8, 6, 7), k=(3, 3, 3))
    y = oracle.conv3d_min_softmax(x, w, b)
    z = F.conv3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(), torch.from_numpy(b).double())
    ref = torch.softmax(torch.min(z, dim=2).values, dim=1).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)


def test_fused_bias_shift_invariance():
    x, w, b = _fused_inputs(4)
    y0 = oracle.conv3d_min_softmax(x, w, b)
    y1 = oracle.conv3d_min_softmax(x, w, b + np.float32(0.25))
    np.testing.assert_allclose(y0, y1, rtol=0, atol=1e-7)


def test_fused_single_depth_is_softmax_of_conv():
    x, w, b = _fused_inputs(5, ins=(3, 6, 6), k=(3, 3, 3))  # output depth 1
    y = oracle.conv3d_min_softmax(x, w, b)
    z = F.conv3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(), torch.from_numpy(b).double())
    ref = torch.softmax(z[:, :, 0], dim=1).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)


def test_fused_argmax_is_argmax_of_min():
    x, w, b = _fused_inputs(6)
    y = oracle.conv3d_min_softmax(x, w, b)
    z = oracle.conv_nd(x, w, b, (1, 1, 1), (0, 0, 0), (1, 1, 1))
    assert np.array_equal(y.argmax(axis=1), z.min(axis=2).argmax(axis=1))


def test_fused_sampled_columns_equal_full():
    x, w, b = _fused_inputs(8)
    y = oracle.conv3d_min_softmax(x, w, b)
    N, C_out, OH, OW = y.shape
    cols = np.array([0, 5, OH * OW - 1, OH * OW, N * OH * OW - 1], np.int64)
    got = oracle.conv3d_min_softmax_at(x, w, b, cols)
    ref = y.transpose(0, 2, 3, 1).reshape(-1, C_out)[cols]
    assert np.array_equal(got, ref)


# ------------------------------------------- fused, min over height or width

@pytest.mark.parametrize("min_dim", [2, 3, 4])
def test_fused_min_dim_matches_torch_float64(min_dim):
    # torch.min(z, dim=min_dim) then softmax over dim 1, on the same 5-D conv
    x, w, b = _fused_inputs(11 + min_dim, N=2, C_in=3, C_out=7, ins=(7, 6, 9), k=(3, 2, 4))
    y = oracle.conv3d_min_softmax(x, w, b, min_dim)
    z = F.conv3d(torch.from_numpy(x).double(), torch.from_numpy(w).double(), torch.from_numpy(b).double())
    ref = torch.softmax(torch.min(z, dim=min_dim).values, dim=1).numpy()
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("min_dim", [3, 4])
def test_fused_min_dim_is_depth_min_of_permuted_problem(min_dim):
    # min over H (W) of conv(x, w) = min over depth of conv(x', w') with the
    # depth axis and the H (W) axis of both x and w exchanged; the kept axes
    # come out in the permuted order
    x, w, b = _fused_inputs(21 + min_dim, N=2, C_in=2, C_out=6, ins=(6, 8, 7), k=(2, 3, 4))
    y = oracle.conv3d_min_softmax(x, w, b, min_dim)
    xp = np.ascontiguousarray(np.swapaxes(x, 2, min_dim))
    wp = np.ascontiguousarray(np.swapaxes(w, 2, min_dim))
    yp = oracle.conv3d_min_softmax(xp, wp, b, 2)
    if min_dim == 4:
        yp = np.swapaxes(yp, 2, 3)  # (H, D) -> (D, H)
    np.testing.assert_allclose(y, yp, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("min_dim", [3, 4])
def test_fused_min_dim_rows_and_sampled_columns(min_dim):
    x, w, b = _fused_inputs(31 + min_dim)
    y = oracle.conv3d_min_softmax(x, w, b, min_dim)
    assert np.abs(y.sum(axis=1) - 1.0).max() < 1e-12
    N, C_out, OA, OB = y.shape
    cols = np.array([0, 3, OA * OB - 1, OA * OB, N * OA * OB - 1], np.int64)
    got = oracle.conv3d_min_softmax_at(x, w, b, cols, min_dim)
    assert np.array_equal(got, y.transpose(0, 2, 3, 1).reshape(-1, C_out)[cols])


def test_fused_rejects_bad_min_dim():
    x, w, b = _fused_inputs(41)
    for bad in (0, 1, 5):
        with pytest.raises(oracle.OracleError):
            oracle.conv3d_min_softmax(x, w, b, bad)


# ---------------------------------------------------------------- groups

@pytest.mark.parametrize("nd,groups,C_in,C_out", [(1, 2, 4, 6), (2, 3, 6, 3), (3, 2, 4, 4), (2, 5, 5, 10),
                                                  (3, 4, 4, 8)])
def test_grouped_matches_torch_float64(nd, groups, C_in, C_out):
    rng = _rng(100 + nd * 10 + groups)
    ins = tuple(int(v) for v in rng.integers(5, 9, nd))
    k = tuple(int(v) for v in rng.integers(1, 4, nd))
    s = tuple(int(v) for v in rng.integers(1, 3, nd))
    p = tuple(int(v) for v in rng.integers(0, 2, nd))
    d = tuple(int(v) for v in rng.integers(1, 3, nd))
    x = rng.standard_normal((2, C_in) + ins).astype(np.float32)
    w = rng.standard_normal((C_out, C_in // groups) + k).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    y = oracle.conv_nd(x, w, b, s, p, d, groups=groups)
    ref = TORCH_CONV[nd](torch.from_numpy(x).double(), torch.from_numpy(w).double(), torch.from_numpy(b).double(),
                         stride=s, padding=p, dilation=d, groups=groups).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_grouped_is_concatenation_of_per_group_convs():
    rng = _rng(120)
    groups, C_in, C_out = 3, 6, 9
    x = rng.standard_normal((2, C_in, 7, 6)).astype(np.float32)
    w = rng.standard_normal((C_out, C_in // groups, 3, 2)).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    y = oracle.conv_nd(x, w, b, (1, 2), (1, 0), (2, 1), groups=groups)
    cg, kg = C_in // groups, C_out // groups
    for g in range(groups):
        part = oracle.conv_nd(x[:, g * cg:(g + 1) * cg], w[g * kg:(g + 1) * kg], b[g * kg:(g + 1) * kg],
                              (1, 2), (1, 0), (2, 1))
        assert np.array_equal(y[:, g * kg:(g + 1) * kg], part)


def test_depthwise_delta_kernel_shifts_each_channel():
    # groups = C_in = C_out, w = 1 at one tap: y[n, c, p] = x[n, c, p*s + k0*d - pad] (0 in the padding)
    rng = _rng(121)
    C, L, k, s, p, d, k0 = 5, 23, 4, 2, 3, 2, 2
    x = rng.standard_normal((3, C, L)).astype(np.float32)
    w = np.zeros((C, 1, k), np.float32)
    w[:, 0, k0] = 1.0
    y = oracle.conv_nd(x, w, None, (s,), (p,), (d,), groups=C)
    (OL,) = oracle.out_dims((L,), (k,), (s,), (p,), (d,))
    ref = np.zeros((3, C, OL))
    for j in range(OL):
        q = j * s + k0 * d - p
        if 0 <= q < L:
            ref[:, :, j] = x[:, :, q]
    assert np.array_equal(y, ref)


def test_grouped_sampled_equals_full_and_rejects_bad_groups():
    rng = _rng(122)
    x = rng.standard_normal((2, 4, 9)).astype(np.float32)
    w = rng.standard_normal((6, 2, 3)).astype(np.float32)
    y = oracle.conv_nd(x, w, None, (2,), (1,), (1,), groups=2)
    idx = np.array([0, 7, y.size // 2, y.size - 1], np.int64)
    assert np.array_equal(oracle.conv_nd_at(x, w, None, (2,), (1,), (1,), idx, groups=2), y.reshape(-1)[idx])
    with pytest.raises(oracle.OracleError):
        oracle.conv_nd(x, w, None, (2,), (1,), (1,), groups=3)


# ---------------------------------------- second formulation: dense im2col

def im2col_conv(x, w, b, stride, pad, dilation, groups=1):
    """The same convolution as an explicit matrix product, written independently of the oracle:
    one column per (batch, output position) holding its zero-padded receptive field (c, k...),
    multiplied by the weights as a [C_out/groups, C_in/groups * prod(k)] matrix per group."""
    x = x.astype(np.float64)
    w = w.astype(np.float64)
    N, C_in = x.shape[:2]
    C_out, Cg = w.shape[:2]
    nd = x.ndim - 2
    ks, ins = w.shape[2:], x.shape[2:]
    outs = [(ins[i] + 2 * pad[i] - dilation[i] * (ks[i] - 1) - 1) // stride[i] + 1 for i in range(nd)]
    xp = np.pad(x, [(0, 0), (0, 0)] + [(pad[i], pad[i]) for i in range(nd)])
    taps = list(itertools.product(*[range(k) for k in ks]))
    positions = list(itertools.product(*[range(o) for o in outs]))
    y = np.zeros((N, C_out, len(positions)))
    Kg = C_out // groups
    for g in range(groups):
        cols = np.zeros((Cg * len(taps), N * len(positions)))
        for n in range(N):
            for j, pos in enumerate(positions):
                r = 0
                for c in range(Cg):
                    for t in taps:
                        idx = tuple(pos[i] * stride[i] + t[i] * dilation[i] for i in range(nd))
                        cols[r, n * len(positions) + j] = xp[(n, g * Cg + c) + idx]
                        r += 1
        wm = w[g * Kg:(g + 1) * Kg].reshape(Kg, -1)
        y[:, g * Kg:(g + 1) * Kg, :] = (wm @ cols).reshape(Kg, N, len(positions)).transpose(1, 0, 2)
    if b is not None:
        y += b.astype(np.float64)[None, :, None]
    return y.reshape((N, C_out) + tuple(outs))


@pytest.mark.parametrize("seed", range(9))
def test_matches_dense_im2col_formulation(seed):
    rng = np.random.default_rng(700 + seed)
    nd = 1 + seed % 3
    groups = 1 + seed % 2
    Cg, Kg = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    k = tuple(int(v) for v in rng.integers(1, 4, nd))
    s = tuple(int(v) for v in rng.integers(1, 3, nd))
    p = tuple(int(v) for v in rng.integers(0, 3, nd))
    d = tuple(int(v) for v in rng.integers(1, 3, nd))
    ins = tuple(int(rng.integers((k[i] - 1) * d[i] + 1, (k[i] - 1) * d[i] + 7)) for i in range(nd))
    x = rng.standard_normal((2, Cg * groups) + ins).astype(np.float32)
    w = rng.standard_normal((Kg * groups, Cg) + k).astype(np.float32)
    b = rng.standard_normal(Kg * groups).astype(np.float32)
    ref = im2col_conv(x, w, b, s, p, d, groups)
    got = oracle.conv_nd(x, w, b, s, p, d, groups=groups)
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_per_dim_hyper_parameters_broadcast_or_must_match_the_rank():
    # an int applies to every dim; a sequence of the wrong length is refused
    # (the C routines read exactly one value per dim)
    x = np.arange(2 * 3 * 5 * 6 * 7, dtype=np.float32).reshape(2, 3, 5, 6, 7) / 100
    w = np.ones((4, 3, 2, 2, 2), np.float32)
    a = oracle.conv_nd(x, w, None, 1, 0, 1)
    b = oracle.conv_nd(x, w, None, (1, 1, 1), (0, 0, 0), (1, 1, 1))
    assert np.array_equal(a, b)
    assert oracle.out_dims((5, 6, 7), 2, 1, 0, 1) == (4, 5, 6)
    with pytest.raises(oracle.OracleError):
        oracle.conv_nd(x, w, None, (1, 1), 0, 1)
    with pytest.raises(oracle.OracleError):
        oracle.out_dims((5, 6, 7), (2, 2), 1, 0, 1)
