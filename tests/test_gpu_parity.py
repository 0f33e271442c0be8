"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle.

Tolerance (from the pages' harness, atol = rtol = 1e-4, restated elementwise):
    |y_gpu - y_oracle| <= 1e-4 * (1 + |y_oracle|)
Shapes must match exactly.  Small cases are compared element by element over
the whole output; the benchmark workloads at full size are compared on
sampled outputs (including the first and last elements and tile edges), which
the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import implicit_gemm_convolution_fwd_gb300 as cf
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4
ALGOS = (cf.CONV_ALGO_DIRECT_FFMA, cf.CONV_ALGO_IGEMM_3XTF32)


@pytest.fixture(scope="module", autouse=True)
def built():
    from implicit_gemm_convolution_fwd_gb300 import build_lib
    build_lib.build()
    cf.load()
    yield
    assert cf.device_status() == 0, "a kernel gave up on a bounded wait"


def assert_close(y, ref, what=""):
    y = np.asarray(y, np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    err = np.abs(y - ref)
    bound = TOL * (1.0 + np.abs(ref))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"gpu {y[i]!r} oracle {ref[i]!r}")


def run_conv(x, w, b, s, p, d, algo=cf.CONV_ALGO_AUTO):
    xt = torch.from_numpy(x).cuda()
    wt = torch.from_numpy(w).cuda()
    bt = None if b is None else torch.from_numpy(b).cuda()
    y = cf.conv_fwd_nd(xt, wt, bt, s, p, d, algo=algo)
    torch.cuda.synchronize()
    return y


def random_case(seed, nd):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 3))
    C_in = int(rng.integers(1, 24))
    C_out = int(rng.integers(1, 70))
    k = tuple(int(v) for v in rng.integers(1, 6, nd))
    s = tuple(int(v) for v in rng.integers(1, 4, nd))
    p = tuple(int(v) for v in rng.integers(0, 4, nd))
    d = tuple(int(v) for v in rng.integers(1, 4, nd))
    ext = [(k[i] - 1) * d[i] + 1 for i in range(nd)]
    hi = {1: 300, 2: 40, 3: 14}[nd]
    ins = tuple(int(rng.integers(max(1, ext[i] - 2 * p[i]), max(ext[i] - 2 * p[i], 1) + hi)) for i in range(nd))
    x = rng.standard_normal((N, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 2 / np.sqrt(C_in * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32) if seed % 2 else None
    return x, w, b, s, p, d


def supported(x, w, s, p, d, algo):
    return cf.algo_supported(x.shape[0], x.shape[1], w.shape[0], x.shape[2:], w.shape[2:], s, p, d, algo)


# ------------------------------------------------------------ small cases

@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("nd", [1, 2, 3])
@pytest.mark.parametrize("seed", range(6))
def test_random_small(algo, nd, seed):
    x, w, b, s, p, d = random_case(1000 * nd + seed, nd)
    if not supported(x, w, s, p, d, algo):
        pytest.skip("shape not supported by this kernel family")
    ref = oracle.conv_nd(x, w, b, s, p, d)
    y = run_conv(x, w, b, s, p, d, algo).cpu().numpy()
    assert_close(y, ref, f"nd={nd} seed={seed} algo={cf.ALGO_NAMES[algo]}")


def random_tc_case(seed):
    """A random problem for the tensor-core family with room for interior warps: C_in 1-40 (multiples of 4
    and not), C_out 16-128 (one or two issuer slots), kernels up to 5, padding 0-2, strides and dilations
    up to 2, spatial sizes up to a few thousand positions per image."""
    rng = np.random.default_rng(50_000 + seed)
    nd = int(rng.integers(1, 4))
    C_in = int(rng.choice([1, 3, 4, 5, 8, 12, 16, 24, 40]))
    C_out = int(rng.integers(16, 129))
    k = tuple(int(v) for v in rng.integers(1, 6, nd))
    s = tuple(int(v) for v in rng.integers(1, 3, nd))
    p = tuple(int(v) for v in rng.integers(0, 3, nd))
    d = tuple(int(v) for v in rng.integers(1, 3, nd))
    lo = {1: 200, 2: 14, 3: 6}[nd]
    hi = {1: 3000, 2: 60, 3: 18}[nd]
    ins = tuple(max(int(rng.integers(lo, hi)), (k[i] - 1) * d[i] + 1) for i in range(nd))
    N = int(rng.integers(1, 4))
    x = rng.standard_normal((N, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 2 / np.sqrt(C_in * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32) if seed % 3 else None
    return x, w, b, s, p, d


@pytest.mark.parametrize("seed", range(24))
def test_random_tensor_core_shapes(seed):
    x, w, b, s, p, d = random_tc_case(seed)
    if not supported(x, w, s, p, d, cf.CONV_ALGO_IGEMM_3XTF32):
        pytest.skip("shape not supported by the tensor-core family")
    ref = oracle.conv_nd(x, w, b, s, p, d)
    y = run_conv(x, w, b, s, p, d, cf.CONV_ALGO_IGEMM_3XTF32).cpu().numpy()
    assert_close(y, ref, f"tensor cores seed={seed} x={x.shape} w={w.shape} s={s} p={p} d={d}")


@pytest.mark.parametrize("algo", ALGOS)
def test_edge_geometries(algo):
    rng = np.random.default_rng(5)
    cases = [
        # (x shape, w shape, stride, pad, dilation)
        ((1, 1, 1), (1, 1, 1), (1,), (0,), (1,)),                    # single output
        ((2, 3, 5), (4, 3, 5), (1,), (0,), (1,)),                    # kernel == input
        ((1, 2, 9), (3, 2, 2), (5,), (3,), (1,)),                    # pad > kernel, stride > kernel
        ((1, 2, 17), (2, 2, 3), (7,), (0,), (3,)),                   # stride skips inputs
        ((1, 3, 4, 5, 6), (5, 3, 1, 1, 1), (1, 1, 1), (0, 0, 0), (1, 1, 1)),  # 1x1x1 kernel
        ((1, 2, 3, 3, 3), (2, 2, 3, 3, 3), (1, 1, 1), (2, 2, 2), (1, 1, 1)),  # pad 2 around 3^3
        ((2, 1, 7, 1, 9), (3, 1, 2, 1, 4), (2, 1, 1), (1, 0, 2), (2, 1, 2)),  # singleton H
        ((1, 4, 130), (67, 4, 3), (1,), (1,), (1,)),                  # C_out not a multiple of any tile
        ((1, 4, 200), (16, 4, 32), (1,), (3,), (1,)),                 # 32 taps along W (a full 32-bit tap mask), padded
        ((1, 2, 3, 40, 8), (16, 2, 1, 32, 3), (1, 1, 1), (0, 2, 1), (1, 1, 1)),  # 32 taps along H, padded
    ]
    for xs, ws, s, p, d in cases:
        x = rng.standard_normal(xs).astype(np.float32)
        w = rng.standard_normal(ws).astype(np.float32) * 0.3
        b = rng.standard_normal(ws[0]).astype(np.float32)
        if not supported(x, w, s, p, d, algo):
            continue
        ref = oracle.conv_nd(x, w, b, s, p, d)
        y = run_conv(x, w, b, s, p, d, algo).cpu().numpy()
        assert_close(y, ref, f"edge {xs} {ws} s={s} p={p} d={d}")


def test_empty_batch_is_a_no_op():
    x = torch.empty((0, 3, 10), device="cuda")
    w = torch.randn((4, 3, 3), device="cuda")
    y = cf.conv_fwd_nd(x, w, None, 1, 0, 1)
    assert tuple(y.shape) == (0, 4, 8)


def test_deterministic_and_stream_ordered():
    x, w, b, s, p, d = random_case(77, 3)
    xt, wt, bt = torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        y1 = cf.conv_fwd_nd(xt, wt, bt, s, p, d, stream=st)
        y2 = cf.conv_fwd_nd(xt, wt, bt, s, p, d, stream=st)
    st.synchronize()
    assert torch.equal(y1, y2)


# ----------------------------------------------- workloads, reduced batch

def workload_inputs(name, N=None):
    wl = synth.WORKLOADS[name]
    if N is not None:
        wl = wl.with_batch(N)
    return (wl,) + wl.make_inputs(seed=0)


@pytest.mark.parametrize("name,N", [("conv1d_tiny", None), ("conv3d_asym", 1), ("conv3d_sweep_a", 1),
                                    ("conv3d_sweep_b", 1), ("conv3d_sweep_b_dil", 1)])
def test_workload_reduced_batch_full_compare(name, N):
    wl, x, w, b = workload_inputs(name, N)
    ref = oracle.conv_nd(x, w, b, wl.stride, wl.pad, wl.dilation)
    y = run_conv(x, w, b, wl.stride, wl.pad, wl.dilation).cpu().numpy()
    assert_close(y, ref, wl.name)


def test_conv1d_long_short_length_full_compare():
    wl = synth.WORKLOADS["conv1d_long"]
    x = synth.uniform((2, 64, 3 * 2000 + 11), 0, 1, 0, synth.TENSOR_X)
    w = synth.uniform(wl.w_shape(), -wl.kaiming_bound, wl.kaiming_bound, 0, synth.TENSOR_W)
    ref = oracle.conv_nd(x, w, None, wl.stride, wl.pad, wl.dilation)
    y = run_conv(x, w, None, wl.stride, wl.pad, wl.dilation).cpu().numpy()
    assert_close(y, ref, "conv1d_long geometry, L=6011")


# ------------------------------------------------- full size, sampled

def sample_indices(shape, count, seed):
    total = int(np.prod(shape))
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, total, count).tolist())
    idx.update([0, total - 1])
    # corners and edges of every (n, o) slab for the first/last batch and channel
    sp = shape[2:]
    for n in (0, shape[0] - 1):
        for o in (0, shape[1] - 1):
            for corner in np.ndindex(*[2] * len(sp)):
                pos = [0 if c == 0 else sp[i] - 1 for i, c in enumerate(corner)]
                idx.add(int(np.ravel_multi_index((n, o) + tuple(pos), shape)))
    return np.array(sorted(idx), np.int64)


@pytest.mark.parametrize("name", ["conv3d_asym", "conv1d_long", "conv3d_sweep_a", "conv3d_sweep_b"])
def test_workload_full_size_sampled(name):
    wl, x, w, b = workload_inputs(name)
    y = run_conv(x, w, b, wl.stride, wl.pad, wl.dilation)
    idx = sample_indices(tuple(y.shape), 4000, 123)
    got = y.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy()
    del y
    ref = oracle.conv_nd_at(x, w, b, wl.stride, wl.pad, wl.dilation, idx)
    assert_close(got, ref, f"{name} full size, {idx.size} sampled outputs")


def test_indexing_beyond_int32():
    # x and y both hold more than 2^31 elements (each dim fits int32): element
    # offsets must be 64-bit.
    L = (1 << 30) + 1000
    x = synth.uniform((2, 1, L), 0, 1, 3, synth.TENSOR_X)
    w = np.array([[[0.25, -0.5, 1.0]]], np.float32)
    y = run_conv(x, w, None, (1,), (0,), (1,))
    total = y.numel()
    assert total > (1 << 31)
    idx = np.array([0, 1, L - 3, L - 2, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, total - 1], np.int64)
    got = y.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy()
    del y
    ref = oracle.conv_nd_at(x, w, None, (1,), (0,), (1,), idx)
    assert_close(got, ref, "int64 indexing")


# ------------------------------------------------------------------ fused

FFMA, TC = cf.CONV_ALGO_DIRECT_FFMA, cf.CONV_ALGO_IGEMM_3XTF32


def run_fused(x, w, b, algo=cf.CONV_ALGO_AUTO):
    xt = torch.from_numpy(x).cuda()
    wt = torch.from_numpy(w).cuda()
    bt = None if b is None else torch.from_numpy(b).cuda()
    y = cf.conv3d_min_softmax(xt, wt, bt, 2, algo=algo)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("algo", [FFMA, TC])
@pytest.mark.parametrize("C_out", [1, 5, 12, 13, 24, 25, 32, 48, 49, 96])
@pytest.mark.parametrize("k", [(3, 3, 3), (2, 3, 5)])
def test_fused_small(C_out, k, algo):
    if algo == TC and C_out > 32:
        pytest.skip("the tensor-core fused kernel takes C_out <= 32")
    rng = np.random.default_rng(C_out * 10 + k[2])
    x = rng.random((3, 3, 7, 11, 37)).astype(np.float32)  # W=37: scalar path, 2 column tiles
    w = (rng.random((C_out, 3) + k).astype(np.float32) - 0.5) * 0.4
    b = (rng.random(C_out).astype(np.float32) - 0.5) * 0.4
    ref = oracle.conv3d_min_softmax(x, w, b)
    y = run_fused(x, w, b, algo).cpu().numpy()
    assert_close(y, ref, f"fused C_out={C_out} k={k} algo={algo}")
    assert np.abs(y.sum(axis=1) - 1).max() < 1e-5


@pytest.mark.parametrize("shape,C_in,C_out,k", [
    ((2, 3, 3, 17, 13), 3, 24, (3, 3, 3)),    # one output depth: the min over a single plane
    ((1, 2, 9, 40, 45), 2, 20, (4, 5, 2)),     # 1 image, planes of 36 x 44 = 1584 positions (12.4 tiles)
    ((5, 4, 6, 12, 12), 4, 32, (2, 2, 2)),     # C_out = 32 (every accumulator column), 121-position planes
    ((3, 1, 30, 5, 7), 1, 7, (1, 1, 1)),       # 1x1x1 kernel, 30 depth tiles per column
])
def test_fused_tensor_core_geometries(shape, C_in, C_out, k):
    rng = np.random.default_rng(sum(shape) + C_out)
    x = rng.standard_normal(shape).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 0.5).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    ref = oracle.conv3d_min_softmax(x, w, b)
    assert_close(run_fused(x, w, b, TC).cpu().numpy(), ref, f"fused tensor cores {shape} k={k}")
    assert_close(run_fused(x, w, None, TC).cpu().numpy(), oracle.conv3d_min_softmax(x, w, None),
                 f"fused tensor cores no bias {shape}")


@pytest.mark.parametrize("shape,C_out,k", [
    ((2, 64, 6, 10, 12), 32, (3, 3, 3)),    # 1728 reduction columns: weights (hi + lo) exceed shared memory
    ((1, 40, 5, 9, 140), 20, (3, 3, 3)),    # 1080 columns, rows of 138 outputs (2 column tiles per row)
    ((2, 128, 4, 6, 7), 7, (2, 2, 2)),      # 1024 columns, 7 channels
])
def test_fused_tensor_core_streamed_weights(shape, C_out, k):
    rng = np.random.default_rng(shape[1] + C_out)
    x = rng.standard_normal(shape).astype(np.float32)
    w = ((rng.random((C_out, shape[1]) + k) - 0.5) * 2 / np.sqrt(shape[1] * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    ref = oracle.conv3d_min_softmax(x, w, b)
    y = run_fused(x, w, b, TC).cpu().numpy()
    assert_close(y, ref, f"fused tensor cores, streamed weights {shape} C_out={C_out}")
    # long reductions: the planner takes the tensor cores (where the FFMA kernels can hold the
    # weights at all, they must agree with the oracle too)
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    try:
        yf = cf.conv3d_min_softmax(xt, wt, bt, 2, algo=FFMA)
        assert_close(yf.cpu().numpy(), ref, f"fused FFMA {shape} C_out={C_out}")
    except cf.ConvError as e:
        assert e.status == cf.CONV_ERR_UNSUPPORTED
    assert torch.equal(cf.conv3d_min_softmax(xt, wt, bt, 2), torch.from_numpy(y).cuda())


# The tensor-core fused kernel gathers each input plane along the reduced axis
# once when its receptive-field columns (C_in x the other two kernel extents)
# number at most 32, sharing it among the KR tiles that read it: a single tile
# per column (R = 1), a kernel extent of 1 and of 5 along the reduced axis
# (16-column slabs, up to 8 in the ring), exactly 32 and 17 columns, a ragged
# last column, two channel blocks, and both reduced axes it serves.
SLAB_CASES = [
    ((2, 3, 3, 12, 17), 24, (3, 3, 3)),      # R = 1 over depth
    ((3, 2, 5, 11, 13), 16, (1, 3, 3)),      # KR = 1
    ((2, 1, 9, 10, 14), 24, (5, 3, 3)),      # KR = 5, 9 columns (16-column slabs)
    ((2, 2, 6, 9, 12), 32, (2, 4, 4)),       # 32 columns
    ((2, 17, 6, 8, 9), 8, (3, 1, 1)),        # 17 columns (padded to 32)
    ((3, 3, 7, 13, 11), 40, (3, 3, 3)),      # two channel blocks, ragged last column
]


@pytest.mark.parametrize("min_dim", [2, 3, 4])
@pytest.mark.parametrize("shape,C_out,k", SLAB_CASES)
def test_fused_tensor_core_shared_planes(shape, C_out, k, min_dim):
    rng = np.random.default_rng(shape[1] * 100 + C_out + k[0])
    x = rng.standard_normal(shape).astype(np.float32)
    w = ((rng.random((C_out, shape[1]) + k) - 0.5) * 0.4).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    y = cf.conv3d_min_softmax(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(),
                              min_dim, algo=TC)
    assert_close(y.cpu().numpy(), oracle.conv3d_min_softmax(x, w, b, min_dim),
                 f"shared planes {shape} {C_out} {k} min_dim={min_dim}")


@pytest.mark.parametrize("min_dim", [2, 3, 4])
def test_fused_planner_takes_the_tensor_cores(min_dim):
    """AUTO equals the tensor-core result bit for bit (the two families differ in rounding):
    on the page's C_in = 3, C_out = 24 shape (reduced batch, planes gathered once), on a 27-column
    reduction and on 40 channels over C_in = 8 (two channel blocks, no shared planes)."""
    wl, x, w, b = workload_inputs("conv3d_min_softmax", 2)
    rng = np.random.default_rng(11)
    cases = [(x, w, b),
             (rng.random((2, 1, 10, 20, 20)).astype(np.float32),
              ((rng.random((24, 1, 3, 3, 3)) - 0.5) * 0.2).astype(np.float32), None),
             (rng.random((2, 8, 8, 12, 14)).astype(np.float32),
              ((rng.random((40, 8, 3, 3, 3)) - 0.5) * 0.2).astype(np.float32), None)]
    for xc, wc, bc in cases:
        assert cf.fused_select_algo(xc.shape, wc.shape, min_dim) == TC
        xt, wt = torch.from_numpy(xc).cuda(), torch.from_numpy(wc).cuda()
        bt = None if bc is None else torch.from_numpy(bc).cuda()
        auto, tc, ffma = (cf.conv3d_min_softmax(xt, wt, bt, min_dim, algo=a) for a in (cf.CONV_ALGO_AUTO, TC, FFMA))
        assert torch.equal(auto, tc) and not torch.equal(auto, ffma)
        ref = oracle.conv3d_min_softmax(xc, wc, bc, min_dim)
        assert_close(auto.cpu().numpy(), ref, f"fused AUTO {xc.shape} {wc.shape} min_dim={min_dim}")


@pytest.mark.parametrize("min_dim", [2, 3, 4])
@pytest.mark.parametrize("shape,C_out,k", [
    ((2, 3, 6, 11, 37), 40, (3, 3, 3)),     # two channel blocks (32 + 8)
    ((1, 4, 5, 9, 20), 100, (2, 3, 9)),     # four blocks, kernel extent 9 along W (beyond the FFMA kernels)
    ((2, 40, 4, 7, 9), 70, (3, 3, 3)),      # blocks with streamed weights (1080 reduction columns)
])
def test_fused_tensor_core_wide_layers(shape, C_out, k, min_dim):
    rng = np.random.default_rng(C_out + shape[1] + min_dim)
    x = rng.standard_normal(shape).astype(np.float32)
    w = ((rng.random((C_out, shape[1]) + k) - 0.5) * 2 / np.sqrt(shape[1] * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    ref = oracle.conv3d_min_softmax(x, w, b, min_dim)
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    y = cf.conv3d_min_softmax(xt, wt, bt, min_dim, algo=TC)
    yauto = cf.conv3d_min_softmax(xt, wt, bt, min_dim)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, f"fused tensor cores, {C_out} channels, min_dim={min_dim}")
    assert_close(yauto.cpu().numpy(), ref, f"fused planner, {C_out} channels, min_dim={min_dim}")
    assert np.abs(y.sum(dim=1).cpu().numpy() - 1).max() < 1e-5


@pytest.mark.parametrize("min_dim", [3, 4])
@pytest.mark.parametrize("shape,C_out,k", [
    ((2, 3, 7, 11, 37), 24, (3, 3, 3)),     # the page's channel counts on a ragged box
    ((1, 5, 9, 40, 45), 32, (2, 5, 4)),     # 32 channels, kept planes of several 128-position tiles
    ((3, 2, 30, 6, 5), 13, (3, 1, 2)),      # a long reduced axis when the min runs over height
    ((2, 48, 5, 8, 9), 20, (3, 3, 3)),      # 1296 reduction columns: streamed weights
])
def test_fused_tensor_core_min_over_height_and_width(shape, C_out, k, min_dim):
    rng = np.random.default_rng(shape[1] * 7 + C_out + min_dim)
    x = rng.standard_normal(shape).astype(np.float32)
    w = ((rng.random((C_out, shape[1]) + k) - 0.5) * 2 / np.sqrt(shape[1] * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    ref = oracle.conv3d_min_softmax(x, w, b, min_dim)
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    y = cf.conv3d_min_softmax(xt, wt, bt, min_dim, algo=TC)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, f"fused tensor cores min_dim={min_dim} {shape} C_out={C_out}")
    assert np.abs(y.sum(dim=1).cpu().numpy() - 1).max() < 1e-5


def test_fused_vector_path_and_ragged_rows():
    rng = np.random.default_rng(3)
    x = rng.random((3, 3, 6, 9, 40)).astype(np.float32)  # W % 4 == 0, OW = 38 -> 2 column tiles; 7 rows/img
    w = (rng.random((24, 3, 3, 3, 3)).astype(np.float32) - 0.5) * 0.4
    b = (rng.random(24).astype(np.float32) - 0.5) * 0.4
    ref = oracle.conv3d_min_softmax(x, w, b)
    assert_close(run_fused(x, w, b).cpu().numpy(), ref, "fused vector path")
    assert_close(run_fused(x, w, None).cpu().numpy(), oracle.conv3d_min_softmax(x, w, None), "fused no bias")


@pytest.mark.parametrize("algo", [FFMA, TC])
def test_fused_workload_reduced_batch_full_compare(algo):
    wl, x, w, b = workload_inputs("conv3d_min_softmax", 4)
    ref = oracle.conv3d_min_softmax(x, w, b)
    assert_close(run_fused(x, w, b, algo).cpu().numpy(), ref, f"fused workload N=4 algo={algo}")


@pytest.mark.parametrize("algo", [cf.CONV_ALGO_AUTO, FFMA])
def test_fused_workload_full_size_sampled(algo):
    wl, x, w, b = workload_inputs("conv3d_min_softmax")
    y = run_fused(x, w, b, algo)
    N, C_out, OH, OW = y.shape
    rng = np.random.default_rng(9)
    cols = np.unique(np.concatenate([rng.integers(0, N * OH * OW, 1500), [0, OW - 1, OH * OW - 1, N * OH * OW - 1]]))
    yc = y.permute(0, 2, 3, 1).reshape(-1, C_out)[torch.from_numpy(cols).cuda()].cpu().numpy()
    ref = oracle.conv3d_min_softmax_at(x, w, b, cols)
    assert_close(yc, ref, "fused full size sampled")
    assert torch.allclose(y.sum(dim=1), torch.ones((), device="cuda"), atol=1e-5)


# ------------------------------------------- kernel-variant coverage

@pytest.mark.parametrize("kw,dw,pw", [(5, 1, 0), (7, 1, 3), (8, 1, 2), (7, 2, 4), (6, 3, 1)])
def test_tensor_core_wide_kernels(kw, dw, pw):
    # wide kernels along W with dilation and padding on the tensor-core path
    rng = np.random.default_rng(kw * 100 + dw * 10 + pw)
    x = rng.standard_normal((2, 5, 6, 7, 41)).astype(np.float32)
    w = ((rng.random((37, 5, 2, 3, kw)) - 0.5) * 0.3).astype(np.float32)
    b = rng.standard_normal(37).astype(np.float32)
    s, p, d = (1, 2, 1), (1, 1, pw), (2, 1, dw)
    assert cf.algo_supported(2, 5, 37, x.shape[2:], w.shape[2:], s, p, d, cf.CONV_ALGO_IGEMM_3XTF32)
    ref = oracle.conv_nd(x, w, b, s, p, d)
    y = run_conv(x, w, b, s, p, d, cf.CONV_ALGO_IGEMM_3XTF32).cpu().numpy()
    assert_close(y, ref, f"wide kernel kw={kw} dw={dw} pw={pw}")


# Wide kernels along W at unit stride over several parities of the row, plane
# and batch strides, and the same tensors 4 bytes into a buffer: the gather
# may assume nothing about the alignment of a receptive field's first tap.
TAP_ROW_CASES = [
    # C_in, C_out, k, s, p, d, in dims, N
    (3, 64, (3, 5, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1), (6, 12, 64), 2),   # the headline's kernel, even rows
    (3, 20, (2, 3, 6), (1, 1, 1), (0, 0, 0), (1, 1, 1), (5, 10, 40), 2),   # OW = 35: positions of both parities per warp
    (3, 33, (3, 3, 5), (1, 1, 1), (1, 1, 2), (1, 1, 1), (6, 10, 32), 2),   # padding: border and interior warps
    (2, 16, (1, 3, 8), (1, 2, 1), (0, 0, 0), (1, 1, 1), (1, 20, 70), 3),   # KW = 8, stride along H
    (6, 24, (1, 1, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1), (1, 1, 1000), 3),  # a Conv1d
    (2, 40, (2, 2, 5), (1, 1, 1), (0, 0, 0), (2, 2, 1), (7, 9, 30), 2),    # KW = 5, dilation along D and H
    (1, 8, (1, 1, 6), (1, 1, 1), (0, 0, 0), (1, 1, 1), (3, 4, 50), 2),     # KW = 6, one channel
    (1, 12, (1, 1, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1), (3, 5, 31), 3),    # odd batch stride
    (4, 28, (1, 1, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1), (2, 3, 33), 2),    # odd row stride
]


@pytest.mark.parametrize("C_in,C_out,k,s,p,d,ins,N", TAP_ROW_CASES)
def test_tensor_core_kw_geometries(C_in, C_out, k, s, p, d, ins, N):
    rng = np.random.default_rng(C_in * 1000 + C_out * 10 + k[2])
    x = rng.standard_normal((N, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 2 / np.sqrt(C_in * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    assert supported(x, w, s, p, d, cf.CONV_ALGO_IGEMM_3XTF32)
    ref = oracle.conv_nd(x, w, b, s, p, d)
    y = run_conv(x, w, b, s, p, d, cf.CONV_ALGO_IGEMM_3XTF32).cpu().numpy()
    assert_close(y, ref, f"kw geometry C_in={C_in} k={k} ins={ins}")
    # the same tensor one float into a buffer (4-byte aligned only)
    buf = torch.empty(x.size + 1, device="cuda")
    xm = buf[1:].view(x.shape)
    xm.copy_(torch.from_numpy(x))
    ym = cf.conv_fwd_nd(xm, torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(), s, p, d,
                        algo=cf.CONV_ALGO_IGEMM_3XTF32)
    assert_close(ym.cpu().numpy(), ref, f"kw geometry, x 4-byte aligned, C_in={C_in} k={k}")


def test_tensor_core_non_finite_input_stays_in_its_receptive_fields():
    """Infinite inputs reach only the outputs whose receptive fields hold them: no padding
    column of the reduction reads x (0 * inf would make NaN of a finite output)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 3, 4, 8, 20)).astype(np.float32)
    x[..., 7:9] = np.inf  # W positions 7 and 8: outside the fields of output columns 0 and 9..13
    w = ((rng.random((16, 3, 2, 3, 7)) - 0.5) * 0.3).astype(np.float32)
    s, p, d = (1, 1, 1), (0, 0, 0), (1, 1, 1)
    ref = oracle.conv_nd(x, w, None, s, p, d)
    y = run_conv(x, w, None, s, p, d, cf.CONV_ALGO_IGEMM_3XTF32).cpu().numpy().astype(np.float64)
    finite = np.isfinite(ref)
    assert (np.isfinite(y) == finite).all()
    assert_close(np.where(finite, y, 0.0), np.where(finite, ref, 0.0), "finite outputs beside inf inputs")


def test_fused_staged_multi_image_blocks():
    # output width <= 32, C_out <= 24, KW = 3: the staged kernel; OH = 6 makes a
    # block of output rows span several images; W = 30 is not a multiple of 4
    rng = np.random.default_rng(17)
    for C_out, N in ((13, 5), (24, 9), (1, 3)):
        x = rng.random((N, 2, 6, 9, 30)).astype(np.float32)
        w = ((rng.random((C_out, 2, 2, 4, 3)) - 0.5) * 0.5).astype(np.float32)
        b = ((rng.random(C_out) - 0.5) * 0.5).astype(np.float32)
        ref = oracle.conv3d_min_softmax(x, w, b)
        assert_close(run_fused(x, w, b).cpu().numpy(), ref, f"fused staged C_out={C_out} N={N}")
        assert_close(run_fused(x, w, None).cpu().numpy(), oracle.conv3d_min_softmax(x, w, None),
                     f"fused staged no bias C_out={C_out}")


def test_fused_narrow_rows_and_many_rows_per_sm():
    # W = 8: a short shared-row pitch, so lanes of the garbage columns read
    # past the last row of a ring (into the allocation's slack)
    rng = np.random.default_rng(23)
    x = rng.random((3, 2, 5, 6, 8)).astype(np.float32)
    w = ((rng.random((7, 2, 3, 3, 3)) - 0.5) * 0.5).astype(np.float32)
    b = ((rng.random(7) - 0.5) * 0.5).astype(np.float32)
    assert_close(run_fused(x, w, b).cpu().numpy(), oracle.conv3d_min_softmax(x, w, b), "fused W=8")
    # N * OH = 4200 rows: more rows per CTA than warps, so warps take several rows
    x = rng.random((140, 3, 5, 32, 32)).astype(np.float32)
    w = ((rng.random((24, 3, 3, 3, 3)) - 0.5) * 0.3).astype(np.float32)
    b = ((rng.random(24) - 0.5) * 0.3).astype(np.float32)
    y = run_fused(x, w, b).cpu().numpy()
    assert_close(y, oracle.conv3d_min_softmax(x, w, b), "fused 4200 rows")


# ------------------------------------- fused, min over height or width

@pytest.mark.parametrize("C_out,k,shape", [
    (24, (3, 3, 3), (3, 3, 9, 32, 11)),    # the staged kernel on the transposed problem (KH = 3, OH <= 32)
    (17, (2, 3, 4), (2, 2, 6, 34, 9)),     # OH = 32 exactly, odd channel count
    (13, (2, 4, 3), (2, 2, 7, 10, 37)),    # KH = 4: the generic kernel
    (24, (3, 3, 3), (2, 3, 5, 40, 12)),    # OH = 38 > 32: the generic kernel
])
def test_fused_ffma_min_over_width_paths(C_out, k, shape):
    rng = np.random.default_rng(C_out + shape[3])
    x = rng.random(shape).astype(np.float32)
    w = ((rng.random((C_out, shape[1]) + k) - 0.5) * 0.4).astype(np.float32)
    b = ((rng.random(C_out) - 0.5) * 0.4).astype(np.float32)
    ref = oracle.conv3d_min_softmax(x, w, b, 4)
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    y = cf.conv3d_min_softmax(xt, wt, bt, 4, algo=FFMA)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, f"fused FFMA min over width C_out={C_out} k={k} {shape}")


@pytest.mark.parametrize("min_dim", [3, 4])
@pytest.mark.parametrize("C_out,k,shape", [(24, (3, 3, 3), (3, 3, 9, 11, 32)), (13, (2, 4, 3), (2, 2, 7, 10, 37)),
                                           (49, (3, 3, 5), (2, 3, 6, 9, 12)), (5, (1, 5, 2), (3, 1, 4, 21, 6))])
def test_fused_min_dim_small(min_dim, C_out, k, shape):
    rng = np.random.default_rng(C_out * 7 + min_dim)
    x = rng.random(shape).astype(np.float32)
    w = ((rng.random((C_out, shape[1]) + k) - 0.5) * 0.4).astype(np.float32)
    b = ((rng.random(C_out) - 0.5) * 0.4).astype(np.float32)
    ref = oracle.conv3d_min_softmax(x, w, b, min_dim)
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    y = cf.conv3d_min_softmax(xt, wt, bt, min_dim)
    torch.cuda.synchronize()
    assert tuple(y.shape) == ref.shape
    assert_close(y.cpu().numpy(), ref, f"fused min_dim={min_dim} C_out={C_out} k={k}")
    y0 = cf.conv3d_min_softmax(xt, wt, None, min_dim).cpu().numpy()
    assert_close(y0, oracle.conv3d_min_softmax(x, w, None, min_dim), f"fused min_dim={min_dim} no bias")


@pytest.mark.parametrize("min_dim", [3, 4])
def test_fused_min_dim_workload_sampled(min_dim):
    # the benchmark's fused workload with the min over height / width instead of depth
    wl, x, w, b = workload_inputs("conv3d_min_softmax")
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    y = cf.conv3d_min_softmax(xt, wt, bt, min_dim)
    N, C_out, OA, OB = y.shape
    rng = np.random.default_rng(40 + min_dim)
    cols = np.unique(np.concatenate([rng.integers(0, N * OA * OB, 800), [0, OB - 1, OA * OB - 1, N * OA * OB - 1]]))
    yc = y.permute(0, 2, 3, 1).reshape(-1, C_out)[torch.from_numpy(cols).cuda()].cpu().numpy()
    ref = oracle.conv3d_min_softmax_at(x, w, b, cols, min_dim)
    assert_close(yc, ref, f"fused min_dim={min_dim} full size sampled")
    assert torch.allclose(y.sum(dim=1), torch.ones((), device="cuda"), atol=1e-5)


# ------------------------------------------------------------------ groups

def run_grouped(x, w, b, s, p, d, groups, algo=cf.CONV_ALGO_AUTO):
    xt, wt = torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda()
    bt = None if b is None else torch.from_numpy(b).cuda()
    y = cf.conv_fwd_nd(xt, wt, bt, s, p, d, algo=algo, groups=groups)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("algo", [cf.CONV_ALGO_DIRECT_FFMA, cf.CONV_ALGO_IGEMM_3XTF32])
@pytest.mark.parametrize("nd,groups,C_in,C_out,k,s,p,d", [
    (1, 2, 8, 40, (5,), (2,), (1,), (3,)),
    (2, 3, 24, 48, (3, 3), (1, 2), (1, 1), (1, 1)),
    (3, 4, 16, 64, (3, 3, 3), (1, 1, 1), (1, 0, 1), (1, 2, 1)),
    (3, 2, 6, 34, (2, 3, 5), (1, 1, 2), (0, 1, 2), (1, 1, 1)),
])
def test_grouped_conv_both_families(algo, nd, groups, C_in, C_out, k, s, p, d):
    rng = np.random.default_rng(groups * 100 + nd * 10 + algo)
    ins = {1: (77,), 2: (13, 19), 3: (6, 9, 11)}[nd]
    x = rng.standard_normal((2, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in // groups) + k) - 0.5) * 0.4).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    ref = oracle.conv_nd(x, w, b, s, p, d, groups=groups)
    assert_close(run_grouped(x, w, b, s, p, d, groups, algo), ref, f"grouped nd={nd} G={groups} algo={algo}")
    assert_close(run_grouped(x, w, None, s, p, d, groups, algo), oracle.conv_nd(x, w, None, s, p, d, groups=groups),
                 f"grouped no bias nd={nd} G={groups} algo={algo}")


def test_depthwise_conv():
    # groups = C_in = C_out: one input channel per output channel (direct family)
    rng = np.random.default_rng(77)
    C = 32
    x = rng.standard_normal((3, C, 17, 23)).astype(np.float32)
    w = rng.standard_normal((C, 1, 3, 3)).astype(np.float32)
    b = rng.standard_normal(C).astype(np.float32)
    ref = oracle.conv_nd(x, w, b, (1, 1), (1, 1), (1, 1), groups=C)
    assert_close(run_grouped(x, w, b, (1, 1), (1, 1), (1, 1), C), ref, "depthwise 3x3")
    # channel multiplier 2
    w2 = rng.standard_normal((2 * C, 1, 5, 1)).astype(np.float32)
    ref2 = oracle.conv_nd(x, w2, None, (2, 1), (2, 0), (1, 1), groups=C)
    assert_close(run_grouped(x, w2, None, (2, 1), (2, 0), (1, 1), C), ref2, "depthwise multiplier 2")


def test_grouped_planner_takes_tensor_cores_per_group():
    # 4 groups of 16 -> 32 channels, 3^3 taps: each group's reduction is 432 long, so AUTO
    # picks the tensor-core family and launches it once per group
    rng = np.random.default_rng(78)
    x = rng.random((2, 64, 10, 18, 20)).astype(np.float32)
    w = ((rng.random((128, 16, 3, 3, 3)) - 0.5) * 0.1).astype(np.float32)
    b = ((rng.random(128) - 0.5) * 0.1).astype(np.float32)
    assert cf.select_algo(2, 16, 32, x.shape[2:], w.shape[2:], 1, 1, 1) == cf.CONV_ALGO_IGEMM_3XTF32
    ref = oracle.conv_nd(x, w, b, (1, 1, 1), (1, 1, 1), (1, 1, 1), groups=4)
    assert_close(run_grouped(x, w, b, (1, 1, 1), (1, 1, 1), (1, 1, 1), 4), ref, "grouped tensor-core AUTO")


# ------------------------------------------------------- channels last

def to_channels_last(a):
    """A CUDA tensor with a's logical shape [N, C, *sp] stored as [N, *sp, C]."""
    nd = a.ndim - 2
    t = torch.from_numpy(np.ascontiguousarray(np.moveaxis(a, 1, -1))).cuda()
    return t.permute(0, nd + 1, *range(1, nd + 1))


@pytest.mark.parametrize("nd,groups,C_in,C_out,k,s,p,d,N", [
    (3, 1, 8, 64, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), 2),    # padded, C % 4 == 0: 16-byte gathers
    (3, 1, 32, 32, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), 1),   # the second sweep's channels (K = 864)
    (3, 1, 3, 64, (3, 5, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1), 2),    # the headline's channel count: scalar gathers
    (2, 2, 24, 96, (3, 3), (2, 1), (1, 2), (1, 2), 3),
    (1, 1, 64, 128, (3,), (3,), (0,), (4,), 2),                       # the long Conv1d's geometry, short
    (2, 1, 6, 20, (5, 2), (1, 1), (2, 0), (1, 1), 1),                 # C_out not a multiple of 4: scalar stores
    # C_in % 4 != 0 with padding on every axis: groups of 4 reduction columns straddle taps whose
    # in-bounds tests differ, so border positions must test every column on its own
    (3, 1, 3, 40, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), 2),
    (2, 1, 5, 32, (3, 3), (2, 1), (1, 2), (1, 2), 2),
    # weights beyond shared memory: streamed from a stream-ordered block in one pass
    (3, 1, 64, 128, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), 1),
    (3, 2, 96, 64, (3, 3, 3), (1, 1, 1), (0, 1, 1), (1, 1, 1), 1),
])
def test_channels_last_conv(nd, groups, C_in, C_out, k, s, p, d, N):
    rng = np.random.default_rng(C_in * 13 + C_out + nd)
    ins = {1: (301,), 2: (14, 17), 3: (7, 12, 13)}[nd]
    x = rng.standard_normal((N, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in // groups) + k) - 0.5) * 0.3).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    ref = oracle.conv_nd(x, w, b, s, p, d, groups=groups)
    y = cf.conv_fwd_nd(to_channels_last(x), to_channels_last(w), torch.from_numpy(b).cuda(), s, p, d,
                       groups=groups, channels_last=True)
    torch.cuda.synchronize()
    assert y.permute(0, *range(2, nd + 2), 1).is_contiguous()
    assert_close(y.cpu().numpy(), ref, f"channels last nd={nd} C_in={C_in} C_out={C_out} G={groups}")


@pytest.mark.parametrize("offset", [0, 4, 2, 1])
def test_channels_last_input_alignment(offset):
    """x starting 0, 16, 8 or 4 bytes past a 32-byte boundary: 32-byte channel
    groups, 16-byte groups, or scalar gathers; the same values either way."""
    rng = np.random.default_rng(71 + offset)
    N, C_in, C_out, ins, k = 2, 16, 32, (6, 9, 11), (3, 3, 3)
    x = rng.standard_normal((N, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 0.3).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    ref = oracle.conv_nd(x, w, b, 1, 1, 1)
    xcl = np.ascontiguousarray(np.moveaxis(x, 1, -1)).ravel()
    buf = torch.zeros(xcl.size + 8, dtype=torch.float32, device="cuda")
    assert buf.data_ptr() % 32 == 0
    buf[offset:offset + xcl.size] = torch.from_numpy(xcl).cuda()
    sp = ins[0] * ins[1] * ins[2]
    xt = torch.as_strided(buf, (N, C_in) + ins, (sp * C_in, 1, ins[1] * ins[2] * C_in, ins[2] * C_in, C_in),
                          storage_offset=offset)
    assert xt.data_ptr() % 32 == offset * 4
    y = cf.conv_fwd_nd(xt, to_channels_last(w), torch.from_numpy(b).cuda(), 1, 1, 1, channels_last=True)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, f"channels last, x offset {offset * 4} bytes")


def test_channels_last_rejects_direct_family():
    x = to_channels_last(np.zeros((1, 4, 9), np.float32))
    w = to_channels_last(np.zeros((8, 4, 3), np.float32))
    with pytest.raises(cf.ConvError) as e:
        cf.conv_fwd_nd(x, w, None, 1, 0, 1, algo=cf.CONV_ALGO_DIRECT_FFMA, channels_last=True)
    assert e.value.status == cf.CONV_ERR_UNSUPPORTED


# ------------------------------------------------------------------ bf16

def bf16_inputs(x, w, b, dtype=torch.bfloat16):
    """The 16-bit tensors (CUDA) and their exact values as float32 arrays for the oracle."""
    xt, wt = torch.from_numpy(x).to(dtype), torch.from_numpy(w).to(dtype)
    bt = None if b is None else torch.from_numpy(b).to(dtype)
    back = lambda t: None if t is None else t.float().numpy()
    return (xt.cuda(), wt.cuda(), None if bt is None else bt.cuda()), (back(xt), back(wt), back(bt))


def assert_bf16_close(y, ref, S, K, what, mant=8):
    """y rounded once to a 16-bit type with `mant` fraction bits (bf16 7, fp16 10) from an fp32 sum:
    |y - ref| <= 2^-mant |ref| + K 2^-23 S, with S the sum of |w||x| (+|b|) per output (half an ulp at
    the output, doubled, plus an fp32 summation bound).  mant = 8 is the bf16 bound."""
    y = y.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -mant * np.abs(ref) + K * 2.0 ** -23 * S
    err = np.abs(y - ref)
    assert (err <= tol).all(), f"{what}: max excess {(err - tol).max():.3e}, max err {err.max():.3e}"


@pytest.mark.parametrize("nd,groups,C_in,C_out,k,s,p,d", [
    (1, 1, 64, 128, (3,), (3,), (0,), (4,)),
    (2, 2, 24, 48, (3, 3), (1, 2), (1, 1), (1, 1)),
    (3, 1, 3, 64, (3, 5, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1)),
    (3, 1, 8, 32, (3, 5, 7), (1, 2, 2), (1, 2, 3), (2, 1, 1)),
    (3, 1, 32, 40, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1)),
    # beyond one resident launch: channel blocks of 128, streamed weights, both, and groups
    (3, 1, 8, 200, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1)),
    (3, 1, 64, 128, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1)),
    (3, 1, 48, 160, (3, 3, 3), (1, 1, 1), (0, 1, 1), (1, 1, 1)),
    (3, 2, 128, 256, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1)),
])
def test_bf16_conv(nd, groups, C_in, C_out, k, s, p, d):
    rng = np.random.default_rng(C_in + C_out * 3 + nd)
    ins = {1: (517,), 2: (15, 22), 3: (9, 14, 16)}[nd]
    x = rng.random((2, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in // groups) + k) - 0.5) * 0.2).astype(np.float32)
    b = ((rng.random(C_out) - 0.5) * 0.2).astype(np.float32)
    (xt, wt, bt), (xf, wf, bf) = bf16_inputs(x, w, b)
    y = cf.conv_fwd_nd(xt, wt, bt, s, p, d, groups=groups)
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    ref = oracle.conv_nd(xf, wf, bf, s, p, d, groups=groups)
    S = oracle.conv_nd(np.abs(xf), np.abs(wf), np.abs(bf), s, p, d, groups=groups)
    K = (C_in // groups) * int(np.prod(k))
    assert_bf16_close(y, ref, S, K, f"bf16 nd={nd} C_in={C_in} C_out={C_out}")


# Interior warps take a separate loop over the chunks that end before the
# reduction's padding columns; the rest of the tile (and every border warp) goes
# through the tested gather.  These shapes put that hand-off at every place it
# can fall: no partial chunk at all (reduction a multiple of 32), one partial
# chunk, interior and border warps in the same tile, and two issuer slots.
FAST_LOOP_CASES = [
    # C_in, C_out, k, pad, in dims
    (16, 48, (2, 2, 2), (0, 0, 0), (5, 12, 70)),    # 128 columns: every chunk full
    (3, 64, (3, 5, 7), (0, 0, 0), (4, 9, 75)),      # 315 columns: one partial chunk
    (5, 40, (3, 3, 3), (0, 1, 1), (4, 9, 70)),      # 135 columns, border and interior warps
    (8, 96, (2, 2, 2), (0, 0, 0), (4, 10, 67)),     # 64 columns, two slots
    (12, 24, (1, 3, 3), (0, 1, 0), (3, 11, 90)),    # 108 columns, padding along H only
]


@pytest.mark.parametrize("C_in,C_out,k,pad,ins", FAST_LOOP_CASES)
def test_tensor_core_full_chunk_loop(C_in, C_out, k, pad, ins):
    rng = np.random.default_rng(C_in * 1000 + C_out)
    x = rng.standard_normal((2, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 2 / np.sqrt(C_in * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    s, d = (1, 1, 1), (1, 1, 1)
    assert supported(x, w, s, pad, d, cf.CONV_ALGO_IGEMM_3XTF32)
    ref = oracle.conv_nd(x, w, b, s, pad, d)
    y = run_conv(x, w, b, s, pad, d, cf.CONV_ALGO_IGEMM_3XTF32).cpu().numpy()
    assert_close(y, ref, f"fp32 C_in={C_in} C_out={C_out} k={k} pad={pad}")
    # the 16-bit kernel has the same split between the two loops (32-column chunks)
    xs = (rng.random((2, C_in) + ins) - 0.5).astype(np.float32)
    (xt, wt, bt), (xf, wf, bf) = bf16_inputs(xs, w, b)
    yb = cf.conv_fwd_nd(xt, wt, bt, s, pad, d)
    torch.cuda.synchronize()
    refb = oracle.conv_nd(xf, wf, bf, s, pad, d)
    S = oracle.conv_nd(np.abs(xf), np.abs(wf), np.abs(bf), s, pad, d)
    assert_bf16_close(yb, refb, S, C_in * int(np.prod(k)), f"bf16 C_in={C_in} C_out={C_out} k={k} pad={pad}")


def test_bf16_exact_on_small_integers():
    # integer inputs and weights: every product and partial sum is exact in
    # fp32 and every output is an integer below 256, exactly representable in
    # bf16; any mistake in the operand packing or the descriptors shows as a
    # mismatch
    rng = np.random.default_rng(5)
    x = rng.integers(0, 3, (2, 4, 6, 9, 11)).astype(np.float32)
    w = rng.integers(-1, 2, (20, 4, 2, 3, 3)).astype(np.float32)
    b = rng.integers(-2, 3, 20).astype(np.float32)
    (xt, wt, bt), (xf, wf, bf) = bf16_inputs(x, w, b)
    y = cf.conv_fwd_nd(xt, wt, bt, 1, (0, 1, 1), 1).float().cpu().numpy()
    ref = oracle.conv_nd(xf, wf, bf, (1, 1, 1), (0, 1, 1), (1, 1, 1))
    assert np.abs(ref).max() < 256
    assert np.array_equal(y, ref)


# 16-bit kernel, bit-exact on integer data across kernel widths 4..9 along W:
# reductions that end a chunk early, a partial last tile (its border warps take
# the per-column tested gather), streamed weights, channel blocks, strides and
# dilations along one axis, padding, and fp16.
WIDE_KW_16BIT_CASES = [
    # nd, C_in, C_out, k, stride, pad, dilation, in dims, N
    (3, 3, 64, (3, 5, 7), 1, 0, 1, (6, 9, 40), 2),         # the headline's kernel
    (3, 5, 24, (2, 3, 5), 1, 0, 1, (5, 8, 23), 3),         # KW 5, partial last tile
    (3, 2, 40, (1, 2, 6), (1, 1, 2), 0, 1, (3, 7, 41), 2),  # KW 6, stride 2 along W
    (3, 4, 16, (2, 2, 8), 1, 0, 1, (4, 6, 30), 1),         # KW 8
    (2, 7, 33, (3, 7), 1, 0, (2, 1), (15, 29), 2),          # 2-D, dilation along H only
    (1, 9, 20, (7,), 2, 0, 1, (300,), 2),                   # 1-D, stride 2
    (3, 64, 48, (3, 3, 5), 1, 0, 1, (5, 7, 20), 2),        # 2880 columns: weights stream
    (3, 4, 160, (1, 3, 7), 1, 0, 1, (3, 8, 25), 2),        # two channel blocks
    (3, 3, 16, (2, 3, 4), 1, 0, 1, (4, 7, 19), 2),         # KW 4
    (3, 3, 16, (2, 3, 9), 1, 0, 1, (4, 7, 19), 2),         # KW 9
    (3, 3, 16, (2, 3, 7), 1, 0, (1, 1, 2), (4, 7, 25), 2),  # dilation along W
    (3, 3, 16, (2, 3, 7), 1, (0, 1, 3), 1, (4, 7, 19), 2),  # padded
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("nd,C_in,C_out,k,s,p,d,ins,N", WIDE_KW_16BIT_CASES)
def test_16bit_wide_kernels_exact(nd, C_in, C_out, k, s, p, d, ins, N, dtype):
    rng = np.random.default_rng(C_in * 131 + C_out * 7 + k[-1])
    x = rng.integers(0, 2, (N, C_in) + ins).astype(np.float32)
    w = rng.integers(-1, 2, (C_out, C_in) + k).astype(np.float32)
    b = rng.integers(-2, 3, C_out).astype(np.float32)
    (xt, wt, bt), (xf, wf, bf) = bf16_inputs(x, w, b, dtype)
    ref = oracle.conv_nd(xf, wf, bf, s, p, d)
    # every output is an integer small enough for the 16-bit type (bf16: 8 significant bits)
    assert np.abs(ref).max() < 256
    y = cf.conv_fwd_nd(xt, wt, bt, s, p, d).float().cpu().numpy()
    assert np.array_equal(y, ref), f"16-bit case nd={nd} C_in={C_in} k={k}: {np.abs(y - ref).max()}"


@pytest.mark.parametrize("nd,groups,C_in,C_out,k,s,p,d", [
    (1, 1, 64, 128, (3,), (3,), (0,), (4,)),
    (3, 1, 3, 64, (3, 5, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1)),
    (2, 3, 12, 48, (3, 2), (2, 1), (1, 0), (1, 2)),
])
def test_f16_conv(nd, groups, C_in, C_out, k, s, p, d):
    rng = np.random.default_rng(C_in * 5 + C_out + nd)
    ins = {1: (517,), 2: (15, 22), 3: (9, 14, 16)}[nd]
    x = rng.random((2, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in // groups) + k) - 0.5) * 0.2).astype(np.float32)
    b = ((rng.random(C_out) - 0.5) * 0.2).astype(np.float32)
    (xt, wt, bt), (xf, wf, bf) = bf16_inputs(x, w, b, torch.float16)
    y = cf.conv_fwd_nd(xt, wt, bt, s, p, d, groups=groups)
    torch.cuda.synchronize()
    assert y.dtype == torch.float16
    ref = oracle.conv_nd(xf, wf, bf, s, p, d, groups=groups)
    S = oracle.conv_nd(np.abs(xf), np.abs(wf), np.abs(bf), s, p, d, groups=groups)
    K = (C_in // groups) * int(np.prod(k))
    assert_bf16_close(y, ref, S, K, f"f16 nd={nd} C_in={C_in} C_out={C_out}", mant=10)


def test_f16_exact_on_small_integers():
    rng = np.random.default_rng(6)
    x = rng.integers(0, 4, (2, 4, 6, 9, 11)).astype(np.float32)
    w = rng.integers(-2, 3, (20, 4, 2, 3, 3)).astype(np.float32)
    b = rng.integers(-3, 4, 20).astype(np.float32)
    (xt, wt, bt), (xf, wf, bf) = bf16_inputs(x, w, b, torch.float16)
    y = cf.conv_fwd_nd(xt, wt, bt, 1, (0, 1, 1), 1).float().cpu().numpy()
    ref = oracle.conv_nd(xf, wf, bf, (1, 1, 1), (0, 1, 1), (1, 1, 1))
    assert np.abs(ref).max() < 2048
    assert np.array_equal(y, ref)



# --------------------------- tensor cores past one tile of channels / weights

@pytest.mark.parametrize("C_in,C_out,k,pad,channels_last,planned", [
    (64, 64, (3, 3, 3), (1, 1, 1), False, True),    # K = 1728: weights (hi + lo) need 4 passes of shared memory
    (12, 200, (2, 3, 3), (0, 1, 1), False, True),   # 200 output channels: blocks of 128 and 72
    (48, 150, (3, 3, 3), (1, 0, 1), True, False),   # both (12 launches: the planner prefers FFMA), channels last
])
def test_tensor_core_reduction_passes_and_channel_blocks(C_in, C_out, k, pad, channels_last, planned):
    rng = np.random.default_rng(C_in * 3 + C_out)
    x = rng.standard_normal((2, C_in, 6, 9, 10)).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 2 / np.sqrt(C_in * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    s, d = (1, 1, 1), (1, 1, 1)
    expect = cf.CONV_ALGO_IGEMM_3XTF32 if planned else cf.CONV_ALGO_DIRECT_FFMA
    assert cf.select_algo(2, C_in, C_out, x.shape[2:], k, s, pad, d) == expect
    ref = oracle.conv_nd(x, w, b, s, pad, d)
    if channels_last:
        y = cf.conv_fwd_nd(to_channels_last(x), to_channels_last(w), torch.from_numpy(b).cuda(), s, pad, d,
                           channels_last=True)
    else:
        y = cf.conv_fwd_nd(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(), s,
                           pad, d, algo=cf.CONV_ALGO_IGEMM_3XTF32)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, f"tensor cores C_in={C_in} C_out={C_out} k={k}")


# ---------------------------------------------------------- streamed weights

@pytest.mark.parametrize("C_in,C_out,k,pad,groups", [
    (64, 64, (3, 3, 3), (1, 1, 1), 1),     # K = 1728 with 64 channels: 4 shared-memory passes without a workspace
    (64, 128, (3, 3, 3), (1, 1, 1), 1),    # 128 channels: two issuer slots, 32-column chunks
    (96, 48, (3, 3, 3), (0, 1, 1), 2),     # two groups, each with its own part of the workspace
    (40, 20, (5, 5, 5), (2, 2, 2), 1),     # K = 5000: a reduction length not a multiple of 32
])
def test_streamed_weights_workspace(C_in, C_out, k, pad, groups):
    rng = np.random.default_rng(C_in + 7 * C_out + groups)
    x = rng.standard_normal((2, C_in, 5, 8, 9)).astype(np.float32)
    w = ((rng.random((C_out, C_in // groups) + k) - 0.5) * 2 / np.sqrt(C_in // groups * np.prod(k))).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    s, d = (1, 1, 1), (1, 1, 1)
    need = cf.workspace_bytes(2, C_in, C_out, x.shape[2:], k, s, pad, d, groups)
    assert need > 0
    ws = torch.full((need + 256,), 255, dtype=torch.uint8, device="cuda")  # garbage: the call must write it
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    y = cf.conv_fwd_nd_ws(xt, wt, bt, s, pad, d, workspace=ws, groups=groups)
    torch.cuda.synchronize()
    ref = oracle.conv_nd(x, w, b, s, pad, d, groups=groups)
    assert_close(y.cpu().numpy(), ref, f"streamed weights C_in={C_in} C_out={C_out} k={k} G={groups}")
    assert cf.device_status() == 0
    with pytest.raises(cf.ConvError) as e:
        cf.conv_fwd_nd_ws(xt, wt, bt, s, pad, d, workspace=ws[:need // 2], groups=groups)
    assert e.value.status == cf.CONV_ERR_ARG
    # the plain call streams them too, from a stream-ordered block of its own (on a side stream
    # here, so the block's lifetime follows that stream); no workspace: passes of shared memory
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        yp = cf.conv_fwd_nd(xt, wt, bt, s, pad, d, groups=groups, stream=side)
    yn = cf.conv_fwd_nd_ws(xt, wt, bt, s, pad, d, groups=groups, no_workspace=True)
    torch.cuda.synchronize()
    assert_close(yp.cpu().numpy(), ref, f"plain call, streamed weights C_in={C_in} k={k} G={groups}")
    assert_close(yn.cpu().numpy(), ref, f"no workspace, passes C_in={C_in} k={k} G={groups}")
    if cf.select_algo(2, C_in, C_out, x.shape[2:], k, s, pad, d) == cf.CONV_ALGO_IGEMM_3XTF32 and groups == 1:
        assert torch.equal(yp, y), "the plain call's streamed weights must match the caller-workspace call"


def test_cuda_graph_capture_and_replay():
    """Each family launched inside a CUDA graph capture (the design replaces a tracing compiler with
    graphs): a plain tensor-core layer, one with streamed weights (its block then comes from the
    device's default pool, as graphs need) and an FFMA layer; replays match the eager results."""
    rng = np.random.default_rng(21)
    cases = [((2, 3, 6, 12, 40), (32, 3, 3, 5, 7), 0),   # tensor cores, weights resident
             ((1, 64, 4, 6, 6), (128, 64, 3, 3, 3), 1),  # tensor cores, streamed weights
             ((2, 4, 300), (8, 4, 3), 0)]                # FFMA direct
    for xs, ws_, pad in cases:
        x = torch.from_numpy(rng.standard_normal(xs).astype(np.float32)).cuda()
        w = torch.from_numpy(((rng.random(ws_) - 0.5) * 0.1).astype(np.float32)).cuda()
        ref = cf.conv_fwd_nd(x, w, None, 1, pad, 1)
        y = torch.empty_like(ref)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            cf.conv_fwd_nd(x, w, None, 1, pad, 1, out=y)  # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(g):
            cf.conv_fwd_nd(x, w, None, 1, pad, 1, out=y)
        y.zero_()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"graph replay differs for x {xs}"
        x.mul_(2.0)  # the graph reads x at replay time
        g.replay()
        ref2 = cf.conv_fwd_nd(x, w, None, 1, pad, 1)
        torch.cuda.synchronize()
        assert torch.equal(y, ref2)


def test_concurrent_streams_and_threads():
    """Calls from four host threads, each on its own stream, interleaved: streamed-weight layers
    (blocks from the library's pool), resident-weight layers and the host-buffer pipeline.  Every
    result equals the same call made alone (each family is deterministic)."""
    import threading
    rng = np.random.default_rng(33)
    shapes = [((1, 64, 4, 6, 6), (128, 64, 3, 3, 3), 1), ((2, 3, 6, 12, 40), (64, 3, 3, 5, 7), 0)]
    inputs = []
    for t in range(4):
        xs, ws_, pad = shapes[t % 2]
        x = torch.from_numpy(rng.standard_normal(xs).astype(np.float32)).cuda()
        w = torch.from_numpy(((rng.random(ws_) - 0.5) * 0.1).astype(np.float32)).cuda()
        inputs.append((x, w, pad))
    alone = [cf.conv_fwd_nd(x, w, None, 1, pad, 1) for x, w, pad in inputs]
    xh = torch.from_numpy(rng.standard_normal((4, 3, 6, 12, 40)).astype(np.float32)).pin_memory()
    wh = torch.from_numpy(((rng.random((32, 3, 3, 5, 7)) - 0.5) * 0.1).astype(np.float32))
    host_alone = cf.conv_fwd_nd_host(xh, wh, None, 1, 0, 1, chunk=1)
    torch.cuda.synchronize()
    results, errors = [None] * 4, []

    def worker(t):
        try:
            st = torch.cuda.Stream()
            x, w, pad = inputs[t]
            with torch.cuda.stream(st):
                for _ in range(5):
                    y = cf.conv_fwd_nd(x, w, None, 1, pad, 1, stream=st)
                yh = cf.conv_fwd_nd_host(xh, wh, None, 1, 0, 1, chunk=1, stream=st)
            st.synchronize()
            results[t] = (y, yh)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(4):
        assert torch.equal(results[t][0], alone[t]), f"thread {t}"
        assert torch.equal(results[t][1], host_alone), f"thread {t} host path"
    assert cf.device_status() == 0


def test_plan_log_names_the_family_and_plan():
    """CONVFWD_LOG=1: one stderr line per launching call with the problem and the plan."""
    import subprocess, sys, os
    code = ("import torch, implicit_gemm_convolution_fwd_gb300 as cf\n"
            "x = torch.rand(2, 3, 6, 12, 40, device='cuda'); w = torch.rand(64, 3, 3, 5, 7, device='cuda')\n"
            "cf.conv_fwd_nd(x, w, None, 1, 0, 1)\n"
            "cf.conv_fwd_nd(torch.rand(1, 4, 99, device='cuda'), torch.rand(8, 4, 3, device='cuda'), None, 1, 0, 1)\n"
            "cf.conv_fwd_nd(torch.rand(1, 64, 4, 6, 6, device='cuda'), torch.rand(128, 64, 3, 3, 3, device='cuda'),"
            " None, 1, 1, 1)\n"
            "x = torch.rand(2, 3, 8, 10, 10, device='cuda'); w = torch.rand(24, 3, 3, 3, 3, device='cuda')\n"
            "cf.conv3d_min_softmax(x, w, None, 2)\n"
            "torch.cuda.synchronize()\n")
    env = dict(os.environ, CONVFWD_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stderr.splitlines() if l.startswith("convfwd: ")]
    assert len(lines) == 4, r.stderr[-2000:]
    assert "-> igemm_3xtf32 tiles=" in lines[0] and "Kred=315" in lines[0] and "weights=resident" in lines[0]
    assert "-> direct_ffma" in lines[1]
    assert "weights=streamed" in lines[2] and "passes=1" in lines[2]
    assert "conv3d_min_softmax(min over depth)" in lines[3] and "-> fused igemm_3xtf32" in lines[3]
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                       env={k: v for k, v in os.environ.items() if k != "CONVFWD_LOG"},
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0 and "convfwd: " not in r.stderr


def test_plain_call_streamed_weights_release_their_block():
    # a layer with streamed weights called many times: the stream-ordered blocks are freed
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((1, 64, 4, 6, 6)).astype(np.float32)).cuda()
    w = torch.from_numpy(((rng.random((128, 64, 3, 3, 3)) - 0.5) * 0.05).astype(np.float32)).cuda()
    assert cf.workspace_bytes(1, 64, 128, (4, 6, 6), (3, 3, 3), 1, 1, 1) > 0
    y = cf.conv_fwd_nd(x, w, None, 1, 1, 1)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(200):
        cf.conv_fwd_nd(x, w, None, 1, 1, 1, out=y)
    torch.cuda.synchronize()
    assert free0 - torch.cuda.mem_get_info()[0] < 64 << 20


@pytest.mark.parametrize("C,mult,ins,k,pad", [
    (16, 1, (9, 13, 37), (3, 3, 3), (1, 1, 1)),   # tiles cut by every output edge
    (8, 3, (5, 17, 70), (3, 5, 7), (1, 2, 3)),    # channel multiplier 3, a 3x5x7 kernel
    (4, 1, (3, 4, 5), (1, 1, 1), (0, 0, 0)),      # 1x1x1 depthwise: a per-channel scale plus bias
])
def test_depthwise_3d_tiled(C, mult, ins, k, pad):
    rng = np.random.default_rng(C * 11 + mult)
    x = rng.standard_normal((2, C) + ins).astype(np.float32)
    w = rng.standard_normal((C * mult, 1) + k).astype(np.float32)
    b = rng.standard_normal(C * mult).astype(np.float32)
    ref = oracle.conv_nd(x, w, b, (1, 1, 1), pad, (1, 1, 1), groups=C)
    assert_close(run_grouped(x, w, b, (1, 1, 1), pad, (1, 1, 1), C), ref, f"depthwise 3-D C={C} x{mult} k={k}")


# ------------------------------------------ empty batches and side streams

def test_empty_batch_every_entry_point():
    x = torch.empty((0, 8, 6, 7, 9), device="cuda")
    w = torch.randn((16, 4, 3, 3, 3), device="cuda")
    assert tuple(cf.conv_fwd_nd(x, w, None, 1, 1, 1, groups=2).shape) == (0, 16, 6, 7, 9)
    xcl = x.to(memory_format=torch.channels_last_3d)
    wcl = torch.randn((16, 8, 3, 3, 3), device="cuda").to(memory_format=torch.channels_last_3d)
    assert tuple(cf.conv_fwd_nd(xcl, wcl, None, 1, 1, 1, channels_last=True).shape) == (0, 16, 6, 7, 9)
    xh, wh = x.to(torch.bfloat16), w.to(torch.bfloat16)
    assert tuple(cf.conv_fwd_nd(xh, wh, None, 1, 1, 1, groups=2).shape) == (0, 16, 6, 7, 9)
    wbig = torch.randn((64, 8, 7, 7, 7), device="cuda")
    assert tuple(cf.conv_fwd_nd_ws(x, wbig, None, 1, 3, 1).shape) == (0, 64, 6, 7, 9)
    xf = torch.empty((0, 3, 5, 8, 8), device="cuda")
    wf = torch.randn((24, 3, 3, 3, 3), device="cuda")
    for md in (2, 3, 4):
        y = cf.conv3d_min_softmax(xf, wf, None, md)
        assert y.shape[0] == 0 and y.shape[1] == 24


def test_side_stream_matches_default_stream_for_each_family():
    rng = np.random.default_rng(31)
    x = torch.from_numpy(rng.standard_normal((2, 16, 6, 9, 10)).astype(np.float32)).cuda()
    w = torch.from_numpy(((rng.random((32, 16, 3, 3, 3)) - 0.5) * 0.1).astype(np.float32)).cuda()
    wide = torch.from_numpy(((rng.random((64, 64, 3, 3, 3)) - 0.5) * 0.05).astype(np.float32)).cuda()
    xw = torch.from_numpy(rng.standard_normal((2, 64, 5, 8, 9)).astype(np.float32)).cuda()
    calls = [
        lambda st: cf.conv_fwd_nd(x, w, None, 1, 1, 1, algo=cf.CONV_ALGO_IGEMM_3XTF32, stream=st),
        lambda st: cf.conv_fwd_nd(x, w, None, 1, 1, 1, algo=cf.CONV_ALGO_DIRECT_FFMA, stream=st),
        lambda st: cf.conv_fwd_nd(x.to(torch.bfloat16), w.to(torch.bfloat16), None, 1, 1, 1, stream=st),
        lambda st: cf.conv_fwd_nd_ws(xw, wide, None, 1, 1, 1, stream=st),
        lambda st: cf.conv_fwd_nd(x, w[:, :4].contiguous(), None, 1, 1, 1, groups=4, stream=st),
    ]
    st = torch.cuda.Stream()
    for call in calls:
        ref = call(None)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            got = call(st)
        st.synchronize()
        assert torch.equal(got, ref)


# ------------------------------------------------- host buffers, chunked batch

@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("shape", [
    # N, C_in, C_out, groups, in dims, k, stride, pad, dilation, chunk, bias
    (5, 3, 64, 1, (6, 10, 13), (3, 5, 7), (1, 1, 1), (0, 0, 0), (1, 1, 1), 2, True),    # tensor cores, ragged chunk
    (4, 8, 12, 2, (7, 9, 8), (3, 3, 3), (1, 2, 1), (1, 1, 1), (1, 1, 2), 1, False),     # direct kernel, grouped
    (3, 64, 128, 1, (301,), (3,), (3,), (0,), (4,), 0, True),                          # one chunk, Conv1d
])
def test_host_buffers_match_device_call(shape, pinned):
    N, C_in, C_out, groups, ins, k, s, p, d, chunk, with_bias = shape
    rng = np.random.default_rng(N * 100 + C_in)
    x = torch.from_numpy(rng.standard_normal((N, C_in) + ins).astype(np.float32))
    w = torch.from_numpy(((rng.random((C_out, C_in // groups) + k) - 0.5) * 0.3).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal(C_out).astype(np.float32)) if with_bias else None
    if pinned:
        x, w = x.pin_memory(), w.pin_memory()
        b = None if b is None else b.pin_memory()
    y = cf.conv_fwd_nd_host(x, w, b, s, p, d, groups=groups, chunk=chunk)
    torch.cuda.synchronize()
    assert y.device.type == "cpu" and y.is_pinned() == pinned
    yd = cf.conv_fwd_nd(x.cuda(), w.cuda(), None if b is None else b.cuda(), s, p, d, groups=groups)
    torch.cuda.synchronize()
    # same kernels on each chunk: the same arithmetic as the one-call device path
    assert torch.equal(y, yd.cpu())
    ref = oracle.conv_nd(x.numpy(), w.numpy(), None if b is None else b.numpy(), s, p, d, groups=groups)
    assert_close(y.numpy(), ref, f"host buffers {shape}")


def test_host_buffers_reused_workspace_and_stream_order():
    # two calls on one stream sharing one workspace: the second waits for the first's copies
    rng = np.random.default_rng(7)
    s, p, d = (1, 1, 1), (0, 1, 1), (1, 1, 1)
    xs = [torch.from_numpy(rng.standard_normal((6, 4, 5, 8, 9)).astype(np.float32)).pin_memory() for _ in range(2)]
    w = torch.from_numpy(((rng.random((32, 4, 3, 3, 3)) - 0.5) * 0.3).astype(np.float32)).pin_memory()
    need = cf.host_workspace_bytes(6, 4, 32, (5, 8, 9), (3, 3, 3), s, p, d, 1, 2)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    ys = [cf.conv_fwd_nd_host(xx, w, None, s, p, d, chunk=2, workspace=ws, stream=st) for xx in xs]
    st.synchronize()
    for xx, y in zip(xs, ys):
        assert_close(y.numpy(), oracle.conv_nd(xx.numpy(), w.numpy(), None, s, p, d), "reused workspace")


def test_host_buffers_from_concurrent_threads():
    # ctypes drops the GIL during the call, so these enqueue concurrently; each has its own stream
    # and workspace, and the library's per-device lock keeps their event records apart
    import threading
    rng = np.random.default_rng(11)
    s, p, d = (1, 1, 1), (1, 1, 1), (1, 1, 1)
    w = torch.from_numpy(((rng.random((24, 8, 3, 3, 3)) - 0.5) * 0.3).astype(np.float32)).pin_memory()
    xs = [torch.from_numpy(rng.standard_normal((5, 8, 6, 9, 12)).astype(np.float32)).pin_memory() for _ in range(4)]
    out = [None] * len(xs)

    def run(i):
        st = torch.cuda.Stream()
        for _ in range(3):
            out[i] = cf.conv_fwd_nd_host(xs[i], w, None, s, p, d, chunk=2, stream=st)
        st.synchronize()

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(xs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for xx, y in zip(xs, out):
        assert_close(y.numpy(), oracle.conv_nd(xx.numpy(), w.numpy(), None, s, p, d), "concurrent host calls")


def test_host_buffers_empty_batch():
    x = torch.empty((0, 3, 6, 7, 8))
    w = torch.ones((4, 3, 2, 2, 2))
    y = cf.conv_fwd_nd_host(x, w, None, 1, 0, 1, chunk=3)
    torch.cuda.synchronize()
    assert tuple(y.shape) == (0, 4, 5, 6, 7)
