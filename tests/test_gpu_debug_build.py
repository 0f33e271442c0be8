"""The debug build (-DCONVFWD_DEBUG): plan assertions on the host and bounds
checks in every kernel that record into the device status word instead of
trapping, the stand-in for a memory checker.

test_parity_suite_under_the_debug_build runs, in a child process with
CONVFWD_DEBUG=1, the tests of this module that need the debug library, the
whole parity suite (test_gpu_parity.py, full-size workloads included) and the
no-allocation entry point's tests; the conftest fixture then fails any test
that leaves an out-of-range index in the status word.

The checks themselves are tested without touching memory outside a tensor:
conv_debug_shrink_bounds makes the device checks treat the last elements of x
(which exist) as out of range, so those reads are skipped and flagged; where
a skipped read yields 0, the output must equal the oracle's on x with that
tail zeroed.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import implicit_gemm_convolution_fwd_gb300 as cf
import oracle

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOL = 1e-4
IN_DEBUG_CHILD = os.environ.get("CONVFWD_DEBUG", "") not in ("", "0")


def test_parity_suite_under_the_debug_build():
    if IN_DEBUG_CHILD:
        pytest.skip("this is the child")
    from implicit_gemm_convolution_fwd_gb300 import build_lib
    build_lib.build(debug=True)
    env = dict(os.environ, CONVFWD_DEBUG="1")
    here = os.path.abspath(__file__)
    others = [os.path.join(ROOT, "tests", f) for f in ("test_gpu_parity.py", "test_zz_no_alloc.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", here] +
                       others, env=env, cwd=ROOT, capture_output=True, text=True, timeout=2400)
    assert r.returncode == 0, r.stdout[-8000:] + r.stderr[-3000:]
    assert " passed" in r.stdout and " failed" not in r.stdout


@pytest.fixture
def debug_lib():
    if not IN_DEBUG_CHILD:
        pytest.skip("runs in the child process that loads the debug build")
    assert cf.is_debug_build(), "CONVFWD_DEBUG=1 but the release library was loaded"
    cf.device_status()
    yield
    cf.debug_shrink_bounds(0)


def assert_close(y, ref, what):
    y = np.asarray(y, np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    bad = np.abs(y - ref) > TOL * (1 + np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"


def zero_tail(x, s):
    z = x.copy()
    z.reshape(-1)[-s:] = 0
    return z


# (C_in, C_out, in_dims, k, stride, pad, dilation, algo): one case per kernel family
FAMILIES = [
    (3, 64, (6, 12, 40), (3, 5, 7), 1, 0, 1, cf.CONV_ALGO_IGEMM_3XTF32),        # tensor cores, interior gather
    (8, 32, (7, 9, 33), (3, 3, 3), 1, 1, 1, cf.CONV_ALGO_IGEMM_3XTF32),         # padded, tested gather
    (64, 128, (6, 8, 10), (3, 3, 3), 1, 1, 1, cf.CONV_ALGO_IGEMM_3XTF32),       # streamed weights
    (5, 12, (5, 9, 17), (2, 3, 3), (1, 2, 1), 1, (2, 1, 1), cf.CONV_ALGO_DIRECT_FFMA),  # FFMA direct
]


def test_debug_build_only_every_family_is_clean(debug_lib):
    rng = np.random.default_rng(1)
    for C_in, C_out, ins, k, s, p, d, algo in FAMILIES:
        x = rng.standard_normal((2, C_in) + ins).astype(np.float32)
        w = ((rng.random((C_out, C_in) + k) - 0.5) * 0.2).astype(np.float32)
        b = rng.standard_normal(C_out).astype(np.float32)
        y = cf.conv_fwd_nd(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(),
                           s, p, d, algo=algo)
        assert cf.device_status() == 0
        assert_close(y.cpu().numpy(), oracle.conv_nd(x, w, b, s, p, d), f"family {algo} {ins} {k}")


@pytest.mark.parametrize("case", range(len(FAMILIES)))
def test_debug_build_only_shrunk_input_extent_is_flagged_and_read_as_zero(debug_lib, case):
    C_in, C_out, ins, k, s, p, d, algo = FAMILIES[case]
    rng = np.random.default_rng(2 + case)
    x = rng.standard_normal((2, C_in) + ins).astype(np.float32)
    w = ((rng.random((C_out, C_in) + k) - 0.5) * 0.2).astype(np.float32)
    b = rng.standard_normal(C_out).astype(np.float32)
    shrink = int(np.prod(ins)) // 3  # a tail of the last input channel of the last image
    cf.debug_shrink_bounds(shrink)
    y = cf.conv_fwd_nd(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(),
                       s, p, d, algo=algo)
    st = cf.device_status()
    first = cf.debug_first_bad_index()
    cf.debug_shrink_bounds(0)
    assert st & cf.STATUS_BOUNDS_X, f"status {st:#x}"
    assert not (st & (cf.STATUS_BOUNDS_ANY & ~cf.STATUS_BOUNDS_X)), f"status {st:#x}"
    assert x.size - shrink <= first < x.size, (first, x.size, shrink)
    assert_close(y.cpu().numpy(), oracle.conv_nd(zero_tail(x, shrink), w, b, s, p, d), "tail read as zero")


def test_debug_build_only_fused_and_16bit_paths_flag_the_tail(debug_lib):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((3, 3, 9, 12, 32)).astype(np.float32)
    w = ((rng.random((24, 3, 3, 3, 3)) - 0.5) * 0.3).astype(np.float32)
    b = rng.standard_normal(24).astype(np.float32)
    shrink = 500
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    for algo in (cf.CONV_ALGO_DIRECT_FFMA, cf.CONV_ALGO_IGEMM_3XTF32):
        for min_dim in (2, 3, 4):
            cf.debug_shrink_bounds(shrink)
            y = cf.conv3d_min_softmax(xt, wt, bt, min_dim, algo=algo)
            st = cf.device_status()
            cf.debug_shrink_bounds(0)
            assert st & cf.STATUS_BOUNDS_X, (algo, min_dim, f"{st:#x}")
            if algo == cf.CONV_ALGO_IGEMM_3XTF32 and min_dim != 4:
                # the tensor-core gather reads skipped elements as 0
                assert_close(y.cpu().numpy(), oracle.conv3d_min_softmax(zero_tail(x, shrink), w, b, min_dim),
                             f"fused tc min_dim {min_dim}")
            y = cf.conv3d_min_softmax(xt, wt, bt, min_dim, algo=algo)
            assert cf.device_status() == 0
            assert_close(y.cpu().numpy(), oracle.conv3d_min_softmax(x, w, b, min_dim), f"fused {algo} {min_dim}")
    xh, wh = xt.bfloat16(), wt.bfloat16()
    cf.debug_shrink_bounds(shrink)
    cf.conv_fwd_nd(xh, wh, None, 1, 1, 1)
    st = cf.device_status()
    cf.debug_shrink_bounds(0)
    assert st & cf.STATUS_BOUNDS_X, f"{st:#x}"
    cf.conv_fwd_nd(xh, wh, None, 1, 1, 1)
    assert cf.device_status() == 0


def test_debug_build_only_channels_last_and_host_buffers_are_clean(debug_lib):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 8, 6, 10, 12)).astype(np.float32)
    w = ((rng.random((16, 8, 3, 3, 3)) - 0.5) * 0.2).astype(np.float32)
    ref = oracle.conv_nd(x, w, None, 1, 1, 1)
    xc = torch.from_numpy(x).cuda().to(memory_format=torch.channels_last_3d)
    wc = torch.from_numpy(w).cuda().to(memory_format=torch.channels_last_3d)
    y = cf.conv_fwd_nd(xc, wc, None, 1, 1, 1, channels_last=True)
    assert cf.device_status() == 0
    assert_close(y.cpu().numpy(), ref, "channels last")
    yh = cf.conv_fwd_nd_host(torch.from_numpy(x).pin_memory(), torch.from_numpy(w), None, 1, 1, 1, chunk=1)
    torch.cuda.synchronize()
    assert cf.device_status() == 0
    assert_close(yh.numpy(), ref, "host buffers")
