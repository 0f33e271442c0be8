"""Host-only checks of the C-ABI library: it loads, exports every symbol that
include/convfwd.h declares, and rejects invalid requests with the documented
status before touching a device.  No compute call runs here.

Several checks hand the library made-up device addresses and rely on its host
validation to refuse the call first.  So that a validation regression can never
turn one of them into a kernel launch on a real GPU, the checks run in a child
pytest process that sees no CUDA device (CUDA_VISIBLE_DEVICES=""): there a call
that got past validation fails with CONV_ERR_CUDA instead of launching.  In
any other process the module runs only the test that starts that child.
"""
import ctypes
import os
import re
import subprocess
import sys
import types

import numpy as np
import pytest

import implicit_gemm_convolution_fwd_gb300 as cf
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "convfwd.h")
DEVICELESS = os.environ.get("CUDA_VISIBLE_DEVICES") == ""
CHILD_RUNNER = "test_host_checks_run_in_a_deviceless_child"


@pytest.fixture(autouse=True)
def _deviceless_only(request):
    if not DEVICELESS and request.node.name != CHILD_RUNNER:
        pytest.skip("runs in the child process that sees no CUDA device")


def test_host_checks_run_in_a_deviceless_child():
    if DEVICELESS:
        pytest.skip("this is the child")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", os.path.abspath(__file__)],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-3000:]
    assert " passed" in r.stdout and " failed" not in r.stdout


@pytest.fixture(scope="module")
def lib():
    from implicit_gemm_convolution_fwd_gb300 import build_lib
    build_lib.build()
    return cf.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*CONVFWD_API\s+[A-Za-z_][A-Za-z0-9_ ]*?\**\s*\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_surface():
    assert declared_functions() == sorted(cf.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_out_dims_matches_oracle(lib):
    rng = np.random.default_rng(0)
    for _ in range(300):
        nd = int(rng.integers(1, 4))
        ins = rng.integers(1, 40, nd)
        k = rng.integers(1, 6, nd)
        s = rng.integers(1, 4, nd)
        p = rng.integers(0, 4, nd)
        d = rng.integers(1, 4, nd)
        ref = oracle.out_dims(ins, k, s, p, d)
        if min(ref) <= 0:
            with pytest.raises(cf.ConvError) as e:
                cf.out_dims(ins, k, s, p, d)
            assert e.value.status == cf.CONV_ERR_SHAPE
        else:
            assert cf.out_dims(ins, k, s, p, d) == ref


def test_page_worked_shapes_through_library(lib):
    assert cf.out_dims((524280,), (3,), 3, 0, 4) == (174758,)
    assert cf.out_dims((64, 64, 64), (3, 5, 7), 1, 0, 1) == (62, 60, 58)
    assert cf.out_dims((24, 32, 32), (3, 3, 3), 1, 0, 1) == (22, 30, 30)


def _call(lib, x=0x1000, w=0x2000, b=None, y=0x10000000, nd=1, N=1, C=1, K=1, ins=(8,), k=(3,), s=(1,), p=(0,),
          d=(1,), algo=0):
    A = cf._arr
    return lib.conv_fwd_nd_ex(x, w, b, y, nd, N, C, K, A(ins), A(k), A(s), A(p), A(d), algo, None)


def test_validation_statuses(lib):
    # every one of these returns before any CUDA call
    assert _call(lib, x=None) == cf.CONV_ERR_NULL
    assert _call(lib, y=None) == cf.CONV_ERR_NULL
    assert lib.conv_fwd_nd_ex(0x1000, 0x2000, None, 0x3000, 1, 1, 1, 1, None, cf._arr((3,)), cf._arr((1,)),
                              cf._arr((0,)), cf._arr((1,)), 0, None) == cf.CONV_ERR_NULL
    assert _call(lib, nd=0) == cf.CONV_ERR_ARG
    assert _call(lib, nd=4, ins=(8,) * 4, k=(1,) * 4, s=(1,) * 4, p=(0,) * 4, d=(1,) * 4) == cf.CONV_ERR_ARG
    assert _call(lib, N=-1) == cf.CONV_ERR_ARG
    assert _call(lib, C=-1) == cf.CONV_ERR_ARG
    assert _call(lib, s=(0,)) == cf.CONV_ERR_ARG
    assert _call(lib, d=(0,)) == cf.CONV_ERR_ARG
    assert _call(lib, p=(-1,)) == cf.CONV_ERR_ARG
    assert _call(lib, ins=(2,), k=(3,)) == cf.CONV_ERR_SHAPE                    # output length <= 0
    assert _call(lib, ins=(8,), k=(3,), d=(4,)) == cf.CONV_ERR_SHAPE            # dilated extent 9 > 8
    assert _call(lib, x=0x1002) == cf.CONV_ERR_ARG                               # misaligned
    assert _call(lib, y=0x1000 + 4) == cf.CONV_ERR_ARG                           # y overlaps x
    assert _call(lib, algo=7) == cf.CONV_ERR_ARG
    assert _call(lib, N=1 << 40) == cf.CONV_ERR_ARG
    msg = lib.conv_last_error().decode()
    assert "N must be" in msg


def test_status_strings(lib):
    for s in range(7):
        assert lib.conv_status_string(s).decode().startswith("CONV_")
    assert b"INTERNAL" in lib.conv_status_string(cf.CONV_ERR_INTERNAL)
    assert b"unknown" in lib.conv_status_string(99)


@pytest.fixture(scope="module")
def debug_lib():
    """The debug build (-DCONVFWD_DEBUG), loaded beside the release one (its own handle)."""
    from implicit_gemm_convolution_fwd_gb300 import build_lib
    d = ctypes.CDLL(build_lib.build(debug=True))
    for h in (d,):
        h.conv_build_flags.restype = ctypes.c_int
        h.conv_debug_shrink_bounds.argtypes = [ctypes.c_longlong]
        h.conv_debug_first_bad_index.argtypes = [ctypes.POINTER(ctypes.c_longlong)]
        h.conv_last_error.restype = ctypes.c_char_p
    return d


def test_debug_library_exports_every_declared_symbol(debug_lib):
    for name in declared_functions():
        assert hasattr(debug_lib, name), name


def test_build_flags_tell_the_builds_apart(lib, debug_lib):
    assert lib.conv_build_flags() == 0
    assert debug_lib.conv_build_flags() == cf.CONV_BUILD_DEBUG


def test_debug_hooks(lib, debug_lib):
    v = ctypes.c_longlong(7)
    # release build: the hooks exist but refuse
    assert lib.conv_debug_shrink_bounds(5) == cf.CONV_ERR_UNSUPPORTED
    assert b"CONVFWD_DEBUG" in lib.conv_last_error()
    assert lib.conv_debug_first_bad_index(ctypes.byref(v)) == cf.CONV_ERR_UNSUPPORTED and v.value == -1
    assert lib.conv_debug_first_bad_index(None) == cf.CONV_ERR_NULL
    # debug build: nothing recorded yet; the shrink takes non-negative counts
    v.value = 7
    assert debug_lib.conv_debug_first_bad_index(ctypes.byref(v)) == cf.CONV_OK and v.value == -1
    assert debug_lib.conv_debug_shrink_bounds(-1) == cf.CONV_ERR_ARG
    assert debug_lib.conv_debug_shrink_bounds(3) == cf.CONV_OK
    assert debug_lib.conv_debug_shrink_bounds(0) == cf.CONV_OK


def test_debug_build_validates_like_the_release_build(debug_lib):
    dims = (ctypes.c_int64 * 3)(8, 8, 8)
    k = (ctypes.c_int64 * 3)(3, 3, 3)
    one = (ctypes.c_int64 * 3)(1, 1, 1)
    zero = (ctypes.c_int64 * 3)(0, 0, 0)
    vp = ctypes.c_void_p
    f = debug_lib.conv_fwd_nd
    f.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + \
        [ctypes.POINTER(ctypes.c_int64)] * 5 + [vp]
    # NULL x with N > 0, then a C_in of 0: refused on the host, as in the release build
    assert f(None, vp(0x1000), None, vp(0x2000), 3, 1, 2, 4, dims, k, one, zero, one, None) == cf.CONV_ERR_NULL
    assert f(vp(0x1000), vp(0x1000), None, vp(0x2000), 3, 1, 0, 4, dims, k, one, zero, one, None) == cf.CONV_ERR_ARG


def test_fused_validation_statuses(lib):
    T5, T4 = cf.Tensor5, cf.Tensor4
    x = T5(0x1000, (ctypes.c_int64 * 5)(2, 3, 24, 32, 32))
    w = T5(0x100000, (ctypes.c_int64 * 5)(24, 3, 3, 3, 3))
    y = T4(0x40000000, (ctypes.c_int64 * 4)(2, 24, 30, 30))
    f = lib.conv3d_min_softmax
    assert f(None, ctypes.byref(w), None, ctypes.byref(y), 2, None) == cf.CONV_ERR_NULL
    # min_dim 3 / 4 keep (D, W) / (D, H): the [N, C_out, OH, OW] descriptor is the wrong shape for them
    assert f(ctypes.byref(x), ctypes.byref(w), None, ctypes.byref(y), 3, None) == cf.CONV_ERR_SHAPE
    assert f(ctypes.byref(x), ctypes.byref(w), None, ctypes.byref(y), 4, None) == cf.CONV_ERR_SHAPE
    assert f(ctypes.byref(x), ctypes.byref(w), None, ctypes.byref(y), 1, None) == cf.CONV_ERR_ARG
    assert f(ctypes.byref(x), ctypes.byref(w), None, ctypes.byref(y), 5, None) == cf.CONV_ERR_ARG
    wbad = T5(0x100000, (ctypes.c_int64 * 5)(24, 4, 3, 3, 3))
    assert f(ctypes.byref(x), ctypes.byref(wbad), None, ctypes.byref(y), 2, None) == cf.CONV_ERR_SHAPE
    ybad = T4(0x40000000, (ctypes.c_int64 * 4)(2, 24, 30, 29))
    assert f(ctypes.byref(x), ctypes.byref(w), None, ctypes.byref(ybad), 2, None) == cf.CONV_ERR_SHAPE
    # 200 channels (beyond the FFMA kernels) with a 40-wide kernel (beyond the tensor-core plan's 32)
    xwide = T5(0x1000, (ctypes.c_int64 * 5)(2, 3, 24, 32, 64))
    wbig = T5(0x100000, (ctypes.c_int64 * 5)(200, 3, 3, 3, 40))
    ybig = T4(0x40000000, (ctypes.c_int64 * 4)(2, 200, 30, 25))
    assert f(ctypes.byref(xwide), ctypes.byref(wbig), None, ctypes.byref(ybig), 2, None) == cf.CONV_ERR_UNSUPPORTED
    ybig4 = T4(0x40000000, (ctypes.c_int64 * 4)(2, 200, 22, 30))  # the min over W keeps (D, H)
    assert f(ctypes.byref(xwide), ctypes.byref(wbig), None, ctypes.byref(ybig4), 4, None) == cf.CONV_ERR_UNSUPPORTED
    xsmall = T5(0x1000, (ctypes.c_int64 * 5)(2, 3, 2, 32, 32))
    assert f(ctypes.byref(xsmall), ctypes.byref(w), None, ctypes.byref(y), 2, None) == cf.CONV_ERR_SHAPE


def test_fused_select_algo_host_only(lib):
    sel = cf.fused_select_algo
    # the tensor cores wherever they run, from the shortest reductions to the widest layers
    for md in (2, 3, 4):
        for xs, ws in [((128, 3, 24, 32, 32), (24, 3, 3, 3, 3)), ((2, 1, 10, 20, 20), (24, 1, 3, 3, 3)),
                       ((2, 1, 10, 20, 20), (40, 1, 3, 3, 3)), ((2, 8, 10, 20, 20), (64, 8, 3, 3, 3))]:
            assert sel(xs, ws, md) == cf.CONV_ALGO_IGEMM_3XTF32, (xs, ws, md)
    # only one family runs: 100 channels (beyond the FFMA kernels), a kernel extent of 9 along W
    assert sel((1, 4, 5, 9, 20), (100, 4, 2, 3, 9), 2) == cf.CONV_ALGO_IGEMM_3XTF32
    # neither family, and invalid requests
    for shapes, md, status in [(((2, 3, 24, 32, 64), (200, 3, 3, 3, 40)), 2, cf.CONV_ERR_UNSUPPORTED),
                               (((2, 3, 24, 32, 32), (24, 3, 3, 3, 3)), 5, cf.CONV_ERR_ARG),
                               (((2, 3, 24, 32, 32), (24, 4, 3, 3, 3)), 2, cf.CONV_ERR_SHAPE),
                               (((2, 3, 2, 32, 32), (24, 3, 3, 3, 3)), 2, cf.CONV_ERR_SHAPE)]:
        with pytest.raises(cf.ConvError) as e:
            sel(*shapes, md)
        assert e.value.status == status, (shapes, md)
    a = ctypes.c_int(0)
    assert lib.conv3d_min_softmax_select_algo(None, None, 2, ctypes.byref(a)) == cf.CONV_ERR_NULL


def test_select_algo_host_only(lib):
    # tiny reductions always take the FFMA direct path
    assert cf.select_algo(2, 4, 8, (1024,), (3,), 3, 0, 4) == cf.CONV_ALGO_DIRECT_FFMA
    a = cf.select_algo(64, 64, 128, (524280,), (3,), 3, 0, 4)
    assert a in (cf.CONV_ALGO_DIRECT_FFMA, cf.CONV_ALGO_IGEMM_3XTF32)
    # weights beyond shared memory (64 -> 128 channels, 3x3x3): conv_fwd_nd streams them in one
    # tensor-core pass, so the planner takes the tensor cores, not the direct path
    assert cf.workspace_bytes(4, 64, 128, (32, 32, 32), (3, 3, 3), 1, 1, 1) > 0
    assert cf.select_algo(4, 64, 128, (32, 32, 32), (3, 3, 3), 1, 1, 1) == cf.CONV_ALGO_IGEMM_3XTF32


def test_algo_supported_queries(lib):
    assert cf.algo_supported(2, 4, 8, (1024,), (3,), 3, 0, 4, cf.CONV_ALGO_DIRECT_FFMA)
    assert not cf.algo_supported(1, 1, 1, (9999,), (1025,), 1, 0, 1, cf.CONV_ALGO_DIRECT_FFMA)
    with pytest.raises(cf.ConvError):
        cf.algo_supported(1, 1, 1, (2,), (3,), 1, 0, 1, cf.CONV_ALGO_DIRECT_FFMA)


def test_grouped_validation_statuses(lib):
    A = cf._arr
    f = lib.conv_fwd_nd_grouped
    args = lambda C_in, C_out, groups: (0x1000, 0x2000, None, 0x10000000, 1, 1, C_in, C_out, groups, A((8,)), A((3,)),
                                        A((1,)), A((0,)), A((1,)), 0, None)
    assert f(*args(4, 6, 0)) == cf.CONV_ERR_ARG     # groups < 1
    assert f(*args(4, 6, 3)) == cf.CONV_ERR_ARG     # 3 does not divide C_in = 4
    assert f(*args(6, 4, 3)) == cf.CONV_ERR_ARG     # 3 does not divide C_out = 4
    assert "groups" in lib.conv_last_error().decode()



def test_host_entry_point_workspace_and_statuses(lib):
    A = cf._arr
    nbytes = ctypes.c_size_t(0)
    dims = lambda: (A((6, 9, 11)), A((3, 5, 7)), A((1, 1, 1)), A((0, 0, 0)), A((1, 1, 1)))
    # workspace: w (64*3*105 floats) and bias, then two x chunks and two y chunks, 256-byte sections
    up = lambda v: (v + 255) // 256 * 256
    out_sp = 4 * 5 * 5
    for chunk, nb in ((0, 10), (3, 3), (10, 10), (25, 10), (-1, 10)):
        assert lib.conv_host_workspace_bytes(3, 10, 3, 64, 1, *dims(), chunk, ctypes.byref(nbytes)) == cf.CONV_OK
        want = up(64 * 3 * 105 * 4) + up(64 * 4) + 2 * up(nb * 3 * 594 * 4) + 2 * up(nb * 64 * out_sp * 4)
        assert nbytes.value == want, (chunk, nbytes.value, want)
    assert lib.conv_host_workspace_bytes(3, 10, 3, 64, 1, *dims(), 2, None) == cf.CONV_ERR_NULL
    assert lib.conv_host_workspace_bytes(3, 10, 3, 64, 4, *dims(), 2, ctypes.byref(nbytes)) == cf.CONV_ERR_ARG
    # the call itself: argument errors are reported before any copy or stream work
    f = lib.conv_fwd_nd_host
    x, w, y = 0x1000, 0x100000, 0x10000000
    ws = 0x7f0000000000
    big = 1 << 40
    assert f(x, w, None, y, 3, 10, 3, 64, 1, *dims(), 2, None, big, None) == cf.CONV_ERR_NULL   # no workspace
    assert f(x, w, None, y, 3, 10, 3, 64, 1, *dims(), 2, ws + 16, big, None) == cf.CONV_ERR_ARG  # misaligned
    assert f(x, w, None, y, 3, 10, 3, 64, 1, *dims(), 2, ws, 1024, None) == cf.CONV_ERR_ARG     # too small
    assert "conv_host_workspace_bytes" in lib.conv_last_error().decode()
    assert f(None, w, None, y, 3, 10, 3, 64, 1, *dims(), 2, ws, big, None) == cf.CONV_ERR_NULL
    assert f(x, w, None, x, 3, 10, 3, 64, 1, *dims(), 2, ws, big, None) == cf.CONV_ERR_ARG     # y overlaps x
    assert f(x, w, None, y, 3, 10, 3, 64, 1, A((6, 9, 2)), A((3, 5, 7)), A((1, 1, 1)), A((0, 0, 0)), A((1, 1, 1)),
             2, ws, big, None) == cf.CONV_ERR_SHAPE                                            # empty output
    # an empty batch needs no device work at all
    assert f(None, w, None, None, 3, 0, 3, 64, 1, *dims(), 2, ws, big, None) == cf.CONV_OK


def test_bindings_reject_bad_tensors_before_any_device_call(lib):
    # host-only: every check below fires before the binding touches CUDA
    import torch
    x = torch.zeros((1, 4, 10))
    w = torch.zeros((6, 4, 3))
    with pytest.raises(ValueError, match="CUDA tensors"):
        cf.conv_fwd_nd(x, w)                                       # CPU tensors on the device entry point
    with pytest.raises(ValueError, match="same rank"):
        cf.conv_fwd_nd(x, torch.zeros((6, 4, 3, 3)))
    with pytest.raises(ValueError, match="float32, bfloat16 or float16"):
        cf.conv_fwd_nd(x.double(), w.double())
    with pytest.raises(ValueError, match="CPU tensors"):
        cf.conv_fwd_nd_host(x.double(), w.double())                # host entry point: fp32 only
    with pytest.raises(ValueError, match="CPU tensors"):
        cf.conv_fwd_nd_host(x[:, :, ::2], w)                       # non-contiguous
    with pytest.raises(ValueError, match="groups"):
        cf.conv_fwd_nd_host(x, w, groups=3)
    with pytest.raises(ValueError, match="groups"):
        cf.conv_fwd_nd_host(x, torch.zeros((6, 3, 3)), groups=2)   # w.shape[1] must be C_in / groups
    with pytest.raises(ValueError, match="CUDA tensors"):
        cf.conv_fwd_nd_ws(x, w)
    with pytest.raises(ValueError, match="5-D"):
        cf.conv3d_min_softmax(x, w)


def test_noalloc_rejects_oversize_before_any_device_work(lib):
    # two groups of 432 -> 128 channels, 3^3 taps: 2 x 128 x 11680 x 8 bytes (24 MB) of streamed weights
    A = cf._arr
    assert cf.workspace_bytes(1, 864, 256, (12, 12, 12), (3, 3, 3), 1, 0, 1, groups=2) > 16 << 20
    st = lib.conv_fwd_nd_ws_noalloc(0x1000, 0x40000000, None, 0x80000000, 3, 1, 864, 256, 2, A((12, 12, 12)),
                                    A((3, 3, 3)), A((1, 1, 1)), A((0, 0, 0)), A((1, 1, 1)), None)
    assert st == cf.CONV_ERR_UNSUPPORTED
    assert "scratch" in lib.conv_last_error().decode()


def test_a_call_past_validation_cannot_launch_here(lib):
    # the guard this module relies on: valid arguments reach the CUDA runtime, which sees no device
    import torch
    assert not torch.cuda.is_available()
    A = cf._arr
    st = lib.conv_fwd_nd_ex(0x1000, 0x2000, None, 0x10000000, 1, 1, 1, 1, A((8,)), A((3,)), A((1,)), A((0,)),
                            A((1,)), cf.CONV_ALGO_DIRECT_FFMA, None)
    assert st == cf.CONV_ERR_CUDA


def _fake_cuda(index, shape=(1,)):
    import torch
    return types.SimpleNamespace(is_cuda=True, device=torch.device("cuda", index), shape=shape)


def test_bindings_reject_tensors_on_different_devices(lib):
    import torch
    assert cf._one_cuda_device(_fake_cuda(0), _fake_cuda(0), None) == torch.device("cuda", 0)
    with pytest.raises(ValueError, match="one CUDA device"):
        cf._one_cuda_device(_fake_cuda(0), _fake_cuda(1))
    with pytest.raises(ValueError, match="one CUDA device"):
        cf._one_cuda_device(_fake_cuda(0), None, _fake_cuda(0), _fake_cuda(2))
    with pytest.raises(ValueError, match="CUDA tensors"):
        cf._one_cuda_device(_fake_cuda(0), torch.zeros(1))


def test_bindings_check_out_shape_dtype_and_layout(lib):
    import torch
    cf._check_out(torch.zeros((2, 3, 4)), (2, 3, 4), torch.float32)
    with pytest.raises(ValueError, match="shape"):
        cf._check_out(torch.zeros((2, 3, 5)), (2, 3, 4), torch.float32)   # a too-small or too-large out
    with pytest.raises(ValueError, match="dtype"):
        cf._check_out(torch.zeros((2, 3, 4), dtype=torch.float16), (2, 3, 4), torch.float32)
    with pytest.raises(ValueError, match="contiguous"):
        cf._check_out(torch.zeros((2, 4, 3)).transpose(1, 2), (2, 3, 4), torch.float32)
    cl = torch.zeros((1, 5, 2, 3, 4)).to(memory_format=torch.channels_last_3d)
    cf._check_out(cl, (1, 5, 2, 3, 4), torch.float32, channels_last=True)
    with pytest.raises(ValueError, match="channels last"):
        cf._check_out(torch.zeros((1, 5, 2, 3, 4)), (1, 5, 2, 3, 4), torch.float32, channels_last=True)


def test_workspace_bindings_check_groups_and_out(lib):
    import torch
    x = torch.zeros((1, 4, 10))
    with pytest.raises(ValueError, match="groups"):
        cf._check_groups(4, 6, 4, 2)          # w.shape[1] must be C_in / groups
    with pytest.raises(ValueError, match="groups"):
        cf._check_groups(4, 6, 1, 4)          # 4 does not divide C_out = 6
    cf._check_groups(4, 6, 2, 2)
    with pytest.raises(ValueError, match="CUDA tensors"):
        cf.conv_fwd_nd_noalloc(x, torch.zeros((6, 4, 3)))


FORCE_PROBE = r"""
import implicit_gemm_convolution_fwd_gb300 as cf
head = cf.select_algo(16, 3, 64, (64, 64, 64), (3, 5, 7))       # the planner: tensor cores
small = cf.select_algo(2, 4, 8, (1024,), (3,), 3, 0, 4)         # the planner: FFMA direct
fused_tc = cf.fused_select_algo((128, 3, 24, 32, 32), (24, 3, 3, 3, 3), 2)   # the planner: tensor cores
fused_short = cf.fused_select_algo((2, 1, 10, 20, 20), (24, 1, 3, 3, 3), 2)  # the planner: tensor cores
print(head, small, fused_tc, fused_short)
"""


TC_, FF_ = cf.CONV_ALGO_IGEMM_3XTF32, cf.CONV_ALGO_DIRECT_FFMA


@pytest.mark.parametrize("value,expect", [
    ("", (TC_, FF_, TC_, TC_)),
    ("direct_ffma", (FF_, FF_, FF_, FF_)),
    ("igemm_3xtf32", (TC_, TC_, TC_, TC_)),
    ("bogus", (TC_, FF_, TC_, TC_)),
])
def test_force_algo_environment_variable(lib, value, expect):
    # read once per process, so each setting gets a process of its own
    env = dict(os.environ, CONVFWD_FORCE_ALGO=value)
    r = subprocess.run([sys.executable, "-c", FORCE_PROBE], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert tuple(int(v) for v in r.stdout.split()) == expect
    assert ("ignored" in r.stderr) == (value == "bogus")
