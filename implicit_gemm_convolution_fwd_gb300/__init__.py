"""Thin Python binding over the C ABI in ``include/convfwd.h``.

Argument marshalling only: every step of the convolution runs in the CUDA
library ``libconvfwd.so`` (built in-tree by ``build_lib.py``).  PyTorch is
used for device memory and streams.  There is no CPU fallback: if the library
is missing or a call fails, these functions raise.  With ``CONVFWD_DEBUG=1``
in the environment the debug build ``libconvfwd_debug.so`` is loaded instead
(plan assertions, device bounds checks; see ``device_status``).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libconvfwd.so")
DEBUG_LIB_PATH = os.path.join(HERE, "libconvfwd_debug.so")

CONV_OK, CONV_ERR_NULL, CONV_ERR_ARG, CONV_ERR_SHAPE, CONV_ERR_UNSUPPORTED, CONV_ERR_CUDA, CONV_ERR_INTERNAL = range(7)
CONV_BUILD_DEBUG = 1
# device status bits (conv_device_status)
STATUS_WATCHDOG = 1 << 0
STATUS_BOUNDS_X, STATUS_BOUNDS_W, STATUS_BOUNDS_Y, STATUS_BOUNDS_WS, STATUS_BOUNDS_SHARED = (1 << 1, 1 << 2, 1 << 3,
                                                                                          1 << 4, 1 << 5)
STATUS_BOUNDS_ANY = STATUS_BOUNDS_X | STATUS_BOUNDS_W | STATUS_BOUNDS_Y | STATUS_BOUNDS_WS | STATUS_BOUNDS_SHARED
CONV_ALGO_AUTO, CONV_ALGO_DIRECT_FFMA, CONV_ALGO_IGEMM_3XTF32 = 0, 1, 2
ALGO_NAMES = {CONV_ALGO_AUTO: "auto", CONV_ALGO_DIRECT_FFMA: "direct_ffma", CONV_ALGO_IGEMM_3XTF32: "igemm_3xtf32"}

# every symbol include/convfwd.h declares
EXPORTED = ("conv_out_dims", "conv_fwd_nd", "conv_fwd_nd_ex", "conv_fwd_nd_grouped", "conv_fwd_nd_channels_last",
            "conv_fwd_nd_bf16", "conv_fwd_nd_f16", "conv_workspace_bytes", "conv_fwd_nd_ws", "conv_fwd_nd_ws_noalloc",
            "conv_host_workspace_bytes", "conv_fwd_nd_host",
            "conv_select_algo",
            "conv_algo_supported",
            "conv3d_min_softmax", "conv3d_min_softmax_ex", "conv3d_min_softmax_select_algo", "conv_peak_mma",
            "conv_peak_ffma", "conv_debug_set_wait_limit",
            "conv_status_string", "conv_last_error", "conv_device_status",
            "conv_build_flags", "conv_debug_first_bad_index", "conv_debug_shrink_bounds")


class ConvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class Tensor5(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dims", ctypes.c_int64 * 5)]


class Tensor4(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dims", ctypes.c_int64 * 4)]


class PeakResult(ctypes.Structure):
    _fields_ = [("flops", ctypes.c_double), ("seconds", ctypes.c_double), ("event_ms", ctypes.c_double),
                ("sm_mhz", ctypes.c_double), ("cycles_per_op", ctypes.c_double), ("ctas", ctypes.c_int)]


_lib = None


def debug_requested() -> bool:
    """True when CONVFWD_DEBUG asks for the debug build."""
    v = os.environ.get("CONVFWD_DEBUG", "")
    return bool(v) and v != "0"


def load(path: str | None = None):
    """Load (once) and return the ctypes handle of libconvfwd.so (libconvfwd_debug.so when CONVFWD_DEBUG=1);
    raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or (DEBUG_LIB_PATH if debug_requested() else LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run build_lib.build())")
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    arr = ctypes.POINTER(ctypes.c_int64)
    lib.conv_out_dims.argtypes = [i32, arr, arr, arr, arr, arr, arr]
    lib.conv_fwd_nd.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, arr, arr, arr, arr, arr, vp]
    lib.conv_fwd_nd_ex.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, arr, arr, arr, arr, arr, i32, vp]
    lib.conv_fwd_nd_grouped.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, i32, vp]
    lib.conv_fwd_nd_channels_last.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, i32,
                                              vp]
    lib.conv_fwd_nd_bf16.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, vp]
    lib.conv_fwd_nd_f16.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, vp]
    lib.conv_workspace_bytes.argtypes = [i32, i64, i64, i64, i64, arr, arr, arr, arr, arr,
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.conv_fwd_nd_ws.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, vp,
                                   ctypes.c_size_t, vp]
    lib.conv_fwd_nd_ws_noalloc.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, vp]
    lib.conv_host_workspace_bytes.argtypes = [i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, i64,
                                              ctypes.POINTER(ctypes.c_size_t)]
    lib.conv_fwd_nd_host.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, arr, arr, arr, arr, arr, i64, vp,
                                     ctypes.c_size_t, vp]
    lib.conv_select_algo.argtypes = [i32, i64, i64, i64, arr, arr, arr, arr, arr, ctypes.POINTER(ctypes.c_int)]
    lib.conv_algo_supported.argtypes = [i32, i64, i64, i64, arr, arr, arr, arr, arr, i32]
    lib.conv3d_min_softmax.argtypes = [ctypes.POINTER(Tensor5), ctypes.POINTER(Tensor5), vp,
                                       ctypes.POINTER(Tensor4), i32, vp]
    lib.conv3d_min_softmax_ex.argtypes = [ctypes.POINTER(Tensor5), ctypes.POINTER(Tensor5), vp,
                                          ctypes.POINTER(Tensor4), i32, i32, vp]
    lib.conv3d_min_softmax_select_algo.argtypes = [ctypes.POINTER(Tensor5), ctypes.POINTER(Tensor5), i32,
                                                   ctypes.POINTER(ctypes.c_int)]
    lib.conv_peak_mma.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(PeakResult), vp]
    lib.conv_peak_ffma.argtypes = [i32, i32, ctypes.POINTER(PeakResult), vp]
    lib.conv_status_string.argtypes = [i32]
    lib.conv_status_string.restype = ctypes.c_char_p
    lib.conv_last_error.argtypes = []
    lib.conv_last_error.restype = ctypes.c_char_p
    lib.conv_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.conv_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
    lib.conv_build_flags.argtypes = []
    lib.conv_debug_first_bad_index.argtypes = [ctypes.POINTER(ctypes.c_longlong)]
    lib.conv_debug_shrink_bounds.argtypes = [ctypes.c_longlong]
    for f in ("conv_out_dims", "conv_fwd_nd", "conv_fwd_nd_ex", "conv_select_algo", "conv_algo_supported",
              "conv3d_min_softmax", "conv3d_min_softmax_ex", "conv3d_min_softmax_select_algo", "conv_peak_mma",
              "conv_peak_ffma", "conv_debug_set_wait_limit", "conv_device_status", "conv_build_flags",
              "conv_debug_first_bad_index", "conv_debug_shrink_bounds"):
        getattr(lib, f).restype = i32
    _lib = lib
    return lib


def _arr(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_int64 * max(1, len(vals)))(*vals)


def _check(status: int):
    if status != CONV_OK:
        lib = load()
        raise ConvError(status, lib.conv_last_error().decode() or lib.conv_status_string(status).decode())


def _tuple(v, nd):
    if isinstance(v, int):
        return (v,) * nd
    v = tuple(int(a) for a in v)
    if len(v) != nd:
        raise ValueError(f"expected {nd} values, got {v}")
    return v


def out_dims(in_dims, k_dims, stride, pad, dilation):
    """Output spatial dims via the library's conv_out_dims (raises ConvError on invalid input)."""
    nd = len(in_dims)
    out = (ctypes.c_int64 * nd)()
    _check(load().conv_out_dims(nd, _arr(in_dims), _arr(k_dims), _arr(_tuple(stride, nd)),
                                _arr(_tuple(pad, nd)), _arr(_tuple(dilation, nd)), out))
    return tuple(out)


def select_algo(N, C_in, C_out, in_dims, k_dims, stride=1, pad=0, dilation=1) -> int:
    nd = len(in_dims)
    a = ctypes.c_int(-1)
    _check(load().conv_select_algo(nd, N, C_in, C_out, _arr(in_dims), _arr(k_dims), _arr(_tuple(stride, nd)),
                                   _arr(_tuple(pad, nd)), _arr(_tuple(dilation, nd)), ctypes.byref(a)))
    return a.value


def fused_select_algo(x_shape, w_shape, min_dim=2) -> int:
    """Host-only query: the kernel family conv3d_min_softmax takes for these shapes with algo=AUTO."""
    xs, ws = Tensor5(), Tensor5()
    xs.dims[:], ws.dims[:] = [int(v) for v in x_shape], [int(v) for v in w_shape]
    a = ctypes.c_int(-1)
    _check(load().conv3d_min_softmax_select_algo(ctypes.byref(xs), ctypes.byref(ws), int(min_dim), ctypes.byref(a)))
    return a.value


def algo_supported(N, C_in, C_out, in_dims, k_dims, stride=1, pad=0, dilation=1, algo=CONV_ALGO_AUTO) -> bool:
    """Host-only query: can kernel family `algo` run this problem?  Raises ConvError if it is invalid."""
    nd = len(in_dims)
    st = load().conv_algo_supported(nd, N, C_in, C_out, _arr(in_dims), _arr(k_dims), _arr(_tuple(stride, nd)),
                                    _arr(_tuple(pad, nd)), _arr(_tuple(dilation, nd)), int(algo))
    if st == CONV_ERR_UNSUPPORTED:
        return False
    _check(st)
    return True


def _stream_handle(stream, device=None):
    """The cudaStream_t of `stream` (default: the current stream of `device`).  A stream given
    explicitly must belong to `device` when one is named."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and stream.device != device:
        raise ValueError(f"the stream is on {stream.device}, the tensors on {device}")
    return ctypes.c_void_p(stream.cuda_stream)


def _one_cuda_device(*tensors):
    """The single CUDA device holding every tensor given (None entries are skipped).

    The library launches on the calling thread's current device; the bindings make the tensors'
    device current for the call, so all of them must live on it."""
    devs = set()
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("x, w, bias and out must be CUDA tensors")
        devs.add(t.device)
    if len(devs) != 1:
        raise ValueError(f"x, w, bias and out must be on one CUDA device, got {sorted(map(str, devs))}")
    return devs.pop()


def _check_groups(C_in, C_out, w_c, groups):
    if groups < 1 or C_in % groups or C_out % groups or w_c * groups != C_in:
        raise ValueError("groups must divide C_in and C_out, and w.shape[1] must be C_in / groups")


def _check_out(out, shape, dtype, channels_last=False):
    """`out` must have exactly `shape` and `dtype` and the layout the call writes."""
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out has shape {tuple(out.shape)}, the call writes {tuple(shape)}")
    if out.dtype != dtype:
        raise ValueError(f"out has dtype {out.dtype}, the call writes {dtype}")
    if channels_last:
        if _channels_last_view(out) is None:
            raise ValueError("out must be stored channels last")
    elif not out.is_contiguous():
        raise ValueError("out must be contiguous")


def _channels_last_view(t):
    """The [N, *spatial, C] tensor whose memory a channels-last [N, C, *spatial] tensor occupies, or None."""
    nd = t.dim() - 2
    v = t.permute(0, *range(2, nd + 2), 1)
    return v if v.is_contiguous() else None


def conv_fwd_nd(x, w, bias=None, stride=1, pad=0, dilation=1, out=None, algo=CONV_ALGO_AUTO, stream=None,
                groups=1, channels_last=False):
    """y = conv(x, w) + bias for fp32 CUDA tensors x [N,C_in,*in], w [C_out,C_in/groups,*k].
    Default layout: contiguous (N C D H W).  channels_last=True: x, w (and out) keep their logical
    shapes but are stored channels last (torch.channels_last / channels_last_3d, i.e. N D H W C);
    the returned y is allocated the same way.
    bfloat16 or float16 x, w (and bias): the 16-bit tensor-core path, fp32 accumulation, y in the
    input dtype (contiguous layout only; `algo` must be AUTO).
    Every tensor must be on one CUDA device; the call runs with that device current."""
    import torch
    nd = x.dim() - 2
    if nd not in (1, 2, 3) or w.dim() != x.dim():
        raise ValueError("x and w must be 3-D, 4-D or 5-D tensors of the same rank")
    dt = x.dtype
    half = (torch.bfloat16, torch.float16)
    if dt not in (torch.float32,) + half:
        raise ValueError("tensors must be float32, bfloat16 or float16")
    for t in (x, w) + ((bias,) if bias is not None else ()):
        if not (t.is_cuda and t.dtype == dt):
            raise ValueError("x, w and bias must be CUDA tensors of one dtype")
    dev = _one_cuda_device(x, w, bias, out)
    if dt in half and (channels_last or algo != CONV_ALGO_AUTO):
        raise ValueError("16-bit tensors take the contiguous layout and algo=AUTO")
    if bias is not None and (not bias.is_contiguous() or tuple(bias.shape) != (w.shape[0],)):
        raise ValueError("bias must be a contiguous [C_out] tensor")
    if channels_last:
        if _channels_last_view(x) is None or _channels_last_view(w) is None:
            raise ValueError("channels_last=True needs x and w stored channels last")
    elif not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("x and w must be contiguous (or pass channels_last=True)")
    s, p, d = _tuple(stride, nd), _tuple(pad, nd), _tuple(dilation, nd)
    N, C_in = x.shape[:2]
    C_out = w.shape[0]
    _check_groups(C_in, C_out, w.shape[1], groups)
    od = out_dims(x.shape[2:], w.shape[2:], s, p, d)
    if out is None:
        if dt in half:
            out = torch.empty((N, C_out) + od, device=dev, dtype=dt)
        elif channels_last:
            out = torch.empty((N,) + od + (C_out,), device=dev, dtype=torch.float32).permute(0, nd + 1,
                                                                                          *range(1, nd + 1))
        else:
            out = torch.empty((N, C_out) + od, device=dev, dtype=torch.float32)
    else:
        _check_out(out, (N, C_out) + od, dt, channels_last)
    lib = load()
    b = None if bias is None else bias.data_ptr()
    dims = (_arr(x.shape[2:]), _arr(w.shape[2:]), _arr(s), _arr(p), _arr(d))
    with torch.cuda.device(dev):
        if dt in half:
            fn = lib.conv_fwd_nd_bf16 if dt == torch.bfloat16 else lib.conv_fwd_nd_f16
            st = fn(x.data_ptr(), w.data_ptr(), b, out.data_ptr(), nd, N, C_in, C_out, int(groups), *dims,
                    _stream_handle(stream, dev))
        else:
            fn = lib.conv_fwd_nd_channels_last if channels_last else lib.conv_fwd_nd_grouped
            st = fn(x.data_ptr(), w.data_ptr(), b, out.data_ptr(), nd, N, C_in, C_out, int(groups), *dims, int(algo),
                    _stream_handle(stream, dev))
    _check(st)
    return out


def conv3d_min_softmax(x, w, bias=None, min_dim=2, out=None, stream=None, algo=CONV_ALGO_AUTO):
    """softmax over channels of the min over tensor dim `min_dim` (2 = depth, 3 = height, 4 = width)
    of conv3d(x, w) + bias, for contiguous fp32 CUDA tensors (stride 1, no padding).  The result
    keeps the two other spatial dims: [N, C_out, OH, OW], [N, C_out, OD, OW] or [N, C_out, OD, OH].
    The conv's output dims come from the library (conv_out_dims).  `algo`: CONV_ALGO_AUTO (the planner),
    CONV_ALGO_DIRECT_FFMA or CONV_ALGO_IGEMM_3XTF32."""
    import torch
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError("x and w must be 5-D")
    for t in (x, w) + ((bias,) if bias is not None else ()):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
            raise ValueError("x, w and bias must be contiguous float32 CUDA tensors")
    dev = _one_cuda_device(x, w, bias, out)
    N, C_out = x.shape[0], w.shape[0]
    od = out_dims(x.shape[2:], w.shape[2:], 1, 0, 1)
    # min_dim outside 2..4 is refused by the library (CONV_ERR_ARG); the buffer shape is then moot
    keep = [od[i] for i in range(3) if i != min_dim - 2] if min_dim in (2, 3, 4) else list(od[1:])
    shape = (N, C_out, keep[0], keep[1])
    if out is None:
        out = torch.empty(shape, device=dev, dtype=torch.float32)
    else:
        _check_out(out, shape, torch.float32)
    xd = Tensor5(x.data_ptr(), (ctypes.c_int64 * 5)(*x.shape))
    wd = Tensor5(w.data_ptr(), (ctypes.c_int64 * 5)(*w.shape))
    yd = Tensor4(out.data_ptr(), (ctypes.c_int64 * 4)(*out.shape))
    with torch.cuda.device(dev):
        st = load().conv3d_min_softmax_ex(ctypes.byref(xd), ctypes.byref(wd),
                                          None if bias is None else bias.data_ptr(), ctypes.byref(yd), int(min_dim),
                                          int(algo), _stream_handle(stream, dev))
    _check(st)
    return out


def workspace_bytes(N, C_in, C_out, in_dims, k_dims, stride=1, pad=0, dilation=1, groups=1) -> int:
    """Bytes of device workspace conv_fwd_nd_ws can use for this problem (0: none needed)."""
    nd = len(in_dims)
    b = ctypes.c_size_t(0)
    _check(load().conv_workspace_bytes(nd, N, C_in, C_out, int(groups), _arr(in_dims), _arr(k_dims),
                                       _arr(_tuple(stride, nd)), _arr(_tuple(pad, nd)), _arr(_tuple(dilation, nd)),
                                       ctypes.byref(b)))
    return int(b.value)


def _fp32_device_problem(x, w, bias, out, stride, pad, dilation, groups):
    """Shared checks of the fp32 contiguous entry points: tensors, groups, the output buffer.
    Returns (device, nd, (s, p, d), N, C_in, C_out, out_dims)."""
    import torch
    nd = x.dim() - 2
    if nd not in (1, 2, 3) or w.dim() != x.dim():
        raise ValueError("x and w must be 3-D, 4-D or 5-D tensors of the same rank")
    for t in (x, w) + ((bias,) if bias is not None else ()):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
            raise ValueError("tensors must be contiguous float32 CUDA tensors")
    dev = _one_cuda_device(x, w, bias, out)
    N, C_in = x.shape[:2]
    C_out = w.shape[0]
    if bias is not None and tuple(bias.shape) != (C_out,):
        raise ValueError("bias must be a [C_out] tensor")
    _check_groups(C_in, C_out, w.shape[1], groups)
    hp = (_tuple(stride, nd), _tuple(pad, nd), _tuple(dilation, nd))
    od = out_dims(x.shape[2:], w.shape[2:], *hp)
    if out is not None:
        _check_out(out, (N, C_out) + od, torch.float32)
    return dev, nd, hp, N, C_in, C_out, od


def conv_fwd_nd_ws(x, w, bias=None, stride=1, pad=0, dilation=1, workspace=None, out=None, stream=None, groups=1,
                   no_workspace=False):
    """conv_fwd_nd (fp32, contiguous) with a caller workspace for streamed weights: `workspace` is a CUDA
    tensor of at least workspace_bytes(...) bytes (allocated here when None and the problem needs one).
    no_workspace=True passes none (NULL): a layer whose weights exceed shared memory then runs in
    several passes, and nothing is allocated."""
    import torch
    dev, nd, (s, p, d), N, C_in, C_out, od = _fp32_device_problem(x, w, bias, out, stride, pad, dilation, groups)
    need = workspace_bytes(N, C_in, C_out, x.shape[2:], w.shape[2:], s, p, d, groups)
    if no_workspace:
        if workspace is not None:
            raise ValueError("no_workspace=True takes no workspace")
    elif workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if stream is not None:
            workspace.record_stream(stream)  # not reused before the call's work on `stream` is done
    if workspace is not None and workspace.device != dev:
        raise ValueError("the workspace must be on the tensors' device")
    if out is None:
        out = torch.empty((N, C_out) + od, device=dev, dtype=torch.float32)
    wsp = None if workspace is None else workspace.data_ptr()
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = load().conv_fwd_nd_ws(x.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
                                   out.data_ptr(), nd, N, C_in, C_out, int(groups), _arr(x.shape[2:]),
                                   _arr(w.shape[2:]), _arr(s), _arr(p), _arr(d), wsp, wsb,
                                   _stream_handle(stream, dev))
    _check(st)
    return out


def conv_fwd_nd_noalloc(x, w, bias=None, stride=1, pad=0, dilation=1, out=None, stream=None, groups=1):
    """conv_fwd_nd_ws with the library's static scratch instead of a caller workspace: the library
    allocates nothing (pass `out` to keep the whole call free of allocation)."""
    import torch
    dev, nd, (s, p, d), N, C_in, C_out, od = _fp32_device_problem(x, w, bias, out, stride, pad, dilation, groups)
    if out is None:
        out = torch.empty((N, C_out) + od, device=dev, dtype=torch.float32)
    with torch.cuda.device(dev):
        st = load().conv_fwd_nd_ws_noalloc(x.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
                                           out.data_ptr(), nd, N, C_in, C_out, int(groups), _arr(x.shape[2:]),
                                           _arr(w.shape[2:]), _arr(s), _arr(p), _arr(d),
                                           _stream_handle(stream, dev))
    _check(st)
    return out


def host_workspace_bytes(N, C_in, C_out, in_dims, k_dims, stride=1, pad=0, dilation=1, groups=1, chunk=0) -> int:
    """Bytes of device workspace conv_fwd_nd_host needs for this problem and batch chunk."""
    nd = len(in_dims)
    b = ctypes.c_size_t(0)
    _check(load().conv_host_workspace_bytes(nd, N, C_in, C_out, int(groups), _arr(in_dims), _arr(k_dims),
                                            _arr(_tuple(stride, nd)), _arr(_tuple(pad, nd)),
                                            _arr(_tuple(dilation, nd)), int(chunk), ctypes.byref(b)))
    return int(b.value)


def conv_fwd_nd_host(x, w, bias=None, stride=1, pad=0, dilation=1, groups=1, chunk=0, workspace=None, out=None,
                     stream=None, device=None):
    """conv_fwd_nd on HOST tensors (contiguous float32 CPU tensors; page-locked ones let the copies overlap
    the compute): the batch goes through the device in chunks of `chunk` images (0: one chunk), copies in
    and out overlapping the convolution.  `workspace`: a CUDA uint8 tensor of at least
    host_workspace_bytes(...) bytes on `device` (allocated here when None).  Returns y on the host once
    `stream` has completed (the call itself does not wait)."""
    import torch
    nd = x.dim() - 2
    if nd not in (1, 2, 3) or w.dim() != x.dim():
        raise ValueError("x and w must be 3-D, 4-D or 5-D tensors of the same rank")
    s, p, d = _tuple(stride, nd), _tuple(pad, nd), _tuple(dilation, nd)
    N, C_in = x.shape[:2]
    C_out = w.shape[0]
    for t in (x, w) + ((bias,) if bias is not None else ()):
        if not (t.device.type == "cpu" and t.dtype == torch.float32 and t.is_contiguous()):
            raise ValueError("tensors must be contiguous float32 CPU tensors")
    if bias is not None and tuple(bias.shape) != (C_out,):
        raise ValueError("bias must be a [C_out] tensor")
    _check_groups(C_in, C_out, w.shape[1], groups)
    od = out_dims(x.shape[2:], w.shape[2:], s, p, d)
    if out is not None:
        if out.device.type != "cpu":
            raise ValueError("out must be a CPU tensor")
        _check_out(out, (N, C_out) + od, torch.float32)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if dev.type != "cuda":
        raise ValueError("device must be a CUDA device")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        need = host_workspace_bytes(N, C_in, C_out, x.shape[2:], w.shape[2:], s, p, d, groups, chunk)
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        # the copies run on the library's own streams too: keep the block until `stream` (which waits
        # for them) is done
        workspace.record_stream(torch.cuda.current_stream(dev) if stream is None else stream)
    elif workspace.device != dev:
        raise ValueError("the workspace must be on `device`")
    if out is None:
        out = torch.empty((N, C_out) + od, dtype=torch.float32, pin_memory=x.is_pinned())
    with torch.cuda.device(dev):
        st = load().conv_fwd_nd_host(x.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
                                     out.data_ptr(), nd, N, C_in, C_out, int(groups), _arr(x.shape[2:]),
                                     _arr(w.shape[2:]), _arr(s), _arr(p), _arr(d), int(chunk), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    _check(st)
    return out


def _peak_dict(r):
    return {"tflops": r.flops / r.seconds / 1e12 if r.seconds > 0 else 0.0, "seconds": r.seconds,
            "event_ms": r.event_ms, "sm_mhz": r.sm_mhz, "cycles_per_op": r.cycles_per_op, "ctas": r.ctas,
            "flops": r.flops}


def peak_mma(kind="tf32", n=128, issuers=2, a_in_tmem=True, iters=20000, stream=None) -> dict:
    """Measured tensor-core rate: back-to-back tcgen05.mma (M=128, N=n, one K step) from `issuers` warps
    per SM on resident operands.  kind "tf32" or "bf16".  Synchronises the stream."""
    r = PeakResult()
    k = {"tf32": 0, "bf16": 1}[kind]
    _check(load().conv_peak_mma(k, int(n), int(issuers), int(bool(a_in_tmem)), int(iters), ctypes.byref(r),
                                _stream_handle(stream)))
    return _peak_dict(r)


def peak_ffma(packed=False, iters=4000, stream=None) -> dict:
    """Measured FP32 FMA rate over every resident thread (scalar or packed f32x2).  Synchronises the stream."""
    r = PeakResult()
    _check(load().conv_peak_ffma(int(bool(packed)), int(iters), ctypes.byref(r), _stream_handle(stream)))
    return _peak_dict(r)


def set_wait_limit(cycles: int = 0):
    """Test hook: tensor-core launches from now on give up a pipeline wait after `cycles` SM clock cycles
    (0 restores the default, about two seconds).  Process-wide."""
    _check(load().conv_debug_set_wait_limit(int(cycles)))


def device_status() -> int:
    """Synchronise and read/clear the device-side status word (0 = no kernel gave up a wait and, in the debug
    build, no index fell outside its tensor)."""
    v = ctypes.c_uint(0)
    _check(load().conv_device_status(ctypes.byref(v)))
    return v.value


def is_debug_build() -> bool:
    """True when the loaded library is the debug build (plan assertions, device bounds checks)."""
    return bool(load().conv_build_flags() & CONV_BUILD_DEBUG)


def debug_first_bad_index() -> int:
    """Debug build: the first out-of-range element index the last device_status() call found (-1: none)."""
    v = ctypes.c_longlong(-1)
    _check(load().conv_debug_first_bad_index(ctypes.byref(v)))
    return v.value


def debug_shrink_bounds(elems: int = 0):
    """Debug-build test hook: the device checks treat the last `elems` elements of x as out of range (0 resets)."""
    _check(load().conv_debug_shrink_bounds(int(elems)))
