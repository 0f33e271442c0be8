"""conv_fwd_nd_ws_noalloc: the streamed-weights convolution with the library's
static scratch array instead of a caller workspace.  Collected last."""
import ctypes

import numpy as np
import pytest

import implicit_gemm_convolution_fwd_gb300 as cf


def test_noalloc_rejects_oversize_before_any_device_work():
    # two groups of 432 -> 128 channels, 3^3 taps: 2 x 128 x 11680 x 8 bytes (24 MB) of streamed weights
    from implicit_gemm_convolution_fwd_gb300 import build_lib
    build_lib.build()
    lib = cf.load()
    A = cf._arr
    assert cf.workspace_bytes(1, 864, 256, (12, 12, 12), (3, 3, 3), 1, 0, 1, groups=2) > 16 << 20
    st = lib.conv_fwd_nd_ws_noalloc(0x1000, 0x40000000, None, 0x80000000, 3, 1, 864, 256, 2, A((12, 12, 12)),
                                    A((3, 3, 3)), A((1, 1, 1)), A((0, 0, 0)), A((1, 1, 1)), None)
    assert st == cf.CONV_ERR_UNSUPPORTED
    assert "scratch" in lib.conv_last_error().decode()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import torch
    rng = np.random.default_rng(99)
    x = torch.from_numpy(rng.standard_normal((2, 64, 6, 9, 10)).astype(np.float32)).cuda()
    w = torch.from_numpy(((rng.random((96, 64, 3, 3, 3)) - 0.5) * 0.05).astype(np.float32)).cuda()
    b = torch.from_numpy(rng.standard_normal(96).astype(np.float32)).cuda()
    assert cf.workspace_bytes(2, 64, 96, (6, 9, 10), (3, 3, 3), 1, 1, 1) > 0
    ref = cf.conv_fwd_nd_ws(x, w, b, 1, 1, 1)
    for _ in range(2):
        y = cf.conv_fwd_nd_noalloc(x, w, b, 1, 1, 1)
        torch.cuda.synchronize()
        assert torch.equal(y, ref)
    # a second problem through the same scratch, then the first again
    w2 = w[:48].contiguous()
    assert torch.equal(cf.conv_fwd_nd_noalloc(x, w2, None, 1, 1, 1), cf.conv_fwd_nd_ws(x, w2, None, 1, 1, 1))
    assert torch.equal(cf.conv_fwd_nd_noalloc(x, w, b, 1, 1, 1), ref)
    assert cf.device_status() == 0
