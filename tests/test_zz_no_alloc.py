"""conv_fwd_nd_ws_noalloc: the streamed-weights convolution with the library's
static scratch array instead of a caller workspace, for callers that cannot
allocate device memory.  Checked against the fp64 oracle and against the
caller-workspace entry point, over consecutive calls that share the scratch.
Collected last, so that a run stopping at its first failure has already run
every other test."""
import numpy as np
import pytest

import implicit_gemm_convolution_fwd_gb300 as cf
import oracle

TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    from implicit_gemm_convolution_fwd_gb300 import build_lib
    build_lib.build()
    cf.load()


def assert_close(y, ref, what):
    y = np.asarray(y, np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    err = np.abs(y - ref)
    bad = err > TOL * (1.0 + np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {err.size} outside |d| <= 1e-4 (1 + |ref|), max {err.max()}"


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls():
    import torch
    rng = np.random.default_rng(99)
    x = rng.standard_normal((2, 64, 6, 9, 10)).astype(np.float32)
    w = ((rng.random((96, 64, 3, 3, 3)) - 0.5) * 0.05).astype(np.float32)
    b = rng.standard_normal(96).astype(np.float32)
    # a layer whose weights exceed shared memory: it needs the scratch
    assert cf.workspace_bytes(2, 64, 96, (6, 9, 10), (3, 3, 3), 1, 1, 1) > 0
    ref_oracle = oracle.conv_nd(x, w, b, (1, 1, 1), (1, 1, 1), (1, 1, 1))
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    ref_ws = cf.conv_fwd_nd_ws(xt, wt, bt, 1, 1, 1)
    out = torch.empty_like(ref_ws)
    for call in range(2):
        y = cf.conv_fwd_nd_noalloc(xt, wt, bt, 1, 1, 1, out=out)
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), ref_oracle, f"no-alloc call {call}")
        assert torch.equal(y, ref_ws)
    # a second problem through the same scratch, then the first again
    w2 = np.ascontiguousarray(w[:48])
    y2 = cf.conv_fwd_nd_noalloc(xt, torch.from_numpy(w2).cuda(), None, 1, 1, 1)
    torch.cuda.synchronize()
    assert_close(y2.cpu().numpy(), oracle.conv_nd(x, w2, None, (1, 1, 1), (1, 1, 1), (1, 1, 1)), "second problem")
    assert torch.equal(cf.conv_fwd_nd_noalloc(xt, wt, bt, 1, 1, 1), ref_ws)
    assert cf.device_status() == 0
