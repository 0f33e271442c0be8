"""The tensor-core kernels' bounded waits, made to run out on purpose.

With the pipeline-wait limit set to a few hundred SM clock cycles, the first
wait that is not satisfied at once gives up: the kernel raises its abort flag,
every role falls through, the issuers wait (with the full default limit) for
their own MMAs, tensor memory is freed and bit 0 of the device status word is
set.  The call itself succeeds (the launch was valid); the status word reports
the incomplete output, and the next call with the default limit must be
correct.  No fault, trap or hang is involved: every wait is bounded."""
import numpy as np
import pytest

import implicit_gemm_convolution_fwd_gb300 as cf
import oracle

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    from implicit_gemm_convolution_fwd_gb300 import build_lib
    build_lib.build()
    cf.load()
    yield
    cf.set_wait_limit(0)


def _problem():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((2, 8, 10, 12, 14)).astype(np.float32)
    w = ((rng.random((32, 8, 3, 3, 3)) - 0.5) * 0.2).astype(np.float32)
    b = rng.standard_normal(32).astype(np.float32)
    return x, w, b, (1, 1, 1), (1, 1, 1), (1, 1, 1)


def test_short_wait_limit_aborts_cleanly_and_the_next_call_is_correct():
    import torch
    x, w, b, s, p, d = _problem()
    assert cf.algo_supported(2, 8, 32, x.shape[2:], w.shape[2:], s, p, d, cf.CONV_ALGO_IGEMM_3XTF32)
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    assert cf.device_status() == 0
    # A poll (`mbarrier.try_wait`) may itself block until its phase completes,
    # up to a time the hardware chooses, so one launch can see every wait
    # satisfied before the clock is read: up to eight launches, each either
    # complete (status 0) or given up (bit 0).
    cf.set_wait_limit(256)
    st = 0
    try:
        for _ in range(8):
            cf.conv_fwd_nd(xt, wt, bt, s, p, d, algo=cf.CONV_ALGO_IGEMM_3XTF32)
            torch.cuda.synchronize()  # the kernel returned
            st = cf.device_status()
            if st & 1:
                break
    finally:
        cf.set_wait_limit(0)
    assert st & 1, "a wait of a few hundred cycles should have given up"
    assert st & 0x1f00, f"the status word names no wait site: {st:#x}"
    assert st & ~0x1f01 == 0, f"unknown status bits: {st:#x}"
    # the status word was read and cleared; the device and the library still work
    assert cf.device_status() == 0
    ref = oracle.conv_nd(x, w, b, s, p, d)
    for _ in range(2):
        y = cf.conv_fwd_nd(xt, wt, bt, s, p, d, algo=cf.CONV_ALGO_IGEMM_3XTF32).cpu().numpy().astype(np.float64)
        err = np.abs(y - ref)
        assert (err <= TOL * (1 + np.abs(ref))).all(), err.max()
    assert cf.device_status() == 0


def test_wait_limit_argument_checks():
    with pytest.raises(cf.ConvError):
        cf.set_wait_limit(10)  # below 64 cycles
    cf.set_wait_limit(0)
