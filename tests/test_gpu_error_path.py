"""The bounded-wait error path on the GPU (the C ABI's device-timeout
contract): every wait inside the library's kernels gives up after a bounded
time, latches CONV_ERR_DEVICE_TIMEOUT in the device error word and unwinds.

The test hook conv_b200_debug_withhold_stage makes the first CTA of the next
register-gather GEMM launch withhold its producers' arrival for one pipeline
stage: that CTA's MMA issuer then waits for a stage that never fills.  The
kernel must give up (about 2 s), drain its own MMAs, free its tensor memory
and return; conv_b200_check() must report CONV_ERR_DEVICE_TIMEOUT once, and a
normal call on the same stream afterwards must run and match the oracle.
No fault, trap or endless wait is involved: the wait is bounded by design.
"""
import numpy as np
import pytest

import synthetic
from tests.gpu_helpers import assert_within_tol

pytestmark = pytest.mark.gpu

CONV_ERR_DEVICE_TIMEOUT = -7


@pytest.fixture(scope="module")
def cb():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from im2col_convolution_tiled_gb300 import build
    build.build()
    import im2col_convolution_tiled_gb300 as m
    m.load()
    return m


def test_withheld_stage_times_out_then_stream_recovers(cb):
    import time
    import torch
    import oracle
    orc = oracle.get()
    # 16 K stages per tile; whether a tile runs whole or its K range is cut
    # over a cluster (at most 8 pieces of >= 2 stages), CTA 0 runs stage 1
    M, K, N = 512, 512, 512
    A, B = synthetic.matmul_case(M, K, N, 0)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    cb.check()                       # nothing pending before the test
    lib = cb.lib()
    assert lib.conv_b200_debug_withhold_stage(1) == 0
    t0 = time.perf_counter()
    cb.matmul(a, b, 0)               # asynchronous: the call itself succeeds
    with pytest.raises(cb.ConvError) as ei:
        cb.check()
    waited = time.perf_counter() - t0
    assert ei.value.code == CONV_ERR_DEVICE_TIMEOUT
    assert waited < 30.0             # the wait is bounded (about 2 s)
    cb.check()                       # the error word was cleared by the read
    # one-shot: the next launch runs normally on the same stream and is correct
    c = cb.matmul(a, b, 0)
    cb.check()
    ref, ref_abs = orc.matmul(A, B, 0)
    assert_within_tol(c.cpu().numpy(), ref, ref_abs, "matmul after a timed-out launch")


def test_withhold_cancel(cb):
    import torch
    lib = cb.lib()
    A, B = synthetic.matmul_case(256, 64, 256, 0)
    assert lib.conv_b200_debug_withhold_stage(1) == 0
    assert lib.conv_b200_debug_withhold_stage(-1) == 0      # cancelled before any launch
    c = cb.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), 0)
    cb.check()
    assert np.isfinite(c.cpu().numpy()).all()
