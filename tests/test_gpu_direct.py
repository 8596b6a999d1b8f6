"""GPU parity of the direct (CUDA-core) convolution kernels, the page's legacy
shaders.  Each output is a sequence of n fp32 fused multiply-adds (or a fixed
tree over partial sums), so it lies within n * 2^-24 * sum|a_k b_k| of the
exact sum; the tests use max(1e-4, n * 2^-24) * sum|a_k b_k| + 1e-6, with n the
number of terms of the output (forward: inC*k*k + 1; input gradient: outC*k*k;
filter gradient: the positions one thread sums plus the 16-level tree).
"""
import numpy as np
import pytest

import synthetic
from tests.gpu_helpers import dev_in, dev_out
from tests.test_gpu_parity import CONV_SHAPES, conv_inputs

pytestmark = pytest.mark.gpu


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


def within(gpu, ref, ref_abs, n, what):
    tol = max(1e-4, n * 2.0 ** -24) * np.asarray(ref_abs) + 1e-6
    err = np.abs(np.asarray(gpu, np.float64) - ref)
    assert np.isfinite(gpu).all(), what
    assert (err <= tol).all(), "%s: worst err/tol %.3g" % (what, float((err / tol).max()))


SHAPES = CONV_SHAPES + [(2, 1, 28, 28, 6, 5, 1, 2), (3, 6, 14, 14, 16, 5, 1, 0)]


@pytest.mark.parametrize("shape", SHAPES)
def test_direct_conv(cb, orc, shape):
    N, C, H, W, K, R, st, pad = shape
    x, w, b, dy = conv_inputs(shape, 700)
    y, dx, dw = dev_out(orc.conv_fwd(x, w, b, st, pad)[0].shape), dev_out(x.shape), dev_out(w.shape)
    cb.conv_fwd_direct(dev_in(x).t, dev_in(w).t, dev_in(b).t, st, pad, y=y.t)
    cb.conv_bwd_data_direct(dev_in(w).t, dev_in(dy).t, x.shape, st, pad, dx=dx.t)
    cb.conv_bwd_filter_direct(dev_in(x).t, dev_in(dy).t, w.shape, st, pad, dw=dw.t)
    cb.check()
    assert y.guards_intact() and dx.guards_intact() and dw.guards_intact()
    within(y.numpy(), *orc.conv_fwd(x, w, b, st, pad, exact=True), C * R * R + 1, "direct fwd %s" % (shape,))
    within(dx.numpy(), *orc.conv_bwd_data(w, dy, x.shape, st, pad, exact=True), K * R * R,
           "direct dgrad %s" % (shape,))
    npos = N * dy.shape[2] * dy.shape[3]
    within(dw.numpy(), *orc.conv_bwd_filter(x, dy, w.shape, st, pad, exact=True), npos // 4096 + 1 + 56,
           "direct wgrad %s" % (shape,))


def test_direct_matches_implicit_gemm_on_small_ints(cb, orc):
    """Small-integer data: every product and partial sum is exact in fp32, so the
    direct kernels, the implicit-GEMM path and the oracle agree bit for bit."""
    shape = (2, 3, 23, 23, 64, 11, 4, 2)
    N, C, H, W, K, R, st, pad = shape
    x = synthetic.small_ints((N, C, H, W), 710)
    w = synthetic.small_ints((K, C, R, R), 711)
    P = (H + 2 * pad - R) // st + 1
    dy = synthetic.small_ints((N, K, P, P), 712)
    xd, wd, dyd = dev_in(x), dev_in(w), dev_in(dy)
    outs = [cb.conv_fwd_direct(xd.t, wd.t, None, st, pad), cb.conv_fwd(xd.t, wd.t, None, st, pad),
            cb.conv_bwd_data_direct(wd.t, dyd.t, x.shape, st, pad), cb.conv_bwd_data(wd.t, dyd.t, x.shape, st, pad),
            cb.conv_bwd_filter_direct(xd.t, dyd.t, w.shape, st, pad),
            cb.conv_bwd_filter(xd.t, dyd.t, w.shape, st, pad)]
    cb.check()
    o = [t.cpu().numpy() for t in outs]
    assert np.array_equal(o[0], o[1]) and np.array_equal(o[0], orc.conv_fwd(x, w, None, st, pad)[0])
    assert np.array_equal(o[2], o[3]) and np.array_equal(o[2], orc.conv_bwd_data(w, dy, x.shape, st, pad)[0])
    assert np.array_equal(o[4], o[5]) and np.array_equal(o[4], orc.conv_bwd_filter(x, dy, w.shape, st, pad)[0])


def test_direct_limits_rejected(cb):
    big = cb.shape_of((70000, 1, 8, 8), (1, 1, 3, 3), 1, 1)      # batch beyond the grid's z limit
    import ctypes
    rc = cb.lib().conv_fwd_direct(ctypes.byref(big), ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10000),
                                  ctypes.c_void_p(0), ctypes.c_void_p(0x10000), ctypes.c_void_p(0))
    assert rc == -2
