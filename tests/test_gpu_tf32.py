"""GPU parity of the one-product TF32 mode (CONV_MATH_TF32) of the contractions.

Tolerance, derived from the arithmetic: each operand is truncated to TF32 (10
explicit mantissa bits), a relative error below 2^-10, so each product is off
by less than (2 * 2^-10 + 2^-20) |a b| < 1.96e-3 |a b|; the fp32 accumulation
adds at most about K * 2^-24 sum|a b| (< 2.5e-4 for K <= 4096).  Hence
|gpu - oracle| <= 2.5e-3 * sum_k |a_k b_k| + 1e-6 per element.  Small
integers are exact in TF32, so small-integer data stays bit-exact.
"""
import numpy as np
import pytest

import synthetic
from tests.gpu_helpers import dev_in, dev_out
from tests.test_gpu_parity import CONV_SHAPES, MM_SHAPES, conv_inputs

pytestmark = pytest.mark.gpu

TOL = 2.5e-3


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


@pytest.fixture
def tf32(cb):
    prev = cb.set_math_mode(cb.CONV_MATH_TF32)
    yield
    cb.set_math_mode(prev)


def within(gpu, ref, ref_abs, what):
    err = np.abs(np.asarray(gpu, np.float64) - ref)
    tol = TOL * ref_abs + 1e-6
    assert np.isfinite(gpu).all(), what
    assert (err <= tol).all(), "%s: worst err/tol %.3g" % (what, float((err / tol).max()))
    return float((err / (ref_abs + 1e-30)).max())


SHAPES = CONV_SHAPES[:5] + CONV_SHAPES[-4:]


@pytest.mark.parametrize("shape", SHAPES)
def test_conv_tf32(cb, orc, tf32, shape):
    x, w, b, dy = conv_inputs(shape, 500)
    st, pad = shape[6], shape[7]
    y = dev_out(orc.conv_fwd(x, w, b, st, pad)[0].shape)
    dx = dev_out(x.shape)
    dw, db = dev_out(w.shape), dev_out(b.shape)
    cb.conv_fwd(dev_in(x).t, dev_in(w).t, dev_in(b).t, st, pad, y=y.t)
    cb.conv_bwd_data(dev_in(w).t, dev_in(dy).t, x.shape, st, pad, dx=dx.t)
    cb.conv_bwd_filter_bias(dev_in(x).t, dev_in(dy).t, w.shape, st, pad, dw=dw.t, db=db.t)
    cb.check()
    assert y.guards_intact() and dx.guards_intact() and dw.guards_intact()
    within(y.numpy(), *orc.conv_fwd(x, w, b, st, pad, exact=True), "fwd %s" % (shape,))
    within(dx.numpy(), *orc.conv_bwd_data(w, dy, x.shape, st, pad, exact=True), "dgrad %s" % (shape,))
    within(dw.numpy(), *orc.conv_bwd_filter(x, dy, w.shape, st, pad, exact=True), "wgrad %s" % (shape,))


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("M,K,N", MM_SHAPES[:6] + MM_SHAPES[-2:])
def test_matmul_tf32(cb, orc, tf32, M, K, N, flags):
    A, B = synthetic.matmul_case(M, K, N, flags)
    c = dev_out((M, N))
    cb.matmul(dev_in(A).t, dev_in(B).t, flags, C=c.t)
    cb.check()
    assert c.guards_intact()
    within(c.numpy(), *orc.matmul(A, B, flags, exact=True), "matmul %dx%dx%d f%d" % (M, K, N, flags))


def test_small_ints_exact_in_tf32(cb, orc, tf32):
    for flags in range(4):
        A = synthetic.small_ints((300, 77) if not flags & 1 else (77, 300), 31)
        B = synthetic.small_ints((77, 129) if not flags & 2 else (129, 77), 32)
        c = cb.matmul(dev_in(A).t, dev_in(B).t, flags)
        cb.check()
        assert np.array_equal(c.cpu().numpy(), orc.matmul(A, B, flags)[0])
    shape = CONV_SHAPES[3]
    N, C, H, W, K, R, st, pad = shape
    x = synthetic.small_ints((N, C, H, W), 33)
    w = synthetic.small_ints((K, C, R, R), 34)
    y = cb.conv_fwd(dev_in(x).t, dev_in(w).t, None, st, pad)
    cb.check()
    assert np.array_equal(y.cpu().numpy(), orc.conv_fwd(x, w, None, st, pad)[0])


def test_mode_takes_effect(cb, orc):
    """The two modes give different results on fp32 data, TF32's error is the
    larger one, and switching back restores the fp32-faithful result exactly."""
    A, B = synthetic.matmul_case(256, 1600, 256, 0)
    ref, ref_abs = orc.matmul(A, B, 0, exact=True)
    a, b = dev_in(A), dev_in(B)
    c3 = cb.matmul(a.t, b.t, 0).cpu().numpy()
    with cb.math(cb.CONV_MATH_TF32):
        c1 = cb.matmul(a.t, b.t, 0).cpu().numpy()
    c3b = cb.matmul(a.t, b.t, 0).cpu().numpy()
    cb.check()
    assert np.array_equal(c3, c3b)
    e3 = np.abs(c3 - ref).max()
    e1 = np.abs(c1 - ref).max()
    assert e1 > 10 * e3, (e1, e3)
    assert (np.abs(c1 - ref) <= TOL * ref_abs + 1e-6).all()


# ---------------------------------------------------------------------------
# flagged matmul: a subset of the 1176-case sweep (small, ragged and the
# largest sizes, so the 32- to 256-wide tiles all run), sampled entries as in
# tests/test_gpu_matmul_sweep.py, at the TF32 tolerance

from tests.test_gpu_matmul_sweep import pools, run_case  # noqa: E402,F401  (fixture and checker)

TF32_SWEEP_MN = (127, 1024, 9216)
TF32_SWEEP_K = (25, 2304, 4096)


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("M", TF32_SWEEP_MN)
def test_matmul_sweep_subset_tf32(cb, orc, tf32, pools, M, flags):
    worst = 0.0
    for N in TF32_SWEEP_MN:
        for K in TF32_SWEEP_K:
            worst = max(worst, run_case(cb, orc, pools, M, K, N, flags, tol_scale=TOL))
    assert worst <= 1.0
