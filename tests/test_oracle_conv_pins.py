"""Pins of the oracle's convolution pipeline (page "DirectCompute Neural Network
Engine", section "Convolution: The im2col Approach") against things other than
itself: a direct convolution, torch's float64 CPU routines, closed forms, the
im2col/col2im adjoint identity and central finite differences.
"""
import itertools

import numpy as np
import pytest

import synthetic
from oracle import out_size

torch = pytest.importorskip("torch")
F = torch.nn.functional

# (N, C, H, W, Ko, R, stride, pad): tiny shapes covering stride 1-4, pad 0-2,
# k 1-5, non-square images and output extents of 1.
SHAPES = [
    (1, 1, 5, 5, 1, 3, 1, 0),
    (2, 3, 7, 6, 4, 3, 2, 1),
    (1, 2, 9, 9, 3, 5, 1, 2),
    (2, 1, 11, 11, 2, 4, 4, 2),
    (1, 3, 6, 8, 2, 1, 1, 0),
    (3, 2, 5, 7, 3, 2, 3, 1),
    (1, 1, 4, 4, 2, 4, 1, 0),    # output 1x1
    (2, 2, 8, 5, 3, 3, 2, 2),
]


def make(shape, seed, ints=False):
    N, C, H, W, Ko, R, st, pad = shape
    P, Q = out_size(H, R, st, pad), out_size(W, R, st, pad)
    gen = synthetic.small_ints if ints else synthetic.normal
    x = gen((N, C, H, W), seed + 1)
    w = gen((Ko, C, R, R), seed + 2)
    b = gen((Ko,), seed + 3)
    dy = gen((N, Ko, P, Q), seed + 4)
    return x, w, b, dy


def direct_conv(x, w, b, st, pad):
    """Seven nested loops over an explicitly zero-padded input (no im2col)."""
    N, C, H, W = x.shape
    Ko, _, R, _ = w.shape
    xp = np.zeros((N, C, H + 2 * pad, W + 2 * pad))
    xp[:, :, pad:pad + H, pad:pad + W] = x
    P, Q = (H + 2 * pad - R) // st + 1, (W + 2 * pad - R) // st + 1
    y = np.zeros((N, Ko, P, Q))
    for n, k, oh, ow in itertools.product(range(N), range(Ko), range(P), range(Q)):
        acc = float(b[k])
        for c in range(C):
            for r in range(R):
                for s in range(R):
                    acc += float(w[k, c, r, s]) * xp[n, c, oh * st + r, ow * st + s]
        y[n, k, oh, ow] = acc
    return y


@pytest.mark.parametrize("shape", SHAPES)
def test_fwd_matches_direct_conv(orc, shape):
    x, w, b, _ = make(shape, 11)
    st, pad = shape[6], shape[7]
    y, y_abs = orc.conv_fwd(x, w, b, st, pad, exact=True)
    ref = direct_conv(x, w, b, st, pad)
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * (1 + y_abs.max()))


@pytest.mark.parametrize("shape", SHAPES)
def test_fwd_small_ints_exact(orc, shape):
    x, w, b, _ = make(shape, 12, ints=True)
    st, pad = shape[6], shape[7]
    y, _ = orc.conv_fwd(x, w, b, st, pad, exact=True)
    assert np.array_equal(y, direct_conv(x, w, b, st, pad))


def test_fwd_hand_worked():
    """1..9 in a 3x3 image, a 2x2 kernel of ones, stride 1: each output is the
    sum of one 2x2 block; with stride 2 / pad 1 the corners see single pixels."""
    import oracle
    orc = oracle.get()
    x = np.arange(1, 10, dtype=np.float32).reshape(1, 1, 3, 3)
    w = np.ones((1, 1, 2, 2), np.float32)
    y, _ = orc.conv_fwd(x, w, None, 1, 0)
    assert y.reshape(2, 2).tolist() == [[1 + 2 + 4 + 5, 2 + 3 + 5 + 6], [4 + 5 + 7 + 8, 5 + 6 + 8 + 9]]
    y, _ = orc.conv_fwd(x, w, np.array([10], np.float32), 2, 1)
    # windows at rows/cols {-1,0} and {1,2}: (1), (2+3), (4+7), (5+6+8+9), each + 10
    assert y.reshape(2, 2).tolist() == [[11, 15], [21, 38]]


@pytest.mark.parametrize("shape", SHAPES)
def test_fwd_matches_torch_float64(orc, shape):
    x, w, b, _ = make(shape, 13)
    st, pad = shape[6], shape[7]
    y, y_abs = orc.conv_fwd(x, w, b, st, pad, exact=True)
    ref = F.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                   torch.from_numpy(b).double(), stride=st, padding=pad).numpy()
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * (1 + y_abs.max()))


@pytest.mark.parametrize("shape", SHAPES)
def test_delta_kernel_is_strided_shift(orc, shape):
    """A filter that is 1 at (c0, r0, s0) and 0 elsewhere copies the input
    shifted by (r0 - pad, s0 - pad) and subsampled by the stride."""
    N, C, H, W, Ko, R, st, pad = shape
    x, _, _, _ = make(shape, 14)
    P, Q = out_size(H, R, st, pad), out_size(W, R, st, pad)
    xp = np.zeros((N, C, H + 2 * pad, W + 2 * pad), np.float32)
    xp[:, :, pad:pad + H, pad:pad + W] = x
    for (c0, r0, s0) in [(0, 0, 0), (C - 1, R - 1, R - 1), (C // 2, R // 2, 0)]:
        w = np.zeros((1, C, R, R), np.float32)
        w[0, c0, r0, s0] = 1.0
        y, _ = orc.conv_fwd(x, w, None, st, pad)
        expect = xp[:, c0, r0:r0 + st * (P - 1) + 1:st, s0:s0 + st * (Q - 1) + 1:st]
        assert np.array_equal(y[:, 0], expect)


def tap_count_1d(size, R, st, pad):
    """How many (r, o) pairs with 0 <= r < R, 0 <= o < out read position i."""
    out = out_size(size, R, st, pad)
    cnt = np.zeros(size, np.int64)
    for o in range(out):
        for r in range(R):
            i = o * st + r - pad
            if 0 <= i < size:
                cnt[i] += 1
    return cnt


@pytest.mark.parametrize("shape", SHAPES)
def test_col2im_of_ones_is_tap_count(orc, shape):
    N, C, H, W, Ko, R, st, pad = shape
    ones = np.ones((N, C, H, W), np.float32)
    col = orc.im2col(ones, R, st, pad)
    assert col.shape == (C * R * R, N * out_size(H, R, st, pad) * out_size(W, R, st, pad))
    dx, _ = orc.col2im(col, ones.shape, R, st, pad)
    expect = np.outer(tap_count_1d(H, R, st, pad), tap_count_1d(W, R, st, pad))
    assert np.array_equal(dx, np.broadcast_to(expect, dx.shape).astype(np.float32))
    # a column matrix of ones also contains the padding reads, which col2im drops
    dx1, _ = orc.col2im(np.ones_like(col), ones.shape, R, st, pad)
    assert np.array_equal(dx1, dx)


@pytest.mark.parametrize("shape", SHAPES)
def test_col2im_is_adjoint_of_im2col(orc, shape):
    """<im2col(x), Y> == <x, col2im(Y)>, exactly, on small-integer tensors."""
    N, C, H, W, Ko, R, st, pad = shape
    x = synthetic.small_ints((N, C, H, W), 21)
    col = orc.im2col(x, R, st, pad, exact=True)
    Y = synthetic.small_ints(col.shape, 22)
    dx, _ = orc.col2im(Y, x.shape, R, st, pad, exact=True)
    lhs = int(np.sum(col.astype(np.int64) * Y.astype(np.int64)))
    rhs = int(np.sum(x.astype(np.int64) * dx.astype(np.int64)))
    assert lhs == rhs


@pytest.mark.parametrize("shape", SHAPES)
def test_im2col_column_is_patch(orc, shape):
    """Each column of the im2col matrix, reshaped to (C, R, R), is the patch the
    direct convolution multiplies with one filter."""
    N, C, H, W, Ko, R, st, pad = shape
    x, _, _, _ = make(shape, 15)
    P, Q = out_size(H, R, st, pad), out_size(W, R, st, pad)
    col = orc.im2col(x, R, st, pad)
    xp = np.zeros((N, C, H + 2 * pad, W + 2 * pad), np.float32)
    xp[:, :, pad:pad + H, pad:pad + W] = x
    for n, oh, ow in [(0, 0, 0), (N - 1, P - 1, Q - 1), (N // 2, P // 2, Q - 1)]:
        patch = xp[n, :, oh * st:oh * st + R, ow * st:ow * st + R]
        assert np.array_equal(col[:, (n * P + oh) * Q + ow].reshape(C, R, R), patch)


@pytest.mark.parametrize("shape", SHAPES)
def test_bwd_matches_torch_autograd(orc, shape):
    x, w, b, dy = make(shape, 16)
    st, pad = shape[6], shape[7]
    xt = torch.from_numpy(x).double().requires_grad_()
    wt = torch.from_numpy(w).double().requires_grad_()
    bt = torch.from_numpy(b).double().requires_grad_()
    F.conv2d(xt, wt, bt, stride=st, padding=pad).backward(torch.from_numpy(dy).double())
    dx, dx_abs = orc.conv_bwd_data(w, dy, x.shape, st, pad, exact=True)
    dw, dw_abs = orc.conv_bwd_filter(x, dy, w.shape, st, pad, exact=True)
    db, db_abs = orc.conv_bwd_bias(dy, exact=True)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=0, atol=1e-12 * (1 + dx_abs.max()))
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=0, atol=1e-12 * (1 + dw_abs.max()))
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=0, atol=1e-12 * (1 + db_abs.max()))


def abs_grads(x, w, dy, st, pad):
    """Torch float64 autograd of conv2d on |x| and |w| with upstream |dy|.

    Every term of the input gradient dx[i] = sum w*dy and of the filter
    gradient dw[j] = sum dy*x is a product of two such factors, so the
    per-element scale sum |a_k b_k| the tolerance uses is exactly the gradient
    of the convolution of the absolute values (padding taps read zero and
    contribute nothing, as in the page's col2im, which drops them).
    """
    xa = torch.from_numpy(np.abs(x)).double().requires_grad_()
    wa = torch.from_numpy(np.abs(w)).double().requires_grad_()
    F.conv2d(xa, wa, stride=st, padding=pad).backward(torch.from_numpy(np.abs(dy)).double())
    return xa.grad.numpy(), wa.grad.numpy()


@pytest.mark.parametrize("shape", SHAPES)
def test_bwd_abs_scales_match_torch(orc, shape):
    """The tolerance scales of both gradients (full and sampled forms) against
    torch's float64 autograd on absolute values."""
    x, w, b, dy = make(shape, 18)
    st, pad = shape[6], shape[7]
    dx_abs_ref, dw_abs_ref = abs_grads(x, w, dy, st, pad)
    _, dx_abs = orc.conv_bwd_data(w, dy, x.shape, st, pad, exact=True)
    _, dw_abs = orc.conv_bwd_filter(x, dy, w.shape, st, pad, exact=True)
    np.testing.assert_allclose(dx_abs, dx_abs_ref, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(dw_abs, dw_abs_ref, rtol=1e-12, atol=1e-300)
    fx = np.arange(x.size, dtype=np.int64)
    fw = np.arange(w.size, dtype=np.int64)
    _, dx_abs_at = orc.conv_bwd_data_at(w, dy, x.shape, st, pad, fx, exact=True)
    _, dw_abs_at = orc.conv_bwd_filter_at(x, dy, w.shape, st, pad, fw, exact=True)
    np.testing.assert_allclose(dx_abs_at, dx_abs_ref.ravel(), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(dw_abs_at, dw_abs_ref.ravel(), rtol=1e-12, atol=1e-300)


def test_bwd_abs_scale_hand_case(orc):
    """One input channel, one filter of ones, 3x3 image, k 2, stride 1, no pad:
    dx_abs is the tap-count map weighted by |dy| (closed form)."""
    x = np.zeros((1, 1, 3, 3), np.float32)
    w = np.ones((1, 1, 2, 2), np.float32)
    dy = np.array([[[[1, -2], [-3, 4]]]], np.float32)
    _, dx_abs = orc.conv_bwd_data(w, dy, x.shape, 1, 0, exact=True)
    expect = np.array([[1, 3, 2], [4, 10, 6], [3, 7, 4]], np.float64)
    assert np.array_equal(dx_abs[0, 0], expect)


@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[3], SHAPES[5]])
def test_bwd_central_differences(orc, shape):
    """L(x, W, b) = sum(conv(x, W, b) * R) is linear in each argument, so the
    central difference with step 1 equals the gradient up to fp64 rounding."""
    x, w, b, R_ = make(shape, 17)
    st, pad = shape[6], shape[7]
    x, w, b, R_ = (a.astype(np.float64) for a in (x, w, b, R_))

    def L(xx, ww, bb):
        return float(np.sum(orc.conv_fwd(xx, ww, bb, st, pad, exact=True)[0] * R_))

    dx, _ = orc.conv_bwd_data(w, R_, x.shape, st, pad, exact=True)
    dw, _ = orc.conv_bwd_filter(x, R_, w.shape, st, pad, exact=True)
    db, _ = orc.conv_bwd_bias(R_, exact=True)
    scale = 1.0 + float(np.abs(R_).sum() * (np.abs(x).max() + np.abs(w).max() + 1))
    for arr, grad, which in ((x, dx, 0), (w, dw, 1), (b, db, 2)):
        fd = np.empty_like(arr)
        for i in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[i] += 1.0
            minus[i] -= 1.0
            args_p = [x, w, b]
            args_m = [x, w, b]
            args_p[which], args_m[which] = plus, minus
            fd[i] = (L(*args_p) - L(*args_m)) / 2.0
        assert np.max(np.abs(fd - grad)) <= 1e-12 * scale, which


def test_bias_grad_is_total_sum(orc):
    dy = synthetic.small_ints((3, 5, 4, 6), 31)
    db, db_abs = orc.conv_bwd_bias(dy, exact=True)
    for k in range(5):
        assert db[k] == float(sum(int(v) for v in dy[:, k].ravel()))
        assert db_abs[k] == float(sum(abs(int(v)) for v in dy[:, k].ravel()))


@pytest.mark.parametrize("shape", SHAPES[:5])
def test_sampled_entries_match_full(orc, shape):
    """The *_at variants evaluate the same definitions at chosen indices."""
    x, w, b, dy = make(shape, 18)
    st, pad = shape[6], shape[7]
    y, y_abs = orc.conv_fwd(x, w, b, st, pad, exact=True)
    dx, dx_abs = orc.conv_bwd_data(w, dy, x.shape, st, pad, exact=True)
    dw, dw_abs = orc.conv_bwd_filter(x, dy, w.shape, st, pad, exact=True)
    g = np.random.default_rng(0)
    for full, full_abs, fn in (
        (y, y_abs, lambda f: orc.conv_fwd_at(x, w, b, st, pad, f, exact=True)),
        (dx, dx_abs, lambda f: orc.conv_bwd_data_at(w, dy, x.shape, st, pad, f, exact=True)),
        (dw, dw_abs, lambda f: orc.conv_bwd_filter_at(x, dy, w.shape, st, pad, f, exact=True)),
    ):
        flat = np.unique(np.concatenate([[0, full.size - 1], g.integers(0, full.size, 40)]))
        v, v_abs = fn(flat)
        np.testing.assert_allclose(v, full.ravel()[flat], rtol=0, atol=1e-12 * (1 + full_abs.max()))
        np.testing.assert_allclose(v_abs, full_abs.ravel()[flat], rtol=1e-12)
