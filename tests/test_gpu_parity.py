"""GPU parity: every libconv_b200 entry point against the CPU oracle on the same
seeded inputs.  Contractions must be within 1e-4 * sum|a_k b_k| + 1e-6 per
element; im2col, col2im on integer data, max pooling (values, indices and
gradient routing) and SGD must be bit-exact.  Outputs sit between canary
guard zones and inputs between NaN guard zones."""
import numpy as np
import pytest

import synthetic
from oracle import out_size
from tests.gpu_helpers import assert_within_tol, dev_in, dev_out

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


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.get()


def sync_check(cb):
    cb.check()


# ---------------------------------------------------------------------------
# flagged matmul

MM_SHAPES = [(1, 1, 1), (5, 3, 7), (16, 25, 16), (127, 25, 129), (128, 32, 128), (200, 150, 300),
             (64, 363, 1024), (1024, 64, 16), (300, 1000, 257), (129, 4096, 40)]


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("M,K,N", MM_SHAPES)
def test_matmul(cb, orc, M, K, N, flags):
    A, B = synthetic.matmul_case(M, K, N, flags)
    ref, ref_abs = orc.matmul(A, B, flags)
    a, b = dev_in(A), dev_in(B)
    c = dev_out((M, N))
    cb.matmul(a.t, b.t, flags, C=c.t)
    sync_check(cb)
    assert c.guards_intact()
    assert_within_tol(c.numpy(), ref, ref_abs, "matmul %dx%dx%d f%d" % (M, K, N, flags))


def test_matmul_small_ints_exact(cb, orc):
    """Small-integer operands: every product and sum is exact in the 3xTF32
    split and in fp32, so the result must equal the oracle bit for bit."""
    for flags in range(4):
        A = synthetic.small_ints((300, 77) if not flags & 1 else (77, 300), 31)
        B = synthetic.small_ints((77, 129) if not flags & 2 else (129, 77), 32)
        ref, _ = orc.matmul(A, B, flags)
        c = cb.matmul(dev_in(A).t, dev_in(B).t, flags)
        sync_check(cb)
        assert np.array_equal(c.cpu().numpy(), ref)


# ---------------------------------------------------------------------------
# convolution: small shapes (full oracle) covering ragged tiles, padding,
# strides above and below the filter size, 1x1 filters and empty phases

CONV_SHAPES = [
    # N, C, H, W, K, R, stride, pad
    (4, 1, 28, 28, 6, 5, 1, 0),        # the single-layer workload, in full
    (2, 3, 9, 9, 4, 3, 2, 1),
    (3, 2, 11, 13, 5, 3, 1, 1),
    (2, 3, 23, 23, 64, 11, 4, 2),      # AlexNet conv1 geometry, small image
    (1, 64, 27, 27, 192, 5, 1, 2),     # AlexNet conv2 at batch 1
    (1, 192, 13, 13, 384, 3, 1, 1),    # AlexNet conv3 at batch 1 (two column tiles)
    (2, 5, 10, 10, 3, 1, 1, 0),        # 1x1 filter
    (2, 4, 12, 12, 7, 3, 4, 0),        # stride > filter: phases with no tap
    (2, 3, 7, 7, 33, 2, 3, 1),
    (1, 20, 6, 6, 300, 3, 1, 1),       # 300 filters: two 192-wide tiles, ragged
    (2, 16, 9, 9, 40, 3, 2, 1),        # 16 channels (one 16-wide tap group), 40 filters
    (1, 48, 7, 7, 24, 3, 1, 1),        # 48 channels (per-element order), 24 filters
    (1, 96, 8, 8, 17, 2, 2, 0),        # three 32-channel chunks, 17 filters
    # 16 x 35 x 35 = 19600 rows: 154 row tiles, more than one wave on any GB300, so the trailing tiles of the
    # 192-column GEMMs are split along K and their partial tiles added by the reduce kernel
    (16, 64, 35, 35, 192, 3, 1, 1),    # forward: 192 filters
    (16, 192, 35, 35, 64, 3, 1, 1),    # input gradient: 192 columns
    (2, 24, 11, 11, 100, 3, 1, 1),     # 100 filters: 128-wide filter-gradient tiles (A in tensor memory)
    # input gradient stored as one float4 (stride 4) / float2 (stride 2) per (channel, row phase), with a
    # last super-row cut by the image's bottom edge (H % stride != 0)
    (2, 3, 30, 28, 8, 5, 4, 1),
    (1, 5, 11, 10, 6, 3, 2, 1),
    # strided input gradients on the padding-aligned super-pixel grid (phase offset pad mod stride): two float2
    # stores per (channel, row phase) with the image's left and right edges cutting a pair (W % 4 = 0 and 2),
    # and pads of at least the stride
    (2, 3, 28, 28, 16, 11, 4, 2),
    (2, 3, 26, 30, 8, 11, 4, 2),
    (1, 4, 17, 17, 5, 7, 2, 3),
    (1, 3, 20, 20, 8, 11, 4, 6),
    (1, 3, 24, 24, 8, 7, 4, 3),        # stride 4, pad 3: the vector space-to-depth copy at offset 1
    # 160 patch-kernel tiles: a round on 152 SMs plus 8 tiles, which are split along their channel chunks and
    # summed by the reduce kernel (forward: 3 chunks of x, 64 columns; input gradient: 2 chunks of dy, 96 columns)
    (80, 96, 16, 16, 64, 3, 1, 1),
    # input gradient with 5 chunks of dy on 32 columns: the trailing tiles split into five pieces
    (80, 32, 16, 16, 160, 3, 1, 1),
    # 40 channels: a last chunk of 8 channels whose stages take two taps each (forward), split from the full
    # chunk in the trailing tiles (pieces of 9 and 5 stages)
    (80, 40, 16, 16, 64, 3, 1, 1),
]


def conv_inputs(shape, seed):
    N, C, H, W, K, R, st, pad = shape
    P, Q = out_size(H, R, st, pad), out_size(W, R, st, pad)
    x = synthetic.normal((N, C, H, W), seed + 1)
    w = synthetic.normal((K, C, R, R), seed + 2, std=float(1 / np.sqrt(C * R * R)))
    b = synthetic.normal((K,), seed + 3, std=0.1)
    dy = synthetic.normal((N, K, P, Q), seed + 4)
    return x, w, b, dy


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_conv_fwd(cb, orc, shape):
    x, w, b, _ = conv_inputs(shape, 100)
    st, pad = shape[6], shape[7]
    ref, ref_abs = orc.conv_fwd(x, w, b, st, pad)
    y = dev_out(ref.shape)
    cb.conv_fwd(dev_in(x).t, dev_in(w).t, dev_in(b).t, st, pad, y=y.t)
    sync_check(cb)
    assert y.guards_intact()
    assert_within_tol(y.numpy(), ref, ref_abs, "conv_fwd %s" % (shape,))


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_conv_fwd_relu(cb, orc, shape):
    """conv_fwd_relu: within tolerance of max(0, oracle) (ReLU is 1-Lipschitz),
    and bit-for-bit max(0, .) of conv_fwd's own output (same kernels, same
    sums: the ReLU is only applied in the epilogue)."""
    x, w, b, _ = conv_inputs(shape, 120)
    st, pad = shape[6], shape[7]
    ref, ref_abs = orc.conv_fwd(x, w, b, st, pad)
    yr = dev_out(ref.shape)
    xd, wd, bd = dev_in(x), dev_in(w), dev_in(b)
    cb.conv_fwd(xd.t, wd.t, bd.t, st, pad, y=yr.t, relu=True)
    y = cb.conv_fwd(xd.t, wd.t, bd.t, st, pad)
    sync_check(cb)
    assert yr.guards_intact()
    got = yr.numpy()
    assert_within_tol(got, orc.relu(ref), ref_abs, "conv_fwd_relu %s" % (shape,))
    assert np.array_equal(got, orc.relu(y.cpu().numpy()))


def test_conv_fwd_without_bias(cb, orc):
    shape = CONV_SHAPES[2]
    x, w, _, _ = conv_inputs(shape, 110)
    ref, ref_abs = orc.conv_fwd(x, w, None, shape[6], shape[7])
    y = cb.conv_fwd(dev_in(x).t, dev_in(w).t, None, shape[6], shape[7])
    sync_check(cb)
    assert_within_tol(y.cpu().numpy(), ref, ref_abs, "conv_fwd no bias")


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_conv_bwd_data(cb, orc, shape):
    x, w, _, dy = conv_inputs(shape, 200)
    st, pad = shape[6], shape[7]
    ref, ref_abs = orc.conv_bwd_data(w, dy, x.shape, st, pad)
    dx = dev_out(x.shape)
    cb.conv_bwd_data(dev_in(w).t, dev_in(dy).t, x.shape, st, pad, dx=dx.t)
    sync_check(cb)
    assert dx.guards_intact()
    assert_within_tol(dx.numpy(), ref, ref_abs, "conv_bwd_data %s" % (shape,))


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_conv_bwd_filter(cb, orc, shape):
    x, w, _, dy = conv_inputs(shape, 300)
    st, pad = shape[6], shape[7]
    ref, ref_abs = orc.conv_bwd_filter(x, dy, w.shape, st, pad)
    dw = dev_out(w.shape)
    cb.conv_bwd_filter(dev_in(x).t, dev_in(dy).t, w.shape, st, pad, dw=dw.t)
    sync_check(cb)
    assert dw.guards_intact()
    assert_within_tol(dw.numpy(), ref, ref_abs, "conv_bwd_filter %s" % (shape,))


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_conv_bwd_filter_bias(cb, orc, shape):
    """The fused entry point: dw as conv_bwd_filter, db summed in the same pass over dy."""
    x, w, _, dy = conv_inputs(shape, 350)
    st, pad = shape[6], shape[7]
    ref_w, ref_w_abs = orc.conv_bwd_filter(x, dy, w.shape, st, pad)
    ref_b, ref_b_abs = orc.conv_bwd_bias(dy)
    dw, db = dev_out(w.shape), dev_out(ref_b.shape)
    cb.conv_bwd_filter_bias(dev_in(x).t, dev_in(dy).t, w.shape, st, pad, dw=dw.t, db=db.t)
    sync_check(cb)
    assert dw.guards_intact() and db.guards_intact()
    assert_within_tol(dw.numpy(), ref_w, ref_w_abs, "conv_bwd_filter_bias dw %s" % (shape,))
    assert_within_tol(db.numpy(), ref_b, ref_b_abs, "conv_bwd_filter_bias db %s" % (shape,))


@pytest.mark.parametrize("shape", CONV_SHAPES)
def test_conv_bwd_relu_fused(cb, orc, shape):
    """conv_bwd_data_relu and conv_bwd_filter_bias_relu: the ReLU gradient
    (nn_relu_grad) applied where dy is read.  Against the oracle's relu_grad
    followed by its backward convolution, within the contraction tolerance;
    the filter and bias gradients also bit for bit equal to the unfused call
    on relu_bwd's output (same kernels, same sums)."""
    x, w, _, dy = conv_inputs(shape, 500)
    st, pad = shape[6], shape[7]
    a = synthetic.relu_normal(dy.shape, 501)          # a ReLU output: about half exact zeros
    g = orc.relu_grad(dy, a)
    ref_x, ref_x_abs = orc.conv_bwd_data(w, g, x.shape, st, pad)
    ref_w, ref_w_abs = orc.conv_bwd_filter(x, g, w.shape, st, pad)
    ref_b, ref_b_abs = orc.conv_bwd_bias(g)
    xd, wd, dyd, ad = dev_in(x), dev_in(w), dev_in(dy), dev_in(a)
    dx, dw, db = dev_out(x.shape), dev_out(w.shape), dev_out(ref_b.shape)
    cb.conv_bwd_data(wd.t, dyd.t, x.shape, st, pad, dx=dx.t, relu_mask=ad.t)
    cb.conv_bwd_filter_bias(xd.t, dyd.t, w.shape, st, pad, dw=dw.t, db=db.t, relu_mask=ad.t)
    gd = cb.relu_bwd(dyd.t, ad.t)
    dw0, db0 = cb.conv_bwd_filter_bias(xd.t, gd, w.shape, st, pad)
    sync_check(cb)
    assert dx.guards_intact() and dw.guards_intact() and db.guards_intact()
    assert_within_tol(dx.numpy(), ref_x, ref_x_abs, "conv_bwd_data_relu %s" % (shape,))
    assert_within_tol(dw.numpy(), ref_w, ref_w_abs, "conv_bwd_filter_bias_relu dw %s" % (shape,))
    assert_within_tol(db.numpy(), ref_b, ref_b_abs, "conv_bwd_filter_bias_relu db %s" % (shape,))
    assert np.array_equal(dw.numpy(), dw0.cpu().numpy()) and np.array_equal(db.numpy(), db0.cpu().numpy())


@pytest.mark.parametrize("shape", CONV_SHAPES[:4])
def test_conv_bwd_bias(cb, orc, shape):
    _, _, _, dy = conv_inputs(shape, 400)
    ref, ref_abs = orc.conv_bwd_bias(dy)
    db = dev_out(ref.shape)
    cb.conv_bwd_bias(dev_in(dy).t, db=db.t)
    sync_check(cb)
    assert db.guards_intact()
    assert_within_tol(db.numpy(), ref, ref_abs, "conv_bwd_bias %s" % (shape,))


def test_conv_small_ints_exact(cb, orc):
    """Integer data and filters: all three GEMMs must match bit for bit."""
    shape = (2, 3, 11, 11, 8, 3, 2, 1)
    N, C, H, W, K, R, st, pad = shape
    P = out_size(H, R, st, pad)
    x = synthetic.small_ints((N, C, H, W), 41)
    w = synthetic.small_ints((K, C, R, R), 42)
    dy = synthetic.small_ints((N, K, P, P), 43)
    y = cb.conv_fwd(dev_in(x).t, dev_in(w).t, None, st, pad)
    dx = cb.conv_bwd_data(dev_in(w).t, dev_in(dy).t, x.shape, st, pad)
    dw = cb.conv_bwd_filter(dev_in(x).t, dev_in(dy).t, w.shape, st, pad)
    db = cb.conv_bwd_bias(dev_in(dy).t)
    sync_check(cb)
    assert np.array_equal(y.cpu().numpy(), orc.conv_fwd(x, w, None, st, pad)[0])
    assert np.array_equal(dx.cpu().numpy(), orc.conv_bwd_data(w, dy, x.shape, st, pad)[0])
    assert np.array_equal(dw.cpu().numpy(), orc.conv_bwd_filter(x, dy, w.shape, st, pad)[0])
    assert np.array_equal(db.cpu().numpy(), orc.conv_bwd_bias(dy)[0])


def test_bwd_filter_and_bias_deterministic(cb):
    shape = CONV_SHAPES[3]
    x, w, _, dy = conv_inputs(shape, 500)
    xt, dyt = dev_in(x).t, dev_in(dy).t
    a = cb.conv_bwd_filter(xt, dyt, w.shape, shape[6], shape[7]).clone()
    b = cb.conv_bwd_filter(xt, dyt, w.shape, shape[6], shape[7])
    c1 = cb.conv_bwd_bias(dyt).clone()
    c2 = cb.conv_bwd_bias(dyt)
    sync_check(cb)
    assert bool((a == b).all()) and bool((c1 == c2).all())


# ---------------------------------------------------------------------------
# standalone im2col / col2im

IM2COL_SHAPES = CONV_SHAPES[:4] + [
    (2, 2, 5, 7, 1, 3, 1, 1),
    (1, 2, 40, 300, 1, 3, 1, 1),       # 300 columns: output-row bands of 3, the last one short
    (1, 1, 20, 500, 1, 5, 2, 2),       # stride 2, bands of 4 rows over 10
    (1, 2, 50, 400, 1, 11, 4, 2),      # conv1-like stride 4, bands of 3 rows over 11
    (3, 2, 19, 21, 1, 7, 2, 3),        # 7x7 stride 2: 4x4 taps per residue class, images grouped
    (1, 1, 11, 4000, 1, 11, 1, 0),     # staged band too wide for shared memory, odd row length
    (1, 1, 12, 4002, 1, 11, 1, 0),     # the same with a row length divisible by 4
]


@pytest.mark.parametrize("shape", IM2COL_SHAPES)
def test_im2col_bit_exact(cb, orc, shape):
    N, C, H, W, K, R, st, pad = shape
    x = synthetic.normal((N, C, H, W), 600)
    ref = orc.im2col(x, R, st, pad)
    col = dev_out(ref.shape)
    cb.im2col(dev_in(x).t, R, st, pad, col=col.t)
    sync_check(cb)
    assert col.guards_intact()
    assert np.array_equal(col.numpy(), ref)


@pytest.mark.parametrize("shape", IM2COL_SHAPES)
def test_col2im(cb, orc, shape):
    N, C, H, W, K, R, st, pad = shape
    P, Q = out_size(H, R, st, pad), out_size(W, R, st, pad)
    Y = synthetic.small_ints((C * R * R, N * P * Q), 700)
    ref, _ = orc.col2im(Y, (N, C, H, W), R, st, pad)
    dx = dev_out((N, C, H, W))
    cb.col2im(dev_in(Y).t, (N, C, H, W), R, st, pad, dx=dx.t)
    sync_check(cb)
    assert dx.guards_intact()
    assert np.array_equal(dx.numpy(), ref)                      # integer data: exact
    Yf = synthetic.normal(Y.shape, 701)
    ref, ref_abs = orc.col2im(Yf, (N, C, H, W), R, st, pad)
    got = cb.col2im(dev_in(Yf).t, (N, C, H, W), R, st, pad)
    sync_check(cb)
    assert_within_tol(got.cpu().numpy(), ref, ref_abs, "col2im float")


# ---------------------------------------------------------------------------
# max pooling and SGD (bit-exact)

POOL_CASES = [((4, 6, 28, 28), 2, 2), ((4, 16, 10, 10), 2, 2), ((2, 64, 55, 55), 3, 2), ((2, 192, 27, 27), 3, 2),
              ((1, 3, 9, 8), 2, 3), ((1, 2, 5, 5), 5, 1), ((3, 1, 7, 7), 1, 1),
              # backward owner blocks: S = 3 with k = S, odd widths whose last block runs past the row end,
              # windows wider than stride + 1, a 2-wide grid, stride 1, and stride 4 (plain gather kernel)
              ((2, 5, 11, 13), 3, 3), ((2, 4, 7, 9), 4, 2), ((1, 3, 4, 5), 3, 2), ((2, 3, 6, 6), 2, 1),
              ((1, 2, 13, 13), 3, 4),
              # forward column walker (3x3 and 2x2, stride 2): rows below the last window (H = 8), a narrow width
              ((2, 3, 8, 9), 3, 2), ((1, 2, 7, 4), 3, 2),
              # register walkers: odd sizes leave a row and a column outside every 2x2 window; a plane
              # whose single window row spans it all; a batch large enough for several row segments
              ((1, 3, 9, 11), 2, 2), ((3, 2, 3, 17), 3, 2), ((16, 64, 55, 55), 3, 2)]


@pytest.mark.parametrize("shape,k,s", POOL_CASES)
def test_maxpool(cb, orc, shape, k, s):
    x = synthetic.relu_normal(shape, 800)         # half zeros: ties everywhere
    y_ref, i_ref = orc.maxpool_fwd(x, k, s)
    y, idx = dev_out(y_ref.shape), dev_out(y_ref.shape, "int32")
    cb.maxpool2d_fwd(dev_in(x).t, k, s, y=y.t, idx=idx.t)
    sync_check(cb)
    assert y.guards_intact() and idx.guards_intact()
    assert np.array_equal(y.numpy(), y_ref)
    assert np.array_equal(idx.numpy(), i_ref)
    dy = synthetic.normal(y_ref.shape, 801)
    dx_ref = orc.maxpool_bwd(dy, i_ref, shape)
    dx = dev_out(shape)
    cb.maxpool2d_bwd(dev_in(dy).t, idx.t, shape, k, s, dx=dx.t)
    sync_check(cb)
    assert dx.guards_intact()
    assert np.array_equal(dx.numpy(), dx_ref)


@pytest.mark.parametrize("count", [1, 3, 4, 61706, 10007, 1 << 20])
def test_sgd(cb, orc, count):
    p = synthetic.normal((count,), 900)
    g = synthetic.normal((count,), 901, std=2.0)
    ref = orc.sgd(p, g, 0.01, 1.0)
    pt = dev_in(p)
    cb.sgd_step(pt.t, dev_in(g).t, 0.01, 1.0)
    sync_check(cb)
    assert pt.guards_intact()
    assert np.array_equal(pt.numpy(), ref)
