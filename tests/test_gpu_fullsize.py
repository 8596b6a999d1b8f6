"""Full-size parity on the AlexNet-shaped batch-128 layers the benchmark times,
in the same launch configuration: every GPU output is computed in full, and a
sample of it (first and last elements plus random positions) is checked
against the oracle evaluated one element at a time.  Max pooling, bias
gradient, SGD and im2col are checked in full (they are cheap for the oracle or
checked image by image)."""
import numpy as np
import pytest

import synthetic
from tests.gpu_helpers import assert_within_tol

pytestmark = pytest.mark.gpu

SAMPLES = 384


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


def sample_idx(size, seed):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 1, size - 2, size - 1], g.integers(0, size, SAMPLES)]))


@pytest.mark.parametrize("L", synthetic.ALEXNET, ids=lambda L: L.name)
def test_alexnet_layer_sampled(cb, orc, L):
    import torch
    x, w, b, dy = L.make()
    b = synthetic.normal(b.shape, L.seed_base + 7, std=0.1)     # exercise the bias add
    xt, wt, bt, dyt = (torch.from_numpy(a).cuda() for a in (x, w, b, dy))
    y = cb.conv_fwd(xt, wt, bt, L.stride, L.pad)
    dx = cb.conv_bwd_data(wt, dyt, L.x_shape, L.stride, L.pad)
    dw = cb.conv_bwd_filter(xt, dyt, L.w_shape, L.stride, L.pad)
    db = cb.conv_bwd_bias(dyt)
    dw2, db2 = cb.conv_bwd_filter_bias(xt, dyt, L.w_shape, L.stride, L.pad)   # the bench's fused call
    cb.check()
    y, dx, dw, db, dw2, db2 = (t.cpu().numpy() for t in (y, dx, dw, db, dw2, db2))

    f = sample_idx(y.size, 1)
    ref, ref_abs = orc.conv_fwd_at(x, w, b, L.stride, L.pad, f)
    assert_within_tol(y.ravel()[f], ref, ref_abs, L.name + " fwd")
    f = sample_idx(dx.size, 2)
    ref, ref_abs = orc.conv_bwd_data_at(w, dy, L.x_shape, L.stride, L.pad, f)
    assert_within_tol(dx.ravel()[f], ref, ref_abs, L.name + " bwd_data")
    f = sample_idx(dw.size, 3)[:160]
    ref, ref_abs = orc.conv_bwd_filter_at(x, dy, L.w_shape, L.stride, L.pad, f)
    assert_within_tol(dw.ravel()[f], ref, ref_abs, L.name + " bwd_filter")
    assert_within_tol(dw2.ravel()[f], ref, ref_abs, L.name + " bwd_filter (fused with bias)")
    ref, ref_abs = orc.conv_bwd_bias(dy)
    assert_within_tol(db, ref, ref_abs, L.name + " bwd_bias")
    assert_within_tol(db2, ref, ref_abs, L.name + " bwd_bias (fused with filter)")
    for a in (y, dx, dw, dw2, db2):
        assert np.isfinite(a).all()


@pytest.mark.parametrize("L", [L for L in synthetic.ALEXNET if L.pool], ids=lambda L: L.name)
def test_alexnet_pool_full(cb, orc, L):
    import torch
    k, s = L.pool
    xp = synthetic.pool_input(L)
    y_ref, i_ref = orc.maxpool_fwd(xp, k, s)
    y, idx = cb.maxpool2d_fwd(torch.from_numpy(xp).cuda(), k, s)
    dyp = synthetic.pool_grad(y_ref.shape, L.seed_base + 20)
    dx = cb.maxpool2d_bwd(torch.from_numpy(dyp).cuda(), idx, xp.shape, k, s)
    cb.check()
    assert np.array_equal(y.cpu().numpy(), y_ref)
    assert np.array_equal(idx.cpu().numpy(), i_ref)
    assert np.array_equal(dx.cpu().numpy(), orc.maxpool_bwd(dyp, i_ref, xp.shape))


def test_alexnet_sgd_full(cb, orc):
    import torch
    n = sum(int(np.prod(L.w_shape)) + L.outC for L in synthetic.ALEXNET)
    p = synthetic.normal((n,), 77)
    g = synthetic.normal((n,), 78, std=2.0)
    pt = torch.from_numpy(p).cuda()
    cb.sgd_step(pt, torch.from_numpy(g).cuda(), *synthetic.SGD_LR_CLIP)
    cb.check()
    assert np.array_equal(pt.cpu().numpy(), orc.sgd(p, g, *synthetic.SGD_LR_CLIP))


def test_alexnet_conv1_im2col_per_image(cb, orc):
    """Full-batch im2col of conv1 (140M entries): the columns of image n equal
    the oracle's im2col of image n alone, bit for bit (checked for 2 images)."""
    import torch
    L = synthetic.ALEXNET_CONV1
    x, _, _, _ = L.make()
    col = cb.im2col(torch.from_numpy(x).cuda(), L.k, L.stride, L.pad)
    cb.check()
    PQ = L.outH * L.outW
    for n in (0, L.batch - 1):
        ref = orc.im2col(x[n:n + 1], L.k, L.stride, L.pad)
        got = col[:, n * PQ:(n + 1) * PQ].cpu().numpy()
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("L", list(synthetic.LENET) + [synthetic.SINGLE], ids=lambda L: L.name)
def test_small_workloads_full(cb, orc, L):
    """The single-layer and LeNet workloads at their own batch, in full."""
    import torch
    x, w, b, dy = L.make()
    xt, wt, bt, dyt = (torch.from_numpy(a).cuda() for a in (x, w, b, dy))
    y = cb.conv_fwd(xt, wt, bt, L.stride, L.pad)
    dx = cb.conv_bwd_data(wt, dyt, L.x_shape, L.stride, L.pad)
    dw = cb.conv_bwd_filter(xt, dyt, L.w_shape, L.stride, L.pad)
    db = cb.conv_bwd_bias(dyt)
    cb.check()
    assert_within_tol(y.cpu().numpy(), *orc.conv_fwd(x, w, b, L.stride, L.pad), L.name + " fwd")
    assert_within_tol(dx.cpu().numpy(), *orc.conv_bwd_data(w, dy, L.x_shape, L.stride, L.pad), L.name + " dgrad")
    assert_within_tol(dw.cpu().numpy(), *orc.conv_bwd_filter(x, dy, L.w_shape, L.stride, L.pad), L.name + " wgrad")
    assert_within_tol(db.cpu().numpy(), *orc.conv_bwd_bias(dy), L.name + " bias")
