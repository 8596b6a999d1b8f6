"""GPU parity of the training-step pieces and of the LeNet-5 step.

* relu_fwd, relu_bwd, grad_accum, add_bias (with and without ReLU, in place)
  and max pooling are bit-exact against the oracle (single fp32 operations or
  routing);
* bias_grad_rows and the contractions are within 1e-4 * sum|terms| + 1e-6;
* softmax_ce: fp32 exp/log/division carry a few ulp each, and the row sum adds
  one rounding per term, so |p_gpu - p| <= (cols + 8) * 2^-24 <= 1e-6 for
  cols <= 1000, and each row loss is within 4e-6 * (1 + |loss_i|) (its value,
  the max and log(s) each carry a few ulp); the batch sum adds one rounding per
  row on top: tolerance 1e-5 * sum_i (1 + |loss_i|).

The LeNet step is checked operation by operation ("teacher forced"): every
GPU output is compared with the oracle's result on the GPU's own inputs to
that operation, so no error propagates along the chain and every routing
decision (ReLU masks, pooling argmax) is taken on identical inputs on both
sides.  The whole step is then also compared end to end with the oracle's
fp32 program (a sanity bound), and graph replay against eager execution (bit
for bit: every kernel is deterministic).
"""
import numpy as np
import pytest

import oracle.lenet as olenet
import synthetic
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


def ce_tol_check(dz, loss, ref_grad, ref_loss_rows, what):
    err = np.abs(dz.astype(np.float64) - ref_grad)
    assert (err <= 1e-6).all(), "%s: dlogits off by %g" % (what, err.max())
    tol = 1e-5 * np.sum(1.0 + np.abs(ref_loss_rows))
    assert abs(float(loss) - ref_loss_rows.sum()) <= tol, (what, float(loss), ref_loss_rows.sum(), tol)


# ---------------------------------------------------------------------------
# pieces

COUNTS = [1, 3, 4, 5, 1023, 4096, 100003]


@pytest.mark.parametrize("n", COUNTS)
def test_relu_and_grad_bit_exact(cb, orc, n):
    x = synthetic.normal((n,), 900 + n % 97)
    x[: min(n, 3)] = 0.0
    g = synthetic.normal((n,), 901 + n % 89)
    xd, gd = dev_in(x), dev_in(g)
    y = dev_out((n,))
    cb.relu_fwd(xd.t, y.t)
    dx = dev_out((n,))
    cb.relu_bwd(gd.t, xd.t, dx.t)
    cb.check()
    assert y.guards_intact() and dx.guards_intact()
    assert np.array_equal(y.numpy(), orc.relu(x))
    assert np.array_equal(dx.numpy(), orc.relu_grad(g, x))
    # in place, and the mask taken from the output
    z = dev_in(x)
    cb.relu_fwd(z.t, z.t)
    cb.relu_bwd(gd.t, z.t, gd.t)
    cb.check()
    assert np.array_equal(z.numpy(), orc.relu(x))
    assert np.array_equal(gd.numpy(), orc.relu_grad(g, x))


@pytest.mark.parametrize("n", COUNTS)
def test_grad_accum_bit_exact(cb, orc, n):
    a = synthetic.normal((n,), 910)
    g = synthetic.normal((n,), 911)
    ad = dev_in(a)
    cb.grad_accum(ad.t, dev_in(g).t)
    cb.check()
    assert np.array_equal(ad.numpy(), orc.grad_accum(a, g))


@pytest.mark.parametrize("rows,cols", [(1, 1), (64, 120), (64, 84), (64, 10), (7, 33), (300, 1000)])
def test_add_bias_and_bias_grad(cb, orc, rows, cols):
    A = synthetic.normal((rows, cols), 920)
    b = synthetic.normal((cols,), 921)
    out = dev_out((rows, cols))
    cb.add_bias(dev_in(A).t, dev_in(b).t, out=out.t)
    relu_out = dev_out((rows, cols))
    cb.add_bias(dev_in(A).t, dev_in(b).t, out=relu_out.t, relu=True)
    inplace = dev_in(A)
    cb.add_bias(inplace.t, dev_in(b).t, out=inplace.t, relu=True)
    db = dev_out((cols,))
    cb.bias_grad_rows(dev_in(A).t, db=db.t)
    cb.check()
    assert out.guards_intact() and relu_out.guards_intact() and db.guards_intact()
    assert np.array_equal(out.numpy(), orc.add_bias(A, b))
    assert np.array_equal(relu_out.numpy(), orc.relu(orc.add_bias(A, b)))
    assert np.array_equal(inplace.numpy(), orc.relu(orc.add_bias(A, b)))
    ref, ref_abs = orc.bias_grad_rows(A)
    assert_within_tol(db.numpy(), ref, ref_abs, "bias_grad_rows %dx%d" % (rows, cols))


@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 10), (64, 10), (33, 7), (100, 1000), (2000, 10)])
def test_softmax_ce(cb, orc, rows, cols):
    z = synthetic.normal((rows, cols), 930) * np.float32(4.0)
    labels = synthetic.rng(931).integers(0, cols, size=rows).astype(np.int32)
    dz = dev_out((rows, cols))
    probs = dev_out((rows, cols))
    loss = dev_out((1,))
    cb.softmax_ce(dev_in(z).t, dev_in(labels).t, dlogits=dz.t, loss=loss.t, probs=probs.t)
    cb.check()
    assert dz.guards_intact() and probs.guards_intact() and loss.guards_intact()
    g, l = orc.softmax_ce(z, labels)
    ce_tol_check(dz.numpy(), loss.numpy()[0], g, l, "softmax_ce %dx%d" % (rows, cols))
    assert (np.abs(probs.numpy() - orc.softmax(z)) <= 1e-6).all()


def test_softmax_ce_label_out_of_range_reported(cb):
    z = dev_in(synthetic.normal((4, 10), 940))
    labels = dev_in(np.array([1, 2, 10, 3], np.int32))
    cb.softmax_ce(z.t, labels.t)
    with pytest.raises(cb.ConvError) as e:
        cb.check()
    assert e.value.code == -10
    cb.check()        # the error word was cleared


# ---------------------------------------------------------------------------
# the LeNet-5 step

def _np(t):
    return t.detach().cpu().numpy()


@pytest.fixture(scope="module")
def lenet_run(cb):
    """One eager step on the workload batch; keeps the pre-step parameters."""
    from im2col_convolution_tiled_gb300.lenet import LeNet5
    params = synthetic.lenet_params()
    x, labels = synthetic.lenet_batch()
    net = LeNet5(params, batch=x.shape[0])
    net.load_batch(x, labels)
    net.run()
    cb.check()
    return params, x, labels, net


def test_lenet_step_operation_by_operation(cb, orc, lenet_run):
    params, x, labels, net = lenet_run
    t = {k: _np(v) for k, v in net.t.items()}
    G = {k: _np(v) for k, v in net.G.items()}
    P0 = params
    c1, c2 = synthetic.LENET
    tol = assert_within_tol

    # forward: conv + bias + ReLU in one pass; ReLU is 1-Lipschitz, so the
    # contraction tolerance carries over to max(0, .) of the oracle's result
    y1, y1_abs = orc.conv_fwd(x, P0["conv1_w"], P0["conv1_b"], c1.stride, c1.pad)
    tol(t["a1"], orc.relu(y1), y1_abs, "conv1 fwd + relu")
    assert (t["a1"] >= 0).all()
    p1, i1 = orc.maxpool_fwd(t["a1"], *c1.pool)
    assert np.array_equal(t["p1"], p1) and np.array_equal(t["i1"], i1)
    y2, y2_abs = orc.conv_fwd(t["p1"], P0["conv2_w"], P0["conv2_b"], c2.stride, c2.pad)
    tol(t["a2"], orc.relu(y2), y2_abs, "conv2 fwd + relu")
    p2, i2 = orc.maxpool_fwd(t["a2"], *c2.pool)
    assert np.array_equal(t["p2"], p2) and np.array_equal(t["i2"], i2)
    # linear layers: bias (and ReLU) in the matmul's epilogue (its bit-identity
    # with matmul + add_bias is tests/test_gpu_matmul_fused.py's); here against
    # the oracle's fp64 product plus bias, within the product's tolerance
    # widened by |b| (one fp32 rounding of the addition)
    h = t["p2"].reshape(x.shape[0], -1)
    for i, out in ((1, "h1"), (2, "h2"), (3, "z3")):
        C, C_abs = orc.matmul(h, P0["fc%d_w" % i], 0, exact=True)
        b = P0["fc%d_b" % i].astype(np.float64)
        ref = C + b
        tol(t[out], np.maximum(ref, 0.0) if i < 3 else ref, C_abs + np.abs(b), "fc%d" % i)
        if i < 3:
            assert (t[out] >= 0).all()
        h = t[out]
    g, l = orc.softmax_ce(t["z3"], labels)
    ce_tol_check(t["dz3"], t["loss"][0], g, l, "lenet softmax_ce")

    # backward: linear layers
    for i in (3, 2, 1):
        hin = t["h%d" % (i - 1)] if i > 1 else t["p2"].reshape(x.shape[0], -1)
        dz = t["dz%d" % i]
        dh = t["dh%d" % (i - 1)] if i > 1 else t["df"]
        tol(G["fc%d_w" % i], *orc.matmul(hin, dz, 1), "dW fc%d" % i)
        tol(G["fc%d_b" % i], *orc.bias_grad_rows(dz), "db fc%d" % i)
        tol(dh, *orc.matmul(dz, P0["fc%d_w" % i], 2), "dX fc%d" % i)
        if i > 1:
            assert np.array_equal(t["dz%d" % (i - 1)], orc.relu_grad(dh, t["h%d" % (i - 1)])), i
    # conv blocks: the pooled gradient routed to the ReLU output (bit-exact),
    # then the convolution gradients with the ReLU mask fused in, against the
    # oracle's relu_grad followed by its backward convolution
    dp2 = t["df"].reshape(t["p2"].shape)
    assert np.array_equal(t["da2"], orc.maxpool_bwd(dp2, t["i2"], t["a2"].shape))
    dy2 = orc.relu_grad(t["da2"], t["a2"])
    tol(G["conv2_w"], *orc.conv_bwd_filter(t["p1"], dy2, P0["conv2_w"].shape, c2.stride, c2.pad), "dW conv2")
    tol(G["conv2_b"], *orc.conv_bwd_bias(dy2), "db conv2")
    tol(t["dp1"], *orc.conv_bwd_data(P0["conv2_w"], dy2, t["p1"].shape, c2.stride, c2.pad), "dX conv2")
    assert np.array_equal(t["da1"], orc.maxpool_bwd(t["dp1"], t["i1"], t["a1"].shape))
    dy1 = orc.relu_grad(t["da1"], t["a1"])
    tol(G["conv1_w"], *orc.conv_bwd_filter(x, dy1, P0["conv1_w"].shape, c1.stride, c1.pad), "dW conv1")
    tol(G["conv1_b"], *orc.conv_bwd_bias(dy1), "db conv1")

    # SGD, bit-exact on the GPU's own gradients
    lr, clip = synthetic.LENET_SGD
    for k in synthetic.LENET_PARAMS:
        assert np.array_equal(_np(net.P[k]), orc.sgd(P0[k], G[k], lr, clip)), k


def test_lenet_step_end_to_end(orc, lenet_run):
    """Against the oracle's fp32 program run on its own: a bound on the whole
    chain.  A ReLU input within rounding of 0 may take the other side on the
    two paths and move one term of a filter gradient, which SGD scales by
    lr = 0.01, hence the absolute bound on the parameters."""
    params, x, labels, net = lenet_run
    new, loss, _ = olenet.step(params, x, labels, orc=orc)
    assert abs(float(net.t["loss"].item()) - loss) <= 1e-4 * abs(loss)
    for k in synthetic.LENET_PARAMS:
        assert np.allclose(_np(net.P[k]), new[k], rtol=0, atol=1e-4), k


def test_lenet_graph_replay_matches_eager(cb):
    from im2col_convolution_tiled_gb300.lenet import LeNet5
    params = synthetic.lenet_params()
    x, labels = synthetic.lenet_batch()
    eager = LeNet5(params)
    eager.load_batch(x, labels)
    for _ in range(3):
        eager.run()
    graphed = LeNet5(params)
    graphed.load_batch(x, labels)
    graphed.capture()          # one eager warm-up step, then the captured one (not yet run)
    graphed.replay()
    graphed.replay()
    cb.check()
    for k in synthetic.LENET_PARAMS:
        assert np.array_equal(_np(eager.P[k]), _np(graphed.P[k])), k
    assert float(eager.t["loss"].item()) == float(graphed.t["loss"].item())
