"""CPU oracle of one LeNet-5 training step, composed from the oracle's own
operations.  TEST INFRASTRUCTURE: only the tests, the smoke check and the
CPU-baseline leg of the benchmark use it.

Network (page "DirectCompute Neural Network Engine", sections "LeNet on
MNIST", "Convolution: The im2col Approach" and the shader tables; the batch,
padding and widths follow the LeNet-5 workload of the benchmark):

    x (B,1,28,28) -> conv 6@5x5 pad 2 -> ReLU -> maxpool 2/2
                  -> conv 16@5x5       -> ReLU -> maxpool 2/2 -> flatten 400
                  -> linear 400->120 -> ReLU -> linear 120->84 -> ReLU
                  -> linear 84->10 -> softmax + cross-entropy against labels

Backward is the chain rule through the same operations in reverse, with the
conventions the page's shaders give:
  * a linear layer is Y = X W + b (W stored in x out, bias by row broadcast);
    dW = X^T dY (matmul flag 1), dX = dY W^T (matmul flag 2), db = row sums;
  * ReLU's gradient is grad * (x > 0);
  * the loss gradient is softmax - one_hot (no 1/batch factor), i.e. the
    gradient of the batch SUM of the row losses -log p[label];
  * max-pool backward routes each gradient to the saved argmax;
  * the first layer's input needs no gradient, so conv1's input gradient is
    not formed;
then SGD with clip on every parameter.

Each operation's result is rounded once to fp32 (the program the GPU runs,
evaluated operation by operation in exact arithmetic); ``exact=True`` keeps
the contractions and the loss gradient in double instead.
"""
from __future__ import annotations

import numpy as np

import synthetic

from . import get


def _r(a, exact):
    return a if exact else np.asarray(a, dtype=np.float32)


def step(params, x, labels, lr=None, clip=None, exact=False, orc=None):
    """One training step.  Returns (new_params, loss_sum, t) where t holds every
    intermediate tensor by name (forward activations, gradients, pool indices)."""
    o = orc or get()
    if lr is None or clip is None:
        lr, clip = synthetic.LENET_SGD
    c1, c2 = synthetic.LENET
    P = {k: np.asarray(v) for k, v in params.items()}
    t = {"x": x}
    f32 = lambda a: np.asarray(a, dtype=np.float32)

    # forward
    y1, _ = o.conv_fwd(x, P["conv1_w"], P["conv1_b"], c1.stride, c1.pad, exact=exact)
    t["y1"] = y1
    t["a1"] = o.relu(f32(y1))
    t["p1"], t["i1"] = o.maxpool_fwd(t["a1"], *c1.pool)
    y2, _ = o.conv_fwd(t["p1"], P["conv2_w"], P["conv2_b"], c2.stride, c2.pad, exact=exact)
    t["y2"] = y2
    t["a2"] = o.relu(f32(y2))
    t["p2"], t["i2"] = o.maxpool_fwd(t["a2"], *c2.pool)
    h = t["p2"].reshape(x.shape[0], -1)
    t["f"] = h
    for i in (1, 2, 3):
        mm, _ = o.matmul(h, P["fc%d_w" % i], 0, exact=exact)
        if exact:
            z = np.asarray(mm, np.float64) + np.asarray(P["fc%d_b" % i], np.float64)
        else:
            z = o.add_bias(f32(mm), P["fc%d_b" % i])
        t["z%d" % i] = z
        if i < 3:
            h = o.relu(f32(z))
            t["h%d" % i] = h
    dz, losses = o.softmax_ce(t["z3"], labels)
    t["dz3"] = _r(dz, exact)
    loss = float(np.sum(losses))

    # backward: linear layers
    g = {}
    dz = t["dz3"]
    for i in (3, 2, 1):
        hin = t["h%d" % (i - 1)] if i > 1 else t["f"]
        g["fc%d_w" % i] = _r(o.matmul(hin, dz, 1, exact=True)[0], exact)
        g["fc%d_b" % i] = _r(o.bias_grad_rows(dz, exact=True)[0], exact)
        dh = _r(o.matmul(dz, P["fc%d_w" % i], 2, exact=True)[0], exact)
        t["dh%d" % (i - 1) if i > 1 else "df"] = dh
        if i > 1:
            dz = o.relu_grad(f32(dh), f32(t["z%d" % (i - 1)]))
            t["dz%d" % (i - 1)] = dz
    # conv2 block
    dp2 = f32(t["df"]).reshape(t["p2"].shape)
    t["da2"] = o.maxpool_bwd(dp2, t["i2"], t["a2"].shape)
    t["dy2"] = o.relu_grad(t["da2"], f32(t["y2"]))
    g["conv2_w"] = _r(o.conv_bwd_filter(t["p1"], t["dy2"], P["conv2_w"].shape, c2.stride, c2.pad, exact=True)[0],
                      exact)
    g["conv2_b"] = _r(o.conv_bwd_bias(t["dy2"], exact=True)[0], exact)
    t["dp1"] = _r(o.conv_bwd_data(P["conv2_w"], t["dy2"], t["p1"].shape, c2.stride, c2.pad, exact=True)[0], exact)
    # conv1 block (no input gradient: x is the network input)
    t["da1"] = o.maxpool_bwd(f32(t["dp1"]), t["i1"], t["a1"].shape)
    t["dy1"] = o.relu_grad(t["da1"], f32(t["y1"]))
    g["conv1_w"] = _r(o.conv_bwd_filter(x, t["dy1"], P["conv1_w"].shape, c1.stride, c1.pad, exact=True)[0], exact)
    g["conv1_b"] = _r(o.conv_bwd_bias(t["dy1"], exact=True)[0], exact)
    t["grads"] = g

    # SGD
    new = {k: o.sgd(f32(P[k]), f32(g[k]), lr, clip) for k in synthetic.LENET_PARAMS}
    return new, loss, t
