"""Pins for the oracle's training-step pieces and its LeNet-5 step.

Each function is held to something other than itself: torch's float64 CPU
routines (relu, softmax, cross-entropy with autograd, broadcasting add, sums),
central finite differences of the loss, closed-form identities, and, for the
whole step, a float64 torch autograd network built here independently of the
oracle's composition.  Mutants of oracle.c (one plausible mistake each) must
fail at least one pin.
"""
import os
import tempfile

import numpy as np
import pytest

import oracle
import oracle.lenet as olenet
import synthetic

torch = pytest.importorskip("torch")
F = torch.nn.functional

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def piece_failures(orc):
    """Compact pins of relu, relu_grad, add_bias, bias_grad_rows, softmax,
    softmax_ce and grad_accum; returns the names of those that fail."""
    bad = []
    x = synthetic.normal((7, 13), 41)
    x[0, :3] = 0.0
    y = orc.relu(x)
    if not np.array_equal(y, F.relu(torch.from_numpy(x)).numpy()):
        bad.append("relu_vs_torch")
    if not np.array_equal(y - orc.relu(-x), x):                 # relu(x) - relu(-x) = x, exactly
        bad.append("relu_identity")
    g = synthetic.normal(x.shape, 42)
    xt = _t(x).requires_grad_()
    F.relu(xt).backward(_t(g))
    if not np.array_equal(orc.relu_grad(g, x), xt.grad.numpy().astype(np.float32)):
        bad.append("relu_grad_vs_autograd")
    if not np.array_equal(orc.relu_grad(g, y), orc.relu_grad(g, x)):   # output as mask = input as mask
        bad.append("relu_grad_mask_from_output")

    A = synthetic.normal((6, 5), 43)
    b = synthetic.normal((5,), 44)
    if not np.array_equal(orc.add_bias(A, b), (torch.from_numpy(A) + torch.from_numpy(b)).numpy()):
        bad.append("add_bias_vs_torch")

    G = synthetic.normal((9, 4), 45)
    db, db_abs = orc.bias_grad_rows(G, exact=True)
    if not np.allclose(db, _t(G).sum(0).numpy(), rtol=0, atol=1e-12):
        bad.append("bias_grad_rows_vs_torch")
    if not np.allclose(db_abs, np.abs(G.astype(np.float64)).sum(0), rtol=1e-15):
        bad.append("bias_grad_rows_abs")

    z = synthetic.normal((5, 10), 46).astype(np.float64) * 3
    p = orc.softmax(z)
    if not np.allclose(p, torch.softmax(_t(z), 1).numpy(), rtol=0, atol=1e-15):
        bad.append("softmax_vs_torch")
    if not np.allclose(orc.softmax(z + 40.0), p, rtol=0, atol=1e-14):       # shift invariance
        bad.append("softmax_shift")
    lab = np.array([0, 3, 9, 3, 7], np.int32)
    grad, loss = orc.softmax_ce(z, lab)
    zt = _t(z).requires_grad_()
    F.cross_entropy(zt, torch.from_numpy(lab).long(), reduction="sum").backward()
    if not np.allclose(grad, zt.grad.numpy(), rtol=0, atol=1e-14):
        bad.append("ce_grad_vs_autograd")
    if not np.allclose(loss, F.cross_entropy(_t(z), torch.from_numpy(lab).long(), reduction="none").numpy(),
                       rtol=0, atol=1e-13):
        bad.append("ce_loss_vs_torch")
    # central differences of the summed loss against the gradient
    h = 1e-6
    fd = np.empty_like(z)
    for i in range(z.shape[0]):
        for j in range(z.shape[1]):
            zp, zm = z.copy(), z.copy()
            zp[i, j] += h
            zm[i, j] -= h
            fd[i, j] = (orc.softmax_ce(zp, lab)[1].sum() - orc.softmax_ce(zm, lab)[1].sum()) / (2 * h)
    if not np.allclose(fd, grad, rtol=0, atol=1e-7):
        bad.append("ce_finite_differences")

    acc = synthetic.normal((11,), 47)
    gg = synthetic.normal((11,), 48)
    if not np.array_equal(orc.grad_accum(acc, gg), (torch.from_numpy(acc) + torch.from_numpy(gg)).numpy()):
        bad.append("grad_accum_vs_torch")
    return bad


def torch_lenet_step(params, x, labels, lr, clip):
    """Float64 torch autograd LeNet-5 step, written from the network's
    definition (not from the oracle's composition)."""
    c1, c2 = synthetic.LENET
    P = {k: _t(v).requires_grad_() for k, v in params.items()}
    a = F.relu(F.conv2d(_t(x), P["conv1_w"], P["conv1_b"], stride=c1.stride, padding=c1.pad))
    a = F.max_pool2d(a, *c1.pool)
    a = F.relu(F.conv2d(a, P["conv2_w"], P["conv2_b"], stride=c2.stride, padding=c2.pad))
    a = F.max_pool2d(a, *c2.pool).reshape(x.shape[0], -1)
    a = F.relu(a @ P["fc1_w"] + P["fc1_b"])
    a = F.relu(a @ P["fc2_w"] + P["fc2_b"])
    z = a @ P["fc3_w"] + P["fc3_b"]
    loss = F.cross_entropy(z, torch.from_numpy(labels).long(), reduction="sum")
    loss.backward()
    grads = {k: v.grad.numpy() for k, v in P.items()}
    new = {k: (P[k].detach() - lr * torch.clamp(P[k].grad, -clip, clip)).numpy() for k in P}
    return new, float(loss.detach()), grads


def step_failures(orc, batch=6):
    bad = []
    params = synthetic.lenet_params()
    x, labels = synthetic.lenet_batch(batch, seed=2311)
    lr, clip = 0.05, 0.02          # a small clip so that clipping is active on some entries
    new, loss, t = olenet.step(params, x, labels, lr, clip, exact=True, orc=orc)
    tnew, tloss, tgrads = torch_lenet_step(params, x, labels, lr, clip)
    if not np.isclose(loss, tloss, rtol=1e-6):
        bad.append("step_loss")
    for k in synthetic.LENET_PARAMS:
        ref = tgrads[k]
        if not np.allclose(t["grads"][k], ref, rtol=1e-4, atol=1e-5 * np.abs(ref).max()):
            bad.append("step_grad_" + k)
        if not np.allclose(new[k], tnew[k], rtol=1e-5, atol=1e-6):
            bad.append("step_param_" + k)
    if not any(np.abs(np.asarray(tgrads[k])).max() > clip for k in tgrads):
        bad.append("step_clip_inactive")
    return bad


def test_pieces_pinned():
    assert piece_failures(oracle.get()) == []


def test_lenet_step_matches_torch_autograd():
    assert step_failures(oracle.get()) == []


def test_lenet_step_fp32_program_close_to_exact():
    """The fp32-rounded program (what the GPU runs) stays close to the exact one."""
    params = synthetic.lenet_params()
    x, labels = synthetic.lenet_batch(8, seed=2312)
    n32, l32, _ = olenet.step(params, x, labels)
    n64, l64, _ = olenet.step(params, x, labels, exact=True)
    assert np.isclose(l32, l64, rtol=1e-5)
    for k in synthetic.LENET_PARAMS:
        assert np.allclose(n32[k], n64[k], rtol=1e-5, atol=1e-6), k


MUTATIONS = {
    "relu_grad_unmasked": ("dx[i] = grad[i] * (x[i] > 0.0f ? 1.0f : 0.0f);", "dx[i] = grad[i];"),
    "add_bias_row_index": ("out[i] = A[i] + b[i % cols];", "out[i] = A[i] + b[i / cols];"),
    "bias_grad_rows_over_cols": ("acc += G[i * cols + j];\n            acc_abs",
                                 "acc += G[j * rows + i];\n            acc_abs"),
    "softmax_unnormalised": ("for (i64 j = 0; j < cols; ++j) p[i * cols + j] /= s;", ""),
    "ce_one_hot_sign": ("grad[i * cols + l] -= 1.0;", "grad[i * cols + l] += 1.0;"),
    "ce_loss_wrong_class": ("loss[i] = -log(grad[i * cols + l]);", "loss[i] = -log(grad[i * cols]);"),
    "grad_accum_overwrites": ("accum[i] = accum[i] + grad[i];", "accum[i] = grad[i];"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutant(name):
    find, repl = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(find) == 1, "mutation anchor not unique/missing: %s" % name
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(find, repl))
        lib = oracle.load(oracle.build(path, os.path.join(d, "libmutant.so"), force=True))
        orc = oracle.Oracle(lib)
        failures = piece_failures(orc) + step_failures(orc, batch=4)
    assert failures, "mutant %s passed every pin" % name
