"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake (a dropped term, a wrong sign or index, a swapped
operand, a wrong tie rule) in a temporary copy of oracle.c, compiles it with
gcc on the CPU, and checks that at least one pin rejects the mutant.
"""
import os
import re
import tempfile

import numpy as np
import pytest

import oracle
import synthetic
from oracle import out_size

torch = pytest.importorskip("torch")
F = torch.nn.functional

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "im2col_pad_sign": ("i64 h = oh * st + r - pad;\n    i64 w = ow * st + s - pad;\n    (void)C;",
                        "i64 h = oh * st + r + pad;\n    i64 w = ow * st + s - pad;\n    (void)C;"),
    "im2col_r_s_swapped": ("i64 r = (row / R) % R;\n    i64 s = row % R;",
                           "i64 s = (row / R) % R;\n    i64 r = row % R;"),
    "col2im_no_pad": ("i64 w = ow * st + s - pad;\n                        if",
                      "i64 w = ow * st + s;\n                        if"),
    "flag_a_wrong_stride": ("A[col * M + row]", "A[col * K + row]"),
    "flag_b_not_transposed": ("B[col * K + row]", "B[row * K + col]"),
    "bias_dropped": ("Y[k * NPQ + n * PQ + pq] + bias;", "Y[k * NPQ + n * PQ + pq];"),
    "dgrad_flags_0": ("oracle_matmul(CRS, Ko, NPQ, 1u", "oracle_matmul(CRS, Ko, NPQ, 0u"),
    "wgrad_flags_0": ("oracle_matmul(Ko, NPQ, CRS, 2u", "oracle_matmul(Ko, NPQ, CRS, 0u"),
    "grad_reshape_transposed": ("G[k * NPQ + n * PQ + pq] = dy[(n * Ko + k) * PQ + pq];",
                                "G[k * NPQ + n * PQ + pq] = dy[(k * N + n) * PQ + pq];"),
    "maxpool_last_max": ("if (x[at] > m)", "if (x[at] >= m)"),
    "maxpool_bwd_overwrites": ("dx[idx[t]] = dx[idx[t]] + dy[t];", "dx[idx[t]] = dy[t];"),
    "sgd_clip_sign": ("float c = g < -clip ? -clip : g;", "float c = g < -clip ? clip : g;"),
    "col2im_abs_twice": ("col_abs ? col_abs[row * cols + j] : fabs(col[row * cols + j]);",
                         "col_abs ? 2.0 * col_abs[row * cols + j] : fabs(col[row * cols + j]);"),
    "col2im_abs_pad_taps": ("if (h < 0 || h >= H || w < 0 || w >= W)\n                            continue;",
                            "if (h < 0 || h >= H || w < 0 || w >= W) {\n"
                            "                            if (plane_abs && col_abs)\n"
                            "                                plane_abs[(h < 0 ? 0 : h >= H ? H - 1 : h) * W +\n"
                            "                                          (w < 0 ? 0 : w >= W ? W - 1 : w)] +=\n"
                            "                                    col_abs[row * cols + (n * P + oh) * Q + ow];\n"
                            "                            continue;\n"
                            "                        }"),
    "dgrad_at_abs_signed": ("acc_abs += fabs(p);\n                        }\n                    }",
                            "acc_abs += p;\n                        }\n                    }"),
    "wgrad_at_abs_from_x": ("acc_abs += fabs(p);\n        }\n        out[t] = acc;\n        out_abs[t] = acc_abs;\n    }\n}\n\n/* Step A8",
                            "acc_abs += fabs(dy[(n * Ko + k) * PQ + pq]);\n        }\n        out[t] = acc;\n"
                            "        out_abs[t] = acc_abs;\n    }\n}\n\n/* Step A8"),
    "abs_scale_signed": ("acc_abs += fabs(p);\n    }\n    *out = acc;", "acc_abs += p;\n    }\n    *out = acc;"),
}


def pin_failures(orc):
    """A compact run of the pins; returns the names of those that fail."""
    bad = []
    for (N, C, H, W, Ko, R, st, pad) in [(2, 3, 7, 6, 4, 3, 2, 1), (1, 2, 9, 9, 3, 5, 1, 2)]:
        x = synthetic.normal((N, C, H, W), 1)
        w = synthetic.normal((Ko, C, R, R), 2)
        b = synthetic.normal((Ko,), 3)
        dy = synthetic.normal((N, Ko, out_size(H, R, st, pad), out_size(W, R, st, pad)), 4)
        xt = torch.from_numpy(x).double().requires_grad_()
        wt = torch.from_numpy(w).double().requires_grad_()
        bt = torch.from_numpy(b).double().requires_grad_()
        yt = F.conv2d(xt, wt, bt, stride=st, padding=pad)
        yt.backward(torch.from_numpy(dy).double())
        y, y_abs = orc.conv_fwd(x, w, b, st, pad, exact=True)
        if not np.allclose(y, yt.detach().numpy(), rtol=0, atol=1e-10):
            bad.append("fwd_vs_torch")
        ya = F.conv2d(torch.from_numpy(np.abs(x)).double(), torch.from_numpy(np.abs(w)).double(),
                      torch.from_numpy(np.abs(b)).double(), stride=st, padding=pad).numpy()
        if not np.allclose(y_abs, ya, rtol=1e-12):
            bad.append("fwd_abs_scale")
        dx, _ = orc.conv_bwd_data(w, dy, x.shape, st, pad, exact=True)
        dw, _ = orc.conv_bwd_filter(x, dy, w.shape, st, pad, exact=True)
        if not np.allclose(dx, xt.grad.numpy(), rtol=0, atol=1e-10):
            bad.append("dgrad_vs_torch")
        if not np.allclose(dw, wt.grad.numpy(), rtol=0, atol=1e-10):
            bad.append("wgrad_vs_torch")
        xa = torch.from_numpy(np.abs(x)).double().requires_grad_()
        wa = torch.from_numpy(np.abs(w)).double().requires_grad_()
        F.conv2d(xa, wa, stride=st, padding=pad).backward(torch.from_numpy(np.abs(dy)).double())
        _, dx_abs = orc.conv_bwd_data(w, dy, x.shape, st, pad, exact=True)
        _, dw_abs = orc.conv_bwd_filter(x, dy, w.shape, st, pad, exact=True)
        if not np.allclose(dx_abs, xa.grad.numpy(), rtol=1e-12, atol=0):
            bad.append("dgrad_abs_scale")
        if not np.allclose(dw_abs, wa.grad.numpy(), rtol=1e-12, atol=0):
            bad.append("wgrad_abs_scale")
        _, dxa_at = orc.conv_bwd_data_at(w, dy, x.shape, st, pad, np.arange(x.size, dtype=np.int64), exact=True)
        _, dwa_at = orc.conv_bwd_filter_at(x, dy, w.shape, st, pad, np.arange(w.size, dtype=np.int64), exact=True)
        if not np.allclose(dxa_at, xa.grad.numpy().ravel(), rtol=1e-12, atol=0):
            bad.append("dgrad_at_abs_scale")
        if not np.allclose(dwa_at, wa.grad.numpy().ravel(), rtol=1e-12, atol=0):
            bad.append("wgrad_at_abs_scale")
        col = orc.im2col(np.ones_like(x), R, st, pad)
        d1, _ = orc.col2im(col, x.shape, R, st, pad)
        cnt = np.zeros((H, W))
        for oh in range(out_size(H, R, st, pad)):
            for ow in range(out_size(W, R, st, pad)):
                for r in range(R):
                    for s in range(R):
                        h, ww = oh * st + r - pad, ow * st + s - pad
                        if 0 <= h < H and 0 <= ww < W:
                            cnt[h, ww] += 1
        if not np.array_equal(d1[0, 0], cnt):
            bad.append("tap_count")
    for flags in range(4):
        A = synthetic.normal((5, 3), 10)
        B = synthetic.normal((3, 4), 11)
        As = A.T.copy() if flags & 1 else A
        Bs = B.T.copy() if flags & 2 else B
        c, _ = orc.matmul(As, Bs, flags, exact=True)
        if not np.allclose(c, A.astype(np.float64) @ B, rtol=0, atol=1e-12):
            bad.append("matmul_flags_%d" % flags)
    xp = synthetic.relu_normal((2, 2, 9, 9), 20)
    yp, ip = orc.maxpool_fwd(xp, 3, 2)
    yt, it = F.max_pool2d(torch.from_numpy(xp).double(), 3, 2, return_indices=True)
    if not np.array_equal(ip - (np.arange(4) * 81).reshape(2, 2, 1, 1), it.numpy()):
        bad.append("maxpool_idx")
    _, iz = orc.maxpool_fwd(np.zeros((1, 1, 4, 4), np.float32), 2, 2)
    if iz.ravel().tolist() != [0, 2, 8, 10]:
        bad.append("maxpool_ties")
    dyp = synthetic.small_ints(yp.shape, 21)
    xt = torch.from_numpy(xp).double().requires_grad_()
    F.max_pool2d(xt, 3, 2).backward(torch.from_numpy(dyp).double())
    if not np.array_equal(orc.maxpool_bwd(dyp, it.numpy().astype(np.int32) +
                                          (np.arange(4) * 81).reshape(2, 2, 1, 1).astype(np.int32),
                                          xp.shape), xt.grad.numpy().astype(np.float32)):
        bad.append("maxpool_bwd")
    out = orc.sgd(np.ones(3, np.float32), np.array([5, -5, 0.25], np.float32), 0.5, 1.0)
    if out.tolist() != [0.5, 1.5, 0.875]:
        bad.append("sgd_hand")
    return bad


def test_unmutated_oracle_passes_compact_pins():
    assert pin_failures(oracle.get()) == []


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
        failures = pin_failures(oracle.Oracle(lib))
    assert failures, "mutant %s passed every pin" % name
