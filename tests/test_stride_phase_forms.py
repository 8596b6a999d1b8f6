"""The index algebra behind the tensor-core input gradient and the space-to-depth
filter gradient, checked on the CPU in float64 (no GPU, no library call).

The input gradient of the page "DirectCompute Neural Network Engine" (section
"Convolution: The im2col Approach": filters^T x grad, then col2im) is computed
on the GPU as ONE GEMM over a super-pixel grid: input row h = s*hh + a - o
with phase a in [0, s) and offset o = pad mod s, every phase served by the
window of dy rows oh = hh + d, d in [pad div s - T + 1, pad div s],
T = ceil(k / s), through tap r = a + (pad - o) - s*d.  The filter gradient of
strided few-channel layers runs over the space-to-depth tensor X' with GEMM
rows that are the ORIGINAL taps (c, r, q), read from X' channel
(c*s + r mod s)*s + q mod s at tap (r div s, q div s).

Both are written out here literally with numpy loops and compared with the
definitions the oracle follows (and torch's float64 gradient), so a wrong
offset, window or phase mapping in the scheme itself fails on the CPU.
"""
import itertools

import numpy as np
import pytest

import synthetic
from oracle import out_size

torch = pytest.importorskip("torch")

# (N, C, H, W, Ko, k, stride, pad): strides 1-4, pads below, equal to and above
# the stride, filters shorter and longer than the stride, odd and even widths.
SHAPES = [
    (1, 2, 23, 23, 3, 11, 4, 2),
    (1, 2, 26, 30, 2, 11, 4, 2),
    (1, 2, 17, 17, 3, 7, 2, 3),
    (1, 2, 20, 20, 3, 11, 4, 6),
    (1, 2, 9, 9, 2, 3, 2, 1),
    (1, 2, 7, 7, 3, 2, 3, 1),
    (1, 2, 12, 12, 2, 3, 4, 0),
    (1, 2, 11, 10, 2, 3, 2, 1),
    (1, 2, 6, 6, 2, 3, 1, 1),
]


def _inputs(shape, seed):
    N, C, H, W, Ko, k, s, p = shape
    P, Q = out_size(H, k, s, p), out_size(W, k, s, p)
    x = synthetic.normal((N, C, H, W), seed + 1).astype(np.float64)
    w = synthetic.normal((Ko, C, k, k), seed + 2).astype(np.float64)
    dy = synthetic.normal((N, Ko, P, Q), seed + 3).astype(np.float64)
    return x, w, dy, P, Q


@pytest.mark.parametrize("shape", SHAPES)
def test_input_gradient_on_padding_aligned_grid(shape):
    N, C, H, W, Ko, k, s, p = shape
    x, w, dy, P, Q = _inputs(shape, 70)
    o = p % s
    T = (k + s - 1) // s
    d_lo = p // s - T + 1
    Hs, Ws = (H + o + s - 1) // s, (W + o + s - 1) // s
    dx = np.zeros((N, C, H, W))
    hits = np.zeros((N, C, H, W), dtype=np.int64)
    for n, hh, ww in itertools.product(range(N), range(Hs), range(Ws)):
        for c, a, b in itertools.product(range(C), range(s), range(s)):
            acc = 0.0
            for td, te in itertools.product(range(T), range(T)):
                oh, ow = hh + d_lo + td, ww + d_lo + te
                r, q = a + (p - o) - s * (d_lo + td), b + (p - o) - s * (d_lo + te)
                if 0 <= oh < P and 0 <= ow < Q and 0 <= r < k and 0 <= q < k:
                    acc += float(np.dot(dy[n, :, oh, ow], w[:, c, r, q]))
            h, wc = s * hh + a - o, s * ww + b - o
            if 0 <= h < H and 0 <= wc < W:
                dx[n, c, h, wc] += acc
                hits[n, c, h, wc] += 1
    assert (hits == 1).all(), "every input pixel is one GEMM output"
    ref = torch.nn.grad.conv2d_input((N, C, H, W), torch.from_numpy(w), torch.from_numpy(dy), stride=s,
                                     padding=p).numpy()
    np.testing.assert_allclose(dx, ref, rtol=0, atol=1e-9)


@pytest.mark.parametrize("shape", [sh for sh in SHAPES if sh[6] > 1])
def test_filter_gradient_over_original_taps_of_space_to_depth(shape):
    N, C, H, W, Ko, k, s, p = shape
    x, w, dy, P, Q = _inputs(shape, 80)
    T = (k + s - 1) // s
    Hs, Ws = P + T - 1, Q + T - 1
    # X'[n, (c, a, b), hh, ww] = x[n, c, s*hh + a - p, s*ww + b - p], zero outside
    xs = np.zeros((N, C * s * s, Hs, Ws))
    for n, c, a, b, hh, ww in itertools.product(range(N), range(C), range(s), range(s), range(Hs), range(Ws)):
        h, wc = s * hh + a - p, s * ww + b - p
        if 0 <= h < H and 0 <= wc < W:
            xs[n, (c * s + a) * s + b, hh, ww] = x[n, c, h, wc]
    dw = np.zeros((Ko, C, k, k))
    for c, r, q in itertools.product(range(C), range(k), range(k)):
        cp, tr, tq = (c * s + r % s) * s + q % s, r // s, q // s
        # the row's column-matrix values: X' at unit stride, shifted by the tap
        col = xs[:, cp, tr:tr + P, tq:tq + Q]
        dw[:, c, r, q] = np.einsum("nkpq,npq->k", dy, col)
    ref = torch.nn.grad.conv2d_weight(torch.from_numpy(x), (Ko, C, k, k), torch.from_numpy(dy), stride=s,
                                      padding=p).numpy()
    np.testing.assert_allclose(dw, ref, rtol=0, atol=1e-9)
