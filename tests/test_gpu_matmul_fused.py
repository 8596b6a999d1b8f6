"""GPU parity of matmul_fused: the flagged matmul with a linear layer's
element-wise work in its epilogue.  Page "DirectCompute Neural Network
Engine": section "Optimizations" -> "Transpose via Flags" for the product,
the utility shader nn_add_bias and the activation shaders nn_relu /
nn_relu_grad for the epilogue (the page's LeNet trainer chains them).

Two checks per case:
* bit-identity with the unfused chain on the GPU -- matmul, then add_bias
  (with or without ReLU) or relu_fwd, then relu_bwd against the gate: the
  epilogue performs the same fp32 operations in the same order;
* the oracle: its fp64 product, the bias added, ReLU and gate applied, within
  1e-4 * (sum|a_k b_k| + |b|) + 1e-6 (rounding the bias addition costs at most
  2^-24 of |c + b|; ReLU and the 0/1 gate do not enlarge an error).
Shapes cover every tile width (32 to 256 columns), the cluster split (few
tiles, long K), ragged M and N, and gates with exact zeros of both signs.
"""
import numpy as np
import pytest

import synthetic
from tests.gpu_helpers import assert_within_tol

pytestmark = pytest.mark.gpu

SHAPES = [
    # M, K, N
    (64, 400, 120),      # LeNet fc1 forward
    (64, 84, 10),        # LeNet fc3 forward: a 32-wide tile
    (64, 120, 400),      # LeNet fc1 input gradient (flag 2 in the step)
    (127, 1600, 127),    # one tile row, long K: split over a cluster
    (16, 4096, 64),      # skinny, long K
    (300, 257, 1000),    # several 256-wide tiles, ragged
    (1024, 363, 300),
    (129, 33, 31),       # ragged everywhere, one K stage and a half
]

VARIANTS = [
    # bias, relu, gate
    (True, True, False),     # forward of a hidden linear layer
    (True, False, False),    # forward of the output layer
    (False, False, True),    # input gradient of a ReLU-fed layer
    (False, True, False),
    (True, True, True),
]


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


def gate_values(M, N, seed):
    """N(0,1) with exact +0 and -0 sprinkled in (the gate is strict: > 0)."""
    g = synthetic.normal((M, N), seed)
    r = synthetic.rng(seed + 1)
    g[r.random((M, N)) < 0.05] = 0.0
    g[r.random((M, N)) < 0.05] = -0.0
    return g


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("M,K,N", SHAPES)
def test_matmul_fused(cb, orc, M, K, N, flags):
    import torch
    A, B = synthetic.matmul_case(M, K, N, flags)
    bias = synthetic.normal((N,), 8100 + N)
    gate = gate_values(M, N, 8200 + M + N)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    bd, gd = torch.from_numpy(bias).cuda(), torch.from_numpy(gate).cuda()
    C, C_abs = orc.matmul(A, B, flags, exact=True)
    for use_bias, relu, use_gate in VARIANTS:
        what = "matmul_fused %dx%dx%d f%d bias=%d relu=%d gate=%d" % (M, K, N, flags, use_bias, relu, use_gate)
        got = cb.matmul(a, b, flags, bias=bd if use_bias else None, relu=relu, gate=gd if use_gate else None)
        # the unfused chain on the GPU
        ref = cb.matmul(a, b, flags)
        if use_bias:
            ref = cb.add_bias(ref, bd, relu=relu)
        elif relu:
            ref = cb.relu_fwd(ref)
        if use_gate:
            ref = cb.relu_bwd(ref, gd)
        cb.check()
        assert torch.equal(got, ref), what + ": differs from the unfused chain"
        # the oracle, in fp64 throughout
        want = C + bias.astype(np.float64) if use_bias else C.copy()
        if relu:
            want = np.maximum(want, 0.0)
        if use_gate:
            want = want * (gate > 0)
        scale = C_abs + (np.abs(bias.astype(np.float64)) if use_bias else 0.0)
        assert_within_tol(got.cpu().numpy(), want, scale, what)
