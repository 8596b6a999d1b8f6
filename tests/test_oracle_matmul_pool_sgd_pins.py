"""Pins of the oracle's flagged matmul (page "DirectCompute Neural Network
Engine", section "Optimizations" -> "Transpose via Flags"), max pooling
("Pooling Shaders") and SGD ("Utility Shaders", nn_sgd)."""
import numpy as np
import pytest

import synthetic

torch = pytest.importorskip("torch")
F = torch.nn.functional

DIMS = [(1, 1, 1), (3, 5, 2), (16, 25, 7), (9, 4, 13), (33, 17, 8)]


def operands(M, K, N, flags, seed, ints=False):
    gen = synthetic.small_ints if ints else synthetic.normal
    A = gen((M, K), seed + 1)
    B = gen((K, N), seed + 2)
    As = np.ascontiguousarray(A.T) if flags & 1 else A
    Bs = np.ascontiguousarray(B.T) if flags & 2 else B
    return A, B, As, Bs


@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("flags", [1, 2, 3])
def test_flags_equal_explicit_transposes(orc, dims, flags):
    """Reading a transposed buffer through the flags gives bit-for-bit what
    flags 0 gives on the explicitly transposed copy."""
    M, K, N = dims
    A, B, As, Bs = operands(M, K, N, flags, 100)
    c0, a0 = orc.matmul(A, B, 0, exact=True)
    cf, af = orc.matmul(As, Bs, flags, exact=True)
    assert cf.shape == (M, N)
    assert np.array_equal(c0, cf) and np.array_equal(a0, af)


@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("flags", range(4))
def test_matmul_vs_numpy_float64(orc, dims, flags):
    M, K, N = dims
    A, B, As, Bs = operands(M, K, N, flags, 200)
    c, c_abs = orc.matmul(As, Bs, flags, exact=True)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    np.testing.assert_allclose(c, ref, rtol=0, atol=1e-12 * (1 + c_abs.max()))
    np.testing.assert_allclose(c_abs, np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64),
                               rtol=1e-12)


@pytest.mark.parametrize("flags", range(4))
def test_matmul_small_ints_exact_and_rectangular(orc, flags):
    M, K, N = 7, 5, 3
    A, B, As, Bs = operands(M, K, N, flags, 300, ints=True)
    c, _ = orc.matmul(As, Bs, flags)
    expect = [[sum(int(A[i, k]) * int(B[k, j]) for k in range(K)) for j in range(N)] for i in range(M)]
    assert c.astype(np.int64).tolist() == expect


def test_identity_and_permutation(orc):
    A = synthetic.normal((6, 6), 401)
    I = np.eye(6, dtype=np.float32)
    for flags in range(4):
        c, _ = orc.matmul(A if not flags & 1 else np.ascontiguousarray(A.T), I, flags)
        assert np.array_equal(c, A)
    perm = np.array([3, 0, 5, 1, 4, 2])
    Pm = np.eye(6, dtype=np.float32)[perm]           # row i of Pm = e_perm[i]
    c, _ = orc.matmul(Pm, A, 0)
    assert np.array_equal(c, A[perm])                 # rows permuted
    c, _ = orc.matmul(A, Pm, 2)                       # A * Pm^T: columns permuted
    assert np.array_equal(c, A[:, perm])


@pytest.mark.parametrize("flags", range(4))
def test_matmul_at_matches_full(orc, flags):
    M, K, N = 33, 17, 8
    _, _, As, Bs = operands(M, K, N, flags, 500)
    c, c_abs = orc.matmul(As, Bs, flags, exact=True)
    flat = np.array([0, 5, 77, M * N - 1])
    v, v_abs = orc.matmul_at(As, Bs, flags, flat, exact=True)
    assert np.array_equal(v, c.ravel()[flat]) and np.array_equal(v_abs, c_abs.ravel()[flat])


# ----------------------------------------------------------------------------
# max pooling

POOLS = [((2, 3, 8, 8), 2, 2), ((1, 2, 7, 9), 3, 2), ((2, 2, 13, 13), 3, 2), ((1, 1, 5, 5), 5, 1),
         ((1, 2, 6, 6), 2, 1), ((2, 1, 11, 10), 3, 3)]


@pytest.mark.parametrize("shape,k,st", POOLS)
def test_maxpool_fwd_vs_torch(orc, shape, k, st):
    x = synthetic.relu_normal(shape, 600)   # about half zeros: many ties
    y, idx = orc.maxpool_fwd(x, k, st)
    yt, it = F.max_pool2d(torch.from_numpy(x).double(), k, st, return_indices=True)
    N, C, H, W = shape
    assert np.array_equal(y.astype(np.float64), yt.numpy())
    plane_base = (np.arange(N * C) * H * W).reshape(N, C, 1, 1)
    assert np.array_equal(idx - plane_base, it.numpy())
    assert np.array_equal(x.ravel()[idx], y)


def test_maxpool_tie_rule_first_max():
    import oracle
    orc = oracle.get()
    x = np.zeros((1, 1, 4, 4), np.float32)
    y, idx = orc.maxpool_fwd(x, 2, 2)           # all-equal windows -> top-left
    assert idx.ravel().tolist() == [0, 2, 8, 10]
    x = np.array([[1, 5, 5, 0], [5, 2, 0, 0], [0, 0, 3, 3], [0, 0, 3, 3]], np.float32).reshape(1, 1, 4, 4)
    y, idx = orc.maxpool_fwd(x, 2, 2)
    assert y.ravel().tolist() == [5, 5, 0, 3]
    assert idx.ravel().tolist() == [1, 2, 8, 10]  # first maximum in row-major window order
    x = np.arange(16, dtype=np.float32).reshape(1, 1, 4, 4)[:, :, ::-1, ::-1].copy()
    y, idx = orc.maxpool_fwd(x, 3, 1)              # overlapping, strictly decreasing
    assert idx.ravel().tolist() == [0, 1, 4, 5]


@pytest.mark.parametrize("shape,k,st", POOLS)
def test_maxpool_bwd_vs_torch(orc, shape, k, st):
    x = synthetic.relu_normal(shape, 610)
    y, idx = orc.maxpool_fwd(x, k, st)
    dy = synthetic.small_ints(y.shape, 611)        # integer grads: sums are exact
    dx = orc.maxpool_bwd(dy, idx, shape)
    xt = torch.from_numpy(x).double().requires_grad_()
    F.max_pool2d(xt, k, st).backward(torch.from_numpy(dy).double())
    assert np.array_equal(dx.astype(np.float64), xt.grad.numpy())
    assert dx.sum() == dy.sum()                     # every gradient lands somewhere


def test_maxpool_bwd_overlap_hand():
    """3x3 windows, stride 2, on a 5x5 plane: the centre pixel (2,2) is the max
    of all four windows and receives all four gradients."""
    import oracle
    orc = oracle.get()
    x = np.zeros((1, 1, 5, 5), np.float32)
    x[0, 0, 2, 2] = 1.0
    y, idx = orc.maxpool_fwd(x, 3, 2)
    assert idx.ravel().tolist() == [12, 12, 12, 12]
    dx = orc.maxpool_bwd(np.array([1, 2, 4, 8], np.float32).reshape(1, 1, 2, 2), idx, x.shape)
    expect = np.zeros((5, 5), np.float32)
    expect[2, 2] = 15.0
    assert np.array_equal(dx[0, 0], expect)


# ----------------------------------------------------------------------------
# SGD

def test_sgd_hand_cases(orc):
    p = np.array([1.0, 1.0, 1.0, -2.0, 0.5], np.float32)
    g = np.array([5.0, -5.0, 0.25, 1.0, -1.0], np.float32)
    out = orc.sgd(p, g, lr=0.5, clip=1.0)
    # clipped to +1 -> 1 - 0.5; clipped to -1 -> 1 + 0.5; inside -> 1 - 0.125;
    # exactly at +clip; exactly at -clip
    assert out.tolist() == [0.5, 1.5, 0.875, -2.5, 1.0]


def test_sgd_vs_numpy_float32(orc):
    p = synthetic.normal((10007,), 700)
    g = synthetic.normal((10007,), 701, std=3.0)
    lr, clip = np.float32(0.01), np.float32(1.0)
    out = orc.sgd(p, g, float(lr), float(clip))
    ref = p - lr * np.clip(g, -clip, clip)         # numpy fp32: one rounding per op
    assert ref.dtype == np.float32
    assert np.array_equal(out, ref)
