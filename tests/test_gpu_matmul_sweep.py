"""GPU parity of the flagged matmul over its whole sweep: every (M, N, K, flags)
with M, N in {16, 64, 127, 128, 1024, 4096, 9216}, K in {25, 150, 363, 1600,
2304, 4096} and all four transpose flags (page "DirectCompute Neural Network
Engine", section "Optimizations" -> "Transpose via Flags"; the shader table's
small- and large-matrix regimes are both inside the grid).  1176 cases.

The large cases are too big for the full oracle, so each case is checked on
sampled entries, each an exact fp64 dot of the oracle: two full rows (one
random, plus the last, ragged one), two full columns (likewise) and 1024
random elements, within 1e-4 * sum|a_k b_k| + 1e-6.  Besides, the whole C
(NaN-filled before the call) must come back finite -- every entry written --
and the floats right after C must keep their canary (nothing written past it).

Operands are windows of two fixed N(0,1) pools (synthetic.matmul_sweep_case),
uploaded once; the oracle reads the same windows in float64.
"""
import numpy as np
import pytest

import synthetic
from tests.gpu_helpers import assert_within_tol

pytestmark = pytest.mark.gpu

CANARY = -1.2345e30
GUARD = 1024


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


@pytest.fixture(scope="module")
def pools():
    """(host float64 pools, device fp32 pools, device output buffer)."""
    import torch
    host32 = [synthetic.matmul_pool(0), synthetic.matmul_pool(1)]
    host64 = [p.astype(np.float64) for p in host32]
    dev = [torch.from_numpy(p).cuda() for p in host32]
    big = max(synthetic.MATMUL_MN)
    cbuf = torch.empty(big * big + GUARD, dtype=torch.float32, device="cuda")
    return host64, dev, cbuf


def views(arr, M, K, N, flags):
    """This case's A and B as windows of the two pools ``arr`` (numpy arrays or
    torch tensors alike)."""
    oa, ob = synthetic.matmul_sweep_offsets(M, K, N, flags)
    a_shape = (K, M) if flags & 1 else (M, K)
    b_shape = (N, K) if flags & 2 else (K, N)
    return arr[0][oa:oa + M * K].reshape(a_shape), arr[1][ob:ob + K * N].reshape(b_shape)


def sample_flat(M, N, K, flags):
    """Flat C indices checked for one case: rows {random, M-1}, columns
    {random, N-1}, and 1024 random elements."""
    g = synthetic.rng(90000 + ((M * 31 + K) * 31 + N) * 4 + flags)
    rows = sorted({int(g.integers(0, M)), M - 1})
    cols = sorted({int(g.integers(0, N)), N - 1})
    parts = [np.arange(N, dtype=np.int64) + r * N for r in rows]
    parts += [np.arange(M, dtype=np.int64) * N + c for c in cols]
    parts.append(g.integers(0, M * N, size=1024).astype(np.int64))
    return np.concatenate(parts)


def run_case(cb, orc, pools, M, K, N, flags, tol_scale=1e-4):
    import torch
    host64, dev, cbuf = pools
    a, b = views(dev, M, K, N, flags)
    c = cbuf[:M * N].view(M, N)
    c.fill_(float("nan"))
    cbuf[M * N:M * N + GUARD].fill_(CANARY)
    cb.matmul(a, b, flags, C=c)
    cb.check()
    assert bool(torch.isfinite(c).all()), "matmul %dx%dx%d f%d: an entry was not written" % (M, K, N, flags)
    assert bool((cbuf[M * N:M * N + GUARD] == CANARY).all()), "matmul %dx%dx%d f%d: wrote past C" % (M, K, N, flags)
    flat = sample_flat(M, N, K, flags)
    got = c.view(-1)[torch.from_numpy(flat).cuda()].cpu().numpy()
    ha, hb = views(host64, M, K, N, flags)
    ref, ref_abs = orc.matmul_at(ha, hb, flags, flat)
    if tol_scale == 1e-4:
        return assert_within_tol(got, ref, ref_abs, "matmul %dx%dx%d f%d" % (M, K, N, flags))
    err = np.abs(got.astype(np.float64) - ref)
    tol = tol_scale * ref_abs + 1e-6
    assert (err <= tol).all(), "matmul %dx%dx%d f%d: %d sampled entries out of tolerance" % (
        M, K, N, flags, int((err > tol).sum()))
    return float((err / tol).max())


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("M", synthetic.MATMUL_MN)
def test_matmul_sweep(cb, orc, pools, M, flags):
    """All 42 (N, K) cases of one (M, flags) row of the sweep."""
    worst = 0.0
    for N in synthetic.MATMUL_MN:
        for K in synthetic.MATMUL_K:
            worst = max(worst, run_case(cb, orc, pools, M, K, N, flags))
    assert worst <= 1.0


class engine:
    """Context manager over the matmul engine test hook: -1 plan, 0 gather,
    1 TMA wherever the operands qualify."""

    def __init__(self, cb, which):
        self.lib, self.which = cb.lib(), which

    def __enter__(self):
        self.prev = self.lib.conv_b200_debug_matmul_engine(self.which)
        assert self.prev in (-1, 0, 1)

    def __exit__(self, *exc):
        self.lib.conv_b200_debug_matmul_engine(self.prev)


def test_sweep_reaches_every_tiling(cb):
    """Over the sweep, each flag combination meets every tile width (32 to 256
    columns) and both whole tiles and K cut over clusters of 2, 4 and 8 CTAs
    (the cluster split: few tiles, long K).  The plan feeds the large
    K-contiguous cases (flags 2) by TMA in both math modes, and those with one
    rows-contiguous operand in TF32 mode, where that measured faster; forced,
    every flag reaches it."""
    def survey(flags):
        widths, pieces, tma = set(), set(), set()
        for M in synthetic.MATMUL_MN:
            for N in synthetic.MATMUL_MN:
                for K in synthetic.MATMUL_K:
                    bn, p, fed = cb.matmul_tiling(M, K, N, flags, with_tma=True)
                    widths.add(bn)
                    pieces.add(p)
                    tma.add(fed)
        return widths, pieces, tma
    for flags in range(4):
        widths, pieces, tma = survey(flags)
        assert widths == {32, 64, 128, 256}, (flags, widths)
        assert {1, 2, 4, 8} <= pieces, (flags, pieces)
        if flags == 2:
            assert tma == {False, True}, (flags, tma)
        with engine(cb, 1):
            assert survey(flags)[2] == {False, True}, flags   # small or misaligned pitches stay gathered
        with engine(cb, 0):
            assert survey(flags)[2] == {False}, flags
    with cb.math(cb.CONV_MATH_TF32):   # one rows-contiguous operand (A stored K x M)
        assert True in survey(3)[2]


# The TMA-fed path (whole tiles >= 128 wide; K-contiguous operands land as
# they are, rows-contiguous ones are transposed by the converters) on ragged
# shapes: M and N past the last full tile (the boxes zero-fill, the epilogue
# drops rows and columns past C), K not a multiple of the 16-deep stage; every
# flag combination, both math modes.
TMA_SHAPES = [(5000, 1024, 5000), (2500, 2048, 9000), (4096, 100, 4096)]


@pytest.mark.parametrize("which", [1, 0])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("M,K,N", TMA_SHAPES)
def test_engines_ragged(cb, orc, pools, M, K, N, flags, which):
    """Both engines, forced, on the shapes above (which = 1: TMA-fed, 0:
    register gather), in both math modes."""
    a, b = views(pools[1], M, K, N, flags)
    with engine(cb, which):
        assert cb.matmul_tiling(M, K, N, flags, a, b, with_tma=True)[2] == bool(which)
        run_case(cb, orc, pools, M, K, N, flags)
        with cb.math(cb.CONV_MATH_TF32):
            assert run_case(cb, orc, pools, M, K, N, flags, tol_scale=2.5e-3) <= 1.0


# Shapes whose tiles are cut over clusters, checked against the full oracle
# (every entry) and for run-to-run bit-identity (the pieces are added in a
# fixed order): one tile (16 x 16), ragged tiles (127 x 127, 130 columns) and
# several tiles (128 x 1024), K from 150 to 4096.
SPLIT_SHAPES = [(16, 4096, 16), (127, 1600, 127), (64, 2304, 130), (128, 363, 1024), (127, 4096, 200),
                (16, 150, 64)]


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_cluster_split_full_oracle(cb, orc, flags):
    import torch
    seen = set()
    for M, K, N in SPLIT_SHAPES:
        A, B = synthetic.matmul_case(M, K, N, flags)
        a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        bn, pieces = cb.matmul_tiling(M, K, N, flags)
        seen.add(pieces)
        c1 = cb.matmul(a, b, flags)
        c2 = cb.matmul(a, b, flags)
        cb.check()
        ref, ref_abs = orc.matmul(A.astype(np.float64), B.astype(np.float64), flags)
        assert_within_tol(c1.cpu().numpy(), ref, ref_abs, "matmul %dx%dx%d f%d (%d pieces)" % (M, K, N, flags, pieces))
        assert torch.equal(c1, c2), "matmul %dx%dx%d f%d: not bit-identical run to run" % (M, K, N, flags)
    assert len(seen - {1}) >= 2, seen
