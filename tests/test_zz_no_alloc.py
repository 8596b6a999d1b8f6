"""conv_fwd_noalloc: the forward convolution for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Called here
through the C ABI directly, twice in a row on different shapes, and checked
bit for bit against conv_fwd's output (and against the oracle within the
parity tolerance); shapes too large for the built-in array must be refused.
This file is collected last on purpose: it must pass alone in a fresh process
as well as after every other test."""
import ctypes

import numpy as np
import pytest

import synthetic

pytestmark = pytest.mark.gpu

CONV_ERR_SCRATCH_LIMIT = -9


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from im2col_convolution_tiled_gb300 import build
    build.build()
    import im2col_convolution_tiled_gb300 as cb
    import oracle
    return cb, cb.load(), oracle.get(), torch


def run_noalloc(env, L):
    cb, lib, orc, torch = env
    x, w, b, _ = L.make()
    b = synthetic.normal(b.shape, L.seed_base + 7, std=0.1)
    xt, wt, bt = (torch.from_numpy(a).cuda() for a in (x, w, b))
    s = cb.shape_of(L.x_shape, L.w_shape, L.stride, L.pad)
    y_ref = cb.conv_fwd(xt, wt, bt, L.stride, L.pad)          # the existing entry point
    y = torch.empty(L.y_shape, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.conv_fwd_noalloc(ctypes.byref(s), ctypes.c_void_p(xt.data_ptr()), ctypes.c_void_p(wt.data_ptr()),
                              ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(y.data_ptr()), stream)
    assert rc == 0, lib.conv_b200_strerror(rc)
    cb.check()
    got, ref = y.cpu().numpy(), y_ref.cpu().numpy()
    assert np.isfinite(got).all()
    # the same kernels on the same inputs: bit for bit conv_fwd's result, so a
    # stale region of the shared scratch would show even if it moved results slightly
    assert np.array_equal(got, ref)
    if orc is not None:
        ref64, y_abs = orc.conv_fwd(x, w, b, L.stride, L.pad, exact=True)   # and within the parity tolerance
        assert (np.abs(got.astype(np.float64) - ref64) <= 1e-4 * y_abs + 1e-6).all()


def test_noalloc_two_calls_match_conv_fwd(env):
    # two different layers back to back: the second call must not see the first's scratch
    run_noalloc(env, synthetic.ALEXNET_CONV2_5[0].with_batch(2))   # 192 x 1600 filters, chunked channels
    run_noalloc(env, synthetic.ALEXNET_CONV1.with_batch(2))        # 64 x 363 filters, stride 4, tap groups


def test_noalloc_alexnet_batch128_limits(env):
    """At batch 128 the scratch of a forward call includes the batch-sized
    staged copy of x: only conv2's fits the array; the others are refused
    before any launch.  conv2 itself must then run and equal conv_fwd."""
    cb, lib, orc, torch = env
    fits = []
    for L in synthetic.ALEXNET:
        s = cb.shape_of(L.x_shape, L.w_shape, L.stride, L.pad)
        need = cb.workspace_bytes(0, s)
        if need <= 8 << 20:
            fits.append(L.name)
        else:
            fake = ctypes.c_void_p(0x10000)   # never touched: refused first
            assert lib.conv_fwd_noalloc(ctypes.byref(s), fake, fake, fake, fake, None) == CONV_ERR_SCRATCH_LIMIT
    assert fits == ["alexnet_conv2_b128"]
    run_noalloc((cb, lib, None, torch), synthetic.ALEXNET_CONV2_5[0])


def test_noalloc_refuses_oversized_shape(env):
    cb, lib, _, _ = env
    s = cb.ConvShape(1, 512, 8, 8, 512, 3, 1, 1, 8, 8)           # 512 x 4608 filters: ~19 MB of tiles
    need = cb.workspace_bytes(0, s)
    assert need > 8 << 20
    fake = ctypes.c_void_p(0x10000)                               # never touched: refused first
    assert lib.conv_fwd_noalloc(ctypes.byref(s), fake, fake, fake, fake, None) == CONV_ERR_SCRATCH_LIMIT
