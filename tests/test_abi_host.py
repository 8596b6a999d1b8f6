"""Host-only checks of the C ABI: the library loads, exports every entry point
declared in include/*.h, and rejects bad arguments with the documented codes
before touching the GPU (these run without a GPU)."""
import ctypes
import os
import re

import pytest

import im2col_convolution_tiled_gb300 as cb
from im2col_convolution_tiled_gb300 import ConvShape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONV_OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_OVERFLOW, ERR_WORKSPACE = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def lib():
    from im2col_convolution_tiled_gb300 import build
    build.build()
    return cb.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, re.M):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["conv_fwd", "conv_fwd_relu", "conv_bwd_data", "conv_bwd_filter", "conv_bwd_filter_bias", "conv_bwd_bias", "im2col",
              "col2im", "matmul", "matmul_tiling", "matmul_fused",
              "maxpool2d_fwd", "maxpool2d_bwd", "sgd_step", "conv_b200_strerror", "conv_b200_check",
              "conv_b200_workspace_bytes", "relu_fwd", "relu_bwd", "grad_accum", "add_bias", "bias_grad_rows",
              "softmax_ce", "conv_b200_set_math_mode", "conv_b200_math_mode", "conv_fwd_direct",
              "conv_bwd_data_direct", "conv_bwd_filter_direct"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def good_shape():
    return ConvShape(2, 3, 9, 9, 4, 3, 2, 1, 5, 5)


FAKE = ctypes.c_void_p(0x10000)       # aligned, never dereferenced (validation fails first)
MIS = ctypes.c_void_p(0x10004)        # misaligned
NULL = ctypes.c_void_p(0)


def test_shape_validation(lib):
    s = good_shape()
    bad = ConvShape(2, 3, 9, 9, 4, 3, 2, 1, 6, 5)            # outH inconsistent
    assert lib.conv_fwd(ctypes.byref(bad), FAKE, FAKE, NULL, FAKE, FAKE, 1 << 20, NULL) == ERR_SHAPE
    for field in ["batch", "inC", "inH", "inW", "outC", "kH", "stride"]:
        t = good_shape()
        setattr(t, field, 0)
        assert lib.conv_fwd(ctypes.byref(t), FAKE, FAKE, NULL, FAKE, FAKE, 1 << 20, NULL) == ERR_SHAPE, field
    t = good_shape()
    t.padding = -1
    assert lib.conv_bwd_data(ctypes.byref(t), FAKE, FAKE, FAKE, FAKE, 1 << 20, NULL) == ERR_SHAPE
    t = ConvShape(1, 1, 2, 2, 1, 5, 1, 0, 0, 0)               # kernel larger than padded input
    assert lib.im2col(ctypes.byref(t), FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.conv_fwd(None, FAKE, FAKE, NULL, FAKE, FAKE, 0, NULL) == ERR_NULL
    assert lib.conv_b200_workspace_bytes(0, ctypes.byref(bad)) == 0
    assert lib.conv_b200_workspace_bytes(7, ctypes.byref(s)) == 0


def test_pointer_validation(lib):
    s = good_shape()
    assert lib.conv_fwd(ctypes.byref(s), NULL, FAKE, NULL, FAKE, FAKE, 1 << 20, NULL) == ERR_NULL
    assert lib.conv_fwd(ctypes.byref(s), MIS, FAKE, NULL, FAKE, FAKE, 1 << 20, NULL) == ERR_ALIGN
    assert lib.conv_fwd(ctypes.byref(s), FAKE, FAKE, MIS, FAKE, FAKE, 1 << 20, NULL) == ERR_ALIGN
    assert lib.conv_bwd_filter(ctypes.byref(s), FAKE, NULL, FAKE, FAKE, 1 << 20, NULL) == ERR_NULL
    assert lib.conv_bwd_bias(ctypes.byref(s), FAKE, NULL, NULL) == ERR_NULL
    assert lib.conv_bwd_filter_bias(ctypes.byref(s), FAKE, FAKE, FAKE, NULL, FAKE, 1 << 20, NULL) == ERR_NULL
    assert lib.conv_bwd_filter_bias(ctypes.byref(s), FAKE, FAKE, FAKE, MIS, FAKE, 1 << 20, NULL) == ERR_ALIGN
    assert lib.col2im(ctypes.byref(s), FAKE, MIS, NULL) == ERR_ALIGN
    assert lib.matmul(4, 4, 4, 0, FAKE, NULL, FAKE, NULL) == ERR_NULL
    assert lib.maxpool2d_fwd(1, 1, 4, 4, 2, 2, 2, 2, FAKE, FAKE, MIS, NULL) == ERR_ALIGN
    assert lib.sgd_step(8, 0.1, 1.0, NULL, FAKE, NULL) == ERR_NULL


def test_workspace_validation(lib):
    s = ConvShape(2, 3, 9, 9, 4, 3, 1, 1, 9, 9)
    need = lib.conv_b200_workspace_bytes(0, ctypes.byref(s))
    assert need > 0
    assert lib.conv_fwd(ctypes.byref(s), FAKE, FAKE, NULL, FAKE, NULL, need, NULL) == ERR_WORKSPACE
    assert lib.conv_fwd(ctypes.byref(s), FAKE, FAKE, NULL, FAKE, FAKE, need - 1, NULL) == ERR_WORKSPACE
    assert lib.conv_b200_workspace_bytes(1, ctypes.byref(s)) > 0


def test_size_validation(lib):
    assert lib.matmul(0, 4, 4, 0, FAKE, FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.matmul(4, 4, 4, 4, FAKE, FAKE, FAKE, NULL) == ERR_SHAPE          # flags > 3
    assert lib.matmul(65536, 65536, 4, 0, FAKE, FAKE, FAKE, NULL) == ERR_OVERFLOW
    assert lib.maxpool2d_fwd(1, 1, 4, 4, 2, 2, 3, 2, FAKE, FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.maxpool2d_bwd(1, 1, 4, 4, 5, 2, 1, 1, FAKE, FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.sgd_step(-1, 0.1, 1.0, FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.sgd_step(0, 0.1, 1.0, NULL, NULL, NULL) == CONV_OK              # nothing to do
    big = ConvShape(1024, 1024, 64, 64, 8, 1, 1, 0, 64, 64)                    # x has 2^32 elements
    assert lib.conv_fwd(ctypes.byref(big), FAKE, FAKE, NULL, FAKE, FAKE, 1 << 30, NULL) == ERR_OVERFLOW


def test_training_piece_validation(lib):
    assert lib.relu_fwd(-1, FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.relu_fwd(0, NULL, NULL, NULL) == CONV_OK                       # nothing to do
    assert lib.relu_fwd(8, NULL, FAKE, NULL) == ERR_NULL
    assert lib.relu_bwd(8, FAKE, MIS, FAKE, NULL) == ERR_ALIGN
    assert lib.grad_accum(8, FAKE, NULL, NULL) == ERR_NULL
    assert lib.add_bias(0, 4, FAKE, FAKE, FAKE, 0, NULL) == ERR_SHAPE
    assert lib.add_bias(4, 4, FAKE, NULL, FAKE, 1, NULL) == ERR_NULL
    assert lib.add_bias(65536, 65536, FAKE, FAKE, FAKE, 0, NULL) == ERR_OVERFLOW
    assert lib.bias_grad_rows(4, 0, FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.bias_grad_rows(4, 4, FAKE, MIS, NULL) == ERR_ALIGN
    assert lib.softmax_ce(4, 10, FAKE, NULL, NULL, FAKE, FAKE, NULL) == ERR_NULL     # labels
    assert lib.softmax_ce(4, 10, FAKE, FAKE, MIS, FAKE, FAKE, NULL) == ERR_ALIGN     # probs (optional)
    assert lib.softmax_ce(4, 10, FAKE, FAKE, NULL, FAKE, NULL, NULL) == ERR_NULL     # loss
    assert lib.softmax_ce(-4, 10, FAKE, FAKE, NULL, FAKE, FAKE, NULL) == ERR_SHAPE


def test_matmul_engine_hook_validation(lib):
    """The engine test hook defaults to the plan (-1), returns the previous
    setting and rejects values outside -1..1 (no launch happens here)."""
    assert lib.conv_b200_debug_matmul_engine(2) == ERR_SHAPE
    assert lib.conv_b200_debug_matmul_engine(-2) == ERR_SHAPE
    assert lib.conv_b200_debug_matmul_engine(1) == -1
    assert lib.conv_b200_debug_matmul_engine(0) == 1
    assert lib.conv_b200_debug_matmul_engine(-1) == 0


def test_matmul_fused_validation(lib):
    """matmul_fused validates like matmul; bias and gate are optional."""
    assert lib.matmul_fused(4, 4, 4, 0, NULL, FAKE, NULL, 1, NULL, FAKE, NULL) == ERR_NULL
    assert lib.matmul_fused(4, 4, 4, 0, FAKE, FAKE, NULL, 1, NULL, MIS, NULL) == ERR_ALIGN
    assert lib.matmul_fused(0, 4, 4, 0, FAKE, FAKE, NULL, 0, NULL, FAKE, NULL) == ERR_SHAPE
    assert lib.matmul_fused(4, 4, 4, 4, FAKE, FAKE, FAKE, 0, FAKE, FAKE, NULL) == ERR_SHAPE
    assert lib.matmul_fused(65536, 65536, 4, 0, FAKE, FAKE, NULL, 0, NULL, FAKE, NULL) == ERR_OVERFLOW


def test_matmul_tiling_validation(lib):
    """The tiling query validates its arguments before it looks for a device."""
    bn, pieces, tma = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    assert lib.matmul_tiling(4, 4, 4, 0, NULL, NULL, NULL, ctypes.byref(pieces), ctypes.byref(tma)) == ERR_NULL
    assert lib.matmul_tiling(4, 4, 4, 0, NULL, NULL, ctypes.byref(bn), NULL, ctypes.byref(tma)) == ERR_NULL
    assert lib.matmul_tiling(4, 4, 4, 0, NULL, NULL, ctypes.byref(bn), ctypes.byref(pieces), NULL) == ERR_NULL
    assert lib.matmul_tiling(0, 4, 4, 0, NULL, NULL, ctypes.byref(bn), ctypes.byref(pieces),
                             ctypes.byref(tma)) == ERR_SHAPE
    assert lib.matmul_tiling(4, 4, 4, 4, NULL, NULL, ctypes.byref(bn), ctypes.byref(pieces),
                             ctypes.byref(tma)) == ERR_SHAPE


def test_math_mode_switch(lib):
    assert lib.conv_b200_math_mode() == 0                        # 3xTF32 by default
    assert lib.conv_b200_set_math_mode(2) == ERR_SHAPE           # unknown: rejected, nothing changes
    assert lib.conv_b200_math_mode() == 0
    assert lib.conv_b200_set_math_mode(1) == 0                   # returns the previous mode
    assert lib.conv_b200_math_mode() == 1
    assert lib.conv_b200_set_math_mode(0) == 1
    with cb.math(cb.CONV_MATH_TF32):
        assert cb.math_mode() == cb.CONV_MATH_TF32
    assert cb.math_mode() == cb.CONV_MATH_FP32


def test_withhold_hook_validation(lib):
    """The bounded-wait test hook is off by default, rejects k < -1 and can be
    cancelled (no launch happens here)."""
    assert lib.conv_b200_debug_withhold_stage(-2) == ERR_SHAPE
    assert lib.conv_b200_debug_withhold_stage(3) == CONV_OK
    assert lib.conv_b200_debug_withhold_stage(-1) == CONV_OK


def test_relu_fused_gradient_validation(lib):
    """conv_bwd_data_relu / conv_bwd_filter_bias_relu validate like the unfused
    calls, including the mask pointer (db may be NULL in the filter call)."""
    s = good_shape()
    ws = ctypes.c_size_t(1 << 30)
    assert lib.conv_bwd_data_relu(ctypes.byref(s), FAKE, FAKE, NULL, FAKE, FAKE, ws, None) == ERR_NULL
    assert lib.conv_bwd_data_relu(ctypes.byref(s), FAKE, FAKE, MIS, FAKE, FAKE, ws, None) == ERR_ALIGN
    assert lib.conv_bwd_filter_bias_relu(ctypes.byref(s), FAKE, FAKE, NULL, FAKE, NULL, FAKE, ws, None) == ERR_NULL
    assert lib.conv_bwd_filter_bias_relu(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, MIS, FAKE, ws, None) == ERR_ALIGN
    bad = ConvShape(2, 3, 9, 9, 4, 3, 2, 1, 6, 5)
    assert lib.conv_bwd_data_relu(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, ws, None) == ERR_SHAPE


def test_strerror(lib):
    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10, -99]:
        assert isinstance(lib.conv_b200_strerror(code), bytes)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(OSError):
        cb.load(str(tmp_path / "nope.so"))
