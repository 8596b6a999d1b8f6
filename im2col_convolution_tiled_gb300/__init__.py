"""im2col_convolution_tiled_gb300 -- Python binding of libconv_b200.

libconv_b200 is the im2col convolution pipeline of the page "DirectCompute
Neural Network Engine" (directcompute-nn 0.1.0) -- forward
(im2col -> filters x columns -> conv_reshape + bias) and backward (filter,
input and bias gradients), its flagged matmul, max pooling and SGD -- as
hand-written sm_103a CUDA kernels behind a C ABI (include/conv_b200.h).

This module only marshals arguments: it checks tensors, allocates outputs and
scratch with torch (device memory and streams are all torch is used for),
builds the shape struct and calls the C entry point of the same name on the
current CUDA stream.  Every step of the computation runs in the library's
kernels; there is no fallback of any kind -- if the shared library cannot be
loaded, the import of the entry points raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "ConvShape", "lib", "load", "conv_fwd", "conv_bwd_data", "conv_bwd_filter", "conv_bwd_filter_bias",
    "conv_bwd_bias",
    "im2col", "col2im", "matmul", "matmul_tiling", "maxpool2d_fwd", "maxpool2d_bwd", "sgd_step", "workspace_bytes",
    "check", "ConvError", "out_size", "LIB_PATH", "launch_count", "relu_fwd", "relu_bwd", "grad_accum", "add_bias",
    "bias_grad_rows", "softmax_ce", "set_math_mode", "math_mode", "math", "CONV_MATH_FP32", "CONV_MATH_TF32",
    "conv_fwd_direct", "conv_bwd_data_direct", "conv_bwd_filter_direct",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libconv_b200.so")

CONV_OP_FWD, CONV_OP_BWD_DATA, CONV_OP_BWD_FILTER = 0, 1, 2


class ConvShape(ctypes.Structure):
    """conv_shape_t: the page's im2col parameter set plus outC."""
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "inC", "inH", "inW", "outC", "kH", "stride", "padding", "outH", "outW")]


class ConvError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = lib().conv_b200_strerror(code).decode() if _lib is not None else str(code)
        super().__init__("%s failed: %s (%d)" % (fn, msg, code))


_lib = None
_P = ctypes.c_void_p
_SHAPE = ctypes.POINTER(ConvShape)
_SIGS = {
    "conv_fwd": ([_SHAPE, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "conv_fwd_relu": ([_SHAPE, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "conv_bwd_data": ([_SHAPE, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "conv_bwd_filter": ([_SHAPE, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "conv_bwd_filter_bias": ([_SHAPE, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "conv_bwd_bias": ([_SHAPE, _P, _P, _P], ctypes.c_int),
    "conv_bwd_data_relu": ([_SHAPE, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "conv_bwd_filter_bias_relu": ([_SHAPE, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "conv_b200_workspace_bytes": ([ctypes.c_int, _SHAPE], ctypes.c_size_t),
    "im2col": ([_SHAPE, _P, _P, _P], ctypes.c_int),
    "col2im": ([_SHAPE, _P, _P, _P], ctypes.c_int),
    "matmul": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32, _P, _P, _P, _P], ctypes.c_int),
    "matmul_tiling": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32, _P, _P, _P, _P, _P],
                      ctypes.c_int),
    "matmul_fused": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32, _P, _P, _P, ctypes.c_int32, _P,
                      _P, _P], ctypes.c_int),
    "maxpool2d_fwd": ([ctypes.c_int32] * 8 + [_P, _P, _P, _P], ctypes.c_int),
    "maxpool2d_bwd": ([ctypes.c_int32] * 8 + [_P, _P, _P, _P], ctypes.c_int),
    "sgd_step": ([ctypes.c_int64, ctypes.c_float, ctypes.c_float, _P, _P, _P], ctypes.c_int),
    "conv_b200_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "conv_b200_check": ([_P], ctypes.c_int),
    "conv_b200_launch_count": ([], ctypes.c_uint64),
    "conv_b200_debug_withhold_stage": ([ctypes.c_int64], ctypes.c_int),
    "conv_fwd_noalloc": ([_SHAPE, _P, _P, _P, _P, _P], ctypes.c_int),
    "relu_fwd": ([ctypes.c_int64, _P, _P, _P], ctypes.c_int),
    "relu_bwd": ([ctypes.c_int64, _P, _P, _P, _P], ctypes.c_int),
    "grad_accum": ([ctypes.c_int64, _P, _P, _P], ctypes.c_int),
    "add_bias": ([ctypes.c_int32, ctypes.c_int32, _P, _P, _P, ctypes.c_int32, _P], ctypes.c_int),
    "bias_grad_rows": ([ctypes.c_int32, ctypes.c_int32, _P, _P, _P], ctypes.c_int),
    "softmax_ce": ([ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "conv_fwd_direct": ([_SHAPE, _P, _P, _P, _P, _P], ctypes.c_int),
    "conv_bwd_data_direct": ([_SHAPE, _P, _P, _P, _P], ctypes.c_int),
    "conv_bwd_filter_direct": ([_SHAPE, _P, _P, _P, _P], ctypes.c_int),
    "conv_b200_set_math_mode": ([ctypes.c_int], ctypes.c_int),
    "conv_b200_math_mode": ([], ctypes.c_int),
}


def load(path: str | None = None):
    """Load libconv_b200.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is None or path is not None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError("libconv_b200.so not found at %s: build it with "
                          "`python -m im2col_convolution_tiled_gb300.build`" % p)
        l = ctypes.CDLL(p)
        for name, (args, res) in _SIGS.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = res
        if path is not None:
            return l
        _lib = l
    return _lib


def lib():
    return load()


def out_size(size: int, k: int, stride: int, pad: int) -> int:
    return (size + 2 * pad - k) // stride + 1


# ---------------------------------------------------------------------------
# marshalling helpers (torch is imported lazily: the C ABI itself needs none)

def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _want(t, name, dtype=None):
    torch = _torch()
    dtype = dtype or torch.float32
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _call(fn, *args):
    rc = getattr(lib(), fn)(*args)
    if rc != 0:
        raise ConvError(fn, rc)


def shape_of(x_shape, w_shape, stride, padding) -> ConvShape:
    N, C, H, W = x_shape
    K, C2, R, R2 = w_shape
    if C2 != C or R2 != R:
        raise ValueError("filters must be (outC, inC, k, k) with inC matching x")
    return ConvShape(N, C, H, W, K, R, stride, padding, out_size(H, R, stride, padding),
                     out_size(W, R, stride, padding))


def workspace_bytes(op: int, s: ConvShape) -> int:
    return int(lib().conv_b200_workspace_bytes(op, ctypes.byref(s)))


def _workspace(op, s, workspace):
    torch = _torch()
    need = workspace_bytes(op, s)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    return workspace, max(need, workspace.numel())


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)

def conv_fwd(x, w, b, stride=1, padding=0, y=None, workspace=None, stream=None, relu=False):
    """y = conv(x, w) + b, NCHW fp32 (b may be None); relu=True: max(0, .) fused
    into the epilogue (conv_fwd_relu)."""
    torch = _torch()
    _want(x, "x"), _want(w, "w")
    if b is not None:
        _want(b, "b")
    s = shape_of(x.shape, w.shape, stride, padding)
    if y is None:
        y = torch.empty((s.batch, s.outC, s.outH, s.outW), dtype=torch.float32, device=x.device)
    _want(y, "y")
    ws, nbytes = _workspace(CONV_OP_FWD, s, workspace)
    _call("conv_fwd_relu" if relu else "conv_fwd", ctypes.byref(s), _ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(ws),
          nbytes, _stream(stream))
    return y


def conv_bwd_data(w, dy, x_shape, stride=1, padding=0, dx=None, workspace=None, stream=None, relu_mask=None):
    """dx = gradient of the convolution with respect to its input.  With
    relu_mask (the ReLU output that followed the convolution, shaped like dy)
    the convolution's gradient is dy * (relu_mask > 0), formed as dy is read
    (conv_bwd_data_relu)."""
    torch = _torch()
    _want(w, "w"), _want(dy, "dy")
    if relu_mask is not None:
        _want(relu_mask, "relu_mask")
    s = shape_of(tuple(x_shape), w.shape, stride, padding)
    if dx is None:
        dx = torch.empty(tuple(x_shape), dtype=torch.float32, device=dy.device)
    _want(dx, "dx")
    ws, nbytes = _workspace(CONV_OP_BWD_DATA, s, workspace)
    if relu_mask is not None:
        _call("conv_bwd_data_relu", ctypes.byref(s), _ptr(w), _ptr(dy), _ptr(relu_mask), _ptr(dx), _ptr(ws), nbytes,
              _stream(stream))
    else:
        _call("conv_bwd_data", ctypes.byref(s), _ptr(w), _ptr(dy), _ptr(dx), _ptr(ws), nbytes, _stream(stream))
    return dx


def conv_bwd_filter(x, dy, w_shape, stride=1, padding=0, dw=None, workspace=None, stream=None):
    """dw = gradient of the convolution with respect to its filters."""
    torch = _torch()
    _want(x, "x"), _want(dy, "dy")
    s = shape_of(x.shape, tuple(w_shape), stride, padding)
    if dw is None:
        dw = torch.empty(tuple(w_shape), dtype=torch.float32, device=x.device)
    _want(dw, "dw")
    ws, nbytes = _workspace(CONV_OP_BWD_FILTER, s, workspace)
    _call("conv_bwd_filter", ctypes.byref(s), _ptr(x), _ptr(dy), _ptr(dw), _ptr(ws), nbytes, _stream(stream))
    return dw


def conv_bwd_filter_bias(x, dy, w_shape, stride=1, padding=0, dw=None, db=None, workspace=None, stream=None,
                         relu_mask=None):
    """(dw, db): filter and bias gradients from one pass over dy.  With
    relu_mask the convolution's gradient is dy * (relu_mask > 0), formed as dy
    is read (conv_bwd_filter_bias_relu)."""
    torch = _torch()
    _want(x, "x"), _want(dy, "dy")
    if relu_mask is not None:
        _want(relu_mask, "relu_mask")
    s = shape_of(x.shape, tuple(w_shape), stride, padding)
    if dw is None:
        dw = torch.empty(tuple(w_shape), dtype=torch.float32, device=x.device)
    if db is None:
        db = torch.empty((w_shape[0],), dtype=torch.float32, device=x.device)
    _want(dw, "dw"), _want(db, "db")
    ws, nbytes = _workspace(CONV_OP_BWD_FILTER, s, workspace)
    if relu_mask is not None:
        _call("conv_bwd_filter_bias_relu", ctypes.byref(s), _ptr(x), _ptr(dy), _ptr(relu_mask), _ptr(dw), _ptr(db),
              _ptr(ws), nbytes, _stream(stream))
    else:
        _call("conv_bwd_filter_bias", ctypes.byref(s), _ptr(x), _ptr(dy), _ptr(dw), _ptr(db), _ptr(ws), nbytes,
              _stream(stream))
    return dw, db


def conv_bwd_bias(dy, db=None, stream=None):
    """db[k] = sum of dy[:, k] over batch and space."""
    torch = _torch()
    _want(dy, "dy")
    N, K, P, Q = dy.shape
    # any consistent input geometry gives the same sums: a 1x1 filter on a PxQ input
    s = ConvShape(N, 1, P, Q, K, 1, 1, 0, P, Q)
    if db is None:
        db = torch.empty((K,), dtype=torch.float32, device=dy.device)
    _want(db, "db")
    _call("conv_bwd_bias", ctypes.byref(s), _ptr(dy), _ptr(db), _stream(stream))
    return db


def im2col(x, k, stride=1, padding=0, col=None, stream=None):
    torch = _torch()
    _want(x, "x")
    N, C, H, W = x.shape
    s = ConvShape(N, C, H, W, 1, k, stride, padding, out_size(H, k, stride, padding), out_size(W, k, stride, padding))
    if col is None:
        col = torch.empty((C * k * k, N * s.outH * s.outW), dtype=torch.float32, device=x.device)
    _want(col, "col")
    _call("im2col", ctypes.byref(s), _ptr(x), _ptr(col), _stream(stream))
    return col


def col2im(col, x_shape, k, stride=1, padding=0, dx=None, stream=None):
    torch = _torch()
    _want(col, "col")
    N, C, H, W = x_shape
    s = ConvShape(N, C, H, W, 1, k, stride, padding, out_size(H, k, stride, padding), out_size(W, k, stride, padding))
    if dx is None:
        dx = torch.empty(tuple(x_shape), dtype=torch.float32, device=col.device)
    _want(dx, "dx")
    _call("col2im", ctypes.byref(s), _ptr(col), _ptr(dx), _stream(stream))
    return dx


def matmul(A, B, flags=0, C=None, stream=None, bias=None, relu=False, gate=None):
    """C = op(A) op(B); flags bit 0: A stored K x M, bit 1: B stored N x K.
    With bias ([N]), relu or gate ([M, N]) the epilogue adds the bias per
    column, applies max(0, .) and multiplies by (gate > 0), in that order, in
    the same pass (matmul_fused)."""
    torch = _torch()
    _want(A, "A"), _want(B, "B")
    if flags & 1:
        K, M = A.shape
    else:
        M, K = A.shape
    if flags & 2:
        N, K2 = B.shape
    else:
        K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _want(C, "C")
    if bias is None and gate is None and not relu:
        _call("matmul", M, K, N, flags, _ptr(A), _ptr(B), _ptr(C), _stream(stream))
        return C
    if bias is not None:
        _want(bias, "bias")
        if tuple(bias.shape) != (N,):
            raise ValueError("bias must have shape (%d,)" % N)
    if gate is not None:
        _want(gate, "gate")
        if tuple(gate.shape) != (M, N):
            raise ValueError("gate must have shape (%d, %d)" % (M, N))
    _call("matmul_fused", M, K, N, flags, _ptr(A), _ptr(B), _ptr(bias) if bias is not None else None,
          1 if relu else 0, _ptr(gate) if gate is not None else None, _ptr(C), _stream(stream))
    return C


def matmul_tiling(M, K, N, flags=0, A=None, B=None, with_tma=False):
    """(tile columns, K pieces per tile) that matmul uses for this shape, plus
    whether the operands arrive by TMA when with_tma (A and B: the operand
    tensors, whose alignment decides; 16-byte aligned when omitted)."""
    bn, pieces, tma = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    pa = ctypes.c_void_p(A.data_ptr()) if A is not None else ctypes.c_void_p(0)
    pb = ctypes.c_void_p(B.data_ptr()) if B is not None else ctypes.c_void_p(0)
    _call("matmul_tiling", M, K, N, flags, pa, pb, ctypes.addressof(bn), ctypes.addressof(pieces),
          ctypes.addressof(tma))
    return (bn.value, pieces.value, bool(tma.value)) if with_tma else (bn.value, pieces.value)


def maxpool2d_fwd(x, k, stride, y=None, idx=None, stream=None):
    torch = _torch()
    _want(x, "x")
    N, C, H, W = x.shape
    P, Q = (H - k) // stride + 1, (W - k) // stride + 1
    if y is None:
        y = torch.empty((N, C, P, Q), dtype=torch.float32, device=x.device)
    if idx is None:
        idx = torch.empty((N, C, P, Q), dtype=torch.int32, device=x.device)
    _want(y, "y"), _want(idx, "idx", torch.int32)
    _call("maxpool2d_fwd", N, C, H, W, k, stride, P, Q, _ptr(x), _ptr(y), _ptr(idx), _stream(stream))
    return y, idx


def maxpool2d_bwd(dy, idx, x_shape, k, stride, dx=None, stream=None):
    torch = _torch()
    _want(dy, "dy"), _want(idx, "idx", torch.int32)
    N, C, H, W = x_shape
    _, _, P, Q = dy.shape
    if dx is None:
        dx = torch.empty(tuple(x_shape), dtype=torch.float32, device=dy.device)
    _want(dx, "dx")
    _call("maxpool2d_bwd", N, C, H, W, k, stride, P, Q, _ptr(dy), _ptr(idx), _ptr(dx), _stream(stream))
    return dx


def sgd_step(param, grad, lr, clip, stream=None):
    """param -= lr * clamp(grad, -clip, clip), in place."""
    _want(param, "param"), _want(grad, "grad")
    if param.numel() != grad.numel():
        raise ValueError("param and grad sizes differ")
    _call("sgd_step", param.numel(), lr, clip, _ptr(param), _ptr(grad), _stream(stream))
    return param


def relu_fwd(x, y=None, stream=None):
    """y = max(0, x) (y may be x)."""
    torch = _torch()
    _want(x, "x")
    y = torch.empty_like(x) if y is None else y
    _want(y, "y")
    if y.numel() != x.numel():
        raise ValueError("x and y sizes differ")
    _call("relu_fwd", x.numel(), _ptr(x), _ptr(y), _stream(stream))
    return y


def relu_bwd(dy, x, dx=None, stream=None):
    """dx = dy * (x > 0); x is the ReLU's input or output (dx may be dy)."""
    torch = _torch()
    _want(dy, "dy"), _want(x, "x")
    dx = torch.empty_like(dy) if dx is None else dx
    _want(dx, "dx")
    if not (dy.numel() == x.numel() == dx.numel()):
        raise ValueError("dy, x and dx sizes differ")
    _call("relu_bwd", dy.numel(), _ptr(dy), _ptr(x), _ptr(dx), _stream(stream))
    return dx


def grad_accum(accum, grad, stream=None):
    """accum += grad, in place."""
    _want(accum, "accum"), _want(grad, "grad")
    if accum.numel() != grad.numel():
        raise ValueError("accum and grad sizes differ")
    _call("grad_accum", accum.numel(), _ptr(grad), _ptr(accum), _stream(stream))
    return accum


def add_bias(a, b, out=None, relu=False, stream=None):
    """out[i, j] = a[i, j] + b[j] (then max(0, .) when relu); out may be a."""
    torch = _torch()
    _want(a, "a"), _want(b, "b")
    rows, cols = a.shape
    if b.numel() != cols:
        raise ValueError("bias length must equal the number of columns")
    out = torch.empty_like(a) if out is None else out
    _want(out, "out")
    _call("add_bias", rows, cols, _ptr(a), _ptr(b), _ptr(out), 1 if relu else 0, _stream(stream))
    return out


def bias_grad_rows(grad, db=None, stream=None):
    """db[j] = sum_i grad[i, j] (a linear layer's bias gradient)."""
    torch = _torch()
    _want(grad, "grad")
    rows, cols = grad.shape
    db = torch.empty(cols, dtype=torch.float32, device=grad.device) if db is None else db
    _want(db, "db")
    _call("bias_grad_rows", rows, cols, _ptr(grad), _ptr(db), _stream(stream))
    return db


def softmax_ce(logits, labels, dlogits=None, loss=None, probs=None, stream=None):
    """(dlogits, loss): dlogits = softmax(logits) - one_hot(labels) per row and
    loss (a 1-element tensor) = sum over rows of -log softmax(logits)[label]."""
    torch = _torch()
    _want(logits, "logits"), _want(labels, "labels", torch.int32)
    rows, cols = logits.shape
    if labels.numel() != rows:
        raise ValueError("one label per row")
    dlogits = torch.empty_like(logits) if dlogits is None else dlogits
    loss = torch.empty(1, dtype=torch.float32, device=logits.device) if loss is None else loss
    _want(dlogits, "dlogits"), _want(loss, "loss")
    if probs is not None:
        _want(probs, "probs")
    _call("softmax_ce", rows, cols, _ptr(logits), _ptr(labels), _ptr(probs), _ptr(dlogits), _ptr(loss),
          _stream(stream))
    return dlogits, loss


def conv_fwd_direct(x, w, b, stride=1, padding=0, y=None, stream=None):
    """Direct (CUDA-core) forward convolution; same result definition as conv_fwd."""
    torch = _torch()
    _want(x, "x"), _want(w, "w")
    if b is not None:
        _want(b, "b")
    s = shape_of(x.shape, w.shape, stride, padding)
    if y is None:
        y = torch.empty((s.batch, s.outC, s.outH, s.outW), dtype=torch.float32, device=x.device)
    _want(y, "y")
    _call("conv_fwd_direct", ctypes.byref(s), _ptr(x), _ptr(w), _ptr(b), _ptr(y), _stream(stream))
    return y


def conv_bwd_data_direct(w, dy, x_shape, stride=1, padding=0, dx=None, stream=None):
    torch = _torch()
    _want(w, "w"), _want(dy, "dy")
    s = shape_of(tuple(x_shape), w.shape, stride, padding)
    if dx is None:
        dx = torch.empty(tuple(x_shape), dtype=torch.float32, device=dy.device)
    _want(dx, "dx")
    _call("conv_bwd_data_direct", ctypes.byref(s), _ptr(w), _ptr(dy), _ptr(dx), _stream(stream))
    return dx


def conv_bwd_filter_direct(x, dy, w_shape, stride=1, padding=0, dw=None, stream=None):
    torch = _torch()
    _want(x, "x"), _want(dy, "dy")
    s = shape_of(x.shape, tuple(w_shape), stride, padding)
    if dw is None:
        dw = torch.empty(tuple(w_shape), dtype=torch.float32, device=x.device)
    _want(dw, "dw")
    _call("conv_bwd_filter_direct", ctypes.byref(s), _ptr(x), _ptr(dy), _ptr(dw), _stream(stream))
    return dw


CONV_MATH_FP32, CONV_MATH_TF32 = 0, 1


def set_math_mode(mode) -> int:
    """Select the contractions' arithmetic (process-wide): CONV_MATH_FP32 (3xTF32,
    the default) or CONV_MATH_TF32 (one TF32 product).  Returns the previous mode."""
    prev = int(lib().conv_b200_set_math_mode(int(mode)))
    if prev < 0:
        raise ConvError("conv_b200_set_math_mode", prev)
    return prev


def math_mode() -> int:
    return int(lib().conv_b200_math_mode())


class math:
    """Context manager: ``with math(CONV_MATH_TF32): ...`` restores the previous mode on exit."""

    def __init__(self, mode):
        self.mode = mode

    def __enter__(self):
        self.prev = set_math_mode(self.mode)
        return self

    def __exit__(self, *exc):
        set_math_mode(self.prev)


def launch_count() -> int:
    """Kernels launched by the library so far (see conv_b200_launch_count)."""
    return int(lib().conv_b200_launch_count())


def check(stream=None):
    """Synchronise the stream and raise if a kernel latched a device error."""
    _call("conv_b200_check", _stream(stream))
