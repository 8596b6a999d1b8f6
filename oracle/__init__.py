"""CPU oracle for the im2col convolution pipeline of the page
"DirectCompute Neural Network Engine" (directcompute-nn 0.1.0).

TEST INFRASTRUCTURE.  This package is the slow, obviously-correct yardstick the
CUDA library is checked against.  Only the test suite, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` may import it; the library itself never
does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation, OpenMP over
independent outputs).  This module only compiles it, marshals numpy arrays and
rounds each double result once to fp32.

Contraction entries return ``(value_fp32, abs_scale)`` where ``abs_scale`` is
sum_k |a_k b_k| in double: the per-element tolerance of the parity tests is
``1e-4 * abs_scale + 1e-6``.

Parity pins (tests/test_oracle_*.py) hold every function here to something
other than itself: direct convolution, torch's float64 CPU routines, the
im2col/col2im adjoint identity, closed forms and central finite differences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_I64 = ctypes.c_int64
_DP = ctypes.POINTER(ctypes.c_double)
_FP = ctypes.POINTER(ctypes.c_float)
_IP = ctypes.POINTER(ctypes.c_int32)
_LP = ctypes.POINTER(ctypes.c_int64)


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP, no FMA contraction)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    sig = {
        "oracle_im2col": [_I64] * 9 + [_DP, _DP],
        "oracle_col2im": [_I64] * 9 + [_DP, _DP, _DP, _DP],
        "oracle_matmul": [_I64, _I64, _I64, ctypes.c_uint, _DP, _DP, _DP, _DP],
        "oracle_matmul_at": [_I64, _I64, _I64, ctypes.c_uint, _DP, _DP, _I64, _LP, _DP, _DP],
        "oracle_conv_fwd": [_I64] * 10 + [_DP, _DP, _DP, _DP, _DP],
        "oracle_conv_fwd_at": [_I64] * 10 + [_DP, _DP, _DP, _I64, _LP, _DP, _DP],
        "oracle_conv_bwd_data": [_I64] * 10 + [_DP, _DP, _DP, _DP],
        "oracle_conv_bwd_data_at": [_I64] * 10 + [_DP, _DP, _I64, _LP, _DP, _DP],
        "oracle_conv_bwd_filter": [_I64] * 10 + [_DP, _DP, _DP, _DP],
        "oracle_conv_bwd_filter_at": [_I64] * 10 + [_DP, _DP, _I64, _LP, _DP, _DP],
        "oracle_conv_bwd_bias": [_I64] * 4 + [_DP, _DP, _DP],
        "oracle_maxpool_fwd": [_I64] * 8 + [_FP, _FP, _IP],
        "oracle_maxpool_bwd": [_I64] * 6 + [_FP, _IP, _FP],
        "oracle_sgd": [_I64, ctypes.c_float, ctypes.c_float, _FP, _FP],
        "oracle_relu": [_I64, _FP, _FP],
        "oracle_relu_grad": [_I64, _FP, _FP, _FP],
        "oracle_add_bias": [_I64, _I64, _FP, _FP, _FP],
        "oracle_bias_grad_rows": [_I64, _I64, _DP, _DP, _DP],
        "oracle_softmax": [_I64, _I64, _DP, _DP],
        "oracle_softmax_ce": [_I64, _I64, _DP, _IP, _DP, _DP],
        "oracle_grad_accum": [_I64, _FP, _FP],
        "oracle_threads": [],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int if name == "oracle_threads" else None
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the compiled oracle."""
    global _lib
    with _lock:
        if path is not None:
            return _declare(ctypes.CDLL(path))
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


# ---------------------------------------------------------------------------
# helpers

def out_size(size: int, k: int, stride: int, pad: int) -> int:
    """Output extent: floor((size + 2*pad - k) / stride) + 1 (zero padding)."""
    return (size + 2 * pad - k) // stride + 1


def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a, t=_DP):
    return a.ctypes.data_as(t)


def _f32(a):
    """Round double results once to fp32 (IEEE round-to-nearest-even)."""
    return a.astype(np.float32)


class Oracle:
    """Thin marshalling layer over the C oracle.  ``lib`` may point at a
    differently-compiled copy (the mutation tests use that)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def threads(self) -> int:
        return int(self.lib.oracle_threads())

    # -- A1 / A7 ------------------------------------------------------------
    def im2col(self, x, R, stride, pad, exact=False):
        x = _d(x)
        N, C, H, W = x.shape
        P, Q = out_size(H, R, stride, pad), out_size(W, R, stride, pad)
        col = np.empty((C * R * R, N * P * Q), np.float64)
        self.lib.oracle_im2col(N, C, H, W, R, stride, pad, P, Q, _p(x), _p(col))
        return col if exact else _f32(col)

    def col2im(self, col, x_shape, R, stride, pad, exact=False):
        N, C, H, W = x_shape
        P, Q = out_size(H, R, stride, pad), out_size(W, R, stride, pad)
        col = _d(col)
        assert col.shape == (C * R * R, N * P * Q)
        dx = np.empty((N, C, H, W), np.float64)
        dx_abs = np.empty_like(dx)
        self.lib.oracle_col2im(N, C, H, W, R, stride, pad, P, Q, _p(col),
                               ctypes.cast(None, _DP), _p(dx), _p(dx_abs))
        return (dx, dx_abs) if exact else (_f32(dx), dx_abs)

    # -- A9 ------------------------------------------------------------------
    @staticmethod
    def _mm_dims(A, B, flags):
        if flags & 1:
            K, M = A.shape
        else:
            M, K = A.shape
        if flags & 2:
            N, K2 = B.shape
        else:
            K2, N = B.shape
        assert K == K2, "inner dimensions differ"
        return M, K, N

    def matmul(self, A, B, flags=0, exact=False):
        A, B = _d(A), _d(B)
        M, K, N = self._mm_dims(A, B, flags)
        C = np.empty((M, N), np.float64)
        C_abs = np.empty_like(C)
        self.lib.oracle_matmul(M, K, N, flags, _p(A), _p(B), _p(C), _p(C_abs))
        return (C, C_abs) if exact else (_f32(C), C_abs)

    def matmul_at(self, A, B, flags, flat, exact=False):
        A, B = _d(A), _d(B)
        M, K, N = self._mm_dims(A, B, flags)
        flat = np.ascontiguousarray(flat, dtype=np.int64)
        out = np.empty(flat.shape, np.float64)
        out_abs = np.empty_like(out)
        self.lib.oracle_matmul_at(M, K, N, flags, _p(A), _p(B), flat.size,
                                  _p(flat, _LP), _p(out), _p(out_abs))
        return (out, out_abs) if exact else (_f32(out), out_abs)

    # -- conv: A1-A8 -----------------------------------------------------------
    @staticmethod
    def _conv_dims(x_shape, w_shape, stride, pad):
        N, C, H, W = x_shape
        Ko, C2, R, R2 = w_shape
        assert C == C2 and R == R2, "filters must be (outC, inC, k, k)"
        return N, C, H, W, Ko, R, stride, pad, out_size(H, R, stride, pad), out_size(W, R, stride, pad)

    def conv_fwd(self, x, w, b, stride, pad, exact=False):
        x, w = _d(x), _d(w)
        dims = self._conv_dims(x.shape, w.shape, stride, pad)
        N, Ko, P, Q = dims[0], dims[4], dims[8], dims[9]
        y = np.empty((N, Ko, P, Q), np.float64)
        y_abs = np.empty_like(y)
        bb = _d(b) if b is not None else None
        bp = _p(bb) if bb is not None else ctypes.cast(None, _DP)
        self.lib.oracle_conv_fwd(*dims, _p(x), _p(w), bp, _p(y), _p(y_abs))
        return (y, y_abs) if exact else (_f32(y), y_abs)

    def conv_fwd_at(self, x, w, b, stride, pad, flat, exact=False):
        x, w = _d(x), _d(w)
        dims = self._conv_dims(x.shape, w.shape, stride, pad)
        flat = np.ascontiguousarray(flat, dtype=np.int64)
        out = np.empty(flat.shape, np.float64)
        out_abs = np.empty_like(out)
        bb = _d(b) if b is not None else None
        bp = _p(bb) if bb is not None else ctypes.cast(None, _DP)
        self.lib.oracle_conv_fwd_at(*dims, _p(x), _p(w), bp, flat.size,
                                    _p(flat, _LP), _p(out), _p(out_abs))
        return (out, out_abs) if exact else (_f32(out), out_abs)

    def conv_bwd_data(self, w, dy, x_shape, stride, pad, exact=False):
        w, dy = _d(w), _d(dy)
        dims = self._conv_dims(x_shape, w.shape, stride, pad)
        assert dy.shape == (dims[0], dims[4], dims[8], dims[9])
        dx = np.empty(x_shape, np.float64)
        dx_abs = np.empty_like(dx)
        self.lib.oracle_conv_bwd_data(*dims, _p(w), _p(dy), _p(dx), _p(dx_abs))
        return (dx, dx_abs) if exact else (_f32(dx), dx_abs)

    def conv_bwd_data_at(self, w, dy, x_shape, stride, pad, flat, exact=False):
        w, dy = _d(w), _d(dy)
        dims = self._conv_dims(x_shape, w.shape, stride, pad)
        flat = np.ascontiguousarray(flat, dtype=np.int64)
        out = np.empty(flat.shape, np.float64)
        out_abs = np.empty_like(out)
        self.lib.oracle_conv_bwd_data_at(*dims, _p(w), _p(dy), flat.size,
                                         _p(flat, _LP), _p(out), _p(out_abs))
        return (out, out_abs) if exact else (_f32(out), out_abs)

    def conv_bwd_filter(self, x, dy, w_shape, stride, pad, exact=False):
        x, dy = _d(x), _d(dy)
        dims = self._conv_dims(x.shape, w_shape, stride, pad)
        assert dy.shape == (dims[0], dims[4], dims[8], dims[9])
        dw = np.empty(w_shape, np.float64)
        dw_abs = np.empty_like(dw)
        self.lib.oracle_conv_bwd_filter(*dims, _p(x), _p(dy), _p(dw), _p(dw_abs))
        return (dw, dw_abs) if exact else (_f32(dw), dw_abs)

    def conv_bwd_filter_at(self, x, dy, w_shape, stride, pad, flat, exact=False):
        x, dy = _d(x), _d(dy)
        dims = self._conv_dims(x.shape, w_shape, stride, pad)
        flat = np.ascontiguousarray(flat, dtype=np.int64)
        out = np.empty(flat.shape, np.float64)
        out_abs = np.empty_like(out)
        self.lib.oracle_conv_bwd_filter_at(*dims, _p(x), _p(dy), flat.size,
                                           _p(flat, _LP), _p(out), _p(out_abs))
        return (out, out_abs) if exact else (_f32(out), out_abs)

    def conv_bwd_bias(self, dy, exact=False):
        dy = _d(dy)
        N, Ko, P, Q = dy.shape
        db = np.empty(Ko, np.float64)
        db_abs = np.empty_like(db)
        self.lib.oracle_conv_bwd_bias(N, Ko, P, Q, _p(dy), _p(db), _p(db_abs))
        return (db, db_abs) if exact else (_f32(db), db_abs)

    # -- A10 / A11 -------------------------------------------------------------
    def maxpool_fwd(self, x, k, stride):
        x = np.ascontiguousarray(x, dtype=np.float32)
        N, C, H, W = x.shape
        P, Q = out_size(H, k, stride, 0), out_size(W, k, stride, 0)
        y = np.empty((N, C, P, Q), np.float32)
        idx = np.empty((N, C, P, Q), np.int32)
        self.lib.oracle_maxpool_fwd(N, C, H, W, k, stride, P, Q, _p(x, _FP),
                                    _p(y, _FP), _p(idx, _IP))
        return y, idx

    def maxpool_bwd(self, dy, idx, x_shape):
        dy = np.ascontiguousarray(dy, dtype=np.float32)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        N, C, H, W = x_shape
        _, _, P, Q = dy.shape
        dx = np.empty(x_shape, np.float32)
        self.lib.oracle_maxpool_bwd(N, C, H, W, P, Q, _p(dy, _FP), _p(idx, _IP), _p(dx, _FP))
        return dx

    # -- A12 ---------------------------------------------------------------------
    def sgd(self, param, grad, lr, clip):
        p = np.array(param, dtype=np.float32, copy=True)
        g = np.ascontiguousarray(grad, dtype=np.float32)
        assert p.shape == g.shape
        self.lib.oracle_sgd(p.size, lr, clip, _p(p, _FP), _p(g, _FP))
        return p

    # -- training-step pieces (LeNet-5 step) -------------------------------------
    def relu(self, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty_like(x)
        self.lib.oracle_relu(x.size, _p(x, _FP), _p(y, _FP))
        return y

    def relu_grad(self, grad, x):
        g = np.ascontiguousarray(grad, dtype=np.float32)
        x = np.ascontiguousarray(x, dtype=np.float32)
        assert g.shape == x.shape
        dx = np.empty_like(g)
        self.lib.oracle_relu_grad(g.size, _p(g, _FP), _p(x, _FP), _p(dx, _FP))
        return dx

    def add_bias(self, A, b):
        A = np.ascontiguousarray(A, dtype=np.float32)
        b = np.ascontiguousarray(b, dtype=np.float32)
        rows, cols = A.shape
        assert b.shape == (cols,)
        out = np.empty_like(A)
        self.lib.oracle_add_bias(rows, cols, _p(A, _FP), _p(b, _FP), _p(out, _FP))
        return out

    def bias_grad_rows(self, G, exact=False):
        G = _d(G)
        rows, cols = G.shape
        db = np.empty(cols, np.float64)
        db_abs = np.empty_like(db)
        self.lib.oracle_bias_grad_rows(rows, cols, _p(G), _p(db), _p(db_abs))
        return (db, db_abs) if exact else (_f32(db), db_abs)

    def softmax(self, z):
        z = _d(z)
        rows, cols = z.shape
        p = np.empty_like(z)
        self.lib.oracle_softmax(rows, cols, _p(z), _p(p))
        return p

    def softmax_ce(self, z, labels):
        """(grad, per-row losses), both in double: grad = softmax(z) - one_hot,
        loss_i = -log softmax(z)_i[label_i]."""
        z = _d(z)
        rows, cols = z.shape
        lab = np.ascontiguousarray(labels, dtype=np.int32)
        assert lab.shape == (rows,) and lab.min() >= 0 and lab.max() < cols
        grad = np.empty_like(z)
        loss = np.empty(rows, np.float64)
        self.lib.oracle_softmax_ce(rows, cols, _p(z), _p(lab, _IP), _p(grad), _p(loss))
        return grad, loss

    def grad_accum(self, accum, grad):
        acc = np.array(accum, dtype=np.float32, copy=True)
        g = np.ascontiguousarray(grad, dtype=np.float32)
        assert acc.shape == g.shape
        self.lib.oracle_grad_accum(acc.size, _p(g, _FP), _p(acc, _FP))
        return acc


_default = None


def get() -> Oracle:
    """The process-wide oracle over the default build."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
