"""Helpers for the GPU parity tests: guard-zone buffers, transfers and the
per-element tolerance check against the oracle."""
import numpy as np

GUARD = 4096            # floats of slack on each side of every buffer
CANARY = np.float32(-1.2345e30)


def torch():
    import torch as t
    return t


class Guarded:
    """A device tensor living in the middle of a larger allocation.  Outputs
    get canary-filled slack (checked afterwards: nothing may be written
    outside); inputs get NaN-filled slack (an out-of-bounds read would make
    NaNs show up in the results)."""

    def __init__(self, shape, dtype="float32", fill=None, data=None):
        t = torch()
        self.shape = tuple(shape)
        n = int(np.prod(self.shape)) if self.shape else 1
        tdtype = {"float32": t.float32, "int32": t.int32}[dtype]
        self.base = t.empty(n + 2 * GUARD, dtype=tdtype, device="cuda")
        if fill is None:
            fill = float("nan") if (data is not None and dtype == "float32") else CANARY
        if dtype == "int32":
            fill = -7 if fill is CANARY or (isinstance(fill, float) and np.isnan(fill)) else int(fill)
        self.fill = fill
        self.base.fill_(fill)
        self.t = self.base[GUARD:GUARD + n].view(self.shape)
        if data is not None:
            self.t.copy_(t.from_numpy(np.ascontiguousarray(data)))

    def guards_intact(self):
        t = torch()
        lo, hi = self.base[:GUARD], self.base[-GUARD:]
        if self.base.dtype == t.float32 and isinstance(self.fill, float) and np.isnan(self.fill):
            return bool(t.isnan(lo).all() and t.isnan(hi).all())
        return bool((lo == self.fill).all() and (hi == self.fill).all())

    def numpy(self):
        return self.t.cpu().numpy()


def dev_in(a):
    """Input tensor with NaN slack on both sides."""
    return Guarded(a.shape, "int32" if a.dtype == np.int32 else "float32", data=a)


def dev_out(shape, dtype="float32"):
    return Guarded(shape, dtype)


def assert_within_tol(gpu, ref, ref_abs, what=""):
    """|gpu - oracle| <= 1e-4 * sum|a_k b_k| + 1e-6, element by element."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), "%s: non-finite output" % what
    err = np.abs(gpu - ref)
    tol = 1e-4 * np.asarray(ref_abs, np.float64) + 1e-6
    bad = err > tol
    if bad.any():
        i = np.argmax(err - tol)
        raise AssertionError("%s: %d/%d elements out of tolerance; worst at flat %d: gpu %r oracle %r tol %r"
                             % (what, int(bad.sum()), bad.size, i, gpu.ravel()[i], ref.ravel()[i], tol.ravel()[i]))
    return float((err / tol).max()) if err.size else 0.0
