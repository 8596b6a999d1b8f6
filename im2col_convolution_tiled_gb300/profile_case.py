"""Run one library entry point on one workload a few times -- a small, fixed
command for a profiler (for example Nsight Compute) to attach to.

    python -m im2col_convolution_tiled_gb300.profile_case --layer alexnet_conv2_b128 --op fwd --reps 3

--op is one of fwd, dgrad, wgrad, bias, pool, im2col, col2im, matmul (matmul
uses --mnk M,N,K and --flags).  Inputs are the seeded synthetic workload
tensors; nothing is checked.  With --time N the command then times N more
back-to-back calls between CUDA events on the launching stream and prints the
mean time per call (and, for the HBM-bound ops, the algorithmic bytes per call
and the rate they imply).
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    import im2col_convolution_tiled_gb300 as cb
    import synthetic

    ap = argparse.ArgumentParser()
    ap.add_argument("--layer", default="alexnet_conv2_b128")
    ap.add_argument("--op", default="fwd",
                    choices=["fwd", "dgrad", "wgrad", "bias", "pool", "im2col", "col2im", "matmul"])
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--mnk", default="4096,4096,4096")
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--time", type=int, default=0)
    a = ap.parse_args(argv)

    cb.load()
    layers = {L.name: L for L in synthetic.ALEXNET + synthetic.LENET + (synthetic.SINGLE,)}
    if a.op == "matmul":
        M, N, K = (int(v) for v in a.mnk.split(","))
        A, B = synthetic.matmul_case(M, K, N, a.flags)
        At, Bt = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        C = torch.empty((M, N), device="cuda")
        run = lambda: cb.matmul(At, Bt, a.flags, C=C)
    else:
        L = layers[a.layer]
        x, w, b, dy = L.make()
        xt, wt, bt, dyt = (torch.from_numpy(v).cuda() for v in (x, w, b, dy))
        s = cb.shape_of(L.x_shape, L.w_shape, L.stride, L.pad)
        ws = torch.empty(max(cb.workspace_bytes(op, s) for op in range(3)) + 16, dtype=torch.uint8, device="cuda")
        y = torch.empty(L.y_shape, device="cuda")
        dx = torch.empty(L.x_shape, device="cuda")
        dw = torch.empty(L.w_shape, device="cuda")
        if a.op == "fwd":
            run = lambda: cb.conv_fwd(xt, wt, bt, L.stride, L.pad, y=y, workspace=ws)
        elif a.op == "dgrad":
            run = lambda: cb.conv_bwd_data(wt, dyt, L.x_shape, L.stride, L.pad, dx=dx, workspace=ws)
        elif a.op == "wgrad":
            run = lambda: cb.conv_bwd_filter(xt, dyt, L.w_shape, L.stride, L.pad, dw=dw, workspace=ws)
        elif a.op == "bias":
            db = torch.empty(L.outC, device="cuda")
            run = lambda: cb.conv_bwd_bias(dyt, db=db)
        elif a.op == "pool":
            k, st = L.pool or (2, 2)
            xp = torch.from_numpy(synthetic.pool_input(L)).cuda()
            yp, idx = cb.maxpool2d_fwd(xp, k, st)
            dyp = torch.from_numpy(synthetic.pool_grad(tuple(yp.shape), 5)).cuda()
            dxp = torch.empty(L.y_shape, device="cuda")
            run = lambda: (cb.maxpool2d_fwd(xp, k, st, y=yp, idx=idx),
                           cb.maxpool2d_bwd(dyp, idx, L.y_shape, k, st, dx=dxp))
        elif a.op == "im2col":
            col = torch.empty((L.inC * L.k * L.k, L.batch * L.outH * L.outW), device="cuda")
            run = lambda: cb.im2col(xt, L.k, L.stride, L.pad, col=col)
        else:
            col = torch.from_numpy(synthetic.normal((L.inC * L.k * L.k, L.batch * L.outH * L.outW), 6)).cuda()
            run = lambda: cb.col2im(col, L.x_shape, L.k, L.stride, L.pad, dx=dx)
    for _ in range(a.reps):
        run()
    cb.check()
    print("profile_case done: %s %s x%d" % (a.layer if a.op != "matmul" else a.mnk, a.op, a.reps))
    if a.time > 0:
        # algorithmic bytes of the HBM-bound ops (4-byte elements)
        nbytes = None
        if a.op != "matmul":
            xe, ce, ye = L.batch * L.inC * L.inH * L.inW, L.inC * L.k * L.k * L.batch * L.outH * L.outW, \
                L.batch * L.outC * L.outH * L.outW
            if a.op in ("im2col", "col2im"):
                nbytes = 4 * (xe + ce)
            elif a.op == "bias":
                nbytes = 4 * ye
            elif a.op == "pool":   # forward (read x, write y and idx) + backward (read dy and idx, write dx)
                nbytes = 4 * 2 * (ye + 2 * yp.numel())
        # The calls are captured once into a CUDA graph and replayed, so that
        # host-side issue cost does not hide short kernels (outputs are
        # preallocated, so a call allocates nothing); plain issue otherwise.
        graph = None
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                run()
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(a.time):
                    run()
        except RuntimeError:
            graph = None
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for _ in range(a.time):
                run()
        e1.record(stream)
        torch.cuda.synchronize()
        cb.check()
        us = e0.elapsed_time(e1) * 1e3 / a.time
        line = "time: %.2f us per call (%d calls, %s)" % (us, a.time, "graph" if graph is not None else "eager")
        if nbytes:
            line += ", %.1f MB algorithmic, %.1f GB/s" % (nbytes / 1e6, nbytes / us / 1e3)
        print(line)


if __name__ == "__main__":
    main()
