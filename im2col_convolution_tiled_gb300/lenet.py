"""LeNet-5 training step on the GPU, composed from the library's entry points.

Page "DirectCompute Neural Network Engine", section "LeNet on MNIST" (the
trainer) with the convolution of section "Convolution: The im2col Approach"
and the activation/loss and utility shaders:

    x (B,1,28,28) -> conv 6@5x5 pad 2 -> ReLU -> maxpool 2/2
                  -> conv 16@5x5       -> ReLU -> maxpool 2/2 -> flatten 400
                  -> linear 400->120 -> ReLU -> linear 120->84 -> ReLU
                  -> linear 84->10 -> softmax + cross-entropy against labels
    backward through the same operations, then SGD with clip on every parameter.

Every operation is one call into libconv_b200 on one stream; nothing is
computed in Python or by torch (torch only owns the buffers).  All buffers are
allocated once, so the whole step can be captured into one CUDA graph and
replayed: the counterpart of the page's dispatch pipelining
(section "Performance Notes"), without its per-dispatch host round trips.

Conventions (as the page's shaders give them):
  * linear: Y = X W + b with W stored in x out; dW = X^T dY (matmul flag 1),
    dX = dY W^T (matmul flag 2), db = row sums of dY; the bias add and the
    ReLU run in the forward matmul's epilogue (matmul_fused: the same fp32
    operations as add_bias, bit for bit).  The ReLU gradient behind a linear
    layer stays a relu_bwd pass: gating the dX matmul's epilogue instead
    measured 1-12 us slower per graph-replayed step (programmatic dependent
    launch already hides the separate pass);
  * the convolutions' ReLU runs in their epilogue (conv_fwd_relu);
  * the ReLU gradient is masked by the ReLU's output (> 0 exactly where its
    input is); behind a convolution the mask is applied inside the
    convolution's gradient calls, where they first read the routed gradient
    (conv_bwd_data_relu, conv_bwd_filter_bias_relu), so it costs no pass;
  * the loss gradient is softmax - one_hot, the gradient of the batch SUM of
    the row cross-entropies, which is what `loss` holds;
  * the first layer's input gradient is not formed (x is the network input).
"""
from __future__ import annotations

from collections import namedtuple

from . import (CONV_OP_BWD_DATA, CONV_OP_BWD_FILTER, CONV_OP_FWD, bias_grad_rows, conv_bwd_data,
               conv_bwd_filter_bias, conv_fwd, matmul, maxpool2d_bwd, maxpool2d_fwd, relu_bwd, sgd_step, shape_of,
               softmax_ce, workspace_bytes)

# The network.  Conv: outC filters k x k, stride, padding, then a k_pool/s_pool
# max pool; linear layers (in, out); SGD learning rate and clip.
Conv = namedtuple("Conv", "inC outC k stride pad pool")
CONVS = (Conv(1, 6, 5, 1, 2, (2, 2)), Conv(6, 16, 5, 1, 0, (2, 2)))
FCS = ((400, 120), (120, 84), (84, 10))
IMAGE = (1, 28, 28)
LR, CLIP = 0.01, 1.0
PARAMS = ("conv1_w", "conv1_b", "conv2_w", "conv2_b", "fc1_w", "fc1_b", "fc2_w", "fc2_b", "fc3_w", "fc3_b")


def _out(n, k, stride, pad):
    return (n + 2 * pad - k) // stride + 1


class LeNet5:
    """Parameters, gradients and every activation of one LeNet-5 step, resident
    on the GPU.  ``params`` maps the names in PARAMS to fp32 arrays (numpy or
    torch): conv filters (outC, inC, k, k), linear weights (in, out), biases (out,)."""

    def __init__(self, params, batch=64, lr=LR, clip=CLIP, device="cuda"):
        import torch

        self.torch = torch
        self.B = batch
        self.lr, self.clip = lr, clip
        c1, c2 = CONVS
        f32 = dict(dtype=torch.float32, device=device)
        # Parameters and gradients each live in one flat buffer (every tensor a
        # view starting on a 16-byte boundary), so the SGD step over all of them
        # is one launch.  The few padding slots between views hold 0 in both
        # buffers and stay 0: SGD leaves p unchanged where g = 0.
        shapes = {k: tuple(torch.as_tensor(params[k]).shape) for k in PARAMS}
        offs, n = {}, 0
        for k in PARAMS:
            offs[k] = n
            size = 1
            for d in shapes[k]:
                size *= d
            n += (size + 3) // 4 * 4
        self.flat_p = torch.zeros(n, **f32)
        self.flat_g = torch.zeros(n, **f32)
        self.P, self.G = {}, {}
        for k in PARAMS:
            size = 1
            for d in shapes[k]:
                size *= d
            self.P[k] = self.flat_p[offs[k]:offs[k] + size].view(shapes[k])
            self.G[k] = self.flat_g[offs[k]:offs[k] + size].view(shapes[k])
            self.P[k].copy_(torch.as_tensor(params[k]).to(device=device, dtype=torch.float32))
        B = batch
        e = torch.empty
        t = {}
        t["x"] = e((B,) + IMAGE, **f32)
        t["labels"] = e((B,), dtype=torch.int32, device=device)
        H = IMAGE[1]
        H1 = _out(H, c1.k, c1.stride, c1.pad)
        H1p = _out(H1, c1.pool[0], c1.pool[1], 0)
        H2 = _out(H1p, c2.k, c2.stride, c2.pad)
        H2p = _out(H2, c2.pool[0], c2.pool[1], 0)
        t["a1"] = e((B, c1.outC, H1, H1), **f32)        # ReLU(conv1 + bias), one fused pass
        t["p1"] = e((B, c1.outC, H1p, H1p), **f32)      # max pool
        t["i1"] = torch.empty_like(t["p1"], dtype=torch.int32)
        t["a2"] = e((B, c2.outC, H2, H2), **f32)
        t["p2"] = e((B, c2.outC, H2p, H2p), **f32)
        t["i2"] = torch.empty_like(t["p2"], dtype=torch.int32)
        t["f"] = t["p2"].view(B, -1)                    # flatten (a view: no copy)
        for i, (fin, fout) in enumerate(FCS, 1):
            t["dz%d" % i] = e((B, fout), **f32)         # gradient at X W + b
            t["df" if i == 1 else "dh%d" % (i - 1)] = e((B, fin), **f32)   # gradient at X
        t["h1"] = e((B, FCS[0][1]), **f32)              # ReLU(X W + b), layers 1 and 2
        t["h2"] = e((B, FCS[1][1]), **f32)
        t["z3"] = e((B, FCS[2][1]), **f32)              # logits
        t["loss"] = e((1,), **f32)
        t["dp2"] = t["df"].view(t["p2"].shape)
        t["da2"] = torch.empty_like(t["a2"])            # gradient at the ReLU output a2 (routed by the pool)
        t["dp1"] = torch.empty_like(t["p1"])
        t["da1"] = torch.empty_like(t["a1"])
        self.t = t
        s1 = shape_of(t["x"].shape, self.P["conv1_w"].shape, c1.stride, c1.pad)
        s2 = shape_of(t["p1"].shape, self.P["conv2_w"].shape, c2.stride, c2.pad)
        need = max(workspace_bytes(CONV_OP_FWD, s1), workspace_bytes(CONV_OP_BWD_FILTER, s1),
                   workspace_bytes(CONV_OP_FWD, s2), workspace_bytes(CONV_OP_BWD_DATA, s2),
                   workspace_bytes(CONV_OP_BWD_FILTER, s2), 16)
        self.ws = e((need,), dtype=torch.uint8, device=device)
        self.graph = None

    # -- the step --------------------------------------------------------------
    def load_batch(self, x, labels):
        """Copy a batch into the step's input buffers (host or device arrays)."""
        torch = self.torch
        self.t["x"].copy_(torch.as_tensor(x), non_blocking=True)
        self.t["labels"].copy_(torch.as_tensor(labels).to(torch.int32), non_blocking=True)

    def run(self, stream=None):
        """Issue the whole step on `stream` (torch's current stream by default)."""
        t, P, G, ws, st = self.t, self.P, self.G, self.ws, stream
        c1, c2 = CONVS
        # forward
        conv_fwd(t["x"], P["conv1_w"], P["conv1_b"], c1.stride, c1.pad, y=t["a1"], workspace=ws, stream=st,
                 relu=True)
        maxpool2d_fwd(t["a1"], *c1.pool, y=t["p1"], idx=t["i1"], stream=st)
        conv_fwd(t["p1"], P["conv2_w"], P["conv2_b"], c2.stride, c2.pad, y=t["a2"], workspace=ws, stream=st,
                 relu=True)
        maxpool2d_fwd(t["a2"], *c2.pool, y=t["p2"], idx=t["i2"], stream=st)
        h = t["f"]
        for i, out in ((1, "h1"), (2, "h2"), (3, "z3")):
            matmul(h, P["fc%d_w" % i], 0, C=t[out], bias=P["fc%d_b" % i], relu=i < 3, stream=st)
            h = t[out]
        softmax_ce(t["z3"], t["labels"], dlogits=t["dz3"], loss=t["loss"], stream=st)
        # backward: linear layers
        for i in (3, 2, 1):
            hin = t["h%d" % (i - 1)] if i > 1 else t["f"]
            dz = t["dz%d" % i]
            matmul(hin, dz, 1, C=G["fc%d_w" % i], stream=st)
            bias_grad_rows(dz, db=G["fc%d_b" % i], stream=st)
            dh = t["dh%d" % (i - 1)] if i > 1 else t["df"]
            matmul(dz, P["fc%d_w" % i], 2, C=dh, stream=st)
            if i > 1:
                relu_bwd(dh, t["h%d" % (i - 1)], dx=t["dz%d" % (i - 1)], stream=st)
        # conv2 block: route the pooled gradient to the ReLU output, then the
        # convolution's gradients with the ReLU mask (a2 > 0) applied as they
        # read it -- the page's order (pool backward, relu_grad, conv backward)
        # with the relu_grad pass fused away
        maxpool2d_bwd(t["dp2"], t["i2"], t["a2"].shape, *c2.pool, dx=t["da2"], stream=st)
        conv_bwd_filter_bias(t["p1"], t["da2"], P["conv2_w"].shape, c2.stride, c2.pad, dw=G["conv2_w"],
                             db=G["conv2_b"], workspace=ws, stream=st, relu_mask=t["a2"])
        conv_bwd_data(P["conv2_w"], t["da2"], t["p1"].shape, c2.stride, c2.pad, dx=t["dp1"], workspace=ws,
                      stream=st, relu_mask=t["a2"])
        # conv1 block
        maxpool2d_bwd(t["dp1"], t["i1"], t["a1"].shape, *c1.pool, dx=t["da1"], stream=st)
        conv_bwd_filter_bias(t["x"], t["da1"], P["conv1_w"].shape, c1.stride, c1.pad, dw=G["conv1_w"],
                             db=G["conv1_b"], workspace=ws, stream=st, relu_mask=t["a1"])
        # SGD over every parameter at once
        sgd_step(self.flat_p, self.flat_g, self.lr, self.clip, stream=st)

    # -- CUDA graph --------------------------------------------------------------
    def capture(self):
        """Capture run() into a CUDA graph (after one eager warm-up step, which
        also sets every kernel attribute outside the capture).  Note: the
        warm-up step updates the parameters like any other step."""
        torch = self.torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.run()
        return self.graph

    def replay(self):
        self.graph.replay()

    def params_numpy(self):
        return {k: v.detach().cpu().numpy() for k, v in self.P.items()}
