"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the convolution method: it only draws
random arrays (numpy PCG64, fp32) with the shapes and value distributions of
the LeNet- and AlexNet-shaped workloads, plus the flagged-matmul sweep.  The
seed of every tensor is ``1000 * workload_id + tensor_id`` so each array is
reproducible on any machine.

Distributions: "N(0, v)" is read as variance v; He-normal uses
std = sqrt(2 / (inC * k * k)); post-ReLU activations are max(N(0,1), 0), which
makes about half of them exactly zero (that is what makes max-pool ties common).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform01(shape, seed):
    return rng(seed).random(shape, dtype=np.float32)


def normal(shape, seed, std=1.0):
    return (rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def relu_normal(shape, seed):
    a = normal(shape, seed)
    np.maximum(a, np.float32(0.0), out=a)
    return a


def he_normal(shape, seed):
    fan_in = int(np.prod(shape[1:]))
    return normal(shape, seed, std=math.sqrt(2.0 / fan_in))


def small_ints(shape, seed, lo=-4, hi=5):
    """Small-integer-valued fp32 tensors: every sum of products stays exact."""
    return rng(seed).integers(lo, hi, size=shape).astype(np.float32)


@dataclass(frozen=True)
class ConvLayer:
    """One convolution layer workload (NCHW fp32)."""
    name: str
    batch: int
    inC: int
    inH: int
    inW: int
    outC: int
    k: int
    stride: int
    pad: int
    outH: int
    outW: int
    x_dist: str = "normal"      # normal | uniform | relu
    w_dist: str = "he"          # he | normal:<std>
    b_dist: str = "zeros"       # zeros | normal:<std>
    pool: tuple | None = None   # (k, stride) max-pool that follows the layer
    seed_base: int = 0

    @property
    def x_shape(self):
        return (self.batch, self.inC, self.inH, self.inW)

    @property
    def w_shape(self):
        return (self.outC, self.inC, self.k, self.k)

    @property
    def y_shape(self):
        return (self.batch, self.outC, self.outH, self.outW)

    @property
    def gemm_flops(self) -> int:
        """2 * outC * (inC*k*k) * (batch*outH*outW): one of the three GEMMs."""
        return 2 * self.outC * self.inC * self.k * self.k * self.batch * self.outH * self.outW

    def with_batch(self, batch: int) -> "ConvLayer":
        d = dict(self.__dict__)
        d["batch"] = batch
        return ConvLayer(**d)

    def make(self):
        """(x, w, b, dy) as fp32 numpy arrays."""
        s = self.seed_base
        if self.x_dist == "uniform":
            x = uniform01(self.x_shape, s + 1)
        elif self.x_dist == "relu":
            x = relu_normal(self.x_shape, s + 1)
        else:
            x = normal(self.x_shape, s + 1)
        if self.w_dist == "he":
            w = he_normal(self.w_shape, s + 2)
        else:
            w = normal(self.w_shape, s + 2, float(self.w_dist.split(":")[1]))
        if self.b_dist == "zeros":
            b = np.zeros((self.outC,), np.float32)
        else:
            b = normal((self.outC,), s + 3, float(self.b_dist.split(":")[1]))
        dy = normal(self.y_shape, s + 4)
        return x, w, b, dy


# Workload 1: single conv layer, batch 4, 1x28x28 -> 6@5x5 -> 6x24x24.
SINGLE = ConvLayer("single_conv_b4", 4, 1, 28, 28, 6, 5, 1, 0, 24, 24,
                   x_dist="uniform", w_dist="normal:0.2", b_dist="normal:0.1",
                   seed_base=1000)

# Workload 2: LeNet-5 conv stack, batch 64 (conv1 pad 2, ReLU, pool 2/2, conv2, ReLU, pool 2/2).
LENET = (
    ConvLayer("lenet_conv1_b64", 64, 1, 28, 28, 6, 5, 1, 2, 28, 28,
              x_dist="uniform", pool=(2, 2), seed_base=2000),
    ConvLayer("lenet_conv2_b64", 64, 6, 14, 14, 16, 5, 1, 0, 10, 10,
              x_dist="relu", pool=(2, 2), seed_base=2100),
)
LENET_FC = ((400, 120), (120, 84), (84, 10))
LENET_SGD = (0.01, 1.0)   # lr, clip
LENET_CLASSES = 10

# Parameter order of the LeNet-5 step: conv filters are (outC, inC, k, k);
# linear weights are stored in x out (Y = X W), biases per output.
LENET_PARAMS = ("conv1_w", "conv1_b", "conv2_w", "conv2_b",
                "fc1_w", "fc1_b", "fc2_w", "fc2_b", "fc3_w", "fc3_b")


def lenet_params(seed_base=2200):
    """He-normal weights (std sqrt(2 / fan_in)), zero biases: 61,706 fp32 values."""
    c1, c2 = LENET
    p = {"conv1_w": he_normal(c1.w_shape, seed_base + 1), "conv1_b": np.zeros((c1.outC,), np.float32),
         "conv2_w": he_normal(c2.w_shape, seed_base + 2), "conv2_b": np.zeros((c2.outC,), np.float32)}
    for i, (fin, fout) in enumerate(LENET_FC):
        p["fc%d_w" % (i + 1)] = normal((fin, fout), seed_base + 3 + i, std=math.sqrt(2.0 / fin))
        p["fc%d_b" % (i + 1)] = np.zeros((fout,), np.float32)
    return p


def lenet_batch(batch=64, seed=2300):
    """(x, labels): x (batch, 1, 28, 28) U[0,1); labels int32 uniform over the 10 classes."""
    x = uniform01((batch, 1, 28, 28), seed)
    labels = rng(seed + 1).integers(0, LENET_CLASSES, size=(batch,)).astype(np.int32)
    return x, labels

# Workload 3: AlexNet conv1, batch 128.
ALEXNET_CONV1 = ConvLayer("alexnet_conv1_b128", 128, 3, 224, 224, 64, 11, 4, 2, 55, 55,
                          x_dist="normal", pool=(3, 2), seed_base=3000)

# Workload 4: AlexNet conv2-5, batch 128, post-ReLU inputs.
ALEXNET_CONV2_5 = (
    ConvLayer("alexnet_conv2_b128", 128, 64, 27, 27, 192, 5, 1, 2, 27, 27,
              x_dist="relu", pool=(3, 2), seed_base=4000),
    ConvLayer("alexnet_conv3_b128", 128, 192, 13, 13, 384, 3, 1, 1, 13, 13,
              x_dist="relu", seed_base=4100),
    ConvLayer("alexnet_conv4_b128", 128, 384, 13, 13, 256, 3, 1, 1, 13, 13,
              x_dist="relu", seed_base=4200),
    ConvLayer("alexnet_conv5_b128", 128, 256, 13, 13, 256, 3, 1, 1, 13, 13,
              x_dist="relu", seed_base=4300),
)
ALEXNET = (ALEXNET_CONV1,) + ALEXNET_CONV2_5

SGD_LR_CLIP = (0.01, 1.0)

# Workload 5: flagged matmul sweep.
MATMUL_MN = (16, 64, 127, 128, 1024, 4096, 9216)
MATMUL_K = (25, 150, 363, 1600, 2304, 4096)


def matmul_case(M, K, N, flags, seed_base=5000):
    """A (M x K, or K x M when flags bit 0) and B (K x N, or N x K when bit 1), N(0,1)."""
    tag = ((M * 31 + K) * 31 + N) * 4 + flags
    a_shape = (K, M) if flags & 1 else (M, K)
    b_shape = (N, K) if flags & 2 else (K, N)
    s = seed_base + (tag % 997) * 2
    return normal(a_shape, s + 1), normal(b_shape, s + 2)


def matmul_sweep():
    """Every (M, N, K, flags) of the sweep: 7 * 7 * 6 * 4 = 1176 cases."""
    for M in MATMUL_MN:
        for N in MATMUL_MN:
            for K in MATMUL_K:
                for flags in range(4):
                    yield M, K, N, flags


# The sweep's 1176 cases would need 7e9 fresh N(0,1) draws; instead every case
# reads its operands out of two fixed N(0,1) pools (one for A, one for B), at a
# case-dependent offset (a multiple of 4 floats, so views stay 16-byte aligned).
# Any such window of i.i.d. N(0,1) draws is itself i.i.d. N(0,1).
MATMUL_POOL_FLOATS = max(MATMUL_MN) * max(MATMUL_K) + 4096
_MATMUL_POOLS = {}


def matmul_pool(which):
    """Pool 0 (A operands) or 1 (B operands): MATMUL_POOL_FLOATS N(0,1) fp32 draws."""
    if which not in _MATMUL_POOLS:
        _MATMUL_POOLS[which] = normal((MATMUL_POOL_FLOATS,), 5900 + which)
    return _MATMUL_POOLS[which]


def matmul_sweep_offsets(M, K, N, flags):
    """(offset of A in pool 0, offset of B in pool 1), in floats, for one sweep case."""
    tag = ((M * 31 + K) * 31 + N) * 4 + flags
    offs = []
    for i, size in enumerate((M * K, K * N)):
        room = (MATMUL_POOL_FLOATS - size) // 4
        offs.append(4 * int(rng(7000 + 2 * tag + i).integers(0, room + 1)))
    return tuple(offs)


def matmul_sweep_case(M, K, N, flags):
    """A (M x K, or K x M when flags bit 0) and B (K x N, or N x K when bit 1) of
    one sweep case: contiguous views into the two pools."""
    oa, ob = matmul_sweep_offsets(M, K, N, flags)
    a_shape = (K, M) if flags & 1 else (M, K)
    b_shape = (N, K) if flags & 2 else (K, N)
    return (matmul_pool(0)[oa:oa + M * K].reshape(a_shape), matmul_pool(1)[ob:ob + K * N].reshape(b_shape))


def pool_input(layer: ConvLayer, seed_offset=10):
    """Input of the max-pool after ``layer``: post-ReLU activations of the layer's
    output shape (about half zeros, so ties are frequent)."""
    return relu_normal(layer.y_shape, layer.seed_base + seed_offset)


def pool_grad(shape, seed):
    return normal(shape, seed)
