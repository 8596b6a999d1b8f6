// direct_conv.cu -- direct (non-im2col) convolution kernels: the page "DirectCompute
// Neural Network Engine", shader table "Legacy / Unused Shaders"
// (nn_conv_forward[_tiled], nn_conv_backprop_filters[_tiled] with
// nn_conv_reduce_filters, nn_conv_backprop_input[_fused]), which the im2col
// pipeline replaced.  Built as a cross-check of the implicit-GEMM path and as
// an ablation for layers with very few input channels, where the GEMM's K
// dimension (inC * k * k) is short.
//
// Plain fp32 CUDA-core arithmetic (fused multiply-adds), every output summed
// by one thread or one fixed reduction tree in a fixed order: deterministic.
//   forward:      y[n,k,oh,ow] = b[k] + sum_{c,r,s} x[n,c,oh*S+r-p,ow*S+s-p] w[k,c,r,s]
//   input grad:   dx[n,c,h,w]  = sum_{k,r,s : h = oh*S+r-p, w = ow*S+s-p} dy[n,k,oh,ow] w[k,c,r,s]
//   filter grad:  dw[k,c,r,s]  = sum_{n,oh,ow} dy[n,k,oh,ow] x[n,c,oh*S+r-p,ow*S+s-p]
// The filter gradient's long sums are spread over a cluster of CTAs and added
// in rank order through distributed shared memory.
#include <cooperative_groups.h>

#include "conv_b200_internal.h"

namespace cg = cooperative_groups;

namespace cb200 {

namespace {

constexpr int kTile = 16;     // output (forward) or input (input grad) tile: 16 x 16 positions, one per thread
constexpr int kKG = 8;        // filters per block (forward) / channels per block (input grad)

// Forward (nn_conv_forward_tiled).  Block = (image n, 8 filters, 16x16 output
// tile); for each input channel in ascending order the block stages the input
// patch the tile reads (zero outside the image) and the 8 filters' k x k
// slices, then every thread adds its pixel's taps for the 8 filters in (r, s)
// order.
__global__ void __launch_bounds__(kTile* kTile) direct_fwd_kernel(const float* __restrict__ x,
                                                                  const float* __restrict__ w,
                                                                  const float* __restrict__ b, float* __restrict__ y,
                                                                  ConvDims d, int tiles_w, int ph, int pw)
{
    extern __shared__ float sm[];
    float* patch = sm;                 // [ph][pw]
    float* filt = sm + ph * pw;        // [kKG][R][R]
    const int tile = blockIdx.x, kg = blockIdx.y, n = blockIdx.z;
    const int oh0 = (tile / tiles_w) * kTile, ow0 = (tile % tiles_w) * kTile;
    const int ty = threadIdx.x / kTile, tx = threadIdx.x % kTile;
    const int oh = oh0 + ty, ow = ow0 + tx;
    const int k0 = kg * kKG;
    const int RR = d.R * d.R;
    float acc[kKG];
#pragma unroll
    for (int j = 0; j < kKG; ++j) acc[j] = 0.f;
    const int h0 = oh0 * d.S - d.pad, w0 = ow0 * d.S - d.pad;
    for (int c = 0; c < d.C; ++c) {
        __syncthreads();
        const float* xc = x + ((size_t)n * d.C + c) * d.H * d.W;
        for (int i = threadIdx.x; i < ph * pw; i += blockDim.x) {
            const int h = h0 + i / pw, ww = w0 + i % pw;
            patch[i] = (unsigned(h) < unsigned(d.H) && unsigned(ww) < unsigned(d.W)) ? __ldg(xc + h * d.W + ww) : 0.f;
        }
        for (int i = threadIdx.x; i < kKG * RR; i += blockDim.x) {
            const int j = i / RR, t = i % RR;
            filt[i] = k0 + j < d.K ? __ldg(w + ((size_t)(k0 + j) * d.C + c) * RR + t) : 0.f;
        }
        __syncthreads();
        const float* pp = patch + (ty * d.S) * pw + tx * d.S;
        for (int r = 0; r < d.R; ++r)
            for (int s = 0; s < d.R; ++s) {
                const float v = pp[r * pw + s];
#pragma unroll
                for (int j = 0; j < kKG; ++j) acc[j] = fmaf(v, filt[j * RR + r * d.R + s], acc[j]);
            }
    }
    if (oh < d.P && ow < d.Q)
#pragma unroll
        for (int j = 0; j < kKG; ++j)
            if (k0 + j < d.K)
                y[(((size_t)n * d.K + k0 + j) * d.P + oh) * d.Q + ow] = acc[j] + (b ? __ldg(b + k0 + j) : 0.f);
}

// Input gradient (nn_conv_backprop_input, gather form).  Block = (image n, 8
// channels, 16x16 tile of dx); a thread owns one dx position and, for each
// filter k in ascending order, adds the taps (r, s) whose output position
// oh = (h + p - r) / S, ow = (w + p - s) / S exists, in (r, s) order, for its
// 8 channels.  dy is read through the cache (each value is shared by the
// thread's neighbours), the filters' k x k slices for the 8 channels are staged.
__global__ void __launch_bounds__(kTile* kTile) direct_dgrad_kernel(const float* __restrict__ w,
                                                                    const float* __restrict__ dy,
                                                                    float* __restrict__ dx, ConvDims d, int tiles_w)
{
    extern __shared__ float filt[];    // [kKG][R][R] of filter k
    const int tile = blockIdx.x, cgrp = blockIdx.y, n = blockIdx.z;
    const int h = (tile / tiles_w) * kTile + threadIdx.x / kTile;
    const int ww = (tile % tiles_w) * kTile + threadIdx.x % kTile;
    const int c0 = cgrp * kKG;
    const int RR = d.R * d.R;
    float acc[kKG];
#pragma unroll
    for (int j = 0; j < kKG; ++j) acc[j] = 0.f;
    const bool inside = h < d.H && ww < d.W;
    for (int k = 0; k < d.K; ++k) {
        __syncthreads();
        for (int i = threadIdx.x; i < kKG * RR; i += blockDim.x) {
            const int j = i / RR, t = i % RR;
            filt[i] = c0 + j < d.C ? __ldg(w + ((size_t)k * d.C + c0 + j) * RR + t) : 0.f;
        }
        __syncthreads();
        if (!inside) continue;
        const float* dyk = dy + ((size_t)n * d.K + k) * d.P * d.Q;
        for (int r = 0; r < d.R; ++r) {
            const int hp = h + d.pad - r;
            if (hp < 0 || hp % d.S) continue;
            const int oh = hp / d.S;
            if (oh >= d.P) continue;
            for (int s = 0; s < d.R; ++s) {
                const int wp = ww + d.pad - s;
                if (wp < 0 || wp % d.S) continue;
                const int ow = wp / d.S;
                if (ow >= d.Q) continue;
                const float g = __ldg(dyk + oh * d.Q + ow);
#pragma unroll
                for (int j = 0; j < kKG; ++j) acc[j] = fmaf(g, filt[j * RR + r * d.R + s], acc[j]);
            }
        }
    }
    if (inside)
#pragma unroll
        for (int j = 0; j < kKG; ++j)
            if (c0 + j < d.C) dx[(((size_t)n * d.C + c0 + j) * d.H + h) * d.W + ww] = acc[j];
}

// Filter gradient (nn_conv_backprop_filters with nn_conv_reduce_filters).
// A cluster of kWgCluster CTAs takes one (k, c) pair and a group of up to 32
// taps; thread t of CTA rank q takes the output positions (n, oh, ow) numbered
// q * 512 + t, then + kWgCluster * 512, ..., in order, keeping one partial sum
// per tap.  Each CTA adds its 512 partials of a tap by a fixed tree (xor
// shuffles inside each warp, then the 16 warp sums in warp order); rank 0
// then adds the CTAs' sums in rank order through distributed shared memory
// (the reduce step), so the result does not depend on scheduling.
constexpr int kWgThreads = 512;
constexpr int kWgTaps = 32;
constexpr int kWgCluster = 8;
__global__ void __launch_bounds__(kWgThreads) direct_wgrad_kernel(const float* __restrict__ x,
                                                                  const float* __restrict__ dy,
                                                                  float* __restrict__ dw, ConvDims d)
{
    __shared__ float part[kWgThreads / 32][kWgTaps];
    __shared__ float cta_sum[kWgTaps];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int k = blockIdx.x / d.C, c = blockIdx.x % d.C;
    const int RR = d.R * d.R;
    const int t0 = blockIdx.y * kWgTaps;
    const int nt = min(kWgTaps, RR - t0);
    float acc[kWgTaps];
#pragma unroll
    for (int j = 0; j < kWgTaps; ++j) acc[j] = 0.f;
    const int PQ = d.P * d.Q;
    const int npos = d.N * PQ;
    for (int pos = rank * kWgThreads + threadIdx.x; pos < npos; pos += kWgCluster * kWgThreads) {
        const int n = pos / PQ, pq = pos - n * PQ;
        const int oh = pq / d.Q, ow = pq - oh * d.Q;
        const float g = __ldg(dy + ((size_t)n * d.K + k) * PQ + pq);
        const float* xc = x + ((size_t)n * d.C + c) * d.H * d.W;
#pragma unroll
        for (int j = 0; j < kWgTaps; ++j) {
            if (j < nt) {
                const int t = t0 + j, r = t / d.R, s = t - r * d.R;
                const int h = oh * d.S + r - d.pad, ww = ow * d.S + s - d.pad;
                const float v = (unsigned(h) < unsigned(d.H) && unsigned(ww) < unsigned(d.W)) ? __ldg(xc + h * d.W + ww)
                                                                                              : 0.f;
                acc[j] = fmaf(g, v, acc[j]);
            }
        }
    }
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < kWgTaps; ++j) {
        float v = acc[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) part[wp][j] = v;
    }
    __syncthreads();
    if (threadIdx.x < kWgTaps) {
        float s = 0.f;
        for (int q = 0; q < kWgThreads / 32; ++q) s += part[q][threadIdx.x];
        cta_sum[threadIdx.x] = s;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x < nt) {
        float s = 0.f;
        for (int q = 0; q < kWgCluster; ++q) s += cluster.map_shared_rank(cta_sum, q)[threadIdx.x];
        dw[((size_t)k * d.C + c) * RR + t0 + threadIdx.x] = s;
    }
    cluster.sync();   // every CTA's shared memory stays alive until rank 0 has read it
}

}  // namespace

cudaError_t launch_conv_fwd_direct(const ConvDims& d, const float* x, const float* w, const float* b, float* y,
                                   cudaStream_t st)
{
    const int tiles_h = (d.P + kTile - 1) / kTile, tiles_w = (d.Q + kTile - 1) / kTile;
    const int ph = (kTile - 1) * d.S + d.R, pw = ph;
    const size_t smem = size_t(ph * pw + kKG * d.R * d.R) * sizeof(float);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(direct_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   int(smem));
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(tiles_h * tiles_w, (d.K + kKG - 1) / kKG, d.N);
    direct_fwd_kernel<<<grid, kTile * kTile, smem, st>>>(x, w, b, y, d, tiles_w, ph, pw);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_conv_dgrad_direct(const ConvDims& d, const float* w, const float* dy, float* dx, cudaStream_t st)
{
    const int tiles_h = (d.H + kTile - 1) / kTile, tiles_w = (d.W + kTile - 1) / kTile;
    const size_t smem = size_t(kKG * d.R * d.R) * sizeof(float);
    const dim3 grid(tiles_h * tiles_w, (d.C + kKG - 1) / kKG, d.N);
    direct_dgrad_kernel<<<grid, kTile * kTile, smem, st>>>(w, dy, dx, d, tiles_w);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_conv_wgrad_direct(const ConvDims& d, const float* x, const float* dy, float* dw, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.K * d.C, (d.R * d.R + kWgTaps - 1) / kWgTaps, kWgCluster);
    cfg.blockDim = dim3(kWgThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = kWgCluster;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, direct_wgrad_kernel, x, dy, dw, d);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace cb200
