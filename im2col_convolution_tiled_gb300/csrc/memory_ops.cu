// memory_ops.cu -- the HBM-bound steps of the page "DirectCompute Neural
// Network Engine": the standalone im2col / col2im shaders (section
// "Convolution Shaders"), max pooling forward/backward ("Pooling Shaders"),
// SGD and the bias gradient ("Utility Shaders").
//
// All of them are pure data movement or short per-element arithmetic, so they
// are written for bandwidth: grids sized to the SM count, consecutive threads
// on consecutive output addresses, 16-byte stores where rows allow it, and
// every output element produced by exactly one thread in a fixed order (no
// atomics; results are deterministic and, for the integer/routing work,
// bit-exact).
#include <cooperative_groups.h>

#include "gemm_tc.cuh"

namespace cg = cooperative_groups;

namespace cb200 {

static int grid_for(long long work, int per_block)
{
    long long b = (work + per_block - 1) / per_block;
    const long long cap = 16LL * sm_count();
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return int(b);
}

// ---------------------------------------------------------------------------
// im2col: col[(c, r, q)][(n, oh, ow)] = x[n, c, oh*s + r - pad, ow*s + q - pad].
// One thread writes 4 consecutive columns of one row (a 16-byte store when
// the row length NPQ is a multiple of 4); its (n, oh, ow) is decoded once and
// advanced incrementally.

__global__ void im2col_kernel(const float* __restrict__ x, float* __restrict__ col, int C, int H, int W, int S,
                              int pad, int P, int Q, FastDiv f_pq, FastDiv f_q, FastDiv f_rr, FastDiv f_r,
                              FastDiv f_npq4, int total4)
{
    const int npq = int(f_npq4.d) * 4;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total4; t += gridDim.x * blockDim.x) {
        uint32_t row, j4;
        f_npq4.divmod(uint32_t(t), row, j4);
        const int j0 = int(j4) * 4;
        uint32_t c, rem, r, q;
        f_rr.divmod(row, c, rem);
        f_r.divmod(rem, r, q);
        uint32_t n, pq, oh, ow;
        f_pq.divmod(uint32_t(j0), n, pq);
        f_q.divmod(pq, oh, ow);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int h = int(oh) * S + int(r) - pad;
            const int w = int(ow) * S + int(q) - pad;
            v[e] = (unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W))
                       ? __ldg(x + ((int(n) * C + int(c)) * H + h) * W + w)
                       : 0.f;
            if (++ow == uint32_t(Q)) {
                ow = 0;
                if (++oh == uint32_t(P)) { oh = 0; ++n; }
            }
        }
        *reinterpret_cast<float4*>(col + size_t(row) * npq + j0) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// Scalar variant for row lengths that are not a multiple of 4.
__global__ void im2col_scalar_kernel(const float* __restrict__ x, float* __restrict__ col, int C, int H, int W,
                                     int S, int pad, FastDiv f_npq, FastDiv f_pq, FastDiv f_q, FastDiv f_rr,
                                     FastDiv f_r, int total)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t row, j, c, rem, r, q, n, pq, oh, ow;
        f_npq.divmod(uint32_t(t), row, j);
        f_rr.divmod(row, c, rem);
        f_r.divmod(rem, r, q);
        f_pq.divmod(j, n, pq);
        f_q.divmod(pq, oh, ow);
        const int h = int(oh) * S + int(r) - pad;
        const int w = int(ow) * S + int(q) - pad;
        col[t] = (unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W))
                     ? __ldg(x + ((int(n) * C + int(c)) * H + h) * W + w)
                     : 0.f;
    }
}

cudaError_t launch_im2col(const ConvDims& d, const float* x, float* col, cudaStream_t st)
{
    const int NPQ = d.N * d.P * d.Q;
    const int CRS = d.C * d.R * d.R;
    const FastDiv f_pq(d.P * d.Q), f_q(d.Q), f_rr(d.R * d.R), f_r(d.R);
    if (NPQ % 4 == 0) {
        const long long total4 = (long long)CRS * (NPQ / 4);
        im2col_kernel<<<grid_for(total4, 256), 256, 0, st>>>(x, col, d.C, d.H, d.W, d.S, d.pad, d.P, d.Q, f_pq,
                                                             f_q, f_rr, f_r, FastDiv(NPQ / 4), int(total4));
    note_launch();
    } else {
        const long long total = (long long)CRS * NPQ;
        im2col_scalar_kernel<<<grid_for(total, 256), 256, 0, st>>>(x, col, d.C, d.H, d.W, d.S, d.pad, FastDiv(NPQ),
                                                                    f_pq, f_q, f_rr, f_r, int(total));
    note_launch();
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// col2im as a gather: dx[n, c, h, w] = sum over taps r == (h + pad) mod s
// (ascending), q likewise, of col[(c, r, q)][(n, (h + pad - r)/s, (w + pad - q)/s)]
// where that output position exists.  One thread per dx element, fixed order.

__global__ void col2im_kernel(const float* __restrict__ col, float* __restrict__ dx, int R, int S, int pad, int P,
                              int Q, int NPQ, FastDiv f_w, FastDiv f_h, FastDiv f_c, int total)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t r1, w, r2, h, n, c;
        f_w.divmod(uint32_t(t), r1, w);
        f_h.divmod(r1, r2, h);
        f_c.divmod(r2, n, c);
        const int hp = int(h) + pad, wp = int(w) + pad;
        float acc = 0.f;
        // taps with r <= h + pad only: oh = (h + pad - r) / S must be >= 0
        for (int r = hp % S; r < R && r <= hp; r += S) {
            const int oh = (hp - r) / S;
            if (oh >= P) continue;
            for (int q = wp % S; q < R && q <= wp; q += S) {
                const int ow = (wp - q) / S;
                if (ow >= Q) continue;
                acc += __ldg(col + size_t((int(c) * R + r) * R + q) * NPQ + (int(n) * P + oh) * Q + ow);
            }
        }
        dx[t] = acc;
    }
}

cudaError_t launch_col2im(const ConvDims& d, const float* col, float* dx, cudaStream_t st)
{
    const long long total = (long long)d.N * d.C * d.H * d.W;
    col2im_kernel<<<grid_for(total, 256), 256, 0, st>>>(col, dx, d.R, d.S, d.pad, d.P, d.Q, d.N * d.P * d.Q,
                                                        FastDiv(d.W), FastDiv(d.H), FastDiv(d.C), int(total));
    note_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Max pooling forward: first maximum in row-major window order (strict >).

__global__ void maxpool_fwd_kernel(const float* __restrict__ x, float* __restrict__ y, int32_t* __restrict__ idx,
                                   int H, int W, int k, int S, FastDiv f_q, FastDiv f_p, int total)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t r1, ow, nc, oh;
        f_q.divmod(uint32_t(t), r1, ow);
        f_p.divmod(r1, nc, oh);
        const int corner = (int(nc) * H + int(oh) * S) * W + int(ow) * S;
        int best = corner;
        float m = __ldg(x + corner);
        for (int r = 0; r < k; ++r)
            for (int q = 0; q < k; ++q) {
                const int at = corner + r * W + q;
                const float v = __ldg(x + at);
                if (v > m) {
                    m = v;
                    best = at;
                }
            }
        y[t] = m;
        idx[t] = best;
    }
}

// Plane-staged variant: a block copies whole (n, c) planes of x into shared
// memory with coalesced loads, then each thread scans its windows there and
// writes y / idx coalesced.  x is read from HBM exactly once.
constexpr int kPoolThreads = 256;
constexpr int kPoolSmemFloats = 8192;   // 32 KB of staged planes per block

__global__ void __launch_bounds__(kPoolThreads) maxpool_fwd_plane_kernel(
    const float* __restrict__ x, float* __restrict__ y, int32_t* __restrict__ idx, int NC, int H, int W, int k, int S,
    int P, int Q, int ppb, FastDiv f_pq, FastDiv f_q)
{
    extern __shared__ float sx[];
    const int HW = H * W, PQ = P * Q;
    for (int nc0 = blockIdx.x * ppb; nc0 < NC; nc0 += gridDim.x * ppb) {
        const int np = min(ppb, NC - nc0);
        const float* src = x + size_t(nc0) * HW;
        const int total = np * HW;
#pragma unroll 4
        for (int i = threadIdx.x; i < total; i += kPoolThreads) sx[i] = __ldg(src + i);
        __syncthreads();
        const int nout = np * PQ;
        for (int o = threadIdx.x; o < nout; o += kPoolThreads) {
            uint32_t pl, pq, oh, ow;
            f_pq.divmod(uint32_t(o), pl, pq);
            f_q.divmod(pq, oh, ow);
            const int corner = int(pl) * HW + int(oh) * S * W + int(ow) * S;
            int best = corner;
            float m = sx[corner];
            for (int r = 0; r < k; ++r)
                for (int q = 0; q < k; ++q) {
                    const int at = corner + r * W + q;
                    const float v = sx[at];
                    if (v > m) {
                        m = v;
                        best = at;
                    }
                }
            y[size_t(nc0) * PQ + o] = m;
            idx[size_t(nc0) * PQ + o] = nc0 * HW + best;
        }
        __syncthreads();
    }
}

// Plane-staged backward: a block stages the windows' gradients and indices of
// whole planes, then each thread gathers, in ascending window order, the
// gradients routed to its input pixel and writes dx coalesced.  The window
// rows covering input row h (and columns covering w) come from small tables
// built once per block, so the per-pixel work is table lookups and compares.
__global__ void __launch_bounds__(kPoolThreads) maxpool_bwd_plane_kernel(
    const float* __restrict__ dy, const int32_t* __restrict__ idx, float* __restrict__ dx, int NC, int H, int W,
    int k, int S, int P, int Q, int ppb, FastDiv f_hw, FastDiv f_w)
{
    extern __shared__ float sm[];
    const int HW = H * W, PQ = P * Q;
    float* sdy = sm;
    int* sidx = reinterpret_cast<int*>(sm + ppb * PQ);
    int* hrange = sidx + ppb * PQ;   // (first window row << 16) | last window row, per input row
    int* wrange = hrange + H;        // same per input column
    for (int i = threadIdx.x; i < H + W; i += kPoolThreads) {
        const int v = i < H ? i : i - H;
        const int lim = i < H ? P - 1 : Q - 1;
        const int lo = v - k + 1 <= 0 ? 0 : (v - k + S) / S;
        const int hi = min(v / S, lim);
        (i < H ? hrange[i] : wrange[i - H]) = (lo << 16) | (hi & 0xFFFF);
    }
    for (int nc0 = blockIdx.x * ppb; nc0 < NC; nc0 += gridDim.x * ppb) {
        const int np = min(ppb, NC - nc0);
        const int nwin = np * PQ;
#pragma unroll 4
        for (int i = threadIdx.x; i < nwin; i += kPoolThreads) {
            sdy[i] = __ldg(dy + size_t(nc0) * PQ + i);
            sidx[i] = __ldg(idx + size_t(nc0) * PQ + i);
        }
        __syncthreads();
        const int total = np * HW;
        for (int i = threadIdx.x; i < total; i += kPoolThreads) {
            uint32_t pl, hw, h, w;
            f_hw.divmod(uint32_t(i), pl, hw);
            f_w.divmod(hw, h, w);
            const int flat = nc0 * HW + i;
            const int hr = hrange[h], wr = wrange[w];
            const int oh_lo = hr >> 16, oh_hi = hr & 0xFFFF;   // oh_hi < oh_lo: no window
            const int ow_lo = wr >> 16, ow_hi = wr & 0xFFFF;
            const int* irow = sidx + int(pl) * PQ;
            const float* drow = sdy + int(pl) * PQ;
            float acc = 0.f;
            for (int oh = oh_lo; oh <= oh_hi; ++oh)
                for (int ow = ow_lo; ow <= ow_hi; ++ow) {
                    const int o = oh * Q + ow;
                    if (irow[o] == flat) acc += drow[o];
                }
            dx[size_t(nc0) * HW + i] = acc;
        }
        __syncthreads();
    }
}

cudaError_t launch_maxpool_fwd(int N, int C, int H, int W, int k, int s, int P, int Q, const float* x, float* y,
                               int32_t* idx, cudaStream_t st)
{
    const int NC = N * C;
    if (H * W <= kPoolSmemFloats) {
        const int ppb = kPoolSmemFloats / (H * W) < 8 ? kPoolSmemFloats / (H * W) : 8;
        const int blocks = (NC + ppb - 1) / ppb;
        maxpool_fwd_plane_kernel<<<blocks, kPoolThreads, size_t(ppb) * H * W * sizeof(float), st>>>(
            x, y, idx, NC, H, W, k, s, P, Q, ppb, FastDiv(P * Q), FastDiv(Q));
        note_launch();
        return cudaGetLastError();
    }
    const long long total = (long long)N * C * P * Q;
    maxpool_fwd_kernel<<<grid_for(total, 256), 256, 0, st>>>(x, y, idx, H, W, k, s, FastDiv(Q), FastDiv(P),
                                                             int(total));
    note_launch();
    return cudaGetLastError();
}

// Max pooling backward as a gather: dx[i] = sum, over the windows (ascending
// oh, then ow) that contain i and whose saved index is i, of their gradient.

__global__ void maxpool_bwd_kernel(const float* __restrict__ dy, const int32_t* __restrict__ idx,
                                   float* __restrict__ dx, int k, int S, int P, int Q, FastDiv f_w, FastDiv f_h,
                                   int total)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t r1, w, nc, h;
        f_w.divmod(uint32_t(t), r1, w);
        f_h.divmod(r1, nc, h);
        // windows with oh*S <= h < oh*S + k
        const int oh_lo = int(h) - k + 1 <= 0 ? 0 : (int(h) - k + S) / S;
        const int oh_hi = min(int(h) / S, P - 1);
        const int ow_lo = int(w) - k + 1 <= 0 ? 0 : (int(w) - k + S) / S;
        const int ow_hi = min(int(w) / S, Q - 1);
        float acc = 0.f;
        for (int oh = oh_lo; oh <= oh_hi; ++oh)
            for (int ow = ow_lo; ow <= ow_hi; ++ow) {
                const int o = (int(nc) * P + oh) * Q + ow;
                if (__ldg(idx + o) == t) acc += __ldg(dy + o);
            }
        dx[t] = acc;
    }
}

cudaError_t launch_maxpool_bwd(int N, int C, int H, int W, int k, int s, int P, int Q, const float* dy,
                               const int32_t* idx, float* dx, cudaStream_t st)
{
    const int NC = N * C;
    if (P * Q * 2 + H + W <= kPoolSmemFloats) {
        int ppb = (kPoolSmemFloats - H - W) / (2 * P * Q);
        if (ppb > 8) ppb = 8;
        const int blocks = (NC + ppb - 1) / ppb;
        maxpool_bwd_plane_kernel<<<blocks, kPoolThreads, (size_t(ppb) * P * Q * 2 + H + W) * sizeof(float), st>>>(
            dy, idx, dx, NC, H, W, k, s, P, Q, ppb, FastDiv(H * W), FastDiv(W));
        note_launch();
        return cudaGetLastError();
    }
    const long long total = (long long)N * C * H * W;
    maxpool_bwd_kernel<<<grid_for(total, 256), 256, 0, st>>>(dy, idx, dx, k, s, P, Q, FastDiv(W), FastDiv(H),
                                                             int(total));
    note_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SGD: p = p - lr * clamp(g, -clip, clip), one rounding per operation.

__device__ __forceinline__ float sgd_one(float p, float g, float lr, float clip)
{
    const float c = fminf(fmaxf(g, -clip), clip);
    return __fsub_rn(p, __fmul_rn(lr, c));
}

__global__ void sgd_kernel(float* __restrict__ p, const float* __restrict__ g, long long n4, long long count, float lr,
                           float clip)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    for (long long i = tid; i < n4; i += stride) {
        float4 pv = reinterpret_cast<float4*>(p)[i];
        const float4 gv = __ldg(reinterpret_cast<const float4*>(g) + i);
        pv.x = sgd_one(pv.x, gv.x, lr, clip);
        pv.y = sgd_one(pv.y, gv.y, lr, clip);
        pv.z = sgd_one(pv.z, gv.z, lr, clip);
        pv.w = sgd_one(pv.w, gv.w, lr, clip);
        reinterpret_cast<float4*>(p)[i] = pv;
    }
    for (long long i = n4 * 4 + tid; i < count; i += stride) p[i] = sgd_one(p[i], __ldg(g + i), lr, clip);
}

cudaError_t launch_sgd(int64_t count, float lr, float clip, float* p, const float* g, cudaStream_t st)
{
    if (count == 0) return cudaSuccess;
    const long long n4 = count / 4;
    sgd_kernel<<<grid_for(n4 > 0 ? n4 : 1, 256), 256, 0, st>>>(p, g, n4, count, lr, clip);
    note_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bias gradient: db[k] = sum over (n, oh, ow) of dy[n, k, oh, ow].
// One 8-CTA cluster per filter k: CTA r sums images n = r, r + 8, ... with a
// fixed thread/warp order, then CTA 0 adds the 8 partial sums from the
// cluster's shared memory in rank order.  Deterministic, no atomics.

constexpr int kBiasCluster = 8;
constexpr int kBiasThreads = 512;

__global__ void __cluster_dims__(kBiasCluster, 1, 1) __launch_bounds__(kBiasThreads)
    bias_grad_kernel(const float* __restrict__ dy, float* __restrict__ db, int N, int K, int PQ, FastDiv f_pq)
{
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ float warp_part[kBiasThreads / 32];
    __shared__ float cta_part;
    const int k = blockIdx.x / kBiasCluster;
    const int rank = int(cluster.block_rank());
    // This CTA sums images n = rank, rank + 8, ...: element e of that list is
    // (image rank + 8 * (e / PQ), pixel e % PQ).  Eight independent partial
    // sums per thread keep eight loads in flight; they are combined in a
    // fixed order, so the result is deterministic.
    const int images = (N - rank + kBiasCluster - 1) / kBiasCluster;
    const int total = images * PQ;
    float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int e0 = threadIdx.x; e0 < total; e0 += 8 * kBiasThreads) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * kBiasThreads;
            if (e < total) {
                uint32_t nl, pq;
                f_pq.divmod(uint32_t(e), nl, pq);
                const int n = rank + kBiasCluster * int(nl);
                part[u] += __ldg(dy + (size_t(n) * K + k) * PQ + pq);
            }
        }
    }
    float acc = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < kBiasThreads / 32; ++i) t += warp_part[i];
        cta_part = t;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
        float t = 0.f;
        for (int r = 0; r < kBiasCluster; ++r) t += *cluster.map_shared_rank(&cta_part, r);
        db[k] = t;
    }
    cluster.sync();   // keep every CTA's shared memory alive until rank 0 has read it
}

cudaError_t launch_bias_grad(const ConvDims& d, const float* dy, float* db, cudaStream_t st)
{
    bias_grad_kernel<<<d.K * kBiasCluster, kBiasThreads, 0, st>>>(dy, db, d.N, d.K, d.P * d.Q,
                                                                  FastDiv(d.P * d.Q));
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
