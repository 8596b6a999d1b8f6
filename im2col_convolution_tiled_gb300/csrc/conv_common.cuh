// conv_common.cuh -- pieces shared by the three convolution GEMMs: tile-width
// choice and the kernel that lays a filter matrix out as pre-split,
// pre-swizzled tensor-core tiles for bulk copies.
#pragma once
#include "gemm_tc.cuh"

namespace cb200 {

// Widths the GEMM kernel is instantiated for along B rows (columns of D).
inline int pick_conv_bn(int n_total, int* n_tiles)
{
    const int cands[5] = {32, 64, 128, 192, 256};
    int tiles = (n_total + 255) / 256;
    int per = (n_total + tiles - 1) / tiles;
    int bn = 256;
    for (int i = 0; i < 5; ++i)
        if (cands[i] >= per) { bn = cands[i]; break; }
    *n_tiles = (n_total + bn - 1) / bn;
    return bn;
}

// Size in floats of a pre-split image of an (n_rows x k_total) B operand.
inline size_t bimage_floats(int n_rows, int k_total, int bn)
{
    const size_t n_tiles = (n_rows + bn - 1) / bn;
    const size_t k_stages = (k_total + kBK - 1) / kBK;
    return n_tiles * k_stages * 2 * size_t(bn) * kBK;
}

// Image layout: [n_tile][k_stage][hi, lo][bn x 32 fp32, 128-byte swizzled,
// K-major] -- each (n_tile, k_stage) block is exactly the shared-memory image
// of one pipeline stage's B tiles, so one bulk copy moves it.  Rows past
// n_rows and columns past k_total are zero.
//
// Gen(row, k) returns the (unsplit) B element.  One thread builds one 16-byte
// chunk (4 consecutive k of one row) of the hi and of the lo tile; blockIdx.y
// is the row, so consecutive threads read consecutive k.
// With rowsum non-null the kernel also sums each row's unsplit values: every
// block writes rowsum[row * gridDim.x + blockIdx.x] (its threads' values in a
// fixed order, then lanes, then warps), and rowsum_final_kernel adds a row's
// block partials in block order -- a deterministic row sum from the same pass
// (the filter gradient's dy image gives the bias gradient this way).
constexpr int kBimageThreads = 256;

// Gen may provide load4(row, k0, k_total, v): the four values k0 .. k0+3 of a
// row (zero past k_total) in one go, e.g. with one index division instead of
// four; otherwise they come from gen(row, k) one by one.
template <class Gen>
struct HasLoad4 {
    template <class G>
    static constexpr bool test(decltype(&G::load4)) { return true; }
    template <class G>
    static constexpr bool test(...) { return false; }
    static constexpr bool value = test<Gen>(nullptr);
};

template <class Gen>
__device__ __forceinline__ void bimage_load4(const Gen& gen, int row, int k0, int k_total, float (&v)[4])
{
    if constexpr (HasLoad4<Gen>::value) {
        gen.load4(row, k0, k_total, v);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = k0 + e < k_total ? gen(row, k0 + e) : 0.f;
    }
}

template <class Gen>
__global__ void __launch_bounds__(kBimageThreads) build_bimage_kernel(Gen gen, int n_rows, int k_total, int bn,
                                                                      int k_stages, float* img, float* rowsum)
{
    griddep_wait();
    griddep_launch();
    const int row = blockIdx.y;
    const int chunks = k_stages * (kBK / 4);
    const int nt = row / bn, r = row % bn;
    const int stride = gridDim.x * blockDim.x;
    float part = 0.f;
    auto put = [&](int t, const float (&v)[4]) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_tf32(v[e], hi[e], lo[e]);
        const int ks = t / (kBK / 4), c = t % (kBK / 4);
        float* blk = img + ((size_t(nt) * k_stages + ks) * 2) * size_t(bn) * kBK;
        const uint32_t off = sw128_offset(uint32_t(r), uint32_t(c)) / 4;
        *reinterpret_cast<uint4*>(blk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(blk + size_t(bn) * kBK + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    };
    // two chunks per iteration: both chunks' loads are issued before either
    // is split and stored
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < chunks; t += 2 * stride) {
        const int t2 = t + stride;
        float v[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f};
        if (row < n_rows) {
            bimage_load4(gen, row, t * 4, k_total, v);
            if (t2 < chunks) bimage_load4(gen, row, t2 * 4, k_total, w);
        }
        part += (v[0] + v[1]) + (v[2] + v[3]);
        put(t, v);
        if (t2 < chunks) {
            part += (w[0] + w[1]) + (w[2] + w[3]);
            put(t2, w);
        }
    }
    if (rowsum == nullptr || row >= n_rows) return;   // uniform over the block
    __shared__ float warp_part[kBimageThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < kBimageThreads / 32; ++i) t += warp_part[i];
        rowsum[size_t(row) * gridDim.x + blockIdx.x] = t;
    }
}

// The same image in 16-deep blocks with 64-byte rows (the flat kernel's B
// operand, gemm_flat.cuh): img[n_tile][block][2 * bn rows][16] -- the hi rows
// 0..bn-1 then the lo rows bn..2bn-1 of the block, each row one 64-byte
// swizzled K-major row (16-byte chunk j of row r at (j ^ ((r >> 1) & 3)) * 16).
// A flat K stage is two consecutive blocks (two taps).
template <class Gen>
__global__ void __launch_bounds__(kBimageThreads) build_bimage16_kernel(Gen gen, int n_rows, int k_total, int bn,
                                                                        int k_stages, float* img)
{
    griddep_wait();
    griddep_launch();
    const int row = blockIdx.y;
    const int nt = row / bn, r = row % bn;
    const int chunks = k_stages * 4;   // 4-value chunks of one row
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < chunks; t += gridDim.x * blockDim.x) {
        const int k0 = t * 4;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float v = (row < n_rows && k0 + e < k_total) ? gen(row, k0 + e) : 0.f;
            split_tf32(v, hi[e], lo[e]);
        }
        const int ks = t >> 2, c = t & 3;
        float* blk = img + (size_t(nt) * k_stages + ks) * 2 * size_t(bn) * 16;
        const uint32_t oh = (uint32_t(r) * 64u + ((uint32_t(c) ^ ((uint32_t(r) >> 1) & 3u)) << 4)) / 4u;
        const uint32_t ol = (uint32_t(r + bn) * 64u + ((uint32_t(c) ^ ((uint32_t(r + bn) >> 1) & 3u)) << 4)) / 4u;
        *reinterpret_cast<uint4*>(blk + oh) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(blk + ol) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Floats of build_bimage16's image: n_tiles x k_stages stages of 2 * bn x 16.
inline size_t bimage16_floats(int n_rows, int k_stages, int bn)
{
    return size_t((n_rows + bn - 1) / bn) * size_t(k_stages) * 2 * size_t(bn) * 16;
}

template <class Gen>
cudaError_t build_bimage16(const Gen& gen, int n_rows, int k_stages, int bn, float* img, cudaStream_t st)
{
    const int n_tiles = (n_rows + bn - 1) / bn;
    const int chunks = k_stages * 4;
    int bx = (chunks + kBimageThreads - 1) / kBimageThreads;
    if (bx > 1024) bx = 1024;
    cudaError_t le = launch_pdl(build_bimage16_kernel<Gen>, dim3(bx, n_tiles * bn), dim3(kBimageThreads), 0, st, gen,
                                n_rows, k_stages * 16, bn, k_stages, img);
    if (le != cudaSuccess) return le;
    note_launch();
    return cudaGetLastError();
}

// Blocks per row of build_bimage (so callers can size the row-sum partials).
inline int bimage_grid_x(int k_total)
{
    const int k_stages = (k_total + kBK - 1) / kBK;
    const int chunks = k_stages * (kBK / 4);
    int bx = (chunks + kBimageThreads - 1) / kBimageThreads;
    return bx > 1024 ? 1024 : bx;
}

template <class Gen>
cudaError_t build_bimage(const Gen& gen, int n_rows, int k_total, int bn, float* img, cudaStream_t st,
                         float* rowsum = nullptr)
{
    const int n_tiles = (n_rows + bn - 1) / bn;
    const int k_stages = (k_total + kBK - 1) / kBK;
    dim3 grid(bimage_grid_x(k_total), n_tiles * bn);
    cudaError_t le = launch_pdl(build_bimage_kernel<Gen>, grid, dim3(kBimageThreads), 0, st, gen, n_rows, k_total, bn,
                                k_stages, img, rowsum);
    if (le != cudaSuccess) return le;
    note_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Space-to-depth copy for strided convolutions with few channels: for stride
// S, X'[n, c', hh, ww] = x[n, c, S*hh + a - pad, S*ww + b - pad] with
// c' = c*S*S + a*S + b (zero outside the image), over an Hs x Ws super-pixel
// grid.  BLOCKED writes the channel-blocked layout [n][c'/32][hh][ww][32]
// (zero for c' >= C*S*S) that the tensor-map patch kernel loads; otherwise
// NCHW [n][c'][hh][ww] for the filter gradient's column gather.
//
// A gather with no shared memory and no barriers: one output vector per
// thread, every load it needs issued up front.  (A persistent form that staged
// each super-row's input rows in shared memory through bulk copies ran at a
// third of the copy bandwidth: one block-wide barrier per 15 KB super-row.)
//   BLOCKED: thread t writes float4 t of [n][c'/32][hh][ww][32], i.e. channels
//            c' = 32*cb + 4*g .. + 3 of one super-pixel (g = t % 8): eight
//            threads fill a 128-byte pixel, a warp four whole pixels.
//   NCHW:    thread t = (((n*C + c)*S + a)*Hs + hh)*Ws + ww reads the S
//            consecutive inputs x[n, c, S*hh + a - pad, S*ww - pad ..] and
//            writes them to planes c' = (c*S + a)*S + b, b < S; lanes run
//            along ww, so loads and stores are contiguous per warp.
constexpr int kS2dGatherThreads = 256;
constexpr int kS2dLoads = 8;   // NCHW form: loads issued together

template <bool BLOCKED>
__global__ void __launch_bounds__(kS2dGatherThreads)
    s2d_gather_kernel(const float* __restrict__ x, float* __restrict__ dst, int C, int H, int W, int S, int pad,
                      int Cs, long long total, FastDiv f_ws, FastDiv f_hs, FastDiv f_mid, FastDiv f_s, FastDiv f_ss)
{
    griddep_wait();
    griddep_launch();
    const long long t = (long long)blockIdx.x * kS2dGatherThreads + threadIdx.x;
    if (t >= total) return;
    if constexpr (BLOCKED) {
        // t = (((n * Cb + cb) * Hs + hh) * Ws + ww) * 8 + g; f_mid divides by Cb
        const uint32_t g = uint32_t(t) & 7u;
        uint32_t r, ww, hh, cb, n;
        f_ws.divmod(uint32_t(t >> 3), r, ww);
        f_hs.divmod(r, r, hh);
        f_mid.divmod(r, n, cb);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int cp = int(cb) * 32 + 4 * int(g) + e;
            uint32_t c, ab, a, b;
            f_ss.divmod(uint32_t(cp), c, ab);
            f_s.divmod(ab, a, b);
            const int h = S * int(hh) + int(a) - pad, w = S * int(ww) + int(b) - pad;
            const bool in = cp < Cs && unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W);
            v[e] = in ? __ldg(x + ((size_t(n) * C + c) * H + h) * W + w) : 0.f;
        }
        reinterpret_cast<float4*>(dst)[t] = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        // t = (((n * C + c) * S + a) * Hs + hh) * Ws + ww; f_mid divides by C
        uint32_t r, ww, hh, a, c, n;
        f_ws.divmod(uint32_t(t), r, ww);
        f_hs.divmod(r, r, hh);
        f_s.divmod(r, r, a);
        f_mid.divmod(r, n, c);
        const int Hs = int(f_hs.d), Ws = int(f_ws.d);
        const int h = S * int(hh) + int(a) - pad;
        const bool row_in = unsigned(h) < unsigned(H);
        const float* src = x + ((size_t(n) * C + c) * H + (row_in ? h : 0)) * W;
        float* out = dst + ((size_t(n) * Cs + (int(c) * S + int(a)) * S) * Hs + hh) * Ws + ww;
        if (S <= kS2dLoads) {
            // one pass, fully unrolled (a loop around it measured 6% slower on AlexNet conv1)
            float v[kS2dLoads];
#pragma unroll
            for (int b = 0; b < kS2dLoads; ++b) {
                const int w = S * int(ww) + b - pad;
                v[b] = (b < S && row_in && unsigned(w) < unsigned(W)) ? __ldg(src + w) : 0.f;
            }
#pragma unroll
            for (int b = 0; b < kS2dLoads; ++b)
                if (b < S) out[size_t(b) * Hs * Ws] = v[b];
            return;
        }
        for (int b0 = 0; b0 < S; b0 += kS2dLoads) {
            float v[kS2dLoads];
#pragma unroll
            for (int i = 0; i < kS2dLoads; ++i) {
                const int w = S * int(ww) + b0 + i - pad;
                v[i] = (b0 + i < S && row_in && unsigned(w) < unsigned(W)) ? __ldg(src + w) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kS2dLoads; ++i)
                if (b0 + i < S) out[size_t(b0 + i) * Hs * Ws] = v[i];
        }
    }
}

// The same copy for S = 4, W % 4 == 0 and x 16-byte aligned: the four inputs
// of a (c, a, hh, ww) row segment, x[n, c, 4hh + a - pad, 4ww - pad .. + 3],
// lie in two aligned float4 of the row (each wholly inside or outside the
// image, since W % 4 == 0), at offset OFF = (-pad) mod 4 -- the same for every
// thread, so it is a template parameter.  Lanes run along ww: each load
// instruction reads 512 contiguous bytes.
//   BLOCKED: thread t = ((n*Cb + cb)*Hs + hh)*Ws + ww writes the whole 128-byte
//            pixel of chunk cb (eight (c, a) segments of four channels b).
//   NCHW:    thread t = (((n*C + c)*4 + a)*Hs + hh)*Ws + ww writes its segment
//            to the four planes b.
template <int OFF>
__device__ __forceinline__ float4 s2d_segment(const float* __restrict__ rowp, int a0, int W)
{
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 lo = unsigned(a0) < unsigned(W) ? __ldg(reinterpret_cast<const float4*>(rowp + a0)) : z;
    if constexpr (OFF == 0) return lo;
    const float4 hi = unsigned(a0 + 4) < unsigned(W) ? __ldg(reinterpret_cast<const float4*>(rowp + a0 + 4)) : z;
    if constexpr (OFF == 1) return make_float4(lo.y, lo.z, lo.w, hi.x);
    if constexpr (OFF == 2) return make_float4(lo.z, lo.w, hi.x, hi.y);
    return make_float4(lo.w, hi.x, hi.y, hi.z);
}

template <bool BLOCKED, int OFF>
__global__ void __launch_bounds__(kS2dGatherThreads)
    s2d_gather4_kernel(const float* __restrict__ x, float* __restrict__ dst, int C, int H, int W, int pad, int Cs,
                       long long total, FastDiv f_ws, FastDiv f_hs, FastDiv f_mid)
{
    griddep_wait();
    griddep_launch();
    const long long t = (long long)blockIdx.x * kS2dGatherThreads + threadIdx.x;
    const int Hs = int(f_hs.d), Ws = int(f_ws.d);
    if constexpr (BLOCKED) {
        // The warp's 32 pixels pass through shared memory so that each store
        // instruction writes four whole pixels (512 contiguous bytes) instead
        // of one 16-byte piece of 32 pixels; the 16-byte slots are XOR-swizzled
        // by pixel, so neither side has bank conflicts.
        __shared__ float4 stage[kS2dGatherThreads * 8];
        const int lane = int(threadIdx.x) & 31;
        float4* wst = stage + (threadIdx.x - lane) * 8;
        float4 out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) out[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < total) {
            uint32_t r, ww, hh, cb, n;
            f_ws.divmod(uint32_t(t), r, ww);
            f_hs.divmod(r, r, hh);
            f_mid.divmod(r, n, cb);
            const int a0 = 4 * int(ww) - pad - OFF;   // aligned start of the segment's first float4
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int cp0 = int(cb) * 32 + 4 * j;   // channels cp0 .. cp0 + 3: b = 0..3 of one (c, a)
                const int c = cp0 >> 4, a = (cp0 >> 2) & 3;
                const int h = 4 * int(hh) + a - pad;
                if (cp0 < Cs && unsigned(h) < unsigned(H))
                    out[j] = s2d_segment<OFF>(x + ((size_t(n) * C + c) * H + h) * W, a0, W);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) wst[lane * 8 + (j ^ (lane & 7))] = out[j];
        __syncwarp();
        const long long t0 = t - lane;   // the warp's first pixel
        float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int px = 4 * i + (lane >> 3), j = lane & 7;
            if (t0 + px < total) d[size_t(t0 + px) * 8 + j] = wst[px * 8 + (j ^ (px & 7))];
        }
    } else {
        if (t >= total) return;
        uint32_t r, ww, hh, a, c, n;
        f_ws.divmod(uint32_t(t), r, ww);
        f_hs.divmod(r, r, hh);
        a = r & 3u;
        r >>= 2;
        f_mid.divmod(r, n, c);
        const int h = 4 * int(hh) + int(a) - pad;
        const float4 v = unsigned(h) < unsigned(H)
                             ? s2d_segment<OFF>(x + ((size_t(n) * C + c) * H + h) * W, 4 * int(ww) - pad - OFF, W)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        float* out = dst + ((size_t(n) * Cs + (int(c) * 4 + int(a)) * 4) * Hs + hh) * Ws + ww;
        const size_t plane = size_t(Hs) * Ws;
        out[0] = v.x;
        out[plane] = v.y;
        out[2 * plane] = v.z;
        out[3 * plane] = v.w;
    }
}

template <bool BLOCKED>
cudaError_t launch_s2d_copy(const float* x, float* dst, int N, int C, int H, int W, int S, int pad, int Hs, int Ws,
                            cudaStream_t st)
{
    const int Cs = C * S * S, Cb = (Cs + 31) / 32;
    if (S == 4 && W % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const long long total4 = BLOCKED ? (long long)N * Cb * Hs * Ws : (long long)N * C * 4 * Hs * Ws;
        const unsigned blocks4 = unsigned((total4 + kS2dGatherThreads - 1) / kS2dGatherThreads);
        const int off = ((-pad) % 4 + 4) % 4;
        auto run = [&](auto kern) {
            return launch_pdl(kern, dim3(blocks4), dim3(kS2dGatherThreads), 0, st, x, dst, C, H, W, pad, Cs, total4,
                              FastDiv(uint32_t(Ws)), FastDiv(uint32_t(Hs)), FastDiv(uint32_t(BLOCKED ? Cb : C)));
        };
        cudaError_t le = off == 0   ? run(s2d_gather4_kernel<BLOCKED, 0>)
                         : off == 1 ? run(s2d_gather4_kernel<BLOCKED, 1>)
                         : off == 2 ? run(s2d_gather4_kernel<BLOCKED, 2>)
                                    : run(s2d_gather4_kernel<BLOCKED, 3>);
        if (le != cudaSuccess) return le;
        note_launch();
        return cudaGetLastError();
    }
    const long long total = BLOCKED ? (long long)N * Cb * Hs * Ws * 8 : (long long)N * C * S * Hs * Ws;
    const unsigned blocks = unsigned((total + kS2dGatherThreads - 1) / kS2dGatherThreads);
    cudaError_t le = launch_pdl(s2d_gather_kernel<BLOCKED>, dim3(blocks), dim3(kS2dGatherThreads), 0, st, x, dst, C,
                                H, W, S, pad, Cs, total, FastDiv(uint32_t(Ws)), FastDiv(uint32_t(Hs)),
                                FastDiv(uint32_t(BLOCKED ? Cb : C)), FastDiv(uint32_t(S)), FastDiv(uint32_t(S * S)));
    if (le != cudaSuccess) return le;
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
