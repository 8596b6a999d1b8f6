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

template <class Gen>
__global__ void __launch_bounds__(kBimageThreads) build_bimage_kernel(Gen gen, int n_rows, int k_total, int bn,
                                                                      int k_stages, float* img, float* rowsum)
{
    const int row = blockIdx.y;
    const int chunks = k_stages * (kBK / 4);
    const int nt = row / bn, r = row % bn;
    float part = 0.f;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < chunks; t += gridDim.x * blockDim.x) {
        const int k0 = t * 4;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float v = (row < n_rows && k0 + e < k_total) ? gen(row, k0 + e) : 0.f;
            part += v;
            split_tf32(v, hi[e], lo[e]);
        }
        const int ks = t / (kBK / 4), c = t % (kBK / 4);
        float* blk = img + ((size_t(nt) * k_stages + ks) * 2) * size_t(bn) * kBK;
        const uint32_t off = sw128_offset(uint32_t(r), uint32_t(c)) / 4;
        *reinterpret_cast<uint4*>(blk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(blk + size_t(bn) * kBK + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
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
    build_bimage_kernel<Gen><<<grid, kBimageThreads, 0, st>>>(gen, n_rows, k_total, bn, k_stages, img, rowsum);
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
// Persistent blocks take super-rows (n, hh) in turn.  The C*S input rows of a
// super-row are staged in shared memory, kS2dBufs super-rows deep, so that the
// reads of the next ones are in flight while one is written out: with one bulk
// copy per row (the copy engine, completion on a per-buffer mbarrier) when rows
// start on 16-byte boundaries (W a multiple of 4), else with 4-byte cp.async.
// Shared rows have a pitch of 4 mod 32 floats, so the lanes of a warp reading
// (b, a, c) neighbours hit distinct banks.  Waits are bounded; on give-up the
// block records the error and leaves after its copies have landed.
__host__ __device__ inline int s2d_pitch(int W) { return W + ((4 - W) % 32 + 32) % 32; }

constexpr int kS2dThreads = 256;
constexpr int kS2dBufs = 3;

template <bool BLOCKED>
__global__ void __launch_bounds__(kS2dThreads, 4)
    s2d_copy_kernel(const float* __restrict__ x, float* __restrict__ dst, int C, int H, int W, int S, int pad, int Cs,
                    int Cb, int Hs, int Ws, int items, FastDiv f_s, FastDiv f_ss, FastDiv f_hs, int* err)
{
    extern __shared__ __align__(16) float s2d_rows[];   // kS2dBufs buffers of [c * S + a][pitch]
    __shared__ uint64_t bar[kS2dBufs];
    __shared__ int abort_flag;
    const int CS = C * S, pitch = s2d_pitch(W);
    const int buf_floats = CS * pitch;
    const bool bulk = (W & 3) == 0;
    if (threadIdx.x == 0) {
        for (int b = 0; b < kS2dBufs; ++b) mbar_init(&bar[b], 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // stage super-row `item` into buffer b.  Rows outside the image are
    // zero-filled by every thread; with bulk copies the lanes of warp 0 issue
    // one input row each (the byte count of the stage summed over the warp
    // first), so no single thread walks all C * S rows.
    auto stage = [&](int item, int b) {
        uint32_t n, hh;
        f_hs.divmod(uint32_t(item), n, hh);
        float* buf = s2d_rows + b * buf_floats;
        int c = 0, a = 0;   // (c, a) of row ca, advanced without divisions
        for (int ca = 0; ca < CS; ++ca) {
            const int h = S * int(hh) + a - pad;
            float* row = buf + ca * pitch;
            if (unsigned(h) < unsigned(H)) {
                if (!bulk) {
                    const float* src = x + ((size_t(n) * C + c) * H + h) * W;
                    for (int w = threadIdx.x; w < W; w += kS2dThreads) cp_async4(smem_u32(row + w), src + w);
                }
            } else {
                for (int w = threadIdx.x; w < W; w += kS2dThreads) row[w] = 0.f;
            }
            if (++a == S) { a = 0; ++c; }
        }
        if (bulk && threadIdx.x < 32) {
            const int lane = threadIdx.x;
            fence_proxy_async_smem();   // the buffer's last readers are done (they passed the barrier)
            uint32_t live = 0;
            for (int ca = lane; ca < CS; ca += 32) {
                const int h = S * int(hh) + ca % S - pad;
                live += unsigned(h) < unsigned(H) ? 1u : 0u;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) live += __shfl_xor_sync(0xffffffffu, live, o);
            if (lane == 0) mbar_arrive_expect_tx(&bar[b], live * uint32_t(W) * 4u);
            __syncwarp();
            for (int ca = lane; ca < CS; ca += 32) {
                const int cc = ca / S, aa = ca - cc * S;
                const int h = S * int(hh) + aa - pad;
                if (unsigned(h) < unsigned(H))
                    bulk_g2s(buf + ca * pitch, x + ((size_t(n) * C + cc) * H + h) * W, uint32_t(W) * 4u, &bar[b]);
            }
        }
        if (!bulk) cp_async_commit();
    };
    int it = 0, item = blockIdx.x;
    for (int i = 0; i < kS2dBufs - 1; ++i) {
        const int pre = item + i * int(gridDim.x);
        if (pre < items) stage(pre, i);
        else if (!bulk) cp_async_commit();   // keep one group per buffer slot
    }
    for (; item < items; item += gridDim.x, ++it) {
        bool got = true;
        if (bulk) got = mbar_wait(&bar[it % kS2dBufs], uint32_t(it / kS2dBufs) & 1u, &abort_flag);
        else cp_async_wait_group<kS2dBufs - 2>();   // this thread's copies of the current super-row landed
        if (!__syncthreads_and(got ? 1 : 0)) {      // ... and everybody else's
            if (threadIdx.x == 0) {
                abort_flag = 1;
                atomicOr(err, kDevErrTimeout);
            }
            break;
        }
        // Every thread is past this barrier, hence done reading the buffer of
        // the previous super-row: refill that one with the super-row two ahead.
        const int ahead = item + (kS2dBufs - 1) * int(gridDim.x);
        if (ahead < items) stage(ahead, (it + kS2dBufs - 1) % kS2dBufs);
        else if (!bulk) cp_async_commit();
        const float* buf = s2d_rows + (it % kS2dBufs) * buf_floats;
        uint32_t n, hh;
        f_hs.divmod(uint32_t(item), n, hh);
        // A thread owns four consecutive channels c' = 4g .. 4g + 3 of a 32-channel
        // block: their rows and column offsets are decoded once per block, then
        // each pixel costs four shared loads.  Blocked: g = thread % 8 and eight
        // threads write a pixel; NCHW: g = warp and the lanes run along ww.
        const int g4 = BLOCKED ? (threadIdx.x & 7) : (threadIdx.x >> 5);
        const int ww0 = BLOCKED ? (threadIdx.x >> 3) : (threadIdx.x & 31);
        for (int cb = 0; cb < Cb; ++cb) {
            const float* row[4];
            int boff[4];
            bool live[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t c, ab, a, b;
                f_ss.divmod(uint32_t(cb * 32 + 4 * g4 + e), c, ab);
                f_s.divmod(ab, a, b);
                live[e] = int(c) < C;
                row[e] = buf + (live[e] ? (int(c) * S + int(a)) * pitch : 0);
                boff[e] = int(b) - pad;
            }
            if constexpr (BLOCKED) {
                // eight threads write one 128-byte pixel with 16-byte stores
                float4* out = reinterpret_cast<float4*>(dst + ((size_t(n) * Cb + cb) * Hs + hh) * size_t(Ws) * 32);
                for (int ww = ww0; ww < Ws; ww += 32) {
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int w = S * ww + boff[e];
                        v[e] = (live[e] && unsigned(w) < unsigned(W)) ? row[e][w] : 0.f;
                    }
                    out[ww * 8 + g4] = make_float4(v[0], v[1], v[2], v[3]);
                }
            } else {
                // channels of the block past Cs do not exist in NCHW
                const int cp0 = cb * 32 + 4 * g4;
                for (int ww = ww0; ww < Ws; ww += 32) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (cp0 + e >= Cs) break;
                        const int w = S * ww + boff[e];
                        dst[((size_t(n) * Cs + cp0 + e) * Hs + hh) * size_t(Ws) + ww] =
                            (live[e] && unsigned(w) < unsigned(W)) ? row[e][w] : 0.f;
                    }
                }
            }
        }
    }
    if (!bulk) cp_async_wait_group<0>();
    if (bulk && abort_flag && threadIdx.x == 0) {
        // copies still in flight (the failed super-row's and the next one's:
        // refills happen only after a passed barrier) land before the block's
        // shared memory goes away
        for (int j = 0; j < kS2dBufs - 1; ++j) {
            const int pending = item + j * int(gridDim.x);
            if (pending >= items) break;
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&bar[(it + j) % kS2dBufs], uint32_t((it + j) / kS2dBufs) & 1u) &&
                   globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// Shared memory of s2d_copy_kernel (kS2dBufs buffers of staged rows).
inline size_t s2d_copy_smem(int C, int S, int W) { return kS2dBufs * size_t(C) * S * s2d_pitch(W) * sizeof(float); }
constexpr size_t kS2dMaxSmem = 96 * 1024;

template <bool BLOCKED>
cudaError_t launch_s2d_copy(const float* x, float* dst, int N, int C, int H, int W, int S, int pad, int Hs, int Ws,
                            cudaStream_t st)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(s2d_copy_kernel<BLOCKED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(kS2dMaxSmem));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int Cs = C * S * S, Cb = (Cs + 31) / 32;
    const int items = N * Hs;
    const int grid = items < 4 * sm_count() ? items : 4 * sm_count();
    s2d_copy_kernel<BLOCKED><<<grid, kS2dThreads, s2d_copy_smem(C, S, W), st>>>(
        x, dst, C, H, W, S, pad, Cs, Cb, Hs, Ws, items, FastDiv(uint32_t(S)), FastDiv(uint32_t(S * S)),
        FastDiv(uint32_t(Hs)), device_error_word());
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
