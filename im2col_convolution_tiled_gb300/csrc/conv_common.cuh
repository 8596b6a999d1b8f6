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
template <class Gen>
__global__ void build_bimage_kernel(Gen gen, int n_rows, int k_total, int bn, int k_stages, float* img)
{
    const int row = blockIdx.y;
    const int chunks = k_stages * (kBK / 4);
    const int nt = row / bn, r = row % bn;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < chunks; t += gridDim.x * blockDim.x) {
        const int k0 = t * 4;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float v = (row < n_rows && k0 + e < k_total) ? gen(row, k0 + e) : 0.f;
            split_tf32(v, hi[e], lo[e]);
        }
        const int ks = t / (kBK / 4), c = t % (kBK / 4);
        float* blk = img + ((size_t(nt) * k_stages + ks) * 2) * size_t(bn) * kBK;
        const uint32_t off = sw128_offset(uint32_t(r), uint32_t(c)) / 4;
        *reinterpret_cast<uint4*>(blk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(blk + size_t(bn) * kBK + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

template <class Gen>
cudaError_t build_bimage(const Gen& gen, int n_rows, int k_total, int bn, float* img, cudaStream_t st)
{
    const int n_tiles = (n_rows + bn - 1) / bn;
    const int k_stages = (k_total + kBK - 1) / kBK;
    const int chunks = k_stages * (kBK / 4);
    int bx = (chunks + 255) / 256;
    if (bx > 1024) bx = 1024;
    dim3 grid(bx, n_tiles * bn);
    build_bimage_kernel<Gen><<<grid, 256, 0, st>>>(gen, n_rows, k_total, bn, k_stages, img);
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
