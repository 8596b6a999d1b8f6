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
// Gen(row, k) returns the (unsplit) B element.
template <class Gen>
__global__ void build_bimage_kernel(Gen gen, int n_rows, int k_total, int bn, float* img)
{
    const int k_stages = (k_total + kBK - 1) / kBK;
    const int n_tiles = (n_rows + bn - 1) / bn;
    const long long total = (long long)n_tiles * bn * k_stages * kBK;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int k = int(e % (k_stages * kBK));
        const int row = int(e / (k_stages * kBK));
        float v = (row < n_rows && k < k_total) ? gen(row, k) : 0.f;
        uint32_t hi, lo;
        split_tf32(v, hi, lo);
        const int nt = row / bn, r = row % bn, ks = k / kBK, kk = k % kBK;
        float* blk = img + ((size_t(nt) * k_stages + ks) * 2) * size_t(bn) * kBK;
        const uint32_t off = sw128_offset(uint32_t(r), uint32_t(kk >> 2)) / 4 + (kk & 3);
        reinterpret_cast<uint32_t*>(blk)[off] = hi;
        reinterpret_cast<uint32_t*>(blk)[size_t(bn) * kBK + off] = lo;
    }
}

template <class Gen>
cudaError_t build_bimage(const Gen& gen, int n_rows, int k_total, int bn, float* img, cudaStream_t st)
{
    const long long total = (long long)((n_rows + bn - 1) / bn) * bn * ((k_total + kBK - 1) / kBK) * kBK;
    long long blocks = (total + 255) / 256;
    if (blocks > 4LL * sm_count() * 8) blocks = 4LL * sm_count() * 8;
    build_bimage_kernel<Gen><<<int(blocks), 256, 0, st>>>(gen, n_rows, k_total, bn, img);
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
