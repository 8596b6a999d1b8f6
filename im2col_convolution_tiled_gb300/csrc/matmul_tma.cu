// matmul_tma.cu -- launches of the TMA-fed GEMM (gemm_tma.cuh) for the
// flagged matmul of the page "DirectCompute Neural Network Engine", section
// "Optimizations" -> "Transpose via Flags": the tensor maps of both operands
// and the kernel instantiation for the flags, tile width and math mode.  Its
// own translation unit so that it compiles beside matmul.cu.
#include "gemm_tma.cuh"

namespace cb200 {

static cudaError_t encode_kmajor(CUtensorMap* map, const float* X, int rows, int K, int box_rows)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(K) * 4};
    const cuuint32_t box[2] = {cuuint32_t(kTmaBK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(X), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A rows-contiguous operand (stored K x R): [16 k][32 r] boxes, 128-byte swizzle.
static cudaError_t encode_rmajor(CUtensorMap* map, const float* X, int R, int K)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cuuint64_t(R), cuuint64_t(K)};
    const cuuint64_t strides[1] = {cuuint64_t(R) * 4};
    const cuuint32_t box[2] = {32, cuuint32_t(kTmaBK)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(X), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <unsigned FLAGS, int BN>
static cudaError_t run_tma(int M, int K, int N, const float* A, const float* B, float* C, cudaStream_t st)
{
    constexpr bool AT = (FLAGS & 1u) != 0, BT = (FLAGS & 2u) == 0;
    TmaGemmArgs args{};
    cudaError_t e = AT ? encode_rmajor(&args.ta, A, M, K) : encode_kmajor(&args.ta, A, M, K, kBM);
    if (e != cudaSuccess) return e;
    if ((e = BT ? encode_rmajor(&args.tb, B, N, K) : encode_kmajor(&args.tb, B, N, K, BN)) != cudaSuccess) return e;
    args.C = C;
    args.M = M;
    args.N = N;
    args.K = K;
    args.m_tiles = (M + kBM - 1) / kBM;
    args.n_tiles = (N + BN - 1) / BN;
    args.k_stages = (K + kTmaBK - 1) / kTmaBK;
    args.vec_c = (N % 4 == 0) && aligned16(C);
    return math_terms() == 1 ? launch_tma_gemm_terms<BN, 1, AT, BT>(args, device_error_word(), st)
                             : launch_tma_gemm_terms<BN, 3, AT, BT>(args, device_error_word(), st);
}

cudaError_t launch_matmul_tma(unsigned flags, int bn, int M, int K, int N, const float* A, const float* B, float* C,
                              cudaStream_t st)
{
    switch (flags * 2 + (bn == 256 ? 1u : 0u)) {
    case 0: return run_tma<0, 128>(M, K, N, A, B, C, st);
    case 1: return run_tma<0, 256>(M, K, N, A, B, C, st);
    case 2: return run_tma<1, 128>(M, K, N, A, B, C, st);
    case 3: return run_tma<1, 256>(M, K, N, A, B, C, st);
    case 4: return run_tma<2, 128>(M, K, N, A, B, C, st);
    case 5: return run_tma<2, 256>(M, K, N, A, B, C, st);
    case 6: return run_tma<3, 128>(M, K, N, A, B, C, st);
    default: return run_tma<3, 256>(M, K, N, A, B, C, st);
    }
}

}  // namespace cb200
