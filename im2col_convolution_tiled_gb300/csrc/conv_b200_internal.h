// conv_b200_internal.h -- declarations shared by the library's translation
// units (never installed; the public ABI is include/conv_b200.h).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/conv_b200.h"

namespace cb200 {

// Bits of the device error word.
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrRange = 2;   // a class label outside [0, cols)

// The device error word lives in device memory (one per device, file scope in
// api.cu); kernels receive its address.
int* device_error_word();

// Number of SMs of the current device (cached per device).
int sm_count();

// Tensor-core products per 8-deep K step of every contraction launched now:
// 3 (3xTF32, fp32-faithful; the default) or 1 (one TF32 product), from the
// process-wide mode set by conv_b200_set_math_mode().
int math_terms();

// Count of kernels this library has launched since it was loaded (every
// <<<>>> launch calls note_launch()); exported as conv_b200_launch_count().
void note_launch();

// The stage set by conv_b200_debug_withhold_stage (or -1), taken -- and reset
// to -1 -- by the next launch of the register-gather GEMM kernel.
long long take_withhold_stage();
// The matmul engine test hook: -1 plan, 0 register gather, 1 TMA where eligible.
int matmul_engine_override();

inline cudaStream_t as_cuda(conv_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// Launchers implemented in the .cu files (return cudaError_t of the launch).

struct ConvDims {
    int N, C, H, W, K, R, S, P, Q;   // K = outC, R = kH, S = stride, P/Q = outH/outW
    int pad;
};

// relu: apply max(0, .) after the bias in the epilogue (conv_fwd_relu).
cudaError_t launch_conv_fwd(const ConvDims& d, const float* x, const float* w, const float* b, float* y,
                            void* ws, cudaStream_t st, bool relu = false);
size_t conv_fwd_ws(const ConvDims& d);

// mask non-null: G = dy * (mask > 0) (nn_relu_grad fused where dy is read).
cudaError_t launch_conv_dgrad(const ConvDims& d, const float* w, const float* dy, float* dx, void* ws,
                              cudaStream_t st, const float* mask = nullptr);
size_t conv_dgrad_ws(const ConvDims& d);

// db non-null: also the bias gradient, summed in the same pass over dy.
// mask non-null: G = dy * (mask > 0) (nn_relu_grad fused where dy is read).
cudaError_t launch_conv_wgrad(const ConvDims& d, const float* x, const float* dy, float* dw, void* ws,
                              cudaStream_t st, float* db = nullptr, const float* mask = nullptr);
size_t conv_wgrad_ws(const ConvDims& d);

// Tile width, K pieces per tile (cluster split) and whether the operands
// arrive by TMA, as launch_matmul plans them for operands at A and B.
void matmul_tiling(int M, int K, int N, unsigned flags, const float* A, const float* B, int* bn, int* csplit,
                   int* tma);
// Optional epilogue of matmul_fused: bias [N] added per column, then ReLU,
// then the product with (gate[m][n] > 0); all off by default.
struct MatmulEpi {
    const float* bias = nullptr;
    const float* gate = nullptr;
    int relu = 0;
};
cudaError_t launch_matmul(int M, int K, int N, unsigned flags, const float* A, const float* B, float* C,
                          cudaStream_t st, const MatmulEpi& ep = MatmulEpi{});
// The TMA-fed kernel for a planned matmul (matmul_tma.cu): flags 0..3, tile
// width bn (128 or 256); the caller has checked the operands qualify.
cudaError_t launch_matmul_tma(unsigned flags, int bn, int M, int K, int N, const float* A, const float* B, float* C,
                              cudaStream_t st);

cudaError_t launch_bias_grad(const ConvDims& d, const float* dy, float* db, cudaStream_t st);
cudaError_t launch_im2col(const ConvDims& d, const float* x, float* col, cudaStream_t st);
cudaError_t launch_col2im(const ConvDims& d, const float* col, float* dx, cudaStream_t st);
cudaError_t launch_maxpool_fwd(int N, int C, int H, int W, int k, int s, int P, int Q, const float* x, float* y,
                               int32_t* idx, cudaStream_t st);
cudaError_t launch_maxpool_bwd(int N, int C, int H, int W, int k, int s, int P, int Q, const float* dy,
                               const int32_t* idx, float* dx, cudaStream_t st);
cudaError_t launch_sgd(int64_t count, float lr, float clip, float* p, const float* g, cudaStream_t st);

cudaError_t launch_conv_fwd_direct(const ConvDims& d, const float* x, const float* w, const float* b, float* y,
                                   cudaStream_t st);
cudaError_t launch_conv_dgrad_direct(const ConvDims& d, const float* w, const float* dy, float* dx, cudaStream_t st);
cudaError_t launch_conv_wgrad_direct(const ConvDims& d, const float* x, const float* dy, float* dw, cudaStream_t st);

cudaError_t launch_relu_fwd(int64_t n, const float* x, float* y, cudaStream_t st);
cudaError_t launch_relu_bwd(int64_t n, const float* dy, const float* x, float* dx, cudaStream_t st);
cudaError_t launch_grad_accum(int64_t n, const float* g, float* acc, cudaStream_t st);
cudaError_t launch_add_bias(int rows, int cols, const float* A, const float* b, float* out, int relu,
                            cudaStream_t st);
cudaError_t launch_bias_grad_rows(int rows, int cols, const float* G, float* db, cudaStream_t st);
cudaError_t launch_softmax_ce(int rows, int cols, const float* z, const int32_t* labels, float* probs, float* dz,
                              float* loss, cudaStream_t st);

}  // namespace cb200
