// train_ops.cu -- the element-wise and row-wise steps of a training step
// around the convolutions, from the page "DirectCompute Neural Network
// Engine", shader tables "Activation / Loss Shaders" (nn_relu, nn_relu_grad,
// nn_softmax_ce_grad, nn_loss) and "Utility Shaders" (nn_add_bias,
// nn_bias_grad, nn_grad_accum).
//
// All of them are small next to the convolutions (a LeNet-5 step moves a few
// MB), so they are written to be exact and deterministic first: every output
// is produced by one thread in a fixed order, sums use fixed shuffle trees,
// and fp32 additions/products are explicit (__fadd_rn / __fmul_rn) so no
// multiply-add is formed.  The element-wise kernels use 16-byte accesses.
#include "ptx.cuh"

namespace cb200 {

namespace {

constexpr int kEwThreads = 256;

int ew_grid(long long n4)
{
    long long b = (n4 + kEwThreads - 1) / kEwThreads;
    const long long cap = 8LL * sm_count();
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return int(b);
}

__device__ __forceinline__ float relu1(float v) { return v > 0.f ? v : 0.f; }
__device__ __forceinline__ float relu_grad1(float g, float x) { return __fmul_rn(g, x > 0.f ? 1.f : 0.f); }

// y = max(0, x) (nn_relu); +0 for x <= 0.  y may be x (in place).
__global__ void relu_fwd_kernel(const float* x, float* y, long long n)
{
    griddep_wait();
    griddep_launch();
    const long long n4 = n / 4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = reinterpret_cast<const float4*>(x)[i];
        reinterpret_cast<float4*>(y)[i] = make_float4(relu1(v.x), relu1(v.y), relu1(v.z), relu1(v.w));
    }
    for (long long i = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride)
        y[i] = relu1(x[i]);
}

// dx = dy * (x > 0) (nn_relu_grad); x is the ReLU's input or its output; dx may
// be dy (in place).
__global__ void relu_bwd_kernel(const float* dy, const float* __restrict__ x, float* dx, long long n)
{
    griddep_wait();
    griddep_launch();
    const long long n4 = n / 4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 g = reinterpret_cast<const float4*>(dy)[i];
        const float4 v = reinterpret_cast<const float4*>(x)[i];
        reinterpret_cast<float4*>(dx)[i] =
            make_float4(relu_grad1(g.x, v.x), relu_grad1(g.y, v.y), relu_grad1(g.z, v.z), relu_grad1(g.w, v.w));
    }
    for (long long i = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride)
        dx[i] = relu_grad1(dy[i], x[i]);
}

// acc = acc + g (nn_grad_accum), in place.
__global__ void grad_accum_kernel(const float* __restrict__ g, float* __restrict__ acc, long long n)
{
    griddep_wait();
    griddep_launch();
    const long long n4 = n / 4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 a = reinterpret_cast<const float4*>(acc)[i];
        const float4 b = reinterpret_cast<const float4*>(g)[i];
        reinterpret_cast<float4*>(acc)[i] =
            make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
    }
    for (long long i = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride)
        acc[i] = __fadd_rn(acc[i], g[i]);
}

// out[i][j] = A[i][j] + b[j] (nn_add_bias), optionally followed by max(0, .).
// One thread per element, consecutive threads on consecutive columns; out
// may be A (in place).
__global__ void add_bias_kernel(const float* A, const float* __restrict__ b, float* out, int rows,
                                int cols, int relu)
{
    griddep_wait();
    griddep_launch();
    const long long n = (long long)rows * cols;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride) {
        const float v = __fadd_rn(A[i], b[int(i % cols)]);
        out[i] = relu ? relu1(v) : v;
    }
}

// db[j] = sum_i G[i][j] (nn_bias_grad over the rows of a batch x out
// gradient).  A block takes 32 columns (one per lane, coalesced) and 8 row
// slices (one per warp: rows w, w + 8, ... summed in ascending order); the 8
// slice sums are then added in slice order.  The order is fixed by the shape
// alone, so the result is deterministic.
constexpr int kBgSlices = 8;
__global__ void __launch_bounds__(32 * kBgSlices) bias_grad_rows_kernel(const float* __restrict__ G,
                                                                       float* __restrict__ db, int rows, int cols)
{
    griddep_wait();
    griddep_launch();
    __shared__ float part[kBgSlices][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int j = blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (j < cols)
        for (int i = w; i < rows; i += kBgSlices) acc = __fadd_rn(acc, G[(long long)i * cols + j]);
    part[w][lane] = acc;
    __syncthreads();
    if (w == 0 && j < cols) {
        float s = part[0][lane];
#pragma unroll
        for (int k = 1; k < kBgSlices; ++k) s = __fadd_rn(s, part[k][lane]);
        db[j] = s;
    }
}

// Softmax + cross-entropy (nn_softmax_ce_grad, nn_loss), one block over all
// rows: warp w takes rows w, w + 32, ...  Per row: m = max z, s = sum
// exp(z - m) (lane partials over columns lane, lane + 32, ..., then a fixed
// xor-shuffle tree), p = exp(z - m) / s, dz = p - one_hot(label),
// loss_row = log(s) - (z[label] - m) = -log p[label].  The batch loss is the
// sum of the row losses: each warp adds its rows in ascending order, then the
// 32 warp sums are added in warp order.  A label outside [0, cols) marks the
// device error word (range) and its row gets dz = p and no loss.
constexpr int kCeThreads = 1024;
__global__ void __launch_bounds__(kCeThreads) softmax_ce_kernel(const float* __restrict__ z,
                                                                const int32_t* __restrict__ labels,
                                                                float* __restrict__ probs, float* __restrict__ dz,
                                                                float* __restrict__ loss, int rows, int cols,
                                                                int* err)
{
    griddep_wait();
    griddep_launch();
    __shared__ float warp_loss[kCeThreads / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float my_loss = 0.f;
    for (int r = w; r < rows; r += kCeThreads / 32) {
        const float* zr = z + (long long)r * cols;
        float m = -INFINITY;
        for (int j = lane; j < cols; j += 32) m = fmaxf(m, zr[j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = 0.f;
        for (int j = lane; j < cols; j += 32) s = __fadd_rn(s, expf(__fsub_rn(zr[j], m)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
        s = __shfl_sync(0xffffffffu, s, 0);   // every lane divides by the same (lane 0's) sum
        const int l = labels[r];
        const bool ok = l >= 0 && l < cols;
        if (!ok && lane == 0) atomicOr(err, kDevErrRange);
        for (int j = lane; j < cols; j += 32) {
            const float p = __fdiv_rn(expf(__fsub_rn(zr[j], m)), s);
            if (probs) probs[(long long)r * cols + j] = p;
            dz[(long long)r * cols + j] = (ok && j == l) ? __fsub_rn(p, 1.f) : p;
        }
        if (ok) my_loss = __fadd_rn(my_loss, __fsub_rn(logf(s), __fsub_rn(zr[l], m)));
    }
    if (lane == 0) warp_loss[w] = my_loss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int k = 0; k < kCeThreads / 32; ++k) t = __fadd_rn(t, warp_loss[k]);
        *loss = t;
    }
}

}  // namespace

cudaError_t launch_relu_fwd(int64_t n, const float* x, float* y, cudaStream_t st)
{
    cudaError_t e = launch_pdl(relu_fwd_kernel, dim3(ew_grid(n / 4 + 1)), dim3(kEwThreads), 0, st, x, y, n);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_relu_bwd(int64_t n, const float* dy, const float* x, float* dx, cudaStream_t st)
{
    cudaError_t e = launch_pdl(relu_bwd_kernel, dim3(ew_grid(n / 4 + 1)), dim3(kEwThreads), 0, st, dy, x, dx, n);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_grad_accum(int64_t n, const float* g, float* acc, cudaStream_t st)
{
    cudaError_t e = launch_pdl(grad_accum_kernel, dim3(ew_grid(n / 4 + 1)), dim3(kEwThreads), 0, st, g, acc, n);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_add_bias(int rows, int cols, const float* A, const float* b, float* out, int relu,
                            cudaStream_t st)
{
    cudaError_t e = launch_pdl(add_bias_kernel, dim3(ew_grid((long long)rows * cols)), dim3(kEwThreads), 0, st, A, b, out,
                               rows, cols, relu ? 1 : 0);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_bias_grad_rows(int rows, int cols, const float* G, float* db, cudaStream_t st)
{
    cudaError_t e = launch_pdl(bias_grad_rows_kernel, dim3((cols + 31) / 32), dim3(32 * kBgSlices), 0, st, G, db, rows,
                               cols);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_softmax_ce(int rows, int cols, const float* z, const int32_t* labels, float* probs, float* dz,
                              float* loss, cudaStream_t st)
{
    cudaError_t e = launch_pdl(softmax_ce_kernel, dim3(1), dim3(kCeThreads), 0, st, z, labels, probs, dz, loss, rows, cols,
                               device_error_word());
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
