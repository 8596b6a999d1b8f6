// api.cu -- the extern "C" entry points of libconv_b200 (include/conv_b200.h):
// argument validation, then one or two asynchronous launches on the caller's
// stream.  Nothing here synchronises the host except conv_b200_check().
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "conv_b200_internal.h"

namespace cb200 {

// Device error word: a file-scope device variable, one instance per device
// that loads the library, so no allocation is ever needed for it.
__device__ int g_error_word;

namespace {
constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];
bool g_sm103[kMaxDevices];   // an sm_103 part this library was compiled for
std::once_flag g_once[kMaxDevices];

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    return dev;
}

void init_device(int dev)
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) g_err_ptr[dev] = static_cast<int*>(p);
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
    g_sms[dev] = sms;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        major = minor = 0;
    }
    g_sm103[dev] = major == 10 && minor == 3;
}
}  // namespace

static std::atomic<unsigned long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<int> g_math_mode{CONV_MATH_FP32};

// Test hook of the bounded-wait error path (conv_b200_debug_withhold_stage):
// -1, or the CTA-wide stage whose arrival CTA 0 of the next register-gather
// GEMM launch withholds.  One-shot: the launch that takes it resets it.
static std::atomic<long long> g_withhold_stage{-1};
long long take_withhold_stage() { return g_withhold_stage.exchange(-1, std::memory_order_relaxed); }

// Test hook of the matmul engine choice (conv_b200_debug_matmul_engine).
static std::atomic<int> g_matmul_engine{-1};
int matmul_engine_override() { return g_matmul_engine.load(std::memory_order_relaxed); }
int math_terms() { return g_math_mode.load(std::memory_order_relaxed) == CONV_MATH_TF32 ? 1 : 3; }

int* device_error_word()
{
    const int dev = current_device();
    std::call_once(g_once[dev], init_device, dev);
    return g_err_ptr[dev];
}

int sm_count()
{
    const int dev = current_device();
    std::call_once(g_once[dev], init_device, dev);
    return g_sms[dev];
}

// Is the current device an sm_103 part this library was compiled for?
// (Looked up once per device, under the same once-flag as the rest of the
// per-device state, so concurrent host threads see one consistent answer.)
static bool device_ok()
{
    const int dev = current_device();
    std::call_once(g_once[dev], init_device, dev);
    return g_sm103[dev];
}

static constexpr long long kMaxElems = (1LL << 31) - 1;
static constexpr int kMaxExtent = 16384;   // per spatial axis; keeps every index in int32 with headroom

// Validate a convolution shape and fill ConvDims.
static int check_shape(const conv_shape_t* s, ConvDims* d)
{
    if (!s) return CONV_ERR_NULL;
    if (s->batch <= 0 || s->inC <= 0 || s->inH <= 0 || s->inW <= 0 || s->outC <= 0 || s->kH <= 0 ||
        s->stride <= 0 || s->padding < 0)
        return CONV_ERR_SHAPE;
    if (s->inH > kMaxExtent || s->inW > kMaxExtent || s->kH > kMaxExtent || s->padding > kMaxExtent / 2 ||
        s->stride > 64)
        return CONV_ERR_SHAPE;
    const long long hp = (long long)s->inH + 2LL * s->padding - s->kH;
    const long long wp = (long long)s->inW + 2LL * s->padding - s->kH;
    if (hp < 0 || wp < 0) return CONV_ERR_SHAPE;
    if (s->outH != hp / s->stride + 1 || s->outW != wp / s->stride + 1) return CONV_ERR_SHAPE;
    const long long x = (long long)s->batch * s->inC * s->inH * s->inW;
    const long long y = (long long)s->batch * s->outC * s->outH * s->outW;
    const long long w = (long long)s->outC * s->inC * s->kH * s->kH;
    const long long col = (long long)s->inC * s->kH * s->kH * s->batch * s->outH * s->outW;
    (void)col;
    if (x > kMaxElems || y > kMaxElems || w > kMaxElems) return CONV_ERR_OVERFLOW;
    d->N = s->batch;
    d->C = s->inC;
    d->H = s->inH;
    d->W = s->inW;
    d->K = s->outC;
    d->R = s->kH;
    d->S = s->stride;
    d->pad = s->padding;
    d->P = s->outH;
    d->Q = s->outW;
    return CONV_OK;
}

static int status_of(cudaError_t e)
{
    if (e == cudaSuccess) return CONV_OK;
    cudaGetLastError();
    return CONV_ERR_CUDA;
}

static int check_ptrs(std::initializer_list<const void*> ps)
{
    for (const void* p : ps)
        if (!p) return CONV_ERR_NULL;
    for (const void* p : ps)
        if (!aligned16(p)) return CONV_ERR_ALIGN;
    return CONV_OK;
}

static int check_workspace(size_t need, const void* ws, size_t have)
{
    if (need == 0) return CONV_OK;
    if (!ws || have < need) return CONV_ERR_WORKSPACE;
    if (!aligned16(ws)) return CONV_ERR_ALIGN;
    return CONV_OK;
}

}  // namespace cb200

using namespace cb200;

extern "C" {

size_t conv_b200_workspace_bytes(int op, const conv_shape_t* s)
{
    ConvDims d;
    if (check_shape(s, &d) != CONV_OK) return 0;
    switch (op) {
    case CONV_OP_FWD: return conv_fwd_ws(d);
    case CONV_OP_BWD_DATA: return conv_dgrad_ws(d);
    case CONV_OP_BWD_FILTER: return conv_wgrad_ws(d);
    default: return 0;
    }
}

int conv_fwd(const conv_shape_t* s, const float* x, const float* w, const float* b, float* y, void* workspace,
             size_t workspace_bytes, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, w, y})) != CONV_OK) return rc;
    if (b && !aligned16(b)) return CONV_ERR_ALIGN;
    if ((rc = check_workspace(conv_fwd_ws(d), workspace, workspace_bytes)) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_fwd(d, x, w, b, y, workspace, as_cuda(stream)));
}

int conv_fwd_relu(const conv_shape_t* s, const float* x, const float* w, const float* b, float* y, void* workspace,
                  size_t workspace_bytes, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, w, y})) != CONV_OK) return rc;
    if (b && !aligned16(b)) return CONV_ERR_ALIGN;
    if ((rc = check_workspace(conv_fwd_ws(d), workspace, workspace_bytes)) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_fwd(d, x, w, b, y, workspace, as_cuda(stream), true));
}

int conv_bwd_data(const conv_shape_t* s, const float* w, const float* dy, float* dx, void* workspace,
                  size_t workspace_bytes, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({w, dy, dx})) != CONV_OK) return rc;
    if ((rc = check_workspace(conv_dgrad_ws(d), workspace, workspace_bytes)) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_dgrad(d, w, dy, dx, workspace, as_cuda(stream)));
}

int conv_bwd_filter(const conv_shape_t* s, const float* x, const float* dy, float* dw, void* workspace,
                    size_t workspace_bytes, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, dy, dw})) != CONV_OK) return rc;
    if ((rc = check_workspace(conv_wgrad_ws(d), workspace, workspace_bytes)) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_wgrad(d, x, dy, dw, workspace, as_cuda(stream)));
}

int conv_bwd_filter_bias(const conv_shape_t* s, const float* x, const float* dy, float* dw, float* db,
                         void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, dy, dw, db})) != CONV_OK) return rc;
    if ((rc = check_workspace(conv_wgrad_ws(d), workspace, workspace_bytes)) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_wgrad(d, x, dy, dw, workspace, as_cuda(stream), db));
}

int conv_bwd_data_relu(const conv_shape_t* s, const float* w, const float* dy, const float* a, float* dx,
                       void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({w, dy, a, dx})) != CONV_OK) return rc;
    if ((rc = check_workspace(conv_dgrad_ws(d), workspace, workspace_bytes)) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_dgrad(d, w, dy, dx, workspace, as_cuda(stream), a));
}

int conv_bwd_filter_bias_relu(const conv_shape_t* s, const float* x, const float* dy, const float* a, float* dw,
                              float* db, void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, dy, a, dw})) != CONV_OK) return rc;
    if (db && !aligned16(db)) return CONV_ERR_ALIGN;
    if ((rc = check_workspace(conv_wgrad_ws(d), workspace, workspace_bytes)) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_wgrad(d, x, dy, dw, workspace, as_cuda(stream), db, a));
}

int conv_bwd_bias(const conv_shape_t* s, const float* dy, float* db, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({dy, db})) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_bias_grad(d, dy, db, as_cuda(stream)));
}

int im2col(const conv_shape_t* s, const float* x, float* col, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((long long)d.C * d.R * d.R * d.N * d.P * d.Q > kMaxElems) return CONV_ERR_OVERFLOW;
    if ((rc = check_ptrs({x, col})) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_im2col(d, x, col, as_cuda(stream)));
}

int col2im(const conv_shape_t* s, const float* col, float* dx, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_shape(s, &d);
    if (rc != CONV_OK) return rc;
    if ((long long)d.C * d.R * d.R * d.N * d.P * d.Q > kMaxElems) return CONV_ERR_OVERFLOW;
    if ((rc = check_ptrs({col, dx})) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_col2im(d, col, dx, as_cuda(stream)));
}

int matmul(int32_t M, int32_t K, int32_t N, uint32_t flags, const float* A, const float* B, float* C,
           conv_stream_t stream)
{
    if (M <= 0 || K <= 0 || N <= 0 || flags > 3u) return CONV_ERR_SHAPE;
    if ((long long)M * K > kMaxElems || (long long)K * N > kMaxElems || (long long)M * N > kMaxElems)
        return CONV_ERR_OVERFLOW;
    int rc = check_ptrs({A, B, C});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_matmul(M, K, N, flags, A, B, C, as_cuda(stream)));
}

int matmul_fused(int32_t M, int32_t K, int32_t N, uint32_t flags, const float* A, const float* B, const float* bias,
                 int32_t relu, const float* gate, float* C, conv_stream_t stream)
{
    if (M <= 0 || K <= 0 || N <= 0 || flags > 3u) return CONV_ERR_SHAPE;
    if ((long long)M * K > kMaxElems || (long long)K * N > kMaxElems || (long long)M * N > kMaxElems)
        return CONV_ERR_OVERFLOW;
    int rc = check_ptrs({A, B, C});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    MatmulEpi ep;
    ep.bias = bias;
    ep.gate = gate;
    ep.relu = relu ? 1 : 0;
    return status_of(launch_matmul(M, K, N, flags, A, B, C, as_cuda(stream), ep));
}

int matmul_tiling(int32_t M, int32_t K, int32_t N, uint32_t flags, const float* A, const float* B, int32_t* tile_cols,
                  int32_t* k_pieces, int32_t* tma_fed)
{
    if (!tile_cols || !k_pieces || !tma_fed) return CONV_ERR_NULL;
    if (M <= 0 || K <= 0 || N <= 0 || flags > 3u) return CONV_ERR_SHAPE;
    if (!device_ok()) return CONV_ERR_DEVICE;
    int bn = 0, cs = 0, tma = 0;
    cb200::matmul_tiling(M, K, N, flags, A, B, &bn, &cs, &tma);
    *tile_cols = bn;
    *k_pieces = cs;
    *tma_fed = tma;
    return CONV_OK;
}

static int check_pool(int32_t N, int32_t C, int32_t H, int32_t W, int32_t k, int32_t s, int32_t P, int32_t Q)
{
    if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || k <= 0 || s <= 0 || k > H || k > W) return CONV_ERR_SHAPE;
    if (P != (H - k) / s + 1 || Q != (W - k) / s + 1) return CONV_ERR_SHAPE;
    if ((long long)N * C * H * W > kMaxElems) return CONV_ERR_OVERFLOW;
    return CONV_OK;
}

int maxpool2d_fwd(int32_t batch, int32_t C, int32_t H, int32_t W, int32_t k, int32_t stride, int32_t outH,
                  int32_t outW, const float* x, float* y, int32_t* idx, conv_stream_t stream)
{
    int rc = check_pool(batch, C, H, W, k, stride, outH, outW);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, y, idx})) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_maxpool_fwd(batch, C, H, W, k, stride, outH, outW, x, y, idx, as_cuda(stream)));
}

int maxpool2d_bwd(int32_t batch, int32_t C, int32_t H, int32_t W, int32_t k, int32_t stride, int32_t outH,
                  int32_t outW, const float* dy, const int32_t* idx, float* dx, conv_stream_t stream)
{
    int rc = check_pool(batch, C, H, W, k, stride, outH, outW);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({dy, idx, dx})) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_maxpool_bwd(batch, C, H, W, k, stride, outH, outW, dy, idx, dx, as_cuda(stream)));
}

int sgd_step(int64_t count, float lr, float clip, float* param, const float* grad, conv_stream_t stream)
{
    if (count < 0) return CONV_ERR_SHAPE;
    if (count == 0) return CONV_OK;
    int rc = check_ptrs({param, grad});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_sgd(count, lr, clip, param, grad, as_cuda(stream)));
}

// ---------------------------------------------------------------------------
// direct convolution (legacy shaders; cross-check and small-channel ablation)

static int check_direct(const conv_shape_t* s, ConvDims* d)
{
    int rc = check_shape(s, d);
    if (rc != CONV_OK) return rc;
    // grid limits (batch and 8-wide filter/channel groups on y/z) and the forward patch
    const long long ph = 15LL * d->S + d->R;
    if (d->N > 65535 || (d->K + 7) / 8 > 65535 || (d->C + 7) / 8 > 65535) return CONV_ERR_SHAPE;
    if ((ph * ph + 8LL * d->R * d->R) * 4 > 200 * 1024) return CONV_ERR_SHAPE;
    return CONV_OK;
}

int conv_fwd_direct(const conv_shape_t* s, const float* x, const float* w, const float* b, float* y,
                    conv_stream_t stream)
{
    ConvDims d;
    int rc = check_direct(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, w, y})) != CONV_OK) return rc;
    if (b && !aligned16(b)) return CONV_ERR_ALIGN;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_fwd_direct(d, x, w, b, y, as_cuda(stream)));
}

int conv_bwd_data_direct(const conv_shape_t* s, const float* w, const float* dy, float* dx, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_direct(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({w, dy, dx})) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_dgrad_direct(d, w, dy, dx, as_cuda(stream)));
}

int conv_bwd_filter_direct(const conv_shape_t* s, const float* x, const float* dy, float* dw, conv_stream_t stream)
{
    ConvDims d;
    int rc = check_direct(s, &d);
    if (rc != CONV_OK) return rc;
    if ((rc = check_ptrs({x, dy, dw})) != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_conv_wgrad_direct(d, x, dy, dw, as_cuda(stream)));
}

// ---------------------------------------------------------------------------
// training-step pieces

int relu_fwd(int64_t count, const float* x, float* y, conv_stream_t stream)
{
    if (count < 0) return CONV_ERR_SHAPE;
    if (count == 0) return CONV_OK;
    int rc = check_ptrs({x, y});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_relu_fwd(count, x, y, as_cuda(stream)));
}

int relu_bwd(int64_t count, const float* dy, const float* x, float* dx, conv_stream_t stream)
{
    if (count < 0) return CONV_ERR_SHAPE;
    if (count == 0) return CONV_OK;
    int rc = check_ptrs({dy, x, dx});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_relu_bwd(count, dy, x, dx, as_cuda(stream)));
}

int grad_accum(int64_t count, const float* grad, float* accum, conv_stream_t stream)
{
    if (count < 0) return CONV_ERR_SHAPE;
    if (count == 0) return CONV_OK;
    int rc = check_ptrs({grad, accum});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_grad_accum(count, grad, accum, as_cuda(stream)));
}

int add_bias(int32_t rows, int32_t cols, const float* a, const float* b, float* out, int32_t relu,
             conv_stream_t stream)
{
    if (rows <= 0 || cols <= 0) return CONV_ERR_SHAPE;
    if ((long long)rows * cols > kMaxElems) return CONV_ERR_OVERFLOW;
    int rc = check_ptrs({a, b, out});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_add_bias(rows, cols, a, b, out, relu, as_cuda(stream)));
}

int bias_grad_rows(int32_t rows, int32_t cols, const float* grad, float* db, conv_stream_t stream)
{
    if (rows <= 0 || cols <= 0) return CONV_ERR_SHAPE;
    if ((long long)rows * cols > kMaxElems) return CONV_ERR_OVERFLOW;
    int rc = check_ptrs({grad, db});
    if (rc != CONV_OK) return rc;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_bias_grad_rows(rows, cols, grad, db, as_cuda(stream)));
}

int softmax_ce(int32_t rows, int32_t cols, const float* logits, const int32_t* labels, float* probs,
               float* dlogits, float* loss, conv_stream_t stream)
{
    if (rows <= 0 || cols <= 0) return CONV_ERR_SHAPE;
    if ((long long)rows * cols > kMaxElems) return CONV_ERR_OVERFLOW;
    int rc = check_ptrs({logits, labels, dlogits, loss});
    if (rc != CONV_OK) return rc;
    if (probs && !aligned16(probs)) return CONV_ERR_ALIGN;
    if (!device_ok()) return CONV_ERR_DEVICE;
    return status_of(launch_softmax_ce(rows, cols, logits, labels, probs, dlogits, loss, as_cuda(stream)));
}

uint64_t conv_b200_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int conv_b200_debug_matmul_engine(int32_t engine)
{
    if (engine < -1 || engine > 1) return CONV_ERR_SHAPE;
    return g_matmul_engine.exchange(engine, std::memory_order_relaxed);
}

int conv_b200_debug_withhold_stage(int64_t stage)
{
    if (stage < -1 || stage > (int64_t(1) << 30)) return CONV_ERR_SHAPE;
    g_withhold_stage.store(stage, std::memory_order_relaxed);
    return CONV_OK;
}

int conv_b200_set_math_mode(int mode)
{
    if (mode != CONV_MATH_FP32 && mode != CONV_MATH_TF32) return CONV_ERR_SHAPE;
    return g_math_mode.exchange(mode, std::memory_order_relaxed);
}

int conv_b200_math_mode(void) { return g_math_mode.load(std::memory_order_relaxed); }

const char* conv_b200_strerror(int code)
{
    switch (code) {
    case CONV_OK: return "ok";
    case CONV_ERR_NULL: return "a required pointer is NULL";
    case CONV_ERR_SHAPE: return "invalid or inconsistent sizes";
    case CONV_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case CONV_ERR_OVERFLOW: return "a tensor has 2^31 elements or more";
    case CONV_ERR_WORKSPACE: return "workspace missing or too small";
    case CONV_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case CONV_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
    case CONV_ERR_DEVICE: return "no usable sm_103 device";
    case CONV_ERR_SCRATCH_LIMIT: return "shape needs more scratch than the built-in array holds";
    case CONV_ERR_RANGE: return "a class label lies outside [0, cols)";
    default: return "unknown error";
    }
}

int conv_b200_check(conv_stream_t stream)
{
    if (cudaStreamSynchronize(as_cuda(stream)) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    if (word != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
        if (word & kDevErrTimeout) return CONV_ERR_DEVICE_TIMEOUT;
        return (word & kDevErrRange) ? CONV_ERR_RANGE : CONV_ERR_CUDA;
    }
    return CONV_OK;
}

}  // extern "C"
