/*
 * conv_b200.h -- C ABI of libconv_b200: the im2col convolution pipeline of the
 * page "DirectCompute Neural Network Engine" (directcompute-nn 0.1.0), forward
 * and backward, with its flagged matmul, max pooling and SGD, as hand-written
 * sm_103a CUDA kernels.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are fp32, row-major, NCHW (the page keeps every buffer as a float
 *    StructuredBuffer, section "Buffer Layout"); max-pool indices are int32.
 *  - Every pointer argument is a DEVICE pointer owned by the caller; the
 *    library never frees, keeps or reallocates it.  Outputs are fully
 *    OVERWRITTEN, never accumulated into (the page adds gradients with a
 *    separate grad_accum shader and clears scatter targets first).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  The library never synchronises the host.  Argument errors are
 *    reported before anything is launched.  A device-side failure (a bounded
 *    wait that gave up) is latched in a device error word and reported by the
 *    next conv_b200_check().
 *  - Kernels are launched with programmatic stream serialization: each one
 *    waits (griddepcontrol.wait) for the kernel before it in the stream before
 *    touching memory, and lets the next one be scheduled early.  Stream order
 *    is kept for everything else (events, copies, ordinary kernels); a
 *    caller's own kernel launched the same way right after a call must itself
 *    wait before reading the call's outputs, as that launch mode requires.
 *  - Operands must not alias outputs.  Pointers must be 16-byte aligned
 *    (CONV_ERR_ALIGN otherwise); element counts of every tensor must stay
 *    below 2^31 (CONV_ERR_OVERFLOW otherwise).
 *  - Convolution shape (section "Constant Buffer Convention", the im2col
 *    parameter set batch/inC/inH/inW/kH/stride/padding/outH/outW): square
 *    kH x kH filters, the same stride and zero padding on both axes,
 *    outH = (inH + 2*padding - kH) / stride + 1 (floor) and likewise outW;
 *    inconsistent outH/outW are rejected.
 *  - Contractions (conv_fwd, conv_bwd_data, conv_bwd_filter, matmul) run on
 *    the tcgen05 tensor cores in an fp32-faithful 3xTF32 mode with fp32
 *    accumulation: each result is within 1e-4 * sum_k |a_k b_k| + 1e-6 of the
 *    exact sum (a one-product TF32 mode is selectable: conv_b200_set_math_mode).
 */
#ifndef CONV_B200_H
#define CONV_B200_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (cudaStream_t). */
typedef struct CUstream_st *conv_stream_t;

typedef struct {
    int32_t batch, inC, inH, inW; /* input x: batch x inC x inH x inW            */
    int32_t outC;                 /* number of filters                           */
    int32_t kH;                   /* filter extent (kW == kH)                    */
    int32_t stride, padding;      /* same on both axes; padding reads zero       */
    int32_t outH, outW;           /* output extent, must match the floor formula */
} conv_shape_t;

/* Return codes. */
#define CONV_OK 0
#define CONV_ERR_NULL (-1)           /* a required pointer is NULL                  */
#define CONV_ERR_SHAPE (-2)          /* non-positive or inconsistent sizes, flags>3 */
#define CONV_ERR_ALIGN (-3)          /* a pointer is not 16-byte aligned            */
#define CONV_ERR_OVERFLOW (-4)       /* a tensor has 2^31 elements or more          */
#define CONV_ERR_WORKSPACE (-5)      /* workspace missing or smaller than required  */
#define CONV_ERR_CUDA (-6)           /* a CUDA runtime call or launch failed        */
#define CONV_ERR_DEVICE_TIMEOUT (-7) /* a kernel's bounded wait gave up             */
#define CONV_ERR_DEVICE (-8)         /* no usable sm_103 device                     */
#define CONV_ERR_SCRATCH_LIMIT (-9)  /* shape needs more than the built-in scratch  */
#define CONV_ERR_RANGE (-10)         /* a class label outside [0, cols) (device)    */

/* Operation ids for conv_b200_workspace_bytes. */
#define CONV_OP_FWD 0
#define CONV_OP_BWD_DATA 1
#define CONV_OP_BWD_FILTER 2

/* Forward convolution.  Page section "Convolution: The im2col Approach",
 * forward: im2col -> filters (outC x inC*kH*kW) times the column matrix ->
 * conv_reshape (+ bias) to (batch, outC, outH, outW).  Computed as one
 * implicit GEMM: the column matrix is gathered tile by tile and never stored.
 *   x  [batch][inC][inH][inW]   w [outC][inC][kH][kH]   b [outC] or NULL (no bias)
 *   y  [batch][outC][outH][outW]                              (overwritten)
 *   workspace: device scratch of conv_b200_workspace_bytes(CONV_OP_FWD, s)
 *   bytes (the filters split into tensor-core tiles), owned by the caller,
 *   reused freely after the stream passes the call. */
int conv_fwd(const conv_shape_t *s, const float *x, const float *w, const float *b, float *y, void *workspace,
             size_t workspace_bytes, conv_stream_t stream);

/* Forward convolution with ReLU (nn_relu) fused into the epilogue: exactly
 * max(0, conv_fwd(...)) -- the same sums and the same fp32 bias add, then +0
 * wherever the result is not > 0 -- in one pass over y instead of two.
 * Arguments, workspace (CONV_OP_FWD) and errors as conv_fwd. */
int conv_fwd_relu(const conv_shape_t *s, const float *x, const float *w, const float *b, float *y, void *workspace,
                  size_t workspace_bytes, conv_stream_t stream);

/* Input gradient.  Page section "Convolution: The im2col Approach", backward:
 * filters^T x grad_reshaped -> col2im -> grad_input.  Computed as one implicit
 * GEMM per stride phase that gathers grad_output directly, so the col2im sum
 * happens inside the accumulator and the column-matrix gradient is never
 * stored.
 *   w  [outC][inC][kH][kH]   dy [batch][outC][outH][outW]
 *   dx [batch][inC][inH][inW] (overwritten; pixels no window reads get 0)
 *   workspace: conv_b200_workspace_bytes(CONV_OP_BWD_DATA, s) bytes. */
int conv_bwd_data(const conv_shape_t *s, const float *w, const float *dy, float *dx, void *workspace,
                  size_t workspace_bytes, conv_stream_t stream);

/* Filter gradient.  Page section "Convolution: The im2col Approach", backward:
 * grad_reshaped x im2col_matrix^T.  The column matrix is regathered from x
 * (not read from a saved copy); the batch*outH*outW reduction is split across
 * the GPU and summed in a fixed order (deterministic).
 *   x  [batch][inC][inH][inW]   dy [batch][outC][outH][outW]
 *   dw [outC][inC][kH][kH] (overwritten)
 *   workspace: conv_b200_workspace_bytes(CONV_OP_BWD_FILTER, s) bytes. */
int conv_bwd_filter(const conv_shape_t *s, const float *x, const float *dy, float *dw, void *workspace,
                    size_t workspace_bytes, conv_stream_t stream);

/* Filter and bias gradients from one pass over dy: conv_bwd_filter plus the
 * bias gradient of conv_bwd_bias, the latter summed while dy is re-laid for
 * the filter-gradient GEMM (so dy is read once for both).  Same layouts as
 * conv_bwd_filter and conv_bwd_bias; db [outC] (overwritten).  The bias sums
 * run in a fixed order (deterministic) that differs from conv_bwd_bias's, so
 * the two may differ in the last bits.
 *   workspace: conv_b200_workspace_bytes(CONV_OP_BWD_FILTER, s) bytes. */
int conv_bwd_filter_bias(const conv_shape_t *s, const float *x, const float *dy, float *dw, float *db,
                         void *workspace, size_t workspace_bytes, conv_stream_t stream);

/* The two gradient calls above with the ReLU gradient that precedes them fused
 * in (shader table "Activation / Loss Shaders": nn_relu_grad, grad * (x > 0)).
 * For a layer followed by a ReLU, a = the ReLU's output (or its input: both
 * are > 0 at the same positions) and dy = the gradient at the ReLU's output;
 * the convolution's own output gradient is G = dy * (a > 0), an fp32 product
 * with 1 or 0 -- exactly relu_bwd(dy, a) -- and it is formed where dy is
 * first read (the gather of the input gradient, or the re-layout of dy that
 * the filter gradient and the bias sums read), so no separate pass over dy
 * runs.  Results equal conv_bwd_data / conv_bwd_filter_bias on relu_bwd's
 * output.
 *   a [batch][outC][outH][outW] (same shape as dy; read only)
 *   conv_bwd_filter_bias_relu: db may be NULL (filter gradient only).
 *   workspace: conv_b200_workspace_bytes(CONV_OP_BWD_DATA or CONV_OP_BWD_FILTER, s),
 *   the same sizes as the unfused calls.  Errors as the unfused calls. */
int conv_bwd_data_relu(const conv_shape_t *s, const float *w, const float *dy, const float *a, float *dx,
                       void *workspace, size_t workspace_bytes, conv_stream_t stream);
int conv_bwd_filter_bias_relu(const conv_shape_t *s, const float *x, const float *dy, const float *a, float *dw,
                              float *db, void *workspace, size_t workspace_bytes, conv_stream_t stream);

/* Bias gradient.  Page section "Convolution: The im2col Approach", backward:
 * the sum of grad_reshaped over its columns, i.e. over batch, outH and outW.
 * Fixed-order reduction (deterministic).
 *   dy [batch][outC][outH][outW]   db [outC] (overwritten) */
int conv_bwd_bias(const conv_shape_t *s, const float *dy, float *db, conv_stream_t stream);

/* Scratch bytes the given operation needs for shape s (0 if none).  op is one
 * of CONV_OP_*; returns 0 for an invalid shape or op. */
size_t conv_b200_workspace_bytes(int op, const conv_shape_t *s);

/* Standalone im2col (the nn_im2col shader of section "Convolution Shaders"):
 *   col[(c*kH + r)*kH + q][(n*outH + oh)*outW + ow] = x[n][c][oh*stride + r - padding][ow*stride + q - padding]
 * or 0 where that position lies in the padding.
 *   x [batch][inC][inH][inW]   col [inC*kH*kH][batch*outH*outW] (overwritten) */
int im2col(const conv_shape_t *s, const float *x, float *col, conv_stream_t stream);

/* Standalone col2im (the nn_col2im shader): the adjoint of im2col.  Every
 * column-matrix entry is added to the input position im2col read it from;
 * entries that came from padding are dropped.  Each dx element is summed in a
 * fixed order (ascending r, then q), so the result is deterministic.
 *   col [inC*kH*kH][batch*outH*outW]   dx [batch][inC][inH][inW] (overwritten) */
int col2im(const conv_shape_t *s, const float *col, float *dx, conv_stream_t stream);

/* Flagged matmul.  Page section "Optimizations" -> "Transpose via Flags" and
 * the matmul shader table: C (M x N) = op(A) * op(B), row-major, where
 * flags bit 0 reads A as column-major (A stored K x M) and flags bit 1 reads B
 * as column-major (B stored N x K).  C is overwritten (no alpha/beta).
 * Any M, K, N >= 1 (ragged edges are handled); flags in 0..3. */
int matmul(int32_t M, int32_t K, int32_t N, uint32_t flags, const float *A, const float *B, float *C,
           conv_stream_t stream);

/* Flagged matmul with a fused epilogue: the linear layer of the page's LeNet
 * trainer (section "LeNet on MNIST") without separate element-wise passes.
 * C = op(A) * op(B) exactly as matmul computes it, then per element (i, j),
 * in this order:
 *   bias != NULL:  c = c + bias[j]          one fp32 addition (nn_add_bias, as add_bias)
 *   relu != 0:     c = max(0, c)            +0 for c <= 0 (nn_relu, as relu_fwd)
 *   gate != NULL:  c = c * (gate[i][j] > 0) an fp32 product with 1 or 0 (nn_relu_grad, as relu_bwd)
 * so the result is bit-identical to matmul followed by add_bias and relu_bwd
 * (the forward Y = relu(X W + b); the input gradient of a ReLU-fed layer,
 * dX = (dY W^T) * (X > 0)).  bias [N] and gate [M][N] are optional, read only,
 * and must not overlap C; arguments otherwise as matmul. */
int matmul_fused(int32_t M, int32_t K, int32_t N, uint32_t flags, const float *A, const float *B, const float *bias,
                 int32_t relu, const float *gate, float *C, conv_stream_t stream);

/* How matmul runs an M x K x N product with operands at A and B (a
 * host-side query, no GPU work; only the operands' alignment is looked at,
 * they may be NULL) on the current device and in the current math mode:
 * *tile_cols = width of an output tile (32, 64, 128 or 256 columns; tiles are
 * 128 rows); *k_pieces = number of pieces each tile's K range is cut into when
 * there are too few tiles for the SMs (1: whole tiles) -- the pieces of a tile
 * run on the CTAs of one thread-block cluster and are added in a fixed order
 * through distributed shared memory, so results stay deterministic;
 * *tma_fed = 1 when the operands arrive by TMA tensor copies, 0 when the
 * producer warps gather them.  TMA qualifies when every operand's row pitch
 * is a multiple of 16 bytes (K % 4 == 0 for an operand stored with K
 * contiguous, M or N % 4 == 0 for one stored K-major), the operands are
 * 16-byte aligned, M >= 128 and N >= 128; the plan then picks whichever
 * engine, tile width and split its measured stage costs make fastest.
 * Returns CONV_OK, CONV_ERR_NULL (an output pointer is NULL), CONV_ERR_SHAPE
 * (as matmul) or CONV_ERR_DEVICE. */
int matmul_tiling(int32_t M, int32_t K, int32_t N, uint32_t flags, const float *A, const float *B,
                  int32_t *tile_cols, int32_t *k_pieces, int32_t *tma_fed);

/* Max pooling forward (nn_maxpool_forward, section "Pooling Shaders"):
 * k x k windows, stride `stride`, no padding, outH = (H - k) / stride + 1.
 * y = window maximum; idx = flat offset into the whole NCHW x of the FIRST
 * maximum in row-major window order.
 *   x [batch][C][H][W]   y, idx [batch][C][outH][outW] (overwritten) */
int maxpool2d_fwd(int32_t batch, int32_t C, int32_t H, int32_t W, int32_t k, int32_t stride, int32_t outH,
                  int32_t outW, const float *x, float *y, int32_t *idx, conv_stream_t stream);

/* Max pooling backward (nn_maxpool_backward): dx[i] = sum of dy[o] over the
 * windows o whose saved index is i, in ascending window order (bit-exact and
 * deterministic); 0 where no window routed a gradient.  idx must come from
 * maxpool2d_fwd with the same sizes (every entry must lie inside the window of
 * its own output; others are ignored).
 *   dy, idx [batch][C][outH][outW]   dx [batch][C][H][W] (overwritten) */
int maxpool2d_bwd(int32_t batch, int32_t C, int32_t H, int32_t W, int32_t k, int32_t stride, int32_t outH,
                  int32_t outW, const float *dy, const int32_t *idx, float *dx, conv_stream_t stream);

/* SGD step (nn_sgd, section "Utility Shaders"), in place:
 *   param[i] = param[i] - lr * min(max(grad[i], -clip), clip)
 * each operation rounded to fp32, no fused multiply-add.  count >= 0. */
int sgd_step(int64_t count, float lr, float clip, float *param, const float *grad, conv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Direct convolution: the page's legacy shaders (table "Legacy / Unused
 * Shaders": nn_conv_forward[_tiled], nn_conv_backprop_input[_fused],
 * nn_conv_backprop_filters[_tiled] with nn_conv_reduce_filters), which the
 * im2col pipeline replaced.  Same definitions, layouts and overwrite rule as
 * conv_fwd / conv_bwd_data / conv_bwd_filter, computed with fp32 fused
 * multiply-adds on the CUDA cores (no workspace, no tensor cores), each
 * output summed in a fixed order: a cross-check of the implicit-GEMM path and
 * an ablation for layers with few input channels.  Each result is within
 * n * 2^-24 * sum |a_k b_k| of the exact sum for its n terms.  Extra limits
 * (CONV_ERR_SHAPE): batch <= 65535, and the forward's input patch for a 16x16
 * output tile with 8 filter slices, ((15 * stride + kH)^2 + 8 * kH^2) floats,
 * within 200 KB.
 * ------------------------------------------------------------------------- */
int conv_fwd_direct(const conv_shape_t *s, const float *x, const float *w, const float *b, float *y,
                    conv_stream_t stream);
int conv_bwd_data_direct(const conv_shape_t *s, const float *w, const float *dy, float *dx, conv_stream_t stream);
int conv_bwd_filter_direct(const conv_shape_t *s, const float *x, const float *dy, float *dw, conv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Training-step pieces around the convolutions (shader tables "Activation /
 * Loss Shaders" and "Utility Shaders"; the page's LeNet trainer, section
 * "LeNet on MNIST", chains them with conv, pooling, flagged matmul and SGD).
 * Element counts: count >= 0 (0 is a no-op); rows, cols >= 1.  Unlike the
 * rest of the library these allow the in-place forms named below.
 * ------------------------------------------------------------------------- */

/* ReLU forward (nn_relu): y[i] = max(0, x[i]) (+0 for x <= 0).  y may be x. */
int relu_fwd(int64_t count, const float *x, float *y, conv_stream_t stream);

/* ReLU backward (nn_relu_grad): dx[i] = dy[i] * (x[i] > 0), an fp32 product
 * with 1 or 0.  x may be the ReLU's input or its output (both are > 0 at the
 * same positions).  dx may be dy. */
int relu_bwd(int64_t count, const float *dy, const float *x, float *dx, conv_stream_t stream);

/* Gradient accumulation (nn_grad_accum): accum[i] = accum[i] + grad[i], one
 * fp32 addition each, in place. */
int grad_accum(int64_t count, const float *grad, float *accum, conv_stream_t stream);

/* Bias add (nn_add_bias): out[i][j] = a[i][j] + b[j] over a row-major
 * rows x cols matrix (a linear layer's bias broadcast over the batch rows),
 * one fp32 addition each; relu != 0 then applies max(0, .) (nn_relu fused).
 * out may be a.   a, out [rows][cols]   b [cols] */
int add_bias(int32_t rows, int32_t cols, const float *a, const float *b, float *out, int32_t relu,
             conv_stream_t stream);

/* Bias gradient of a linear layer (nn_bias_grad, "sum-reduces rows"):
 * db[j] = sum_i grad[i][j] over the rows of a rows x cols gradient.  fp32
 * sums in a fixed order set by the shape (deterministic).
 *   grad [rows][cols]   db [cols] (overwritten) */
int bias_grad_rows(int32_t rows, int32_t cols, const float *grad, float *db, conv_stream_t stream);

/* Softmax + cross-entropy (nn_softmax, nn_softmax_ce_grad, nn_loss), per row
 * of rows x cols logits with integer labels: p = exp(z - max z) / sum exp(z -
 * max z) (the numerically stable form), dlogits = p - one_hot(label), and
 * *loss = sum over rows of -log p[label] -- the batch SUM, whose gradient is
 * exactly dlogits (the page's softmax_ce_grad has no 1/rows factor).  probs
 * (nullable) receives p.  A label outside [0, cols) cannot be seen before the
 * kernel runs: its row gets dlogits = p and no loss, and the next
 * conv_b200_check() returns CONV_ERR_RANGE.
 *   logits, probs, dlogits [rows][cols]   labels [rows] (int32)   loss [1] */
int softmax_ce(int32_t rows, int32_t cols, const float *logits, const int32_t *labels, float *probs,
               float *dlogits, float *loss, conv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Arithmetic of the contractions (conv_fwd, conv_bwd_data, conv_bwd_filter,
 * conv_bwd_filter_bias, conv_fwd_noalloc, matmul).
 *   CONV_MATH_FP32 (default): fp32-faithful 3xTF32 -- each operand split into a
 *     TF32 high part and a TF32 remainder, three tensor-core products per
 *     product (hi*hi + hi*lo + lo*hi), fp32 accumulation; within
 *     1e-4 * sum_k |a_k b_k| + 1e-6 of the exact sum.
 *   CONV_MATH_TF32: one tensor-core product of the operands truncated to TF32
 *     (10 explicit mantissa bits), fp32 accumulation: within
 *     2.5e-3 * sum_k |a_k b_k| + 1e-6; the "fast precision" mode, about three
 *     times fewer tensor-core instructions and half the operand traffic.
 * The mode is process-wide and read when a call launches its kernels (a CUDA
 * graph keeps the mode it was captured with).  conv_b200_set_math_mode returns
 * the previous mode, or CONV_ERR_SHAPE for an unknown mode (nothing changes).
 * ------------------------------------------------------------------------- */
#define CONV_MATH_FP32 0
#define CONV_MATH_TF32 1
int conv_b200_set_math_mode(int mode);
int conv_b200_math_mode(void);

/* Number of kernels the library has launched since it was loaded (all
 * devices, all streams).  A diagnostic: callers difference two readings to
 * count the launches of a region of their own code. */
uint64_t conv_b200_launch_count(void);

/* conv_fwd without a workspace argument.  The page has no counterpart: this
 * entry point exists for callers that cannot allocate device memory -- code
 * running under a memory manager that owns the whole device heap, or a
 * latency-critical loop that cannot afford an allocation's implicit device
 * synchronisation.  Such callers pass x, w, b and y exactly as for conv_fwd;
 * the scratch conv_fwd would take from `workspace` comes from a fixed array
 * of CONV_FWD_NOALLOC_SCRATCH_BYTES inside the library instead.  The library
 * allocates nothing for it: the array is part of the loaded module, and every
 * device that loads the library keeps one until the process exits.
 *  - The array must hold the whole scratch conv_fwd would take for the shape,
 *    conv_b200_workspace_bytes(CONV_OP_FWD, s): the filters as pre-split
 *    tensor-core tiles, plus -- for the forms that stage the input through a
 *    copy -- the channel-blocked or space-to-depth copy of x (its size grows
 *    with the batch) and the partial tiles of a split last round of tiles.
 *    Shapes that need more are rejected with CONV_ERR_SCRATCH_LIMIT before
 *    anything is launched; check in advance with conv_b200_workspace_bytes.
 *    Of the AlexNet layers at batch 128 only conv2 fits (2.3 MiB); conv1
 *    (101.8 MiB), conv3 (16.9), conv4 (25.1) and conv5 (22.9) are refused,
 *    while all five fit at batch 2.  Every other argument is validated
 *    exactly as by conv_fwd, with the same codes.
 *  - The first call on each device resolves the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before capturing a stream.
 *  - All calls share the one array.  Each call writes every byte of it that
 *    it later reads, so nothing needs clearing between calls.  Two calls
 *    whose kernels may overlap on the GPU (different streams with no ordering
 *    between them) race on it and can both return garbage: order them.
 *  - The result is identical to conv_fwd's for the same inputs. */
#define CONV_FWD_NOALLOC_SCRATCH_BYTES (8u << 20)
int conv_fwd_noalloc(const conv_shape_t *s, const float *x, const float *w, const float *b, float *y,
                     conv_stream_t stream);

/* Test hook of the bounded-wait error path; the page has no counterpart (its
 * D3D11 runtime has no device-side waits).  Off by default.  After
 * conv_b200_debug_withhold_stage(k) the NEXT launch of the register-gather
 * tensor-core kernel (flagged matmul, and the convolution GEMMs that run on
 * it) withholds, in its first CTA, the producers' arrival for CTA-wide
 * pipeline stage k: that CTA's MMA issuer waits for a stage that never
 * fills, gives up after its bounded wait (about 2 s), and the kernel unwinds
 * -- it drains its own MMAs, frees its tensor memory and returns -- so the
 * next conv_b200_check() returns CONV_ERR_DEVICE_TIMEOUT and the stream stays
 * usable.  The results of that one launch are undefined.  One-shot: the
 * launch that takes the setting resets it; k = -1 cancels it.  Returns
 * CONV_OK, or CONV_ERR_SHAPE for k < -1. */
int conv_b200_debug_withhold_stage(int64_t stage);

/* Test hook choosing the flagged matmul's engine (process-wide, read at each
 * matmul call and by matmul_tiling): -1 (default) lets the plan choose from
 * measured stage costs, 0 always gathers the operands in the producer warps,
 * 1 feeds them by TMA wherever the operands qualify (see matmul_tiling), so
 * that tests reach both engines in both math modes.  Results agree within the
 * matmul's tolerance whichever engine runs.  Returns the previous setting, or
 * CONV_ERR_SHAPE for a value outside -1..1 (nothing changes). */
int conv_b200_debug_matmul_engine(int32_t engine);

/* Text for a return code. */
const char *conv_b200_strerror(int code);

/* Synchronise `stream`, then read and clear the device error word: returns
 * CONV_OK, CONV_ERR_DEVICE_TIMEOUT, CONV_ERR_RANGE, or CONV_ERR_CUDA. */
int conv_b200_check(conv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CONV_B200_H */
