/*
 * oracle.c -- plain CPU oracle for the im2col convolution pipeline described on
 * the page "DirectCompute Neural Network Engine" (directcompute-nn 0.1.0).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct yardstick
 * the CUDA library is checked against.  Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark load it; the CUDA library never does,
 * and the two share no code, headers or tables.
 *
 * Arithmetic: every floating-point value is handled as an IEEE double.  Products
 * of fp32 inputs are exact in double, sums are carried in double, and the caller
 * rounds each output once to fp32.  Next to every contraction output the oracle
 * also returns sum_k |a_k * b_k|, the scale of the per-element tolerance.
 *
 * Index conventions (the page gives the column-matrix shape only; this is the
 * single ordering under which its conv_reshape step is a plain reshape):
 *   column-matrix row    = (c * kH + r) * kW + s          (kW == kH)
 *   column-matrix column = (n * outH + oh) * outW + ow
 *   tensors are NCHW, row-major, fp32 on the page.
 *
 * Max pooling and SGD are fp32 operations on the page and stay fp32 here, with
 * a fixed operation order (build with -ffp-contract=off so no FMA is formed).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

/* ------------------------------------------------------------------------- */
/* Step A1: im2col.  Page section "Convolution: The im2col Approach", forward
 * step 1: patches of the input become the columns of an
 * (inC*kH*kW) x (batch*outH*outW) matrix.  Positions outside the image
 * (padding) read as zero.                                                    */
static double col_entry(const double *x, i64 C, i64 H, i64 W, i64 R, i64 st,
                        i64 pad, i64 P, i64 Q, i64 row, i64 j)
{
    i64 c = row / (R * R);
    i64 r = (row / R) % R;
    i64 s = row % R;
    i64 n = j / (P * Q);
    i64 oh = (j / Q) % P;
    i64 ow = j % Q;
    i64 h = oh * st + r - pad;
    i64 w = ow * st + s - pad;
    (void)C;
    if (h < 0 || h >= H || w < 0 || w >= W)
        return 0.0;
    return x[((n * C + c) * H + h) * W + w];
}

void oracle_im2col(i64 N, i64 C, i64 H, i64 W, i64 R, i64 st, i64 pad, i64 P,
                   i64 Q, const double *x, double *col)
{
    i64 rows = C * R * R, cols = N * P * Q;
#pragma omp parallel for schedule(static)
    for (i64 row = 0; row < rows; ++row)
        for (i64 j = 0; j < cols; ++j)
            col[row * cols + j] = col_entry(x, C, H, W, R, st, pad, P, Q, row, j);
}

/* ------------------------------------------------------------------------- */
/* Step A7: col2im.  Page section "Convolution: The im2col Approach", backward
 * (input gradients) and the shader table entry for nn_col2im ("scatters the
 * column matrix back to image format").  Written as that scatter: every
 * column-matrix entry is added to the image position it was read from by
 * im2col; entries that came from padding are dropped.  The output is fully
 * overwritten (the page clears scatter targets first).  Each (n, c) plane only
 * receives entries from its own rows/columns, so planes are independent.     */
void oracle_col2im(i64 N, i64 C, i64 H, i64 W, i64 R, i64 st, i64 pad, i64 P,
                   i64 Q, const double *col, const double *col_abs,
                   double *dx, double *dx_abs)
{
    i64 cols = N * P * Q;
#pragma omp parallel for schedule(static)
    for (i64 nc = 0; nc < N * C; ++nc) {
        i64 n = nc / C, c = nc % C;
        double *plane = dx + nc * H * W;
        double *plane_abs = dx_abs ? dx_abs + nc * H * W : NULL;
        for (i64 i = 0; i < H * W; ++i) {
            plane[i] = 0.0;
            if (plane_abs)
                plane_abs[i] = 0.0;
        }
        for (i64 r = 0; r < R; ++r)
            for (i64 s = 0; s < R; ++s) {
                i64 row = (c * R + r) * R + s;
                for (i64 oh = 0; oh < P; ++oh)
                    for (i64 ow = 0; ow < Q; ++ow) {
                        i64 h = oh * st + r - pad;
                        i64 w = ow * st + s - pad;
                        if (h < 0 || h >= H || w < 0 || w >= W)
                            continue;
                        i64 j = (n * P + oh) * Q + ow;
                        plane[h * W + w] += col[row * cols + j];
                        if (plane_abs)
                            plane_abs[h * W + w] +=
                                col_abs ? col_abs[row * cols + j] : fabs(col[row * cols + j]);
                    }
            }
    }
}

/* ------------------------------------------------------------------------- */
/* Step A9: matmul with transpose flags.  Page section "Optimizations" ->
 * "Transpose via Flags": C (M x N) = op(A) * op(B), row-major storage; bit 0 of
 * flags reads A as column-major (stored K x M), bit 1 reads B as column-major
 * (stored N x K).  These two accessors are the page's two index formulas.   */
static double a_at(const double *A, i64 M, i64 K, unsigned flags, i64 row, i64 col)
{
    return (flags & 1u) ? A[col * M + row] : A[row * K + col];
}

static double b_at(const double *B, i64 K, i64 N, unsigned flags, i64 row, i64 col)
{
    return (flags & 2u) ? B[col * K + row] : B[row * N + col];
}

static void dot_at(i64 M, i64 K, i64 N, unsigned flags, const double *A,
                   const double *B, i64 i, i64 j, double *out, double *out_abs)
{
    double acc = 0.0, acc_abs = 0.0;
    for (i64 k = 0; k < K; ++k) {
        double p = a_at(A, M, K, flags, i, k) * b_at(B, K, N, flags, k, j);
        acc += p;
        acc_abs += fabs(p);
    }
    *out = acc;
    *out_abs = acc_abs;
}

void oracle_matmul(i64 M, i64 K, i64 N, unsigned flags, const double *A,
                   const double *B, double *C, double *C_abs)
{
#pragma omp parallel for schedule(static)
    for (i64 i = 0; i < M; ++i)
        for (i64 j = 0; j < N; ++j)
            dot_at(M, K, N, flags, A, B, i, j, &C[i * N + j], &C_abs[i * N + j]);
}

/* The same definition evaluated only at the listed flat indices i*N + j. */
void oracle_matmul_at(i64 M, i64 K, i64 N, unsigned flags, const double *A,
                      const double *B, i64 count, const i64 *flat, double *out,
                      double *out_abs)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (i64 t = 0; t < count; ++t)
        dot_at(M, K, N, flags, A, B, flat[t] / N, flat[t] % N, &out[t], &out_abs[t]);
}

/* ------------------------------------------------------------------------- */
/* Forward convolution, page section "Convolution: The im2col Approach",
 * forward steps 1-3: im2col (A1), filters (outC x inC*kH*kW) times the column
 * matrix (A2, matmul flags 0), then conv_reshape: add the bias and reshape
 * (outC x batch*outH*outW) to (batch, outC, outH, outW) (A3).  The bias enters
 * the tolerance scale as one more term |b * 1|.                              */
void oracle_conv_fwd(i64 N, i64 C, i64 H, i64 W, i64 Ko, i64 R, i64 st, i64 pad,
                     i64 P, i64 Q, const double *x, const double *w,
                     const double *b, double *y, double *y_abs)
{
    i64 CRS = C * R * R, NPQ = N * P * Q, PQ = P * Q;
    double *col = (double *)malloc(sizeof(double) * CRS * NPQ);
    double *Y = (double *)malloc(sizeof(double) * Ko * NPQ);
    double *Y_abs = (double *)malloc(sizeof(double) * Ko * NPQ);
    oracle_im2col(N, C, H, W, R, st, pad, P, Q, x, col);   /* A1 */
    oracle_matmul(Ko, CRS, NPQ, 0u, w, col, Y, Y_abs);       /* A2 */
#pragma omp parallel for schedule(static)
    for (i64 nk = 0; nk < N * Ko; ++nk) {                    /* A3 */
        i64 n = nk / Ko, k = nk % Ko;
        double bias = b ? b[k] : 0.0;
        for (i64 pq = 0; pq < PQ; ++pq) {
            y[nk * PQ + pq] = Y[k * NPQ + n * PQ + pq] + bias;
            y_abs[nk * PQ + pq] = Y_abs[k * NPQ + n * PQ + pq] + fabs(bias);
        }
    }
    free(col);
    free(Y);
    free(Y_abs);
}

/* The same forward definition at listed flat NCHW output indices: one column
 * of the im2col matrix, dotted with one filter row, plus the bias.          */
void oracle_conv_fwd_at(i64 N, i64 C, i64 H, i64 W, i64 Ko, i64 R, i64 st,
                        i64 pad, i64 P, i64 Q, const double *x, const double *w,
                        const double *b, i64 count, const i64 *flat, double *out,
                        double *out_abs)
{
    i64 CRS = C * R * R, PQ = P * Q;
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (i64 t = 0; t < count; ++t) {
        i64 n = flat[t] / (Ko * PQ), k = (flat[t] / PQ) % Ko, pq = flat[t] % PQ;
        i64 j = n * PQ + pq;
        double acc = 0.0, acc_abs = 0.0;
        for (i64 row = 0; row < CRS; ++row) {
            double p = w[k * CRS + row] * col_entry(x, C, H, W, R, st, pad, P, Q, row, j);
            acc += p;
            acc_abs += fabs(p);
        }
        double bias = b ? b[k] : 0.0;
        out[t] = acc + bias;
        out_abs[t] = acc_abs + fabs(bias);
    }
}

/* ------------------------------------------------------------------------- */
/* Step A4: conv_grad_reshape, page section "Convolution: The im2col Approach",
 * backward: grad_output (batch, outC, outH, outW) becomes the
 * (outC x batch*outH*outW) matrix G.                                         */
static void grad_reshape(i64 N, i64 Ko, i64 PQ, const double *dy, double *G)
{
    i64 NPQ = N * PQ;
#pragma omp parallel for schedule(static)
    for (i64 k = 0; k < Ko; ++k)
        for (i64 n = 0; n < N; ++n)
            for (i64 pq = 0; pq < PQ; ++pq)
                G[k * NPQ + n * PQ + pq] = dy[(n * Ko + k) * PQ + pq];
}

/* Input gradient, page section "Convolution: The im2col Approach", backward:
 * filters^T x G (A6, matmul flags 1 on the stored outC x inC*kH*kW filters),
 * then col2im (A7).  The column-matrix gradient is kept in double.          */
void oracle_conv_bwd_data(i64 N, i64 C, i64 H, i64 W, i64 Ko, i64 R, i64 st,
                          i64 pad, i64 P, i64 Q, const double *w,
                          const double *dy, double *dx, double *dx_abs)
{
    i64 CRS = C * R * R, NPQ = N * P * Q;
    double *G = (double *)malloc(sizeof(double) * Ko * NPQ);
    double *dcol = (double *)malloc(sizeof(double) * CRS * NPQ);
    double *dcol_abs = (double *)malloc(sizeof(double) * CRS * NPQ);
    grad_reshape(N, Ko, P * Q, dy, G);                                   /* A4 */
    oracle_matmul(CRS, Ko, NPQ, 1u, w, G, dcol, dcol_abs);               /* A6 */
    oracle_col2im(N, C, H, W, R, st, pad, P, Q, dcol, dcol_abs, dx, dx_abs); /* A7 */
    free(G);
    free(dcol);
    free(dcol_abs);
}

/* The same input gradient at listed flat NCHW indices of dx.  A single image
 * position is reached by col2im from every (r, s, oh, ow) with
 * oh*stride + r - pad == h and ow*stride + s - pad == w; each such entry of
 * filters^T x G is a dot over outC.                                         */
void oracle_conv_bwd_data_at(i64 N, i64 C, i64 H, i64 W, i64 Ko, i64 R, i64 st,
                             i64 pad, i64 P, i64 Q, const double *w,
                             const double *dy, i64 count, const i64 *flat,
                             double *out, double *out_abs)
{
    i64 CRS = C * R * R, PQ = P * Q;
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (i64 t = 0; t < count; ++t) {
        i64 n = flat[t] / (C * H * W), c = (flat[t] / (H * W)) % C;
        i64 h = (flat[t] / W) % H, x_w = flat[t] % W;
        double acc = 0.0, acc_abs = 0.0;
        for (i64 r = 0; r < R; ++r)
            for (i64 s = 0; s < R; ++s)
                for (i64 oh = 0; oh < P; ++oh)
                    for (i64 ow = 0; ow < Q; ++ow) {
                        if (oh * st + r - pad != h || ow * st + s - pad != x_w)
                            continue;
                        i64 row = (c * R + r) * R + s;
                        for (i64 k = 0; k < Ko; ++k) {
                            double p = w[k * CRS + row] * dy[(n * Ko + k) * PQ + oh * Q + ow];
                            acc += p;
                            acc_abs += fabs(p);
                        }
                    }
        out[t] = acc;
        out_abs[t] = acc_abs;
    }
}

/* Filter gradient, page section "Convolution: The im2col Approach", backward:
 * G x im2col_matrix^T (A5, matmul flags 2 on the stored column matrix).     */
void oracle_conv_bwd_filter(i64 N, i64 C, i64 H, i64 W, i64 Ko, i64 R, i64 st,
                            i64 pad, i64 P, i64 Q, const double *x,
                            const double *dy, double *dw, double *dw_abs)
{
    i64 CRS = C * R * R, NPQ = N * P * Q;
    double *col = (double *)malloc(sizeof(double) * CRS * NPQ);
    double *G = (double *)malloc(sizeof(double) * Ko * NPQ);
    oracle_im2col(N, C, H, W, R, st, pad, P, Q, x, col);  /* A1 */
    grad_reshape(N, Ko, P * Q, dy, G);                    /* A4 */
    oracle_matmul(Ko, NPQ, CRS, 2u, G, col, dw, dw_abs);  /* A5 */
    free(col);
    free(G);
}

/* The same filter gradient at listed flat indices k*CRS + row of dW. */
void oracle_conv_bwd_filter_at(i64 N, i64 C, i64 H, i64 W, i64 Ko, i64 R, i64 st,
                               i64 pad, i64 P, i64 Q, const double *x,
                               const double *dy, i64 count, const i64 *flat,
                               double *out, double *out_abs)
{
    i64 CRS = C * R * R, PQ = P * Q, NPQ = N * P * Q;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 t = 0; t < count; ++t) {
        i64 k = flat[t] / CRS, row = flat[t] % CRS;
        double acc = 0.0, acc_abs = 0.0;
        for (i64 j = 0; j < NPQ; ++j) {
            i64 n = j / PQ, pq = j % PQ;
            double p = dy[(n * Ko + k) * PQ + pq] *
                       col_entry(x, C, H, W, R, st, pad, P, Q, row, j);
            acc += p;
            acc_abs += fabs(p);
        }
        out[t] = acc;
        out_abs[t] = acc_abs;
    }
}

/* Step A8: bias gradient, page section "Convolution: The im2col Approach",
 * backward: the sum of G over its columns, i.e. over batch and both spatial
 * dimensions (shader table: nn_bias_grad sum-reduces rows).                 */
void oracle_conv_bwd_bias(i64 N, i64 Ko, i64 P, i64 Q, const double *dy,
                          double *db, double *db_abs)
{
    i64 PQ = P * Q, NPQ = N * P * Q;
    double *G = (double *)malloc(sizeof(double) * Ko * NPQ);
    grad_reshape(N, Ko, PQ, dy, G);                       /* A4 */
#pragma omp parallel for schedule(static)
    for (i64 k = 0; k < Ko; ++k) {
        double acc = 0.0, acc_abs = 0.0;
        for (i64 j = 0; j < NPQ; ++j) {
            acc += G[k * NPQ + j];
            acc_abs += fabs(G[k * NPQ + j]);
        }
        db[k] = acc;
        db_abs[k] = acc_abs;
    }
    free(G);
}

/* ------------------------------------------------------------------------- */
/* Step A10: max pooling forward, page shader table "Pooling Shaders":
 * nn_maxpool_forward takes the maximum of each window and stores where it was.
 * Windows are k x k with the given stride, no padding, floor-sized output.
 * Ties keep the first maximum in row-major window order (strict '>').  The
 * stored index is the flat offset into the whole NCHW input.                */
void oracle_maxpool_fwd(i64 N, i64 C, i64 H, i64 W, i64 k, i64 st, i64 P, i64 Q,
                        const float *x, float *y, int32_t *idx)
{
#pragma omp parallel for schedule(static)
    for (i64 nc = 0; nc < N * C; ++nc)
        for (i64 oh = 0; oh < P; ++oh)
            for (i64 ow = 0; ow < Q; ++ow) {
                i64 best = nc * H * W + (oh * st) * W + ow * st;
                float m = x[best];
                for (i64 r = 0; r < k; ++r)
                    for (i64 s = 0; s < k; ++s) {
                        i64 at = nc * H * W + (oh * st + r) * W + (ow * st + s);
                        if (x[at] > m) {
                            m = x[at];
                            best = at;
                        }
                    }
                y[(nc * P + oh) * Q + ow] = m;
                idx[(nc * P + oh) * Q + ow] = (int32_t)best;
            }
}

/* Step A11: max pooling backward, page shader table: nn_maxpool_backward
 * scatters each output gradient to its saved position, after the runtime's
 * ClearBuffer zeroes the target.  Overlapping windows add up; the scatter
 * runs in ascending window order per plane, in fp32.                        */
void oracle_maxpool_bwd(i64 N, i64 C, i64 H, i64 W, i64 P, i64 Q,
                        const float *dy, const int32_t *idx, float *dx)
{
#pragma omp parallel for schedule(static)
    for (i64 nc = 0; nc < N * C; ++nc) {
        for (i64 i = 0; i < H * W; ++i)
            dx[nc * H * W + i] = 0.0f;
        for (i64 t = nc * P * Q; t < (nc + 1) * P * Q; ++t)
            dx[idx[t]] = dx[idx[t]] + dy[t];
    }
}

/* ------------------------------------------------------------------------- */
/* Step A12: SGD, page shader table "Utility Shaders" (nn_sgd):
 * param -= lr * clamp(grad, -clip, clip), elementwise, in fp32:
 * c = min(max(g, -clip), clip); t = lr * c; p = p - t.                      */
void oracle_sgd(i64 count, float lr, float clip, float *param, const float *grad)
{
#pragma omp parallel for schedule(static)
    for (i64 i = 0; i < count; ++i) {
        float g = grad[i];
        float c = g < -clip ? -clip : g;
        c = c > clip ? clip : c;
        float t = lr * c;
        param[i] = param[i] - t;
    }
}

/* ------------------------------------------------------------------------- */
/* Training-step pieces around the convolutions (LeNet-5 step), page shader
 * tables "Activation / Loss Shaders" and "Utility Shaders".                  */

/* nn_relu: y = max(0, x), fp32; the result for x <= 0 is +0.                */
void oracle_relu(i64 count, const float *x, float *y)
{
#pragma omp parallel for schedule(static)
    for (i64 i = 0; i < count; ++i)
        y[i] = x[i] > 0.0f ? x[i] : 0.0f;
}

/* nn_relu_grad: dx = grad * (x > 0), an fp32 product with 1 or 0.  x may be
 * the ReLU's input or its output: both are > 0 at the same positions.       */
void oracle_relu_grad(i64 count, const float *grad, const float *x, float *dx)
{
#pragma omp parallel for schedule(static)
    for (i64 i = 0; i < count; ++i)
        dx[i] = grad[i] * (x[i] > 0.0f ? 1.0f : 0.0f);
}

/* nn_add_bias: out[i] = A[i] + B[i % cols] over a row-major rows x cols
 * matrix, one fp32 addition per element.                                    */
void oracle_add_bias(i64 rows, i64 cols, const float *A, const float *b, float *out)
{
#pragma omp parallel for schedule(static)
    for (i64 i = 0; i < rows * cols; ++i)
        out[i] = A[i] + b[i % cols];
}

/* nn_bias_grad for a linear layer: the sum of the rows of the (batch x out)
 * gradient, db[j] = sum_i G[i][j], in double, with sum_i |G[i][j]|.         */
void oracle_bias_grad_rows(i64 rows, i64 cols, const double *G, double *db, double *db_abs)
{
    for (i64 j = 0; j < cols; ++j) {
        double acc = 0.0, acc_abs = 0.0;
        for (i64 i = 0; i < rows; ++i) {
            acc += G[i * cols + j];
            acc_abs += fabs(G[i * cols + j]);
        }
        db[j] = acc;
        db_abs[j] = acc_abs;
    }
}

/* nn_softmax: per row, subtract the row maximum, exponentiate, divide by the
 * sum (the numerically stable form the page names), in double.              */
void oracle_softmax(i64 rows, i64 cols, const double *z, double *p)
{
    for (i64 i = 0; i < rows; ++i) {
        const double *zr = z + i * cols;
        double m = zr[0];
        for (i64 j = 1; j < cols; ++j)
            if (zr[j] > m) m = zr[j];
        double s = 0.0;
        for (i64 j = 0; j < cols; ++j) {
            p[i * cols + j] = exp(zr[j] - m);
            s += p[i * cols + j];
        }
        for (i64 j = 0; j < cols; ++j) p[i * cols + j] /= s;
    }
}

/* nn_softmax_ce_grad and nn_loss: with p = softmax(z) per row and the row's
 * label l, grad = p - one_hot(l) and loss_i = -log p[l], in double.  The
 * gradient is that of the batch sum of the row losses (no 1/batch factor).   */
void oracle_softmax_ce(i64 rows, i64 cols, const double *z, const int32_t *labels, double *grad,
                       double *loss)
{
    oracle_softmax(rows, cols, z, grad);
    for (i64 i = 0; i < rows; ++i) {
        const i64 l = labels[i];
        loss[i] = -log(grad[i * cols + l]);
        grad[i * cols + l] -= 1.0;
    }
}

/* nn_grad_accum: accum += grad in place, one fp32 addition per element.     */
void oracle_grad_accum(i64 count, const float *grad, float *accum)
{
#pragma omp parallel for schedule(static)
    for (i64 i = 0; i < count; ++i)
        accum[i] = accum[i] + grad[i];
}

/* Number of threads the parallel loops use (for reporting). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
