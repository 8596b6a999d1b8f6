// memory_ops.cu -- the HBM-bound steps of the page "DirectCompute Neural
// Network Engine": the standalone im2col / col2im shaders (section
// "Convolution Shaders"), max pooling forward/backward ("Pooling Shaders"),
// SGD and the bias gradient ("Utility Shaders").
//
// All of them are pure data movement or short per-element arithmetic, so they
// are written for bandwidth: grids sized to the SM count, consecutive threads
// on consecutive output addresses, 16-byte stores where rows allow it, and
// every output element produced by exactly one thread in a fixed order (no
// atomics; results are deterministic and, for the integer/routing work,
// bit-exact).
#include <atomic>
#include <cooperative_groups.h>

#include "gemm_tc.cuh"

namespace cg = cooperative_groups;

namespace cb200 {

static int grid_for(long long work, int per_block)
{
    long long b = (work + per_block - 1) / per_block;
    const long long cap = 16LL * sm_count();
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return int(b);
}

// ---------------------------------------------------------------------------
// Staging of a contiguous element range into shared memory by the bulk-copy
// engine (used by the band col2im and the staged pooling kernels).

// Thread 0: copy elements [start, start + count) of a tensor of `total`
// elements into dst so that element start + i lands at dst[(start & 3) + i].
// The tensor base is 16-byte aligned, so the bulk copy covers whole 16-byte
// blocks; up to 3 elements past the tensor's last 16-byte boundary are
// loaded with plain loads.  Returns the bulk-copied bytes.
__device__ __forceinline__ uint32_t stage_range_bytes(long long start, int count, long long total)
{
    const long long a0 = start & ~3LL;
    long long a1 = (start + count + 3) & ~3LL;
    const long long lim = total & ~3LL;
    if (a1 > lim) a1 = lim;
    return a1 > a0 ? uint32_t((a1 - a0) * 4) : 0u;
}

__device__ __forceinline__ void stage_range(float* dst, const float* base, long long start, int count, long long total,
                                            uint64_t* bar)
{
    const long long a0 = start & ~3LL;
    const uint32_t bytes = stage_range_bytes(start, count, total);
    const long long a1 = a0 + bytes / 4;
    for (long long e = a1 > start ? a1 : start; e < start + count; ++e) dst[e - a0] = __ldg(base + e);
    if (bytes) bulk_g2s(dst, base + a0, bytes, bar);
}

// Bounded wait by every thread of the block on a staging barrier.  The
// outcome is agreed block-wide (a barrier every thread reaches), so either all
// threads go on or all leave the loop together; on give-up the device error
// word is set.
__device__ __forceinline__ bool stage_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err)
{
    const bool got = mbar_wait(bar, parity, abort_flag);
    if (__syncthreads_and(got ? 1 : 0)) return true;
    if (threadIdx.x == 0) {
        *abort_flag = 1;
        atomicOr(err, kDevErrTimeout);
    }
    return false;
}

// ---------------------------------------------------------------------------
// im2col: col[(c, r, q)][(n, oh, ow)] = x[n, c, oh*s + r - pad, ow*s + q - pad].
//
// Staged form.  A block owns one (n, c) plane and a band of Pb output rows
// oh0 .. oh0+Pb-1.  It copies the input rows that band reads -- (Pb-1)*s + R
// of them, Wn = (Q-1)*s + R padded columns each, zeros outside the image -- to
// shared memory once, then writes, for each of the R*R filter taps (r, q), the
// contiguous run of Pb*Q columns of col row (c, r, q) that belong to the band:
// every global store is coalesced and every input element is read from HBM
// once per band.  Each staged row is split by column phase (padded column
// u goes to phase u % s, slot u / s), so the stride-s reads of one tap are
// consecutive shared addresses for any s.  A thread owns up to kIm2colPer
// fixed positions j = tid + k*blockDim of the band, whose shared offsets are
// the same for every tap up to a tap constant.

constexpr int kIm2colThreads = 256;
constexpr int kIm2colPer = 4;
constexpr size_t kIm2colSmem = 72 * 1024;  // three blocks per SM

// Band of pb output rows of one image, or (pb == P) whole images, nb of them
// per block, when a plane is small: the nb images' columns of one col row
// are contiguous too, and a block then has enough positions to amortise its
// set-up.
struct Im2colBand {
    int pb = 0, nband = 0, nb = 0, rows = 0, wph = 0;
    size_t smem = 0;
};

static Im2colBand plan_im2col(const ConvDims& d)
{
    Im2colBand b;
    const int wn = (d.Q - 1) * d.S + d.R;
    b.wph = (wn + d.S - 1) / d.S;
    auto smem_of = [&](int p) { return size_t((p - 1) * d.S + d.R) * d.S * b.wph * sizeof(float); };
    const int cap = kIm2colThreads * kIm2colPer;
    if ((long long)d.P * d.Q <= cap && smem_of(d.P) <= kIm2colSmem) {
        int nb = 1;
        while (nb < d.N && (long long)(nb + 1) * d.P * d.Q <= cap && (nb + 1) * smem_of(d.P) <= kIm2colSmem) ++nb;
        b.nb = nb;
        b.pb = d.P;
        b.nband = 1;
    } else {
        int pb = std::min(d.P, cap / std::max(d.Q, 1));
        while (pb > 1 && smem_of(pb) > kIm2colSmem) --pb;
        if (pb < 1 || smem_of(pb) > 160 * 1024) return b;  // pb == 0: no staged form
        // among the band heights that fit, take the one whose bands leave the
        // fewest idle thread slots over the whole image (each band of nrow rows
        // takes ceil(nrow*Q / threads) passes); ties go to the taller band
        auto use = [&](int h) {
            long long slots = 0;
            for (int oh0 = 0; oh0 < d.P; oh0 += h) {
                const long long pos = (long long)std::min(h, d.P - oh0) * d.Q;
                slots += (pos + kIm2colThreads - 1) / kIm2colThreads * kIm2colThreads;
            }
            return double(d.P) * d.Q / double(slots);
        };
        int best = pb;
        for (int h = pb - 1; h >= std::max(1, pb / 2); --h)
            if (use(h) > use(best) + 0.01) best = h;
        b.pb = best;
        b.nband = (d.P + best - 1) / best;
        b.nb = 1;
    }
    b.rows = (b.pb - 1) * d.S + d.R;
    b.smem = b.nb * smem_of(b.pb);
    return b;
}

__global__ void __launch_bounds__(kIm2colThreads, 6) im2col_band_kernel(
    const float* __restrict__ x, float* __restrict__ col, int N, int C, int H, int W, int S, int R, int pad, int P,
    int Q, int pb, int nband, int nb, int rows, int wph, FastDiv f_s, FastDiv f_q, FastDiv f_iq, FastDiv f_wn,
    FastDiv f_rows, long long npq)
{
    extern __shared__ __align__(16) float tile[];
    // block = (group * C + c) * nband + band
    const int band = blockIdx.x % nband;
    const int rest = blockIdx.x / nband;
    const int c = rest % C;
    const int n0 = (rest / C) * nb;
    const int nbi = min(nb, N - n0);
    const int oh0 = band * pb;
    const int nrow = min(pb, P - oh0);
    const int h0 = oh0 * S - pad;
    const int wn = int(f_wn.d);
    const int rowf = S * wph;          // floats per staged row
    const int imgf = rows * rowf;      // floats per staged image

    // stage rows h0 .. h0+rows-1 of each image, padded columns u = 0 .. wn-1
    // (w = u - pad), zeros outside the image: element e = (img*rows + hl)*wn + u,
    // one asynchronous 4-byte copy each
    const size_t plane = size_t(H) * W;
    const float* xc = x + (size_t(n0) * C + c) * plane;
    const int ne = nbi * rows * wn;
    for (int e = threadIdx.x; e < ne; e += kIm2colThreads) {
        uint32_t ra, u, img, hl, slot, ph;
        f_wn.divmod(uint32_t(e), ra, u);
        f_rows.divmod(ra, img, hl);
        f_s.divmod(u, slot, ph);
        const int h = h0 + int(hl), w = int(u) - pad;
        const bool in = unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W);
        const float* src = in ? xc + size_t(img) * C * plane + size_t(h) * W + w : x;
        cp_async4_zfill(smem_u32(tile + int(img) * imgf + int(hl) * rowf + int(ph) * wph + int(slot)), src, in);
    }
    cp_async_wait_all();
    __syncthreads();

    // position j = (img, oh_l, ow); tap (r, q) reads slot
    // img*imgf + (oh_l*s + r)*rowf + (q % s)*wph + ow + q / s
    const int nj = (nbi - 1) * P * Q + nrow * Q;
    int base[kIm2colPer];
#pragma unroll
    for (int k = 0; k < kIm2colPer; ++k) {
        const int j = threadIdx.x + k * kIm2colThreads;
        uint32_t img, rem, ohl, ow;
        f_iq.divmod(uint32_t(j < nj ? j : 0), img, rem);
        f_q.divmod(rem, ohl, ow);
        base[k] = j < nj ? int(img) * imgf + int(ohl) * S * rowf + int(ow) : -1;
    }
    float* dst = col + size_t(c) * R * R * npq + size_t(n0) * P * Q + size_t(oh0) * Q + threadIdx.x;
    for (int r = 0; r < R; ++r) {
        int toff = r * rowf;  // r*rowf + (q % s)*wph + q / s, advanced with q
        int qp = 0;
        for (int q = 0; q < R; ++q) {
#pragma unroll
            for (int k = 0; k < kIm2colPer; ++k)
                if (base[k] >= 0) dst[k * kIm2colThreads] = tile[base[k] + toff];
            dst += npq;
            if (++qp == S) {
                qp = 0;
                toff += 1 - (S - 1) * wph;
            } else {
                toff += wph;
            }
        }
    }
}

// Unstaged form, for shapes whose band does not fit shared memory.
// One thread writes 4 consecutive columns of one row (a 16-byte store when
// the row length NPQ is a multiple of 4); its (n, oh, ow) is decoded once and
// advanced incrementally.

__global__ void im2col_kernel(const float* __restrict__ x, float* __restrict__ col, int C, int H, int W, int S,
                              int pad, int P, int Q, FastDiv f_pq, FastDiv f_q, FastDiv f_rr, FastDiv f_r,
                              FastDiv f_npq4, int total4)
{
    const int npq = int(f_npq4.d) * 4;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total4; t += gridDim.x * blockDim.x) {
        uint32_t row, j4;
        f_npq4.divmod(uint32_t(t), row, j4);
        const int j0 = int(j4) * 4;
        uint32_t c, rem, r, q;
        f_rr.divmod(row, c, rem);
        f_r.divmod(rem, r, q);
        uint32_t n, pq, oh, ow;
        f_pq.divmod(uint32_t(j0), n, pq);
        f_q.divmod(pq, oh, ow);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int h = int(oh) * S + int(r) - pad;
            const int w = int(ow) * S + int(q) - pad;
            v[e] = (unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W))
                       ? __ldg(x + ((int(n) * C + int(c)) * H + h) * W + w)
                       : 0.f;
            if (++ow == uint32_t(Q)) {
                ow = 0;
                if (++oh == uint32_t(P)) { oh = 0; ++n; }
            }
        }
        *reinterpret_cast<float4*>(col + size_t(row) * npq + j0) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// Scalar variant for row lengths that are not a multiple of 4.
__global__ void im2col_scalar_kernel(const float* __restrict__ x, float* __restrict__ col, int C, int H, int W,
                                     int S, int pad, FastDiv f_npq, FastDiv f_pq, FastDiv f_q, FastDiv f_rr,
                                     FastDiv f_r, int total)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t row, j, c, rem, r, q, n, pq, oh, ow;
        f_npq.divmod(uint32_t(t), row, j);
        f_rr.divmod(row, c, rem);
        f_r.divmod(rem, r, q);
        f_pq.divmod(j, n, pq);
        f_q.divmod(pq, oh, ow);
        const int h = int(oh) * S + int(r) - pad;
        const int w = int(ow) * S + int(q) - pad;
        col[t] = (unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W))
                     ? __ldg(x + ((int(n) * C + int(c)) * H + h) * W + w)
                     : 0.f;
    }
}

cudaError_t launch_im2col(const ConvDims& d, const float* x, float* col, cudaStream_t st)
{
    const int NPQ = d.N * d.P * d.Q;
    const int CRS = d.C * d.R * d.R;
    const FastDiv f_pq(d.P * d.Q), f_q(d.Q), f_rr(d.R * d.R), f_r(d.R);
    const Im2colBand b = plan_im2col(d);
    const long long blocks = (long long)((d.N + std::max(b.nb, 1) - 1) / std::max(b.nb, 1)) * d.C * b.nband;
    if (b.pb > 0 && blocks <= INT32_MAX) {
        if (b.smem > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(im2col_band_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(b.smem));
            if (e != cudaSuccess) return e;
        }
        im2col_band_kernel<<<unsigned(blocks), kIm2colThreads, b.smem, st>>>(
            x, col, d.N, d.C, d.H, d.W, d.S, d.R, d.pad, d.P, d.Q, b.pb, b.nband, b.nb, b.rows, b.wph,
            FastDiv(d.S), FastDiv(d.Q), FastDiv(b.pb * d.Q), FastDiv((d.Q - 1) * d.S + d.R), FastDiv(b.rows), NPQ);
        note_launch();
        return cudaGetLastError();
    }
    if (NPQ % 4 == 0) {
        const long long total4 = (long long)CRS * (NPQ / 4);
        im2col_kernel<<<grid_for(total4, 256), 256, 0, st>>>(x, col, d.C, d.H, d.W, d.S, d.pad, d.P, d.Q, f_pq,
                                                             f_q, f_rr, f_r, FastDiv(NPQ / 4), int(total4));
    note_launch();
    } else {
        const long long total = (long long)CRS * NPQ;
        im2col_scalar_kernel<<<grid_for(total, 256), 256, 0, st>>>(x, col, d.C, d.H, d.W, d.S, d.pad, FastDiv(NPQ),
                                                                    f_pq, f_q, f_rr, f_r, int(total));
    note_launch();
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// col2im as a gather: dx[n, c, h, w] = sum of col[(c, r, q)][(n, oh, ow)] over
// the taps with oh*s + r - pad = h and ow*s + q - pad = w.  With hp = h + pad
// those are r = hp % s + i*s, oh = hp / s - i (and q, ow alike from wp = w +
// pad) for i, j < ceil(R/s), kept when r, q < R and oh, ow fall inside the
// output.  Every thread walks the same (i, j) schedule, masked at the edges,
// so in each step the lanes of a warp that share wp % s read consecutive ow
// of one col row: the reads are coalesced for any stride.  The terms arrive
// in ascending (r, q) order -- a fixed order, so the result is deterministic
// -- and eight loads are issued before the first add.

__global__ void col2im_kernel(const float* __restrict__ col, float* __restrict__ dx, int R, int S, int pad, int P,
                              int Q, long long npq, FastDiv f_s, FastDiv f_w, FastDiv f_h, FastDiv f_c, int total)
{
    const int steps = (R + S - 1) / S;
    const int taps = steps * steps;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t r1, w, r2, h, n, c;
        f_w.divmod(uint32_t(t), r1, w);
        f_h.divmod(r1, r2, h);
        f_c.divmod(r2, n, c);
        uint32_t ohb, r0, owb, q0;
        f_s.divmod(h + uint32_t(pad), ohb, r0);
        f_s.divmod(w + uint32_t(pad), owb, q0);
        // element (i, j): col row (c*R + r0 + i*s)*R + q0 + j*s, column (n*P + ohb - i)*Q + owb - j
        const float* base = col + (size_t(c) * R * R + size_t(r0) * R + q0) * npq + (size_t(n) * P + ohb) * Q + owb;
        float acc = 0.f;
        int i = 0, j = 0;
        for (int k0 = 0; k0 < taps; k0 += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                v[u] = 0.f;
                if (k0 + u < taps) {
                    const int r = int(r0) + i * S, q = int(q0) + j * S;
                    const int oh = int(ohb) - i, ow = int(owb) - j;
                    if (r < R && q < R && oh >= 0 && oh < P && ow >= 0 && ow < Q)
                        v[u] = __ldg(base + (size_t(i) * S * R + size_t(j) * S) * npq - size_t(i) * Q - j);
                    if (++j == steps) {
                        j = 0;
                        ++i;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) acc += v[u];
        }
        dx[t] = acc;
    }
}

// Staged col2im by residue class.  The taps that reach a dx element (h, w)
// all have r = (h + pad) % s (mod s) and q = (w + pad) % s (mod s), so the
// taps split into s*s classes (r0, q0), each of which is a stride-1 problem:
// with a = (h + pad) / s and b = (w + pad) / s, the element sums
// col[(c, r0 + i*s, q0 + j*s)][(n, a - i, b - j)] over i, j < ceil((R - r0)/s)
// (and ceil((R - q0)/s)) wherever a - i, b - j fall inside the output.  Every
// col row belongs to exactly one class.  A block owns one class of one
// channel c for a band of A sub-rows a of one image, or for all sub-rows of
// nb consecutive images; for each of its taps it needs one contiguous run of
// the col row (output rows oa .. ob-1 with a halo of ceil(R/s) - 1 rows, or
// whole images), which one lane of warp 0 stages with a bulk copy.  After
// one bounded wait every thread sums its dx elements from shared memory, taps in
// ascending (r, q) order -- a fixed order, so the result is deterministic --
// and writes them once.

// One item per block: a block stages its item with bulk copies, waits once,
// sums, and exits; three blocks share an SM, so one block's copies overlap
// the others' sums.  (A persistent form with two stages and one block per SM
// measured 1.6x slower: every item then ends in a block-wide barrier that the
// whole SM waits at.)
constexpr int kCol2imThreads = 256;
constexpr size_t kCol2imStage = 74 * 1024;  // three blocks per SM
constexpr int kCol2imMaxPix = 2048;         // dx elements per item when whole images are grouped

struct Col2imPlan {
    int steps = 0, U = 0, V = 0, A = 0, nband = 0, nb = 0, seg = 0, items = 0;
    size_t smem = 0;
};

static Col2imPlan plan_col2im(const ConvDims& d)
{
    Col2imPlan p;
    p.steps = (d.R + d.S - 1) / d.S;
    p.U = (d.H + d.pad + d.S - 1) / d.S;
    p.V = (d.W + d.pad + d.S - 1) / d.S;
    const size_t taps = size_t(p.steps) * p.steps;
    if (taps > 25) return p;  // nb == 0: the taps no longer fit in registers
    const long long PQ = (long long)d.P * d.Q;
    auto seg_of = [](long long count) { return (count + 8 + 3) & ~3LL; };
    // one stage: the staged runs of every tap plus the table of their offsets
    auto bytes_of = [&](long long count) { return taps * (size_t(seg_of(count)) * sizeof(float) + sizeof(int)); };
    if (bytes_of(PQ) <= kCol2imStage) {
        int nb = 1;
        while (nb < d.N && bytes_of((nb + 1) * PQ) <= kCol2imStage &&
               (long long)(nb + 1) * p.U * p.V <= kCol2imMaxPix)
            ++nb;
        p.nb = nb;
        p.A = p.U;
        p.nband = 1;
        p.seg = int(seg_of(nb * PQ));
    } else {
        int A = p.U;
        while (A > 1 && bytes_of((long long)std::min(d.P, A + p.steps - 1) * d.Q) > kCol2imStage) --A;
        if (bytes_of((long long)std::min(d.P, A + p.steps - 1) * d.Q) > kCol2imStage) return p;  // nb == 0: none
        p.nband = (p.U + A - 1) / A;
        p.A = (p.U + p.nband - 1) / p.nband;
        p.nb = 1;
        p.seg = int(seg_of((long long)std::min(d.P, p.A + p.steps - 1) * d.Q));
    }
    const long long items = (long long)((d.N + p.nb - 1) / p.nb) * d.C * p.nband * d.S * d.S;
    if (items > INT32_MAX) {
        p.nb = 0;
        return p;
    }
    p.items = int(items);
    p.smem = taps * (size_t(p.seg) * sizeof(float) + sizeof(int));
    return p;
}

struct Col2imArgs {
    const float* col;
    float* dx;
    int N, C, H, W, S, R, pad, P, Q;
    long long npq, total;
    int steps, A, nband, nb, seg, items;
    FastDiv f_v, f_av;
    int* err;
};

// One work item: class cls of channel c, sub-row band `band`, images n0 .. n0+nbi-1.
struct Col2imItem {
    int n0, nbi, c, r0, q0, ni, nj, a0, oa, ob, count;
    long long start;
    __device__ Col2imItem(const Col2imArgs& g, int item)
    {
        const int SS = g.S * g.S;
        const int cls = item % SS;
        int rest = item / SS;
        const int band = rest % g.nband;
        rest /= g.nband;
        c = rest % g.C;
        n0 = (rest / g.C) * g.nb;
        nbi = min(g.nb, g.N - n0);
        r0 = cls / g.S;
        q0 = cls - r0 * g.S;
        ni = (g.R - r0 + g.S - 1) / g.S;
        nj = (g.R - q0 + g.S - 1) / g.S;
        a0 = band * g.A;
        oa = max(0, a0 - g.steps + 1);
        ob = min(g.P, a0 + g.A);
        start = (long long)n0 * g.P * g.Q + (long long)oa * g.Q;
        count = (nbi - 1) * g.P * g.Q + max(ob - oa, 0) * g.Q;
    }
    __device__ long long tap_start(const Col2imArgs& g, int i, int j) const
    {
        return (((long long)c * g.R + r0 + i * g.S) * g.R + q0 + j * g.S) * g.npq + start;
    }
};

// Sum the dx elements of one staged item whose class has NI x NJ taps.  The
// tap offsets live in registers.  Every element takes the same predicated
// sequence -- a tap counts when its output row a - i and column b - j lie
// inside the output -- so the lanes of a warp never diverge between an
// interior and an edge path.  Terms are added in ascending (i, j), i.e.
// ascending (r, q), order.
template <int NI, int NJ>
__device__ __forceinline__ void col2im_sum_item(const Col2imArgs& g, const Col2imItem& it, const float* buf,
                                                const int* tadj)
{
    constexpr int NT = NI * NJ > 0 ? NI * NJ : 1;
    int tr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) tr[t] = t < NI * NJ ? tadj[t] : 0;
    const int PQ = g.P * g.Q, HW = g.H * g.W, CHW = g.C * HW;
    float* out = g.dx + (size_t(it.n0) * g.C + it.c) * size_t(HW);
    const int npix = it.nbi * g.A * int(g.f_v.d);
    for (int px = threadIdx.x; px < npix; px += kCol2imThreads) {
        uint32_t img, rem, al, bb;
        g.f_av.divmod(uint32_t(px), img, rem);
        g.f_v.divmod(rem, al, bb);
        const int a = it.a0 + int(al), b = int(bb);
        const int h = a * g.S + it.r0 - g.pad, w = b * g.S + it.q0 - g.pad;
        if (a >= it.a0 + g.A || h < 0 || h >= g.H || w < 0 || w >= g.W) continue;
        const float* e = buf + (int(img) * PQ + (a - it.oa) * g.Q + b);
        bool vi[NI > 0 ? NI : 1], vj[NJ > 0 ? NJ : 1];
#pragma unroll
        for (int i = 0; i < NI; ++i) vi[i] = unsigned(a - i) < unsigned(g.P);
#pragma unroll
        for (int j = 0; j < NJ; ++j) vj[j] = unsigned(b - j) < unsigned(g.Q);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j)
                if (vi[i] && vj[j]) acc += e[tr[i * NJ + j]];
        out[int(img) * CHW + h * g.W + w] = acc;
    }
}

// Block = one item.  The 32 lanes of warp 0 issue the item's copies, one tap
// per lane; every thread then waits (bounded) for them and sums.  Shared
// memory holds three blocks per SM; telling the compiler so (rather than
// letting it aim at more blocks with fewer registers) lets it schedule the
// shared loads of a dx element further ahead: 1.4x faster as measured.
// ST = ceil(R/s): the taps of a class are ST or ST - 1 along each axis.
template <int ST>
__global__ void __launch_bounds__(kCol2imThreads, 3) col2im_class_kernel(const __grid_constant__ Col2imArgs g)
{
    extern __shared__ __align__(16) float c2i_smem[];
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    const int taps_max = g.steps * g.steps;
    float* buf = c2i_smem;
    // tadj[t] for tap t = i*nj + j is the buffer offset of (image 0, output row
    // oa, column 0) minus i*Q + j, so that the element a dx position (img, a, b)
    // takes from tap t sits at tadj[t] + img*PQ + (a - oa)*Q + b.
    int* tadj = reinterpret_cast<int*>(c2i_smem + size_t(taps_max) * g.seg);
    const Col2imItem it(g, blockIdx.x);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int nt = it.ni * it.nj;
        uint32_t bytes = 0;
        for (int t = lane; t < nt; t += 32)
            bytes += stage_range_bytes(it.tap_start(g, t / it.nj, t % it.nj), it.count, g.total);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
        if (lane == 0) mbar_arrive_expect_tx(&bar, bytes);
        __syncwarp();
        for (int t = lane; t < nt; t += 32) {
            const int i = t / it.nj, j = t % it.nj;
            const long long st = it.tap_start(g, i, j);
            tadj[t] = t * g.seg + int(st & 3) - i * g.Q - j;
            if (it.count > 0) stage_range(buf + size_t(t) * g.seg, g.col, st, it.count, g.total, &bar);
        }
    }
    if (!stage_wait(&bar, 0, &abort_flag, g.err)) return;
    // a class has ST or ST - 1 taps along each axis
    if (it.ni == ST && it.nj == ST)
        col2im_sum_item<ST, ST>(g, it, buf, tadj);
    else if (it.ni == ST)
        col2im_sum_item<ST, ST - 1>(g, it, buf, tadj);
    else if (it.nj == ST)
        col2im_sum_item<ST - 1, ST>(g, it, buf, tadj);
    else
        col2im_sum_item<ST - 1, ST - 1>(g, it, buf, tadj);
}

cudaError_t launch_col2im(const ConvDims& d, const float* col, float* dx, cudaStream_t st)
{
    const long long NPQ = (long long)d.N * d.P * d.Q;
    const Col2imPlan p = plan_col2im(d);
    if (p.nb > 0 && (reinterpret_cast<uintptr_t>(col) & 15) == 0) {
        Col2imArgs g{col, dx, d.N, d.C, d.H, d.W, d.S, d.R, d.pad, d.P, d.Q, NPQ, NPQ * d.C * d.R * d.R,
                     p.steps, p.A, p.nband, p.nb, p.seg, p.items, FastDiv(p.V), FastDiv(p.A * p.V),
                     device_error_word()};
        auto run = [&](auto kern) {
            if (p.smem > 48 * 1024) {
                const cudaError_t e =
                    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(p.smem));
                if (e != cudaSuccess) return e;
            }
            kern<<<p.items, kCol2imThreads, p.smem, st>>>(g);
            return cudaSuccess;
        };
        const cudaError_t e = p.steps == 1   ? run(col2im_class_kernel<1>)
                              : p.steps == 2 ? run(col2im_class_kernel<2>)
                              : p.steps == 3 ? run(col2im_class_kernel<3>)
                              : p.steps == 4 ? run(col2im_class_kernel<4>)
                                             : run(col2im_class_kernel<5>);
        if (e != cudaSuccess) return e;
        note_launch();
        return cudaGetLastError();
    }
    const long long total = (long long)d.N * d.C * d.H * d.W;
    col2im_kernel<<<grid_for(total, 256), 256, 0, st>>>(col, dx, d.R, d.S, d.pad, d.P, d.Q, NPQ, FastDiv(d.S),
                                                        FastDiv(d.W), FastDiv(d.H), FastDiv(d.C), int(total));
    note_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Max pooling forward: first maximum in row-major window order (strict >).

__global__ void maxpool_fwd_kernel(const float* __restrict__ x, float* __restrict__ y, int32_t* __restrict__ idx,
                                   int H, int W, int k, int S, FastDiv f_q, FastDiv f_p, int total)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t r1, ow, nc, oh;
        f_q.divmod(uint32_t(t), r1, ow);
        f_p.divmod(r1, nc, oh);
        const int corner = (int(nc) * H + int(oh) * S) * W + int(ow) * S;
        int best = corner;
        float m = __ldg(x + corner);
        for (int r = 0; r < k; ++r)
            for (int q = 0; q < k; ++q) {
                const int at = corner + r * W + q;
                const float v = __ldg(x + at);
                if (v > m) {
                    m = v;
                    best = at;
                }
            }
        y[t] = m;
        idx[t] = best;
    }
}

// Staged variants.  Consecutive (n, c) planes are contiguous, so a group of
// `ppb` planes is one contiguous range: a block stages it into shared memory
// with one bulk copy (the tensor engine moves the bytes; no thread issues
// loads) and scans the windows there.  Two stage buffers per block: while
// group i is scanned, group i + 1 is in flight.  Blocks are persistent (a
// few per SM) and take groups blockIdx.x, blockIdx.x + gridDim.x, ...
constexpr int kPoolThreads = 512;
constexpr int kPoolStageFloats = 6144;   // 24 KB per staged range

__global__ void __launch_bounds__(kPoolThreads, 4) maxpool_fwd_staged_kernel(
    const float* __restrict__ x, float* __restrict__ y, int32_t* __restrict__ idx, int NC, int H, int W, int k, int S,
    int P, int Q, int ppb, int stage_floats, FastDiv f_pq, FastDiv f_q, int* err)
{
    extern __shared__ __align__(16) float pool_smem[];
    __shared__ uint64_t bar[2];
    __shared__ int abort_flag;
    const int HW = H * W, PQ = P * Q;
    const long long total = (long long)NC * HW;
    const int groups = (NC + ppb - 1) / ppb;
    auto issue = [&](int g, int b) {
        const int nc0 = g * ppb, np = min(ppb, NC - nc0);
        const long long start = (long long)nc0 * HW;
        mbar_arrive_expect_tx(&bar[b], stage_range_bytes(start, np * HW, total));
        stage_range(pool_smem + b * stage_floats, x, start, np * HW, total, &bar[b]);
    };
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        abort_flag = 0;
        mbar_fence_init();
        for (int i = 0; i < 2; ++i)
            if (int(blockIdx.x) + i * int(gridDim.x) < groups) issue(blockIdx.x + i * gridDim.x, i);
    }
    __syncthreads();
    int i = 0, g = blockIdx.x;
    for (; g < groups; g += gridDim.x, ++i) {
        const int b = i & 1;
        if (!stage_wait(&bar[b], uint32_t(i >> 1) & 1u, &abort_flag, err)) break;
        const int nc0 = g * ppb, np = min(ppb, NC - nc0);
        const float* sx = pool_smem + b * stage_floats + ((long long)nc0 * HW & 3);
        const int nout = np * PQ;
        for (int o = threadIdx.x; o < nout; o += kPoolThreads) {
            uint32_t pl, pq, oh, ow;
            f_pq.divmod(uint32_t(o), pl, pq);
            f_q.divmod(pq, oh, ow);
            const int corner = int(pl) * HW + int(oh) * S * W + int(ow) * S;
            int best = corner;
            float m = sx[corner];
            for (int r = 0; r < k; ++r)
                for (int q = 0; q < k; ++q) {
                    const int at = corner + r * W + q;
                    const float v = sx[at];
                    if (v > m) {
                        m = v;
                        best = at;
                    }
                }
            y[size_t(nc0) * PQ + o] = m;
            idx[size_t(nc0) * PQ + o] = nc0 * HW + best;
        }
        __syncthreads();   // buffer b fully read
        if (threadIdx.x == 0 && g + 2 * int(gridDim.x) < groups) {
            fence_proxy_async_smem();
            issue(g + 2 * gridDim.x, b);
        }
    }
    if (abort_flag && threadIdx.x == 0) {
        // let copies still in flight (groups g and g + gridDim.x) land before
        // the block's memory goes away
        for (int j = 0; j < 2 && g + j * int(gridDim.x) < groups; ++j) {
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&bar[(i + j) & 1], uint32_t((i + j) >> 1) & 1u) &&
                   globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// Staged backward: a group's window gradients and saved indices (two
// contiguous ranges) are staged per buffer.  Each thread owns an S x S block
// of input pixels (rows S*i .., columns S*j ..).  It visits, in ascending
// (oh, ow) order, the windows that can reach its block -- oh from
// ceil((S*i - k + 1) / S) to i, the same for ow -- and adds each window's
// gradient to the pixel of the block its saved index names, if any.  Every
// pixel therefore sums its contributions in ascending window order (the
// oracle's order) with a handful of compares per window and no per-pixel
// division; the S*S results are written with coalesced stores.
template <int S>
__global__ void __launch_bounds__(kPoolThreads, 3) maxpool_bwd_staged_kernel(
    const float* __restrict__ dy, const int32_t* __restrict__ idx, float* __restrict__ dx, int NC, int H, int W,
    int k, int P, int Q, int ppb, int stage_floats, int BH, int BW, FastDiv f_blk, FastDiv f_bw, int* err)
{
    extern __shared__ __align__(16) float pool_smem[];
    __shared__ uint64_t bar[2];
    __shared__ int abort_flag;
    const int HW = H * W, PQ = P * Q;
    // per buffer (2 * stage_floats): [gradients (stage_floats)][indices (stage_floats)]
    const long long total = (long long)NC * PQ;
    const int groups = (NC + ppb - 1) / ppb;
    auto issue = [&](int g, int b) {
        const int nc0 = g * ppb, np = min(ppb, NC - nc0);
        const long long start = (long long)nc0 * PQ;
        mbar_arrive_expect_tx(&bar[b], 2 * stage_range_bytes(start, np * PQ, total));
        float* sb = pool_smem + 2 * b * stage_floats;
        stage_range(sb, dy, start, np * PQ, total, &bar[b]);
        stage_range(sb + stage_floats, reinterpret_cast<const float*>(idx), start, np * PQ, total, &bar[b]);
    };
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        abort_flag = 0;
        mbar_fence_init();
        for (int i = 0; i < 2; ++i)
            if (int(blockIdx.x) + i * int(gridDim.x) < groups) issue(blockIdx.x + i * gridDim.x, i);
    }
    __syncthreads();
    const int nblk_plane = BH * BW;
    int it = 0, g = blockIdx.x;
    for (; g < groups; g += gridDim.x, ++it) {
        const int b = it & 1;
        if (!stage_wait(&bar[b], uint32_t(it >> 1) & 1u, &abort_flag, err)) break;
        const int nc0 = g * ppb, np = min(ppb, NC - nc0);
        const int sh = int((long long)nc0 * PQ & 3);
        const float* sdy = pool_smem + 2 * b * stage_floats + sh;
        const int* sidx = reinterpret_cast<const int*>(sdy + stage_floats);
        const int nblk = np * nblk_plane;
        for (int t = threadIdx.x; t < nblk; t += kPoolThreads) {
            uint32_t pl, ij, bi, bj;
            f_blk.divmod(uint32_t(t), pl, ij);
            f_bw.divmod(ij, bi, bj);
            const int h0 = S * int(bi), w0 = S * int(bj);
            const int base = (nc0 + int(pl)) * HW + h0 * W + w0;   // flat index of the block's first pixel
            const int oh_lo = h0 - k + 1 <= 0 ? 0 : (h0 - k + S) / S;
            const int oh_hi = min(int(bi), P - 1);
            const int ow_lo = w0 - k + 1 <= 0 ? 0 : (w0 - k + S) / S;
            const int ow_hi = min(int(bj), Q - 1);
            float acc[S * S];
#pragma unroll
            for (int a = 0; a < S * S; ++a) acc[a] = 0.f;
            const int* irow = sidx + int(pl) * PQ;
            const float* drow = sdy + int(pl) * PQ;
            for (int oh = oh_lo; oh <= oh_hi; ++oh)
                for (int ow = ow_lo; ow <= ow_hi; ++ow) {
                    const int o = oh * Q + ow;
                    const int d = irow[o] - base;
                    const float v = drow[o];
#pragma unroll
                    for (int dh = 0; dh < S; ++dh)
#pragma unroll
                        for (int dw = 0; dw < S; ++dw)
                            if (w0 + dw < W && d == dh * W + dw) acc[dh * S + dw] += v;   // no wrap into the next row
                }
            float* out = dx + base;
#pragma unroll
            for (int dh = 0; dh < S; ++dh)
#pragma unroll
                for (int dw = 0; dw < S; ++dw)
                    if (h0 + dh < H && w0 + dw < W) out[dh * W + dw] = acc[dh * S + dw];
        }
        __syncthreads();
        if (threadIdx.x == 0 && g + 2 * int(gridDim.x) < groups) {
            fence_proxy_async_smem();
            issue(g + 2 * gridDim.x, b);
        }
    }
    if (abort_flag && threadIdx.x == 0) {
        for (int j = 0; j < 2 && g + j * int(gridDim.x) < groups; ++j) {
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&bar[(it + j) & 1], uint32_t((it + j) >> 1) & 1u) &&
                   globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Register walkers for K x K windows with stride S and K <= 2S (the 3x3/2 and
// 2x2/2 pools).  No shared memory and no barriers: a thread walks down one
// column of windows (forward) or one column of S-wide pixel blocks
// (backward) and keeps what neighbouring rows share in registers.  Loads for
// kWalkChunk rows of windows are issued before any of them is used, so each
// thread has a few dozen independent loads in flight.  Work item = (plane,
// row segment, column), column fastest, so a warp's loads and stores run
// along a row.
constexpr int kWalkThreads = 256;
constexpr int kWalkChunk = 4;
constexpr int kFwdWalkChunk = 8;   // the forward walk is load-latency bound: more windows' rows in flight

// Forward: window oh combines the first maxima of its K input rows
// (rows oh*S .. oh*S + K - 1, each the first maximum over its K columns);
// taking rows in order with a strict > gives the first maximum of the window
// in row-major order.  Rows shared with the previous window (K - S of them)
// are carried.
template <int K, int S>
__global__ void __launch_bounds__(kWalkThreads) maxpool_fwd_walk_kernel(
    const float* __restrict__ x, float* __restrict__ y, int32_t* __restrict__ idx, int H, int W, int P, int Q,
    int seglen, FastDiv f_q, FastDiv f_seg, int items)
{
    static_assert(S <= K && K <= 2 * S, "walker covers windows at most two strides wide");
    griddep_wait();
    griddep_launch();
    const int t = int(blockIdx.x) * kWalkThreads + int(threadIdx.x);
    if (t >= items) return;
    uint32_t rest, ow, plane, seg;
    f_q.divmod(uint32_t(t), rest, ow);
    f_seg.divmod(rest, plane, seg);
    const int oh0 = int(seg) * seglen;
    const int oh1 = min(oh0 + seglen, P);
    const int col0 = int(plane) * H * W + int(ow) * S;   // flat index of the column's first window corner
    float rm[K];
    int ri[K];
    // the K - S rows the segment's first window shares with the window above it
#pragma unroll
    for (int r = 0; r < K - S; ++r) {
        const int at = col0 + (oh0 * S + r) * W;
        rm[r] = __ldg(x + at);
        ri[r] = at;
#pragma unroll
        for (int c = 1; c < K; ++c) {
            const float v = __ldg(x + at + c);
            if (v > rm[r]) {
                rm[r] = v;
                ri[r] = at + c;
            }
        }
    }
    float* yo = y + size_t(plane) * P * Q + ow;
    int32_t* io = idx + size_t(plane) * P * Q + ow;
    for (int oh = oh0; oh < oh1; oh += kFwdWalkChunk) {
        // rows oh*S + K - S + u, u < kFwdWalkChunk*S: the S new rows of each window of the chunk
        float v[kFwdWalkChunk * S][K];
#pragma unroll
        for (int u = 0; u < kFwdWalkChunk * S; ++u)
            if (oh + u / S < oh1) {
                const int at = col0 + (oh * S + K - S + u) * W;
#pragma unroll
                for (int c = 0; c < K; ++c) v[u][c] = __ldg(x + at + c);
            }
#pragma unroll
        for (int i = 0; i < kFwdWalkChunk; ++i) {
            if (oh + i >= oh1) break;
#pragma unroll
            for (int r = 0; r < S; ++r) {
                const float* row = v[i * S + r];
                const int at = col0 + ((oh + i) * S + K - S + r) * W;
                float m = row[0];
                int a = at;
#pragma unroll
                for (int c = 1; c < K; ++c)
                    if (row[c] > m) {
                        m = row[c];
                        a = at + c;
                    }
                rm[K - S + r] = m;
                ri[K - S + r] = a;
            }
            float m = rm[0];
            int a = ri[0];
#pragma unroll
            for (int r = 1; r < K; ++r)
                if (rm[r] > m) {
                    m = rm[r];
                    a = ri[r];
                }
            yo[size_t(oh + i) * Q] = m;
            io[size_t(oh + i) * Q] = a;
            // the next window's first K - S rows are this window's last ones
#pragma unroll
            for (int r = 0; r < K - S; ++r) {
                rm[r] = rm[r + S];
                ri[r] = ri[r + S];
            }
        }
    }
}

// Add gradient v of a window to the pixel its saved index iv names, if that
// pixel is one of the walking thread's cells: rows r < K below its block
// origin p00 (rows >= S belong to the next block row and go to the carry),
// columns c < CM (S for the thread's own window column, K - S for the window
// column to its left, the part of that window over this block column).  All
// those cells lie inside the window, so a match is also the window check: the
// index is compared with each cell's offset instead of being decoded.
template <int K, int S, int KC, int CM>
__device__ __forceinline__ void pool_route(float v, int iv, int p00, int W, float (&acc)[S][S], float (&nxt)[KC][S])
{
    const int d = iv - p00;
#pragma unroll
    for (int r = 0; r < K; ++r)
#pragma unroll
        for (int c = 0; c < CM; ++c)
            if (d == r * W + c) {
                if (r < S)
                    acc[r][c] += v;
                else
                    nxt[r - S < KC ? r - S : 0][c] += v;
            }
}

// Backward: a thread owns the column of S x S pixel blocks j (pixel columns
// S*j .. S*j + S - 1) and walks down its block rows b.  With K <= 2S only the
// windows (b, j - 1) and (b, j) of window row b reach block (b, j), and
// window row b reaches block row b (its first S rows) and block row b + 1
// (its last K - S rows, carried to the next step).  A pixel of block (b, j)
// therefore receives, in this order, (b-1, j-1) and (b-1, j) through the
// carry, then (b, j-1) and (b, j): ascending window order, each added in
// fp32 to a sum that starts at zero -- bit-for-bit the ClearBuffer-then-
// scatter result.  A saved index outside its window routes nothing.
template <int K, int S>
__global__ void __launch_bounds__(kWalkThreads) maxpool_bwd_walk_kernel(
    const float* __restrict__ dy, const int32_t* __restrict__ idx, float* __restrict__ dx, int H, int W, int P,
    int Q, int BH, int seglen, FastDiv f_bw, FastDiv f_seg, int items)
{
    static_assert(S <= K && K <= 2 * S, "walker covers windows at most two strides wide");
    griddep_wait();
    griddep_launch();
    constexpr int KC = K - S > 0 ? K - S : 1;   // carried rows (at least one slot)
    const int t = int(blockIdx.x) * kWalkThreads + int(threadIdx.x);
    if (t >= items) return;
    uint32_t rest, j, plane, seg;
    f_bw.divmod(uint32_t(t), rest, j);
    f_seg.divmod(rest, plane, seg);
    const int b0 = int(seg) * seglen;
    const int b1 = min(b0 + seglen, BH);
    const int pbase = int(plane) * H * W;
    const float* dyp = dy + size_t(plane) * P * Q;
    const int32_t* ip = idx + size_t(plane) * P * Q;
    const bool has_l = j >= 1 && int(j) - 1 < Q;   // window column j - 1 exists
    const bool has_r = int(j) < Q;                 // window column j exists

    float carry[KC][S];
#pragma unroll
    for (int r = 0; r < KC; ++r)
#pragma unroll
        for (int c = 0; c < S; ++c) carry[r][c] = 0.f;
    if (K > S && b0 >= 1 && b0 - 1 < P) {
        // the segment starts mid-plane: window row b0 - 1's contributions to block row b0
        float unused[S][S] = {};
        const int oh = b0 - 1;
        const int p00 = pbase + oh * S * W + int(j) * S;
        if (has_l) pool_route<K, S, KC, K - S>(__ldg(dyp + oh * Q + j - 1), __ldg(ip + oh * Q + j - 1), p00, W, unused, carry);
        if (has_r) pool_route<K, S, KC, S>(__ldg(dyp + oh * Q + j), __ldg(ip + oh * Q + j), p00, W, unused, carry);
    }
    const int wend = min(b1, P);   // window rows this segment reads: [b0, wend)
    float* out = dx + pbase + int(j) * S;
    for (int b = b0; b < b1; b += kWalkChunk) {
        float vl[kWalkChunk], vr[kWalkChunk];
        int il[kWalkChunk], ir[kWalkChunk];
#pragma unroll
        for (int u = 0; u < kWalkChunk; ++u)
            if (b + u < wend) {
                const int o = (b + u) * Q + int(j);
                if (has_l) {
                    vl[u] = __ldg(dyp + o - 1);
                    il[u] = __ldg(ip + o - 1);
                }
                if (has_r) {
                    vr[u] = __ldg(dyp + o);
                    ir[u] = __ldg(ip + o);
                }
            }
#pragma unroll
        for (int u = 0; u < kWalkChunk; ++u) {
            const int bb = b + u;
            if (bb >= b1) break;
            float acc[S][S], nxt[KC][S];
#pragma unroll
            for (int r = 0; r < S; ++r)
#pragma unroll
                for (int c = 0; c < S; ++c) acc[r][c] = (K > S && r < K - S) ? carry[r < KC ? r : 0][c] : 0.f;
#pragma unroll
            for (int r = 0; r < KC; ++r)
#pragma unroll
                for (int c = 0; c < S; ++c) nxt[r][c] = 0.f;
            if (bb < wend) {
                const int p00 = pbase + bb * S * W + int(j) * S;
                if (has_l) pool_route<K, S, KC, K - S>(vl[u], il[u], p00, W, acc, nxt);
                if (has_r) pool_route<K, S, KC, S>(vr[u], ir[u], p00, W, acc, nxt);
            }
#pragma unroll
            for (int r = 0; r < S; ++r) {
                const int h = bb * S + r;
                if (h < H) {
#pragma unroll
                    for (int c = 0; c < S; ++c)
                        if (int(j) * S + c < W) out[h * W + c] = acc[r][c];
                }
            }
#pragma unroll
            for (int r = 0; r < KC; ++r)
#pragma unroll
                for (int c = 0; c < S; ++c) carry[r][c] = nxt[r][c];
        }
    }
}

// Rows per segment for a walker with `per_seg_items` threads per segment and
// `resident` threads resident on the GPU at once.  The walk is latency-bound
// (long-scoreboard stalls), so it wants every SM full until the end: of the
// segment counts that keep at least two load chunks of rows per segment (a
// shorter walk does not amortise its start), take the fewest whose last wave
// of threads is nearly as full as the best (within 5 points).  AlexNet pool1:
// one whole-plane walk per column is 1.42 waves (the second 42% full); two
// half-plane segments are 2.84 waves (forward 0.65 -> 0.68, backward 0.56 ->
// 0.60 of the copy bandwidth).  Pool2's 13-row planes stay whole (three
// 5-row segments measured 0.78 -> 0.71).
static int walk_seglen(int rows, long long per_seg_items, long long resident)
{
    const long long max_seg = rows / (2 * kWalkChunk) > 1 ? rows / (2 * kWalkChunk) : 1;
    int best = 1;
    double best_eff = 0.0;
    for (int nseg = 1; nseg <= max_seg && nseg <= 8; ++nseg) {
        const double waves = double(per_seg_items) * nseg / double(resident);
        const double eff = waves / double((long long)(waves + 0.999999));
        if (eff > best_eff + 0.05) {
            best_eff = eff;
            best = nseg;
        }
    }
    return (rows + best - 1) / best;
}

// Threads of a walker kernel resident on the GPU at once (from the occupancy
// the compiled kernel allows).
template <class Kern>
static long long walk_resident(Kern kern)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWalkThreads, 0) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        per_sm = 4;
    }
    return (long long)sm_count() * per_sm * kWalkThreads;
}

template <int K, int S>
static cudaError_t launch_pool_fwd_walk(int NC, int H, int W, int P, int Q, const float* x, float* y, int32_t* idx,
                                        cudaStream_t st)
{
    static const long long resident = walk_resident(maxpool_fwd_walk_kernel<K, S>);
    const int seglen = walk_seglen(P, (long long)NC * Q, resident);
    const int nseg = (P + seglen - 1) / seglen;
    const long long items = (long long)NC * nseg * Q;
    cudaError_t e = launch_pdl(maxpool_fwd_walk_kernel<K, S>, dim3(unsigned((items + kWalkThreads - 1) / kWalkThreads)),
                               dim3(kWalkThreads), 0, st, x, y, idx, H, W, P, Q, seglen, FastDiv(uint32_t(Q)),
                               FastDiv(uint32_t(nseg)), int(items));
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

template <int K, int S>
static cudaError_t launch_pool_bwd_walk(int NC, int H, int W, int P, int Q, const float* dy, const int32_t* idx,
                                        float* dx, cudaStream_t st)
{
    const int BH = (H + S - 1) / S, BW = (W + S - 1) / S;
    static const long long resident = walk_resident(maxpool_bwd_walk_kernel<K, S>);
    const int seglen = walk_seglen(BH, (long long)NC * BW, resident);
    const int nseg = (BH + seglen - 1) / seglen;
    const long long items = (long long)NC * nseg * BW;
    cudaError_t e = launch_pdl(maxpool_bwd_walk_kernel<K, S>, dim3(unsigned((items + kWalkThreads - 1) / kWalkThreads)),
                               dim3(kWalkThreads), 0, st, dy, idx, dx, H, W, P, Q, BH, seglen, FastDiv(uint32_t(BW)),
                               FastDiv(uint32_t(nseg)), int(items));
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

// Blocks per SM for a staged kernel using `smem` bytes of dynamic shared memory.
static int staged_grid(int groups, size_t smem, int max_per_sm = 4)
{
    static std::atomic<bool> attr_set{false};   // set once; racing setters are harmless
    if (!attr_set) {
        cudaFuncSetAttribute(maxpool_fwd_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
        attr_set = true;
    }
    int per_sm = int((200 * 1024) / (smem + 1024));
    if (per_sm > max_per_sm) per_sm = max_per_sm;
    if (per_sm < 1) per_sm = 1;
    const int cap = per_sm * sm_count();
    return groups < cap ? groups : cap;
}

cudaError_t launch_maxpool_fwd(int N, int C, int H, int W, int k, int s, int P, int Q, const float* x, float* y,
                               int32_t* idx, cudaStream_t st)
{
    const int NC = N * C;
    const int HW = H * W;
    if (k == 3 && s == 2) return launch_pool_fwd_walk<3, 2>(NC, H, W, P, Q, x, y, idx, st);
    if (k == 2 && s == 2) return launch_pool_fwd_walk<2, 2>(NC, H, W, P, Q, x, y, idx, st);
    if (HW + 4 <= kPoolStageFloats) {
        const int ppb = (kPoolStageFloats - 4) / HW < 64 ? (kPoolStageFloats - 4) / HW : 64;
        const int stage = (ppb * HW + 4 + 3) & ~3;   // floats per buffer (room for the 16-byte shift)
        const size_t smem = 2 * size_t(stage) * sizeof(float);
        const int groups = (NC + ppb - 1) / ppb;
        maxpool_fwd_staged_kernel<<<staged_grid(groups, smem), kPoolThreads, smem, st>>>(
            x, y, idx, NC, H, W, k, s, P, Q, ppb, stage, FastDiv(P * Q), FastDiv(Q), device_error_word());
        note_launch();
        return cudaGetLastError();
    }
    const long long total = (long long)N * C * P * Q;
    maxpool_fwd_kernel<<<grid_for(total, 256), 256, 0, st>>>(x, y, idx, H, W, k, s, FastDiv(Q), FastDiv(P),
                                                             int(total));
    note_launch();
    return cudaGetLastError();
}

// Max pooling backward as a gather: dx[i] = sum, over the windows (ascending
// oh, then ow) that contain i and whose saved index is i, of their gradient.

__global__ void maxpool_bwd_kernel(const float* __restrict__ dy, const int32_t* __restrict__ idx,
                                   float* __restrict__ dx, int k, int S, int P, int Q, FastDiv f_w, FastDiv f_h,
                                   int total)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        uint32_t r1, w, nc, h;
        f_w.divmod(uint32_t(t), r1, w);
        f_h.divmod(r1, nc, h);
        // windows with oh*S <= h < oh*S + k
        const int oh_lo = int(h) - k + 1 <= 0 ? 0 : (int(h) - k + S) / S;
        const int oh_hi = min(int(h) / S, P - 1);
        const int ow_lo = int(w) - k + 1 <= 0 ? 0 : (int(w) - k + S) / S;
        const int ow_hi = min(int(w) / S, Q - 1);
        float acc = 0.f;
        for (int oh = oh_lo; oh <= oh_hi; ++oh)
            for (int ow = ow_lo; ow <= ow_hi; ++ow) {
                const int o = (int(nc) * P + oh) * Q + ow;
                if (__ldg(idx + o) == t) acc += __ldg(dy + o);
            }
        dx[t] = acc;
    }
}

cudaError_t launch_maxpool_bwd(int N, int C, int H, int W, int k, int s, int P, int Q, const float* dy,
                               const int32_t* idx, float* dx, cudaStream_t st)
{
    const int NC = N * C;
    const int PQ = P * Q;
    if (k == 3 && s == 2) return launch_pool_bwd_walk<3, 2>(NC, H, W, P, Q, dy, idx, dx, st);
    if (k == 2 && s == 2) return launch_pool_bwd_walk<2, 2>(NC, H, W, P, Q, dy, idx, dx, st);
    if (PQ + 4 <= kPoolStageFloats / 2 && s >= 1 && s <= 3) {
        const int ppb = (kPoolStageFloats / 2 - 4) / PQ < 64 ? (kPoolStageFloats / 2 - 4) / PQ : 64;
        const int stage = (ppb * PQ + 4 + 3) & ~3;
        const size_t smem = 4 * size_t(stage) * sizeof(float);
        const int groups = (NC + ppb - 1) / ppb;
        const int BH = (H + s - 1) / s, BW = (W + s - 1) / s;
        const int grid = staged_grid(groups, smem, 3);  // three blocks per SM (register bound)
        const FastDiv f_blk{uint32_t(BH * BW)}, f_bw{uint32_t(BW)};
        auto run = [&](auto kern) {
            kern<<<grid, kPoolThreads, smem, st>>>(dy, idx, dx, NC, H, W, k, P, Q, ppb, stage, BH, BW, f_blk, f_bw,
                                                   device_error_word());
        };
        switch (s) {
        case 1: run(maxpool_bwd_staged_kernel<1>); break;
        case 2: run(maxpool_bwd_staged_kernel<2>); break;
        default: run(maxpool_bwd_staged_kernel<3>); break;
        }
        note_launch();
        return cudaGetLastError();
    }
    const long long total = (long long)N * C * H * W;
    maxpool_bwd_kernel<<<grid_for(total, 256), 256, 0, st>>>(dy, idx, dx, k, s, P, Q, FastDiv(W), FastDiv(H),
                                                             int(total));
    note_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SGD: p = p - lr * clamp(g, -clip, clip), one rounding per operation.

__device__ __forceinline__ float sgd_one(float p, float g, float lr, float clip)
{
    const float c = fminf(fmaxf(g, -clip), clip);
    return __fsub_rn(p, __fmul_rn(lr, c));
}

__global__ void sgd_kernel(float* __restrict__ p, const float* __restrict__ g, long long n4, long long count, float lr,
                           float clip)
{
    griddep_wait();
    griddep_launch();
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    for (long long i = tid; i < n4; i += stride) {
        float4 pv = reinterpret_cast<float4*>(p)[i];
        const float4 gv = __ldg(reinterpret_cast<const float4*>(g) + i);
        pv.x = sgd_one(pv.x, gv.x, lr, clip);
        pv.y = sgd_one(pv.y, gv.y, lr, clip);
        pv.z = sgd_one(pv.z, gv.z, lr, clip);
        pv.w = sgd_one(pv.w, gv.w, lr, clip);
        reinterpret_cast<float4*>(p)[i] = pv;
    }
    for (long long i = n4 * 4 + tid; i < count; i += stride) p[i] = sgd_one(p[i], __ldg(g + i), lr, clip);
}

cudaError_t launch_sgd(int64_t count, float lr, float clip, float* p, const float* g, cudaStream_t st)
{
    if (count == 0) return cudaSuccess;
    const long long n4 = count / 4;
    cudaError_t e = launch_pdl(sgd_kernel, dim3(grid_for(n4 > 0 ? n4 : 1, 256)), dim3(256), 0, st, p, g, n4, count, lr,
                               clip);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bias gradient: db[k] = sum over (n, oh, ow) of dy[n, k, oh, ow].
// One cluster of CS CTAs (T threads each) per filter k.  CTA r of the cluster
// sums the planes (n, k) of images n = r, r + CS, ...: thread t takes elements
// t, t + T, ... of that list of planes, sixteen loads in flight at a time,
// into four accumulators; the position in the list is advanced incrementally,
// without divisions.  The accumulators, the warp lanes, the warps and finally
// the cluster's CTAs (read through distributed shared memory by CTA 0) are
// combined in fixed orders, so the result is deterministic; no atomics.
// (T, CS) are chosen per call so that the grid is about one wave of resident
// CTAs: a call on small planes (13 x 13) moves only 22-33 MB, and a second,
// partial wave of short CTAs cost as much as the first.

constexpr int kBiasMaxThreads = 512;
constexpr int kBiasMaxCluster = 8;
constexpr int kBiasBatch = 16;   // loads in flight per thread

__global__ void __launch_bounds__(kBiasMaxThreads, 3)
    bias_grad_kernel(const float* __restrict__ dy, float* __restrict__ db, int N, int K, int PQ)
{
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ float warp_part[kBiasMaxThreads / 32];
    __shared__ float cta_part;
    griddep_wait();
    griddep_launch();
    const int T = int(blockDim.x);
    const int cs = int(cluster.num_blocks());
    const int rank = int(cluster.block_rank());
    const int k = blockIdx.x / cs;
    const int images = (N - rank + cs - 1) / cs;          // planes this CTA sums
    const int img_stride = cs * K * PQ;                   // elements between its consecutive planes
    const int step_n = T / PQ, step_e = T % PQ;
    int nl = int(threadIdx.x) / PQ, e = int(threadIdx.x) % PQ;
    unsigned off = unsigned((rank * K + k) * PQ + nl * img_stride + e);   // may run past the end once nl >= images: never loaded
    float part[4] = {0.f, 0.f, 0.f, 0.f};
    while (nl < images) {
        float v[kBiasBatch];
#pragma unroll
        for (int u = 0; u < kBiasBatch; ++u) {
            v[u] = nl < images ? __ldg(dy + off) : 0.f;
            nl += step_n;
            e += step_e;
            off += unsigned(step_n * img_stride + step_e);
            if (e >= PQ) {
                e -= PQ;
                ++nl;
                off += unsigned(img_stride - PQ);
            }
        }
#pragma unroll
        for (int u = 0; u < kBiasBatch; ++u) part[u & 3] += v[u];
    }
    float acc = (part[0] + part[1]) + (part[2] + part[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < T / 32; ++i) t += warp_part[i];
        cta_part = t;
        if (cs == 1) db[k] = t;   // launched without a cluster
    }
    if (cs == 1) return;
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
        float t = 0.f;
        for (int r = 0; r < cs; ++r) t += *cluster.map_shared_rank(&cta_part, r);
        db[k] = t;
    }
    cluster.sync();   // keep every CTA's shared memory alive until rank 0 has read it
}

// CTAs of `threads` threads of bias_grad_kernel resident on the GPU at once.
static int bias_resident(int threads)
{
    static std::atomic<int> cached[2] = {0, 0};
    std::atomic<int>& c = cached[threads == kBiasMaxThreads ? 1 : 0];
    int r = c.load();
    if (r > 0) return r;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bias_grad_kernel, threads, 0) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        per_sm = (2048 / threads) / 2;
    }
    r = per_sm * sm_count();
    c.store(r);
    return r;
}

struct BiasPlan {
    int threads, cluster;
};

// Of 512- and 256-thread CTAs, the (threads, cluster size) whose grid fills
// its last wave of resident CTAs best (ties to 512); a cluster is at most 8
// CTAs, at most one per image, and no larger than gives each thread 8
// elements.  AlexNet batch 128: conv1 (64 filters, 55 x 55) 512 x 8; conv2
// (192, 27 x 27) 512 x 3; conv3 (384, 13 x 13) 256 x 3; conv4/5 (256) 512 x 2.
static BiasPlan plan_bias(const ConvDims& d)
{
    const long long per_k = (long long)d.N * d.P * d.Q;
    BiasPlan best{kBiasMaxThreads, 1};
    double best_fill = -1.0;
    for (int threads : {kBiasMaxThreads, kBiasMaxThreads / 2}) {
        const long long resident = bias_resident(threads);
        long long cs = resident / d.K;
        const long long by_work = per_k / (8LL * threads);
        if (cs > by_work) cs = by_work;
        if (cs > kBiasMaxCluster) cs = kBiasMaxCluster;
        if (cs > d.N) cs = d.N;
        if (cs < 1) cs = 1;
        const long long ctas = (long long)d.K * cs;
        const long long waves = (ctas + resident - 1) / resident;
        const double fill = double(ctas) / double(waves * resident);
        if (fill > best_fill + 1e-9) {
            best_fill = fill;
            best = BiasPlan{threads, int(cs)};
        }
    }
    return best;
}

cudaError_t launch_bias_grad(const ConvDims& d, const float* dy, float* db, cudaStream_t st)
{
    const BiasPlan bp = plan_bias(d);
    cudaError_t e = launch_pdl_cluster(bias_grad_kernel, dim3(unsigned(d.K * bp.cluster)), dim3(unsigned(bp.threads)), 0,
                                       st, bp.cluster, dy, db, d.N, d.K, d.P * d.Q);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
