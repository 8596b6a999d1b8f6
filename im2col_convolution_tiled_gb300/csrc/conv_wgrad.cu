// conv_wgrad.cu -- filter gradient of the page "DirectCompute Neural Network
// Engine", section "Convolution: The im2col Approach" (backward: grad_reshaped
// x im2col_matrix^T), as an implicit GEMM on the tcgen05 tensor cores:
//
//   dW[k, crs] = sum_j G[k, j] * col[crs, j],   j = (n, oh, ow)
//
// Rows of the accumulator are filter taps crs (A = the column matrix,
// regathered from x), columns are filters k (B = G, read straight from dy in
// NCHW: conv_grad_reshape is only an index map).  The reduction over j is long
// (batch*outH*outW) and the output small, so j is split into contiguous ranges
// spread over the SMs; each range writes its own partial tile and a second
// kernel adds the partials in range order -- a fixed summation order, so the
// result is deterministic.  Each range's tensor-core accumulation chain is
// bounded by its length.
//
// The A operand (column matrix) is gathered ChunkFast: a thread holds 4
// consecutive j of 8 rows, so 8 lanes read 32 consecutive pixels of one row.
// The B operand G is dy itself, re-laid once per call as pre-split hi/lo
// tiles (one streaming pass over dy) and fed by bulk copies, so the producers
// spend their issue slots on the gather that needs them.
#include "conv_common.cuh"

namespace cb200 {

// INTERIOR: no padding and every window inside the image ((P-1)*S + R <= H,
// likewise along W), so the gather tests only the end of the reduction -- the
// space-to-depth form of AlexNet conv1 (X' 57 x 57, 3 x 3 taps, 55 x 55
// outputs).
template <int BN, bool INTERIOR = false>
struct ConvWgradProb {
    static constexpr bool kBBulk = true;
    int terms = 3;   // tensor-core products per K step: 3 (3xTF32) or 1 (TF32)
    static constexpr int kGroups = 2;
    static constexpr Map kAMap = Map::ChunkFast;
    static constexpr Map kBMap = Map::ChunkFast;   // unused (bulk)

    const float* x;
    const float* bimg;   // G as pre-split tiles
    float* out;          // dW (splits == 1) or partials [split][K][CRS]
    int C, H, W, K, R, S, pad, P, Q;
    int PQ, NPQ, CRS, HW, CHW;
    FastDiv f_pq, f_q, f_rr, f_r;
    int m_tiles, n_tiles, k_stages, splits, ks_per_split;
    // Space-to-depth form (s2dS > 1): x is X', the geometry above is the
    // derived stride-1 convolution, and the rows are the ORIGINAL taps
    // (c, r, q), CRS = C_orig * R_orig^2, decoded by f_rr / f_r over R_orig and
    // read from X' channel (c*s2dS + r % s2dS)*s2dS + q % s2dS, tap
    // (r / s2dS, q / s2dS).
    int s2dS = 0;

    __device__ int num_tiles() const { return m_tiles * n_tiles * splits; }
    __device__ Tile tile(int t) const
    {
        const int mn = m_tiles * n_tiles;
        const int split = t / mn;
        const int rem = t % mn;
        Tile r;
        r.n0 = (rem % n_tiles) * BN;
        r.m0 = (rem / n_tiles) * kBM;
        r.ks0 = split * ks_per_split;
        r.ks1 = min(r.ks0 + ks_per_split, k_stages);
        r.grp = split;
        return r;
    }

    // Rows (taps) of this thread: (tid / 8) + 16 p.
    struct AState {
        int rowoff[8];   // c*H*W + r*W + q
        int rq[8];       // (r << 16) | q, or a sentinel that is never inside
    };
    __device__ AState a_setup(const Tile& tl, int tid) const
    {
        AState s;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int crs = tl.m0 + (tid >> 3) + 16 * p;
            if (crs < CRS) {
                uint32_t c, rem, r, q;
                f_rr.divmod(uint32_t(crs), c, rem);
                f_r.divmod(rem, r, q);
                if (s2dS > 1) {
                    const uint32_t S2 = uint32_t(s2dS);
                    c = (c * S2 + r % S2) * S2 + q % S2;
                    r /= S2;
                    q /= S2;
                }
                s.rowoff[p] = int(c) * HW + int(r) * W + int(q);
                s.rq[p] = int((r << 16) | q);
            } else {
                s.rowoff[p] = 0;
                s.rq[p] = 0x7FFF0000;
            }
        }
        return s;
    }

    __device__ void load_a(const AState& s, const Tile&, int ks, int tid, float (&v)[32]) const
    {
        // Pixels j0..j0+3 of this thread's chunk.
        const int j0 = ks * kBK + 4 * (tid & 7);
        int jbase[4], jh[4], jw[4];
        if constexpr (INTERIOR) {
            uint32_t n, pq, oh, ow;
            f_pq.divmod(uint32_t(j0 < NPQ ? j0 : 0), n, pq);
            f_q.divmod(pq, oh, ow);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                jbase[e] = j0 + e < NPQ ? int(n) * CHW + int(oh) * S * W + int(ow) * S : -1;
                if (++ow == uint32_t(Q)) {
                    ow = 0;
                    if (++oh == uint32_t(P)) { oh = 0; ++n; }
                }
            }
#pragma unroll
            for (int p = 0; p < 8; ++p)
#pragma unroll
                for (int e = 0; e < 4; ++e) v[4 * p + e] = ldg_keep_if(x + (jbase[e] + s.rowoff[p]), jbase[e] >= 0);
            return;
        }
        {
            uint32_t n, pq, oh, ow;
            f_pq.divmod(uint32_t(j0 < NPQ ? j0 : 0), n, pq);
            f_q.divmod(pq, oh, ow);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (j0 + e < NPQ) {
                    jh[e] = int(oh) * S - pad;
                    jw[e] = int(ow) * S - pad;
                    jbase[e] = int(n) * CHW + jh[e] * W + jw[e];
                } else {
                    jh[e] = -(1 << 24);
                    jw[e] = 0;
                    jbase[e] = 0;
                }
                if (++ow == uint32_t(Q)) {
                    ow = 0;
                    if (++oh == uint32_t(P)) { oh = 0; ++n; }
                }
            }
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = jh[e] + (s.rq[p] >> 16);
                const int w = jw[e] + (s.rq[p] & 0xFFFF);
                v[4 * p + e] = ldg_keep_if(x + (jbase[e] + s.rowoff[p]), unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W));
            }
        }
    }

    struct BState {};
    __device__ BState b_setup(const Tile&, int) const { return {}; }
    __device__ void load_b(const BState&, const Tile&, int, int, int, float (&)[32]) const {}
    __device__ const float* b_image(const Tile& tl, int ks) const
    {
        return bimg + (size_t(tl.n0 / BN) * k_stages + ks) * 2 * size_t(BN) * kBK;
    }

    struct EState {
        float* o;   // out + crs, filter stride CRS
        bool valid;
    };
    __device__ EState e_setup(const Tile& tl, int row) const
    {
        EState e;
        const int crs = tl.m0 + row;
        e.valid = crs < CRS;
        e.o = out + size_t(tl.grp) * K * CRS + (e.valid ? crs : 0);
        return e;
    }

    __device__ void store(const EState& e, const Tile& tl, int, int c, const uint32_t (&r)[32]) const
    {
        if (!e.valid) return;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int k = tl.n0 + c + i;
            if (k < K) e.o[size_t(k) * CRS] = __uint_as_float(r[i]);
        }
    }
};

// B[k, j] = G[k, j] = dy[n, k, pq] with j = n*PQ + pq (conv_grad_reshape).
struct GradGen {
    const float* dy;
    int K, PQ;
    FastDiv f_pq;
    __device__ float operator()(int k, int j) const
    {
        uint32_t n, pq;
        f_pq.divmod(uint32_t(j), n, pq);
        return __ldg(dy + (size_t(n) * K + k) * PQ + pq);
    }
    // j0 .. j0+3 with one division: offsets step by one pixel, and by
    // (K - 1) * PQ more where the run crosses into the next image (dy has
    // fewer than 2^31 elements, so 32-bit offsets hold)
    __device__ void load4(int k, int j0, int J, float (&v)[4]) const
    {
        uint32_t n, pq;
        f_pq.divmod(uint32_t(j0 < J ? j0 : 0), n, pq);
        uint32_t off = (n * uint32_t(K) + uint32_t(k)) * uint32_t(PQ) + pq;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[e] = j0 + e < J ? __ldg(dy + off) : 0.f;
            ++off;
            if (++pq == uint32_t(PQ)) {
                pq = 0;
                off += uint32_t(K - 1) * uint32_t(PQ);
            }
        }
    }
};

// The same with the ReLU gradient applied as dy is read (nn_relu_grad):
// G[k, j] = dy[n, k, pq] * (mask[n, k, pq] > 0), mask shaped like dy.
struct GradMaskGen {
    const float* dy;
    const float* mask;
    int K, PQ;
    FastDiv f_pq;
    __device__ float operator()(int k, int j) const
    {
        uint32_t n, pq;
        f_pq.divmod(uint32_t(j), n, pq);
        const size_t at = (size_t(n) * K + k) * PQ + pq;
        return __ldg(dy + at) * relu_gate(__ldg(mask + at));
    }
    __device__ void load4(int k, int j0, int J, float (&v)[4]) const
    {
        uint32_t n, pq;
        f_pq.divmod(uint32_t(j0 < J ? j0 : 0), n, pq);
        uint32_t off = (n * uint32_t(K) + uint32_t(k)) * uint32_t(PQ) + pq;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[e] = j0 + e < J ? __ldg(dy + off) * relu_gate(__ldg(mask + off)) : 0.f;
            ++off;
            if (++pq == uint32_t(PQ)) {
                pq = 0;
                off += uint32_t(K - 1) * uint32_t(PQ);
            }
        }
    }
};

// out[row] = sum of rowsum[row * blocks + i] over the blocks i: one warp per
// row (warp `wid` of the grid), lane l adding blocks l, l + 32, ... in order,
// then a fixed shuffle tree (deterministic).
__device__ __forceinline__ void rowsum_final_warp(const float* __restrict__ rowsum, int blocks, int row,
                                                  float* __restrict__ out)
{
    const int lane = threadIdx.x & 31;
    const float* src = rowsum + size_t(row) * blocks;
    float acc = 0.f;
    for (int i = lane; i < blocks; i += 32) acc += __ldg(src + i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) out[row] = acc;
}

__global__ void rowsum_final_kernel(const float* __restrict__ rowsum, int blocks, int rows, float* __restrict__ out)
{
    griddep_wait();
    griddep_launch();
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;   // whole warps leave together
    rowsum_final_warp(rowsum, blocks, row, out);
}

// dW[i] = sum over split s (ascending) of part[s][i].  With db non-null the
// grid's first warps also finish the bias gradient (rowsum_final's work, one
// warp per filter row), saving that launch.
__global__ void wgrad_reduce_kernel(const float* __restrict__ part, int splits, long long count, float* __restrict__ dw,
                                    const float* __restrict__ rowsum, int rs_blocks, int rows, float* __restrict__ db)
{
    griddep_wait();
    griddep_launch();
    if (db) {
        const int wid = int(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
        const int nw = int(gridDim.x) * (blockDim.x >> 5);
        for (int row = wid; row < rows; row += nw) rowsum_final_warp(rowsum, rs_blocks, row, db);
    }
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) acc += __ldg(part + s * count + i);
        dw[i] = acc;
    }
}

// Space-to-depth form (stride S > 1, at most 16 channels): the filter
// gradient of the stride-1 convolution over S x S super-pixels
//   X'[n, c', hh, ww] = x[n, c, S*hh + a - pad, S*ww + b - pad],  c' = c*S*S + a*S + b
// with T = ceil(R / S) taps (see the forward's space-to-depth form), whose
// column-matrix gather reads X' with unit stride instead of x with stride S;
// then dW[k, c, r, s] = dW'[k, (c, r % S, s % S), r / S, s / S].  The GEMM's
// rows are the original taps (c, r, s), each gathering its X' channel and tap:
// the taps past the filter (S*tr + a >= R), zero in W', are not computed
// (AlexNet conv1: 363 rows, three tiles, instead of 48 * 3 * 3 = 432, four).
// X' is written NCHW (rows of ww contiguous) for the gather.
struct WgradS2d {
    bool use;
    int T, Cs, Hs, Ws;
    ConvDims d2;   // the derived stride-1 convolution over X'
};

static WgradS2d plan_wgrad_s2d(const ConvDims& d)
{
    WgradS2d w{};
    w.use = false;
    if (d.S < 2 || d.C > 16) return w;
    w.T = (d.R + d.S - 1) / d.S;
    w.Cs = d.C * d.S * d.S;
    if (w.Cs < 17 || w.Cs > 128) return w;
    w.Hs = d.P + w.T - 1;
    w.Ws = d.Q + w.T - 1;
    if ((long long)d.N * w.Cs * w.Hs * w.Ws >= (1LL << 31)) return w;
    w.d2 = d;
    w.d2.C = w.Cs;
    w.d2.H = w.Hs;
    w.d2.W = w.Ws;
    w.d2.R = w.T;
    w.d2.S = 1;
    w.d2.pad = 0;
    w.use = true;
    return w;
}

struct WgradPlan {
    int bn, m_tiles, n_tiles, k_stages, splits, ks_per_split;
};

// rows: the GEMM's row count (taps of the original convolution)
static WgradPlan plan_wgrad(const ConvDims& d, int rows)
{
    WgradPlan pl;
    pl.bn = pick_conv_bn(d.K, &pl.n_tiles);
    const int CRS = rows;
    const long long NPQ = (long long)d.N * d.P * d.Q;
    pl.m_tiles = (CRS + kBM - 1) / kBM;
    pl.k_stages = int((NPQ + kBK - 1) / kBK);
    const int mn = pl.m_tiles * pl.n_tiles;
    // The persistent grid runs ceil(tiles / SMs) rounds of tiles; a round
    // costs its range length plus a fixed per-tile overhead (pipeline fill,
    // last epilogue).  Pick the split count with the least total, fewest
    // splits on a tie: a 13-tile GEMM on 152 SMs takes 11 splits (one round
    // of 143 tiles), not 12 (156 tiles: a second round for 4 of them).
    const int min_stages = 16;                     // keep each range worth a tile
    const int tile_overhead = 16;                  // in stages
    const long long P = sm_count();
    const int max_splits = pl.k_stages / min_stages > 1 ? pl.k_stages / min_stages : 1;
    long long best = -1;
    pl.splits = 1;
    pl.ks_per_split = pl.k_stages;
    for (int s = 1; s <= max_splits; ++s) {
        const int per = (pl.k_stages + s - 1) / s;
        const int ns = (pl.k_stages + per - 1) / per;   // no empty range
        const long long rounds = ((long long)mn * ns + P - 1) / P;
        const long long cost = rounds * (per + tile_overhead);
        if (best < 0 || cost < best) {
            best = cost;
            pl.splits = ns;
            pl.ks_per_split = per;
        }
    }
    return pl;
}

// Workspace: the G image, then (split-K only) the partial tiles.
static size_t wgrad_image_floats(const ConvDims& d, const WgradPlan& pl)
{
    return bimage_floats(d.K, d.N * d.P * d.Q, pl.bn);
}

static size_t xs2d_floats(const ConvDims& d, const WgradS2d& w)
{
    return w.use ? (size_t(d.N) * w.Cs * w.Hs * w.Ws + 63) & ~size_t(63) : 0;
}

static size_t wgrad_part_floats(const ConvDims& d, const WgradPlan& pl)
{
    return pl.splits > 1 ? size_t(pl.splits) * d.K * d.C * d.R * d.R : 0;
}

// Row-sum partials of the G image (the bias gradient of conv_bwd_filter_bias).
static size_t wgrad_rowsum_floats(const ConvDims& d)
{
    return size_t(d.K) * bimage_grid_x(d.N * d.P * d.Q);
}

// Workspace: [X' (space-to-depth form)] [the G image] [split-K partial tiles]
// [row-sum partials for the bias gradient].
size_t conv_wgrad_ws(const ConvDims& d)
{
    const WgradS2d w = plan_wgrad_s2d(d);
    const ConvDims& g = w.use ? w.d2 : d;
    WgradPlan pl = plan_wgrad(g, d.C * d.R * d.R);
    return (xs2d_floats(d, w) + wgrad_image_floats(g, pl) + wgrad_part_floats(d, pl) + wgrad_rowsum_floats(d)) *
           sizeof(float);
}

// d: the convolution the GEMM runs (the derived one in the space-to-depth
// form, whose rows are then orig's taps); ws: its image and partials.
// With db non-null the G image pass also sums each row of G (the bias
// gradient) into row-sum partials, added in block order by rowsum_final_kernel.
template <int BN, bool INTERIOR = false>
static cudaError_t run_wgrad(const ConvDims& d, const WgradPlan& pl, const float* x, const float* dy, float* dw,
                             void* ws, cudaStream_t st, const ConvDims* orig, float* db, const float* mask)
{
    ConvWgradProb<BN, INTERIOR> p;
    p.terms = math_terms();
    const ConvDims& o = orig ? *orig : d;   // the convolution whose filter gradient is written
    float* img = static_cast<float*>(ws);
    float* part = img + wgrad_image_floats(d, pl);
    float* rowsum = part + wgrad_part_floats(o, pl);
    p.x = x;
    p.bimg = img;
    p.out = pl.splits > 1 ? part : dw;
    p.C = d.C; p.H = d.H; p.W = d.W; p.K = d.K; p.R = d.R; p.S = d.S; p.pad = d.pad; p.P = d.P; p.Q = d.Q;
    p.PQ = d.P * d.Q;
    p.NPQ = d.N * p.PQ;
    p.CRS = o.C * o.R * o.R;
    p.HW = d.H * d.W;
    p.CHW = d.C * p.HW;
    p.f_pq = FastDiv(p.PQ);
    p.f_q = FastDiv(d.Q);
    p.f_rr = FastDiv(o.R * o.R);
    p.f_r = FastDiv(o.R);
    p.s2dS = orig ? orig->S : 0;
    p.m_tiles = pl.m_tiles;
    p.n_tiles = pl.n_tiles;
    p.k_stages = pl.k_stages;
    p.splits = pl.splits;
    p.ks_per_split = pl.ks_per_split;
    cudaError_t e = mask ? build_bimage(GradMaskGen{dy, mask, d.K, p.PQ, FastDiv(uint32_t(p.PQ))}, d.K, p.NPQ, BN,
                                        img, st, db ? rowsum : nullptr)
                         : build_bimage(GradGen{dy, d.K, p.PQ, FastDiv(uint32_t(p.PQ))}, d.K, p.NPQ, BN, img, st,
                                        db ? rowsum : nullptr);
    if (e != cudaSuccess) return e;
    if (db && pl.splits == 1) {   // with split partials the reduce kernel finishes db
        e = launch_pdl(rowsum_final_kernel, dim3((d.K + 7) / 8), dim3(256), 0, st, rowsum, bimage_grid_x(p.NPQ), d.K, db);
        if (e != cudaSuccess) return e;
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    e = launch_tc_gemm<ConvWgradProb<BN, INTERIOR>, BN>(p, p.m_tiles * p.n_tiles * p.splits, device_error_word(), st);
    if (e != cudaSuccess) return e;
    if (pl.splits == 1) return e;
    const long long count = (long long)d.K * p.CRS;
    long long blocks = (count + 255) / 256;
    if (blocks > 8LL * sm_count()) blocks = 8LL * sm_count();
    e = launch_pdl(wgrad_reduce_kernel, dim3(unsigned(blocks)), dim3(256), 0, st, part, pl.splits, count, dw,
                   static_cast<const float*>(rowsum), bimage_grid_x(p.NPQ), d.K, db);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_conv_wgrad(const ConvDims& d, const float* x, const float* dy, float* dw, void* ws,
                              cudaStream_t st, float* db, const float* mask)
{
    const WgradS2d w = plan_wgrad_s2d(d);
    const ConvDims& g = w.use ? w.d2 : d;
    const ConvDims* orig = w.use ? &d : nullptr;
    WgradPlan pl = plan_wgrad(g, d.C * d.R * d.R);
    const float* xg = x;
    void* gws = ws;
    if (w.use) {
        float* xs = static_cast<float*>(ws);
        cudaError_t e = launch_s2d_copy<false>(x, xs, d.N, d.C, d.H, d.W, d.S, d.pad, w.Hs, w.Ws, st);
        if (e != cudaSuccess) return e;
        xg = xs;
        gws = xs + xs2d_floats(d, w);
    }
    // windows that never leave the image (no padding): the gather tests only
    // the reduction's end (instantiated for the 64-wide tiles, AlexNet conv1)
    const bool interior = g.pad == 0 && (g.P - 1) * g.S + g.R <= g.H && (g.Q - 1) * g.S + g.R <= g.W;
    switch (pl.bn) {
    case 32: return run_wgrad<32>(g, pl, xg, dy, dw, gws, st, orig, db, mask);
    case 64:
        return interior ? run_wgrad<64, true>(g, pl, xg, dy, dw, gws, st, orig, db, mask)
                        : run_wgrad<64>(g, pl, xg, dy, dw, gws, st, orig, db, mask);
    case 128: return run_wgrad<128>(g, pl, xg, dy, dw, gws, st, orig, db, mask);
    case 192: return run_wgrad<192>(g, pl, xg, dy, dw, gws, st, orig, db, mask);
    default: return run_wgrad<256>(g, pl, xg, dy, dw, gws, st, orig, db, mask);
    }
}

}  // namespace cb200
