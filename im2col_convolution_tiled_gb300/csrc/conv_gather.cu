// conv_gather.cu -- the forward convolution and the input gradient of the page
// "DirectCompute Neural Network Engine", section "Convolution: The im2col
// Approach", both as one implicit GEMM on the tcgen05 tensor cores whose A
// operand is a convolution-window gather.
//
// Forward (steps 1-3: im2col, filters x columns, conv_reshape + bias):
//   D[(n, oh, ow), k] = sum_(r, q, c) x[n, c, oh*s + r - pad, ow*s + q - pad] * W[k, c, r, q]
//   y[n, k, oh, ow]   = D + b[k]
// The column matrix is the A operand, gathered straight from x (zero in the
// padding) and never stored; the filters are the B operand.
//
// Input gradient (filters^T x grad_reshaped, then col2im): col2im adds, for an
// input pixel h, the contributions of every tap r with oh*s + r - pad = h.
// Write h = a + s*hh with phase a = h mod s; then oh = hh + d with
// d = (a + pad - r) / s, so each dx pixel is
//   dx[n, c, a + s*hh, b + s*ww] = sum_(d, e, k) dy[n, k, hh + d, ww + e] * W[k, c, a + pad - s*d, b + pad - s*e]
// (terms whose tap falls outside 0..kH-1 are zero).  Taking (c, a, b) as the
// GEMM column and (n, hh, ww) as the row makes this a single GEMM for any
// stride: its A operand is again a window gather, now over dy with stride 1
// and the window d in [d_lo, d_lo + T), and the phases widen N (C * s * s
// columns) instead of splitting the problem.  Each dx element is produced by
// exactly one accumulator: col2im needs no scatter, no atomics and no column
// buffer.
//
// K order of both: tap-major, channel-fastest -- k = (tap_r * T + tap_q) * Cp + ci,
// with the channels of the gathered tensor padded to Cp: Cp = Ci when Ci is
// a multiple of 32 (a pipeline stage then holds 32 channels of ONE tap; also
// 32 when 16 < Ci < 32), and the next power of two when Ci <= 16 (a stage
// holds 32 / Cp whole taps).  The
// bounds test is then done once per tap and every element is one add and one
// load.  Any other Ci uses k = (ci * T + tap_r) * T + tap_q with a per-element
// decode shared across the warp.  The B operand (filters, rearranged and
// zero-padded to the same K order) is laid out once per call as pre-split
// hi/lo tiles and fed by bulk copies.
#include "conv_window.cuh"
#include "gemm_patch.cuh"

namespace cb200 {

// The same GEMMs on the patch-staged kernel (gemm_patch.cuh): tiles never
// straddle images, and the K order is chunk-major in 32-channel chunks (or tap
// groups when the gathered tensor has at most 16 channels).
template <int BN>
struct ConvPatchProb {
    int terms = 3;   // tensor-core products per K step: 3 (3xTF32) or 1 (TF32)
    PatchGeom pg;
    OutGeom o;
    const float* bimg;
    int n_tiles, k_stages;
    // Tail split (see plan_patch_tail): units [0, full_units) are whole tiles;
    // each later tile is cut into tail_split pieces along its channel chunks,
    // whose partial tiles go to part_buf [piece][kBM][BN] and are added by
    // tail_reduce_kernel.
    int full_units = 0, tail_split = 1;
    float* part_buf = nullptr;

    __device__ int num_tiles() const
    {
        return full_units + (pg.Nb * pg.tpi * n_tiles - full_units) * tail_split;
    }
    __device__ PatchUnit unit(int t) const
    {
        PatchUnit u{t, 0, pg.nch, -1};
        if (t >= full_units) {
            const int v = t - full_units;
            const int j = v % tail_split;
            u.tt = full_units + v / tail_split;
            u.cc0 = j * pg.nch / tail_split;
            u.cc1 = (j + 1) * pg.nch / tail_split;
            u.part = v;
        }
        return u;
    }
    __device__ Tile tile_t(int t) const
    {
        Tile r;
        r.n0 = (t % n_tiles) * BN;
        r.m0 = 0;
        r.ks0 = 0;
        r.ks1 = k_stages;
        r.grp = t % n_tiles;
        return r;
    }
    __device__ const float* b_image_t(int t, int ks) const
    {
        return bimg + (size_t(t % n_tiles) * k_stages + ks) * 2 * size_t(BN) * kBK;
    }

    using EState = typename ConvGatherProb<BN>::EState;
    __device__ EState e_setup_t(int t, int row) const
    {
        const int mt = t / n_tiles;
        const int n = mt / pg.tpi, ti = mt % pg.tpi;
        const int pix = ti * kBM + row;
        EState e;
        e.valid = pix < pg.GpGq;
        uint32_t p = 0, q = 0;
        if (e.valid) pg.f_gq.divmod(uint32_t(pix), p, q);
        const int h = int(p) * o.so - o.oo, w = int(q) * o.so - o.oo;
        e.hrem = o.Ho - h;
        e.wrem = o.Wo - w;
        e.hmin = -h;
        e.wmin = -w;
        e.opix = o.out + (ptrdiff_t(n) * o.Co * o.HoWo + ptrdiff_t(h) * o.Wo + w);
        return e;
    }
    __device__ void store(const EState& e, const Tile& tl, int row, int c0, const uint32_t (&r)[32]) const
    {
        ConvGatherProb<BN> helper;
        helper.o = o;
        helper.part_buf = part_buf;
        helper.store(e, tl, row, c0, r);
    }
    // epilogue of split trailing tile b, once its pieces are summed
    __device__ void reduce_store(int b, int row, int c0, const uint32_t (&r)[32]) const
    {
        const int tt = full_units + b;
        const Tile tl = tile_t(tt);
        store(e_setup_t(tt, row), tl, row, c0, r);
    }
};

// ---------------------------------------------------------------------------
// B operands (filters in the GEMM's K order)

// K index -> (channel of the gathered tensor, tap index) in one of the three
// orders the gathers use.
struct KDecode {
    int order;         // 0: tap-major, channels padded to Cp fastest; 1: 32-channel chunk, tap, channel; 2: channel, tap;
                       // 3: 16-channel chunk, tap, channel (the flat kernel)
    FastDiv f_cp;      // order 0: Cp
    FastDiv f_chunk;   // order 1: T*T*32; order 3: T*T*16
    FastDiv f_tt;      // order 2: T*T
    // order 1 with a half last chunk (the patch kernel's two-tap stages): from
    // K index half_k0 on, stage j holds taps 2j and 2j + 1, channels
    // half_c0 + 0..15 of each (half_k0 = INT32_MAX: none)
    int half_k0 = 0x7FFFFFFF, half_c0 = 0;
    __device__ __forceinline__ void operator()(int kk, int& c, int& tap) const
    {
        uint32_t a, b;
        if (kk >= half_k0) {
            const int rel = kk - half_k0;
            tap = 2 * (rel >> 5) + ((rel >> 4) & 1);
            c = half_c0 + (rel & 15);
        } else if (order == 0) {
            f_cp.divmod(uint32_t(kk), a, b);
            tap = int(a);
            c = int(b);
        } else if (order == 1) {
            f_chunk.divmod(uint32_t(kk), a, b);
            tap = int(b) >> 5;
            c = int(a) * 32 + (int(b) & 31);
        } else if (order == 3) {
            f_chunk.divmod(uint32_t(kk), a, b);
            tap = int(b) >> 4;
            c = int(a) * 16 + (int(b) & 15);
        } else {
            f_tt.divmod(uint32_t(kk), a, b);
            c = int(a);
            tap = int(b);
        }
    }
};

static KDecode make_kdecode(int order, int cp, int T)
{
    KDecode d{};
    d.order = order;
    d.f_cp = FastDiv(uint32_t(cp > 0 ? cp : 1));
    d.f_chunk = FastDiv(uint32_t(T * T * (order == 3 ? 16 : 32)));
    d.f_tt = FastDiv(uint32_t(T * T));
    return d;
}

struct FwdFilterGen {   // B[k, kk] = W[k, c, r, q] (0 for padded channels)
    const float* w;
    int C, R;
    KDecode dec;
    FastDiv f_r;
    __device__ float operator()(int k, int kk) const
    {
        int c, tap;
        dec(kk, c, tap);
        if (c >= C || tap >= R * R) return 0.f;
        uint32_t r, q;
        f_r.divmod(uint32_t(tap), r, q);
        return __ldg(w + ((size_t(k) * C + c) * R + r) * R + q);
    }
};

struct DgradFilterGen {   // B[(c, a, b), (d, e, kc)] = W[kc, c, a + pad' - s*d, b + pad' - s*e], pad' = pad - oo
    const float* w;
    int C, K, R, S, pad, d_lo;   // pad: pad' (the padding less the grid's phase offset)
    KDecode dec;
    FastDiv f_t, f_ss, f_s;
    __device__ float operator()(int col, int kk) const
    {
        uint32_t c, ab, a, b, td, te;
        f_ss.divmod(uint32_t(col), c, ab);
        f_s.divmod(ab, a, b);
        int kc, tap;
        dec(kk, kc, tap);
        if (kc >= K) return 0.f;
        f_t.divmod(uint32_t(tap), td, te);
        if (int(td) >= int(f_t.d)) return 0.f;   // tap past the window
        const int r = int(a) + pad - S * (d_lo + int(td));
        const int q = int(b) + pad - S * (d_lo + int(te));
        if (r < 0 || r >= R || q < 0 || q >= R) return 0.f;
        return __ldg(w + ((size_t(kc) * C + c) * R + r) * R + q);
    }
};

// The input-gradient GEMM's super-pixel grid.  Input row h is written as
// h = s*hh + a - oo with phase a in [0, s) and oo = pad mod s: the grid is
// aligned with the padding rather than with row 0.  Output row oh reaches h
// through tap r = h + pad - s*oh = s*(hh - oh + pad div s) + a, so with
// d = oh - hh every phase's taps r = a, a + s, ... < R sit at
// d = pad div s - tr, tr in [0, ceil(R / s)): one window of T = ceil(R / s)
// dy rows [d_lo, d_lo + T) serves all phases (a grid aligned with row 0
// needs up to T + 1: 4 instead of 3 for an 11-wide filter at stride 4, pad 2).
// The grid has ceil((H + oo) / s) rows.
static void dgrad_window(const ConvDims& d, int* d_lo, int* T, int* oo)
{
    *oo = d.pad % d.S;
    *T = (d.R + d.S - 1) / d.S;
    *d_lo = d.pad / d.S - *T + 1;
}

static GatherGeom make_gather(const float* in, int Nb, int Ci, int Hi, int Wi, int Gp, int Gq, int sp, int o, int T)
{
    GatherGeom g{};
    g.in = in;
    g.Ci = Ci;
    g.Hi = Hi;
    g.Wi = Wi;
    g.HiWi = Hi * Wi;
    g.CiHiWi = Ci * Hi * Wi;
    g.Gp = Gp;
    g.Gq = Gq;
    g.M = Nb * Gp * Gq;
    g.sp = sp;
    g.o = o;
    g.T = T;
    k_order(Ci, &g.mode, &g.Cp, &g.lcp);
    g.K = T * T * g.Cp;
    g.f_gpq = FastDiv(uint32_t(Gp * Gq));
    g.f_gq = FastDiv(uint32_t(Gq));
    g.f_cchunks = FastDiv(uint32_t(g.mode == 0 ? g.Cp / 32 : 1));
    g.f_tt = FastDiv(uint32_t(T * T));
    g.f_t = FastDiv(uint32_t(T));
    return g;
}

// K extent of the B image for a gather over `ci` channels: chunks of 32
// channels (patch kernel) cover every order the register-gather kernel uses
// when ci > 16; tap groups of 2^ceil(log2 ci) channels otherwise.
static int k_extent(int ci, int T)
{
    if (ci <= 16) {
        int l = 0;
        while ((1 << l) < ci) ++l;
        return T * T * (1 << l);
    }
    return T * T * ((ci + 31) / 32 * 32);
}

static int dgrad_cols(const ConvDims& d) { return d.C * d.S * d.S; }

// Tail split.  A persistent grid of P CTAs takes tiles t, t + P, ...; with
// T = q*P + r tiles (0 < r < P) the last round keeps only r SMs busy for a
// whole tile time.  Instead, the q*P leading tiles run whole and each of the
// r trailing tiles is cut along K into `split` pieces (split*r <= P, at least
// four K stages each), so the last round takes about 1/split of a tile time.
// The pieces write fp32 partial tiles; tail_reduce_kernel adds them in piece
// order (deterministic) and applies the normal epilogue.
struct TailPlan {
    int full_units, split, tail_tiles;
    size_t part_floats;
};

static TailPlan plan_tail(int tiles, int k_stages, int bn)
{
    TailPlan p{tiles, 1, 0, 0};
    const int P = sm_count();
    if (tiles <= P || tiles % P == 0) return p;
    const int rem = tiles % P;
    int split = P / rem;
    if (split > k_stages / 4) split = k_stages / 4;
    if (split < 2) return p;
    p.full_units = tiles - rem;
    p.split = split;
    p.tail_tiles = rem;
    p.part_floats = size_t(rem) * split * kBM * bn;
    return p;
}

// One CTA per (trailing tile, 32-column slice), 1024 threads: thread (row,
// g) adds, in piece order, the 16-byte column group g of its row over the
// pieces (eight threads read one row's 128 bytes: coalesced, and eight times
// the loads in flight of a thread-per-row layout).  The sums meet in shared
// memory, and the 128 row threads hand them to the problem's epilogue.
constexpr int kTailThreads = 1024;

template <class Prob, int BN>
__global__ void __launch_bounds__(kTailThreads) tail_reduce_kernel(const __grid_constant__ Prob prob)
{
    griddep_wait();
    griddep_launch();
    __shared__ float sums[kBM][33];
    const int u0 = blockIdx.x * prob.tail_split;
    const int c0 = blockIdx.y * 32;
    {
        const int row = threadIdx.x >> 3, g = threadIdx.x & 7;
        const float4* src = reinterpret_cast<const float4*>(prob.part_buf + (size_t(u0) * kBM + row) * BN + c0) + g;
        const size_t piece = size_t(kBM) * BN / 4;   // float4s between consecutive pieces
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int j = 0;
        for (; j + 4 <= prob.tail_split; j += 4) {
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = __ldg(src + (j + q) * piece);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc.x += v[q].x;
                acc.y += v[q].y;
                acc.z += v[q].z;
                acc.w += v[q].w;
            }
        }
        for (; j < prob.tail_split; ++j) {
            const float4 v = __ldg(src + j * piece);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        sums[row][4 * g] = acc.x;
        sums[row][4 * g + 1] = acc.y;
        sums[row][4 * g + 2] = acc.z;
        sums[row][4 * g + 3] = acc.w;
    }
    __syncthreads();
    if (threadIdx.x < kBM) {
        const int row = threadIdx.x;
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sums[row][i]);
        prob.reduce_store(int(blockIdx.x), row, c0, r);
    }
}

static size_t round_up_256(size_t b) { return (b + 255) & ~size_t(255); }

template <int BN>
static cudaError_t run_gather(const GatherGeom& g, const OutGeom& o, float* img, float* part, cudaStream_t st)
{
    ConvGatherProb<BN> p;
    p.terms = math_terms();
    p.g = g;
    p.o = o;
    p.bimg = img;
    p.m_tiles = (g.M + kBM - 1) / kBM;
    p.n_tiles = (o.ncols + BN - 1) / BN;
    p.k_stages = (g.K + kBK - 1) / kBK;
    const TailPlan tp = plan_tail(p.m_tiles * p.n_tiles, p.k_stages, BN);
    p.full_units = tp.full_units;
    p.tail_split = tp.split;
    p.part_buf = part;
    const int units = tp.full_units + tp.tail_tiles * tp.split;
    cudaError_t e = launch_tc_gemm<ConvGatherProb<BN>, BN>(p, units, device_error_word(), st);
    if (e != cudaSuccess || tp.tail_tiles == 0) return e;
    e = launch_pdl(tail_reduce_kernel<ConvGatherProb<BN>, BN>, dim3(unsigned(tp.tail_tiles), unsigned(BN / 32)),
                   dim3(kTailThreads), 0, st, p);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

static cudaError_t dispatch_gather(int bn, const GatherGeom& g, const OutGeom& o, float* img, float* part,
                                   cudaStream_t st)
{
    switch (bn) {
    case 32: return run_gather<32>(g, o, img, part, st);
    case 64: return run_gather<64>(g, o, img, part, st);
    case 128: return run_gather<128>(g, o, img, part, st);
    case 192: return run_gather<192>(g, o, img, part, st);
    default: return run_gather<256>(g, o, img, part, st);
    }
}

static PatchGeom make_patch(const float* in, int Nb, int Ci, int Hi, int Wi, int Gp, int Gq, int sp, int o, int T)
{
    PatchGeom pg{};
    pg.in = in;
    pg.Nb = Nb;
    pg.Ci = Ci;
    pg.Hi = Hi;
    pg.Wi = Wi;
    pg.HiWi = Hi * Wi;
    pg.CiHiWi = Ci * Hi * Wi;
    pg.total = (long long)Nb * Ci * Hi * Wi;
    pg.Gp = Gp;
    pg.Gq = Gq;
    pg.GpGq = Gp * Gq;
    pg.tpi = (pg.GpGq + kBM - 1) / kBM;
    pg.sp = sp;
    pg.o = o;
    pg.T = T;
    if (Ci <= 16) {
        int l = 0;
        while ((1 << l) < Ci) ++l;
        pg.mode = 1;
        pg.lcp = l;
        pg.Cp = 1 << l;
        pg.nch = 1;
        pg.spc = (T * T * pg.Cp + kBK - 1) / kBK;
        pg.pc = Ci;
    } else {
        pg.mode = 0;
        pg.lcp = 0;
        pg.Cp = (Ci + 31) / 32 * 32;
        pg.nch = pg.Cp / 32;
        pg.spc = T * T;
        pg.pc = 32;
    }
    pg.half = 0;
    pg.spch = pg.spc;
    pg.f_gq = FastDiv(uint32_t(Gq));
    pg.f_t = FastDiv(uint32_t(T));
    return pg;
}

// Tensor-map form: a last chunk of at most 16 channels takes two taps per
// stage (AlexNet conv1's space-to-depth forward: 48 channels, 2 chunks of 9
// taps -> 9 + 5 stages instead of 18).
static void set_half_chunk(PatchGeom& pg)
{
    const int last = pg.Ci - 32 * (pg.nch - 1);
    if (pg.mode == 0 && last <= 16 && pg.T * pg.T >= 2) {
        pg.half = 1;
        pg.spch = (pg.T * pg.T + 1) / 2;
    }
}

// The patch kernel's K order decode (matching set_half_chunk).
static KDecode patch_kdecode(const PatchGeom& pg)
{
    KDecode dec = make_kdecode(pg.mode == 0 ? 1 : 0, pg.Cp, pg.T);
    if (pg.half) {
        dec.half_k0 = (pg.nch - 1) * pg.spc * kBK;
        dec.half_c0 = (pg.nch - 1) * 32;
    }
    return dec;
}

static int patch_kstages(const PatchGeom& pg) { return pg.stages_range(0, pg.nch); }

static int patch_capacity(int bn)
{
    switch (bn) {
    case 32: return PatchCfg<32>::kPatchFloats;
    case 64: return PatchCfg<64>::kPatchFloats;
    case 128: return PatchCfg<128>::kPatchFloats;
    default: return 0;
    }
}

constexpr int kShortTileStages = 48;   // K stages per tile at or below which 64-wide tiles double-buffer

// Tail split of the patch kernel, by channel chunks.  Worth a reduce launch
// only when the grid runs few rounds of tiles (a round is then a large share
// of the time): AlexNet conv2's input gradient has 768 tiles, five rounds on
// 152 SMs plus 8 tiles, whose round the split cuts to a sixth.
constexpr int kPatchTailMaxRounds = 8;

static TailPlan plan_patch_tail(const PatchGeom& pg, int ncols, int bn)
{
    const int n_tiles = (ncols + bn - 1) / bn;
    const int tiles = pg.Nb * pg.tpi * n_tiles;
    TailPlan p{tiles, 1, 0, 0};
    const int P = sm_count();
    if (tiles <= P || tiles % P == 0 || tiles / P >= kPatchTailMaxRounds) return p;
    const int rem = tiles % P;
    int split = P / rem;
    if (split > pg.nch) split = pg.nch;
    if (split < 2) return p;
    p.full_units = tiles - rem;
    p.split = split;
    p.tail_tiles = rem;
    p.part_floats = size_t(rem) * split * kBM * bn;
    return p;
}

// part: room for plan_patch_tail's partial tiles, or null (no split)
template <int BN, bool TMA>
static cudaError_t run_patch(const PatchGeom& pg, const OutGeom& o, float* img, float* part, cudaStream_t st)
{
    ConvPatchProb<BN> p;
    p.terms = math_terms();
    p.pg = pg;
    p.o = o;
    p.bimg = img;
    p.n_tiles = (o.ncols + BN - 1) / BN;
    p.k_stages = patch_kstages(pg);
    TailPlan tp{pg.Nb * pg.tpi * p.n_tiles, 1, 0, 0};
    if (part) tp = plan_patch_tail(pg, o.ncols, BN);
    p.full_units = tp.full_units;
    p.tail_split = tp.split;
    p.part_buf = part;
    const int units = tp.full_units + tp.tail_tiles * tp.split;
    cudaError_t e;
    // short tiles: double-buffer the accumulators (fewer A stages) so the
    // epilogue overlaps the next tile's MMAs
    bool db2 = false;
    if constexpr (BN == 64) db2 = p.k_stages <= kShortTileStages;
    // Long tiles stack the B tiles (two MMAs per K step instead of three; one
    // accumulator buffer per issuer then): AlexNet conv2's input gradient
    // 0.329 -> 0.298 ms.  Short tiles keep the second buffer instead, which
    // stacking would cost them (conv1's forward measured 13% slower stacked).
    if (db2)
        e = launch_tc_patch<ConvPatchProb<BN>, BN, TMA, BN <= 64>(p, units, device_error_word(), st, false);
    else
        e = launch_tc_patch<ConvPatchProb<BN>, BN, TMA, false>(p, units, device_error_word(), st, true);
    if (e != cudaSuccess || tp.tail_tiles == 0) return e;
    e = launch_pdl(tail_reduce_kernel<ConvPatchProb<BN>, BN>, dim3(unsigned(tp.tail_tiles), unsigned(BN / 32)),
                   dim3(kTailThreads), 0, st, p);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

template <bool TMA>
static cudaError_t dispatch_patch(int bn, const PatchGeom& pg, const OutGeom& o, float* img, float* part,
                                  cudaStream_t st)
{
    switch (bn) {
    case 32: return run_patch<32, TMA>(pg, o, img, part, st);
    case 64: return run_patch<64, TMA>(pg, o, img, part, st);
    default: return run_patch<128, TMA>(pg, o, img, part, st);
    }
}

// ---------------------------------------------------------------------------
// Tensor-map form of the patch kernel (32-channel chunks).

// Box of one (tile, chunk): rows spanned by any tile's window, full window width.
static void patch_box(PatchGeom& pg)
{
    int span = 0;
    for (int ti = 0; ti < pg.tpi; ++ti) {
        const int first = ti * kBM;
        const int last = (first + kBM < pg.GpGq ? first + kBM : pg.GpGq) - 1;
        const int d = last / pg.Gq - first / pg.Gq;
        if (d > span) span = d;
    }
    pg.rowsT = span * pg.sp + pg.T;
    pg.Wt = (pg.Gq - 1) * pg.sp + pg.T;
    pg.Cb = (pg.Ci + 31) / 32;
    pg.tbox = uint32_t(pg.rowsT) * uint32_t(pg.Wt) * 128u;
    pg.tbytes = (pg.tbox + 1023u) & ~1023u;
}

static bool patch_tma_fits(const PatchGeom& pg, int bn)
{
    if (pg.mode != 0 || pg.rowsT > 256 || pg.Wt > 256) return false;
    const size_t cap = PatchCfg<32>::kMaxSmem;
    switch (bn) {
    case 32: return patch_tma_smem<32>(pg.tbytes) <= cap;
    case 64: return patch_tma_smem<64>(pg.tbytes) <= cap;
    case 128: return patch_tma_smem<128>(pg.tbytes) <= cap;
    default: return false;
    }
}

static size_t blocked_bytes(const PatchGeom& pg)
{
    return size_t(pg.Nb) * pg.Cb * pg.Hi * pg.Wi * 32 * sizeof(float);
}

// dst[n][c / 32][h][w][c % 32] = src[n][c][h][w], zero for c >= C.  One block
// per (n, c / 32, group of kBlkRows rows): 32 x 32 (channel x column) tiles of
// every row of the group go through shared memory together, so each thread
// keeps 4 * kBlkRows loads in flight; reads are 128-byte rows along w, writes
// are whole 128-byte pixels (16-byte stores).
constexpr int kBlkRows = 4;

// MASK: each value is multiplied by (mask > 0), mask shaped like src (the
// ReLU gradient fused into the copy the input gradient reads).
template <bool MASK>
__global__ void __launch_bounds__(256, 4) to_blocked32_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                           int C, int Cb, int H, int W, int hgroups,
                                                           const float* __restrict__ mask)
{
    griddep_wait();
    griddep_launch();
    __shared__ float tile[kBlkRows][32][33];
    const int hg = blockIdx.x % hgroups;
    const int ncb = blockIdx.x / hgroups;   // n * Cb + cb
    const int n = ncb / Cb, cb = ncb % Cb;
    const int h0 = hg * kBlkRows;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int w0 = 0; w0 < W; w0 += 32) {
#pragma unroll
        for (int rr = 0; rr < kBlkRows; ++rr) {
            const int h = h0 + rr;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = ty + 8 * i, ch = cb * 32 + c, w = w0 + tx;
                const bool in = h < H && ch < C && w < W;
                const size_t at = ((size_t(n) * C + ch) * H + h) * W + w;
                float v = in ? __ldg(src + at) : 0.f;
                if constexpr (MASK) v *= relu_gate(in ? __ldg(mask + at) : 0.f);
                tile[rr][c][tx] = v;
            }
        }
        __syncthreads();
        // 8 lanes write one pixel's 32 channels as 16-byte chunks: the block
        // covers the tile's 32 pixels in one pass per row
        const int chunk = threadIdx.x & 7, pw = threadIdx.x >> 3, w = w0 + pw;
#pragma unroll
        for (int rr = 0; rr < kBlkRows; ++rr) {
            const int h = h0 + rr;
            if (h < H && w < W) {
                float* dpix = dst + ((size_t(ncb) * H + h) * size_t(W) + w) * 32 + 4 * chunk;
                *reinterpret_cast<float4*>(dpix) = make_float4(tile[rr][4 * chunk][pw], tile[rr][4 * chunk + 1][pw],
                                                               tile[rr][4 * chunk + 2][pw], tile[rr][4 * chunk + 3][pw]);
            }
        }
        __syncthreads();
    }
}


// Lays the gathered tensor out channel-blocked in `blocked` and describes it
// with the box the kernel loads.  Fails (and the caller reports a CUDA error)
// if the driver cannot encode the tensor map.
static cudaError_t encode_patch_tmap(PatchGeom& pg, float* blocked)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[4] = {32, cuuint64_t(pg.Wi), cuuint64_t(pg.Hi), cuuint64_t(pg.Nb) * pg.Cb};
    const cuuint64_t strides[3] = {128, cuuint64_t(pg.Wi) * 128, cuuint64_t(pg.Hi) * pg.Wi * 128};
    const cuuint32_t box[4] = {32, cuuint32_t(pg.Wt), cuuint32_t(pg.rowsT), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(&pg.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, blocked, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static cudaError_t setup_patch_tma(PatchGeom& pg, float* blocked, cudaStream_t st, const float* mask = nullptr)
{
    const int hgroups = (pg.Hi + kBlkRows - 1) / kBlkRows;
    const dim3 grid(unsigned(pg.Nb * pg.Cb * hgroups));
    cudaError_t e = mask ? launch_pdl(to_blocked32_kernel<true>, grid, dim3(256), 0, st, pg.in, blocked, pg.Ci, pg.Cb,
                                      pg.Hi, pg.Wi, hgroups, mask)
                         : launch_pdl(to_blocked32_kernel<false>, grid, dim3(256), 0, st, pg.in, blocked, pg.Ci,
                                      pg.Cb, pg.Hi, pg.Wi, hgroups, mask);
    if (e != cudaSuccess) return e;
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return encode_patch_tmap(pg, blocked);
}

// ---------------------------------------------------------------------------
// The flat kernel (gemm_flat.cuh): a stride-1 window of at least 2 x 2 taps
// over a channel-blocked tensor of at least 16 channels, at most 64 output
// columns (one column tile, BN = the columns rounded up to 16), box and
// stages within shared memory.

struct FlatPlan {
    bool use;
    int bn;
    FlatGeom fg;
};

// The flat kernel runs the forward of a strided few-channel layer in its
// space-to-depth form (AlexNet conv1: 48 channels, 3 x 3 taps, 64 filters),
// where it measured faster than the patch kernel (176 vs 184 us per call in
// 3xTF32, 164 vs 167 us in TF32).  On the input gradients, whose operand
// traffic the patch kernel splits between tensor and shared memory, it was
// slower (conv1 204 vs 178 us, conv2 322 vs 271 us), so they stay on the
// patch kernel.
static FlatPlan plan_flat(int Nb, int Ci, int Hi, int Wi, int Gp, int Gq, int o, int T, int ncols)
{
    FlatPlan f{};
    f.use = false;
    if (T < 2 || Ci < 16 || ncols > 64) return f;
    f.bn = (ncols + 15) / 16 * 16;
    FlatGeom& g = f.fg;
    g.Nb = Nb;
    g.Ci = Ci;
    g.Hi = Hi;
    g.Wi = Wi;
    g.Cb = (Ci + 31) / 32;
    g.nch = (Ci + 15) / 16;
    g.Gp = Gp;
    g.Gq = Gq;
    g.o = o;
    g.T = T;
    g.TT = T * T;
    g.spc = (g.TT + 1) / 2;
    g.Wt = Gq + T - 1;
    g.Rb = flat_box_rows(g.Wt, T);
    if (g.Wt > 256 || g.Rb > 256) return f;
    g.vpi = Gp * g.Wt;
    g.tpi = (g.vpi + kBM - 1) / kBM;
    g.box_bytes = uint32_t(g.Rb) * uint32_t(g.Wt) * 64u;
    g.box_stride = (g.box_bytes + 1023u) & ~1023u;
    size_t smem = 0;
    switch (f.bn) {
    case 16: smem = flat_smem<16>(g.box_stride); break;
    case 32: smem = flat_smem<32>(g.box_stride); break;
    case 48: smem = flat_smem<48>(g.box_stride); break;
    default: smem = flat_smem<64>(g.box_stride); break;
    }
    if (smem > 227 * 1024) return f;
    if ((long long)Nb * g.Cb * Hi * Wi * 32 >= (1LL << 31)) return f;   // 32-bit element offsets in the copy
    g.f_wt = FastDiv(uint32_t(g.Wt));
    g.f_t = FastDiv(uint32_t(T));
    g.f_tt = FastDiv(uint32_t(g.TT));
    f.use = true;
    return f;
}

// The B image: 2 * spc taps (the last padded with zeros when T*T is odd) of
// each 16-channel chunk, one 16-deep block per tap.
static int flat_kblocks(const FlatGeom& g) { return 2 * flat_kstages(g); }

static size_t flat_img_bytes(const FlatPlan& f, int ncols)
{
    return round_up_256(bimage16_floats(ncols, flat_kblocks(f.fg), f.bn) * sizeof(float));
}

// K decode of the flat image: 16-channel chunk, tap (of 2 * spc), channel.
static KDecode flat_kdecode(const FlatGeom& g)
{
    KDecode d = make_kdecode(3, 1, g.T);
    d.f_chunk = FastDiv(uint32_t(2 * g.spc * 16));
    return d;
}

static size_t flat_blocked_bytes(const FlatGeom& g) { return size_t(g.Nb) * g.Cb * g.Hi * g.Wi * 32 * sizeof(float); }

// The box of one (tile, 16-channel chunk) from the channel-blocked copy:
// 16 channels (64 bytes, 64-byte swizzle) x Wt columns x Rb rows.
static cudaError_t encode_flat_tmap(FlatGeom& g, float* blocked)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[4] = {32, cuuint64_t(g.Wi), cuuint64_t(g.Hi), cuuint64_t(g.Nb) * g.Cb};
    const cuuint64_t strides[3] = {128, cuuint64_t(g.Wi) * 128, cuuint64_t(g.Hi) * g.Wi * 128};
    const cuuint32_t box[4] = {16, cuuint32_t(g.Wt), cuuint32_t(g.Rb), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(&g.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, blocked, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


// ---------------------------------------------------------------------------
// Forward convolution with stride S > 1 and few channels, as a stride-1
// convolution over S x S super-pixels (space to depth):
//   y[n, k, p, q] = sum_(c', tr, tq) X'[n, c', p + tr, q + tq] * W'[k, c', tr, tq]
// with c' = (c, a, b) = c*S*S + a*S + b, X'[n, c', hh, ww] = x[n, c, S*hh + a - pad, S*ww + b - pad]
// (zero outside the image) and W'[k, c', tr, tq] = W[k, c, S*tr + a, S*tq + b] (zero past the filter):
// tap r = S*tr + a of output row p reads padded input row S*p + r = S*(p + tr) + a.  The window is
// T = ceil(R / S) super-pixels wide, and C*S*S channels fill 32-channel chunks: the form the
// tensor-map patch kernel runs best (AlexNet conv1: 3 channels, 11 x 11, stride 4 -> 48 channels, 3 x 3).

struct S2dPlan {
    bool use;
    int bn, T, Ci;
    PatchGeom pg;
    FlatPlan fp;   // the flat kernel over the same space-to-depth copy, when it applies
};

static S2dPlan plan_fwd_s2d(const ConvDims& d)
{
    S2dPlan sp{};
    sp.use = false;
    if (d.S < 2 || d.C > 16) return sp;
    sp.T = (d.R + d.S - 1) / d.S;
    sp.Ci = d.C * d.S * d.S;
    if (sp.Ci < 17 || sp.Ci > 128) return sp;
    int n_tiles;
    sp.bn = pick_conv_bn(d.K, &n_tiles);
    if (sp.bn > 128) return sp;
    if ((long long)d.N * ((sp.Ci + 31) / 32) * 32 * (d.P + sp.T - 1) * (d.Q + sp.T - 1) >= (1LL << 31))
        return sp;   // the channel-blocked copy is indexed with 32-bit element offsets
    sp.pg = make_patch(nullptr, d.N, sp.Ci, d.P + sp.T - 1, d.Q + sp.T - 1, d.P, d.Q, 1, 0, sp.T);
    sp.fp = plan_flat(d.N, sp.Ci, d.P + sp.T - 1, d.Q + sp.T - 1, d.P, d.Q, 0, sp.T, d.K);
    if (sp.fp.use) {
        sp.use = true;
        return sp;
    }
    if (sp.pg.mode != 0) return sp;
    patch_box(sp.pg);
    set_half_chunk(sp.pg);
    sp.use = patch_tma_fits(sp.pg, sp.bn);
    return sp;
}

struct FwdS2dFilterGen {   // B[k, kk] = W'[k, c', tr, tq] in the chunk-major K order
    const float* w;
    int C, R, S;
    KDecode dec;
    FastDiv f_t, f_ss, f_s;
    __device__ float operator()(int k, int kk) const
    {
        int cp, tap;
        dec(kk, cp, tap);
        uint32_t c, ab, a, b, tr, tq;
        f_ss.divmod(uint32_t(cp), c, ab);
        f_s.divmod(ab, a, b);
        f_t.divmod(uint32_t(tap), tr, tq);
        if (int(c) >= C || int(tr) >= int(f_t.d)) return 0.f;
        const int r = S * int(tr) + int(a), q = S * int(tq) + int(b);
        if (r >= R || q >= R) return 0.f;
        return __ldg(w + ((size_t(k) * C + c) * R + r) * R + q);
    }
};

// Which kernel a convolution-window GEMM runs on, and the workspace it needs:
// the patch-staged kernel when the output tile is at most 128 wide and every
// tile's patch fits its shared-memory buffer, otherwise the register-gather
// kernel (which may add a tail split's partial tiles).  A patch GEMM over
// 32-channel chunks whose box fits takes the tensor-map form.  Workspace
// layout: [B image, 256-byte aligned][partial tiles | channel-blocked copy].
struct WindowPlan {
    int bn;
    bool patch, tma;
    size_t img_bytes, part_bytes, blocked_bytes;
};

// masked: the gathered tensor is multiplied by a ReLU mask where it is first
// read -- in the channel-blocked copy of the tensor-map form, or in the
// register gather -- so the per-channel bulk-copied patch form (which reads
// the tensor straight into shared memory) is not used.
static WindowPlan plan_window(int Nb, int Ci, int Hi, int Wi, int Gp, int Gq, int sp, int o, int T, int ncols,
                              bool masked = false)
{
    WindowPlan w{};
    int n_tiles;
    w.bn = pick_conv_bn(ncols, &n_tiles);
    w.patch = w.tma = false;
    w.blocked_bytes = 0;
    if (w.bn <= 128) {
        PatchGeom pg = make_patch(nullptr, Nb, Ci, Hi, Wi, Gp, Gq, sp, o, T);
        patch_box(pg);
        w.tma = patch_tma_fits(pg, w.bn);
        w.patch = w.tma || (!masked && max_patch_floats(pg) <= patch_capacity(w.bn));
        if (w.tma) w.blocked_bytes = blocked_bytes(pg);
        if (w.patch) w.part_bytes = round_up_256(plan_patch_tail(pg, ncols, w.bn).part_floats * sizeof(float));
    }
    w.img_bytes = round_up_256(bimage_floats(ncols, k_extent(Ci, T), w.bn) * sizeof(float));
    if (!w.patch) {
        const GatherGeom g = make_gather(nullptr, Nb, Ci, Hi, Wi, Gp, Gq, sp, o, T);
        const TailPlan tp = plan_tail(((g.M + kBM - 1) / kBM) * n_tiles, (g.K + kBK - 1) / kBK, w.bn);
        w.part_bytes = tp.part_floats * sizeof(float);
    }
    return w;
}

// One convolution-window GEMM over the gathered tensor `in` [Nb][Ci][Hi][Wi]:
// rows = the (Gp x Gq) grid of each image, window h = p*sp + o + tap.
// MakeGen(KDecode) builds the B-operand generator in the matching K order.
// mask (nullable): multiply the gathered tensor by (mask > 0) as it is read.
template <class MakeGen>
static cudaError_t run_window_gemm(const float* in, int Nb, int Ci, int Hi, int Wi, int Gp, int Gq, int sp, int o,
                                   int T, const OutGeom& og, void* ws, MakeGen make_gen, cudaStream_t st,
                                   const float* mask = nullptr)
{
    const WindowPlan wp = plan_window(Nb, Ci, Hi, Wi, Gp, Gq, sp, o, T, og.ncols, mask != nullptr);
    float* img = static_cast<float*>(ws);
    const int bn = wp.bn;

    if (wp.patch) {
        PatchGeom pg = make_patch(in, Nb, Ci, Hi, Wi, Gp, Gq, sp, o, T);
        if (wp.tma) set_half_chunk(pg);
        const KDecode dec = patch_kdecode(pg);
        const int k_total = pg.mode == 0 ? patch_kstages(pg) * kBK : T * T * pg.Cp;   // padded taps excluded
        cudaError_t e = build_bimage(make_gen(dec), og.ncols, k_total, bn, img, st);
        if (e != cudaSuccess) return e;
        // workspace: [B image][channel-blocked copy (tensor-map form)][tail partial tiles]
        float* part = wp.part_bytes ? reinterpret_cast<float*>(static_cast<char*>(ws) + wp.img_bytes +
                                                               wp.blocked_bytes)
                                    : nullptr;
        if (wp.tma) {
            patch_box(pg);
            e = setup_patch_tma(pg, reinterpret_cast<float*>(static_cast<char*>(ws) + wp.img_bytes), st, mask);
            if (e != cudaSuccess) return e;
            return dispatch_patch<true>(bn, pg, og, img, part, st);
        }
        return dispatch_patch<false>(bn, pg, og, img, part, st);
    }
    GatherGeom g = make_gather(in, Nb, Ci, Hi, Wi, Gp, Gq, sp, o, T);
    g.mask = mask;
    const KDecode dec = make_kdecode(g.mode == 2 ? 2 : 0, g.Cp, T);
    cudaError_t e = build_bimage(make_gen(dec), og.ncols, g.K, bn, img, st);
    if (e != cudaSuccess) return e;
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + wp.img_bytes);
    return dispatch_gather(bn, g, og, img, part, st);
}

size_t conv_fwd_ws(const ConvDims& d)
{
    const S2dPlan sp = plan_fwd_s2d(d);
    if (sp.use && sp.fp.use) return flat_img_bytes(sp.fp, d.K) + flat_blocked_bytes(sp.fp.fg);
    if (sp.use)
        return round_up_256(bimage_floats(d.K, patch_kstages(sp.pg) * kBK, sp.bn) * sizeof(float)) +
               blocked_bytes(sp.pg);
    const WindowPlan wp = plan_window(d.N, d.C, d.H, d.W, d.P, d.Q, d.S, -d.pad, d.R, d.K);
    return wp.img_bytes + wp.part_bytes + wp.blocked_bytes;
}

size_t conv_dgrad_ws(const ConvDims& d)
{
    int d_lo, T, oo;
    dgrad_window(d, &d_lo, &T, &oo);
    const int Hs = (d.H + oo + d.S - 1) / d.S, Ws = (d.W + oo + d.S - 1) / d.S;
    // room for either plan: the masked one (conv_bwd_data_relu) may take the
    // register-gather form where the plain one takes the per-channel patch form
    const WindowPlan wp = plan_window(d.N, d.K, d.P, d.Q, Hs, Ws, 1, d_lo, T, dgrad_cols(d));
    const WindowPlan wm = plan_window(d.N, d.K, d.P, d.Q, Hs, Ws, 1, d_lo, T, dgrad_cols(d), true);
    const size_t a = wp.img_bytes + wp.part_bytes + wp.blocked_bytes, b = wm.img_bytes + wm.part_bytes + wm.blocked_bytes;
    return a > b ? a : b;
}

cudaError_t launch_conv_fwd(const ConvDims& d, const float* x, const float* w, const float* b, float* y, void* ws,
                            cudaStream_t st, bool relu)
{
    OutGeom o{};
    o.out = y;
    o.bias = b;
    o.relu = relu ? 1 : 0;
    o.Co = d.K;
    o.Ho = d.P;
    o.Wo = d.Q;
    o.HoWo = d.P * d.Q;
    o.so = 1;
    o.ncols = d.K;
    S2dPlan sp = plan_fwd_s2d(d);
    if (sp.use && sp.fp.use) {
        FlatGeom& fg = sp.fp.fg;
        const FwdS2dFilterGen gen{w,   d.C, d.R, d.S, flat_kdecode(fg), FastDiv(uint32_t(sp.T)),
                                  FastDiv(uint32_t(d.S * d.S)), FastDiv(uint32_t(d.S))};
        float* img = static_cast<float*>(ws);
        cudaError_t e = build_bimage16(gen, d.K, flat_kblocks(fg), sp.fp.bn, img, st);
        if (e != cudaSuccess) return e;
        float* blocked = reinterpret_cast<float*>(static_cast<char*>(ws) + flat_img_bytes(sp.fp, d.K));
        e = launch_s2d_copy<true>(x, blocked, d.N, d.C, d.H, d.W, d.S, d.pad, fg.Hi, fg.Wi, st);
        if (e != cudaSuccess) return e;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = encode_flat_tmap(fg, blocked)) != cudaSuccess) return e;
        return dispatch_flat(sp.fp.bn, fg, o, img, st);
    }
    if (sp.use) {
        PatchGeom& pg = sp.pg;
        const int k_total = patch_kstages(pg) * kBK;
        const FwdS2dFilterGen gen{w,   d.C, d.R, d.S, patch_kdecode(pg), FastDiv(uint32_t(sp.T)),
                                  FastDiv(uint32_t(d.S * d.S)), FastDiv(uint32_t(d.S))};
        float* img = static_cast<float*>(ws);
        cudaError_t e = build_bimage(gen, d.K, k_total, sp.bn, img, st);
        if (e != cudaSuccess) return e;
        float* blocked = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                                  round_up_256(bimage_floats(d.K, k_total, sp.bn) * sizeof(float)));
        e = launch_s2d_copy<true>(x, blocked, d.N, d.C, d.H, d.W, d.S, d.pad, pg.Hi, pg.Wi, st);
        if (e != cudaSuccess) return e;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = encode_patch_tmap(pg, blocked)) != cudaSuccess) return e;
        return dispatch_patch<true>(sp.bn, pg, o, img, nullptr, st);
    }
    auto make_gen = [&](const KDecode& dec) { return FwdFilterGen{w, d.C, d.R, dec, FastDiv(uint32_t(d.R))}; };
    return run_window_gemm(x, d.N, d.C, d.H, d.W, d.P, d.Q, d.S, -d.pad, d.R, o, ws, make_gen, st);
}

cudaError_t launch_conv_dgrad(const ConvDims& d, const float* w, const float* dy, float* dx, void* ws,
                              cudaStream_t st, const float* mask)
{
    int d_lo, T, oo;
    dgrad_window(d, &d_lo, &T, &oo);
    const int Hs = (d.H + oo + d.S - 1) / d.S, Ws = (d.W + oo + d.S - 1) / d.S;
    OutGeom o{};
    o.out = dx;
    o.bias = nullptr;
    o.Co = d.C;
    o.Ho = d.H;
    o.Wo = d.W;
    o.HoWo = d.H * d.W;
    o.so = d.S;
    o.oo = oo;
    o.ncols = dgrad_cols(d);
    const uintptr_t ax = reinterpret_cast<uintptr_t>(dx);
    o.vec = (d.S == 4 || d.S == 2) && oo == 0 && d.W % d.S == 0 && (ax & 15) == 0 ? 1
            : (d.S == 4 && oo == 2 && d.W % 2 == 0 && (ax & 7) == 0)           ? 2
                                                                               : 0;
    auto make_gen = [&](const KDecode& dec) {
        return DgradFilterGen{w,   d.C, d.K, d.R, d.S, d.pad - oo, d_lo, dec, FastDiv(uint32_t(T)),
                              FastDiv(uint32_t(d.S * d.S)), FastDiv(uint32_t(d.S))};
    };
    return run_window_gemm(dy, d.N, d.K, d.P, d.Q, Hs, Ws, 1, d_lo, T, o, ws, make_gen, st, mask);
}

}  // namespace cb200
