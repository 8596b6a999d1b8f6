// conv_dgrad.cu -- input gradient of the page "DirectCompute Neural Network
// Engine", section "Convolution: The im2col Approach" (backward: filters^T x
// grad_reshaped, then col2im), as implicit GEMMs on the tcgen05 tensor cores.
//
// col2im sums, for each input pixel (h, w), the column-matrix gradient
// entries of every (r, q, oh, ow) with oh*stride + r - pad = h and
// ow*stride + q - pad = w.  Solving for oh: only taps r == (h + pad) mod stride
// contribute, r = r0 + stride*i, and then oh = (h + pad - r0)/stride - i.  So
// the input pixels split into stride x stride phases (h mod stride,
// w mod stride); inside one phase every pixel sees the same taps and
//
//   dx[n, c, a + s*hh, b + s*ww] =
//       sum_{k, i, j} W[k, c, r0 + s*i, q0 + s*j] * dy[n, k, hh + da - i, ww + db - j]
//
// is a GEMM with rows = pixels of the phase, columns = input channels and
// reduction over (k, i, j).  The A operand gathers dy directly (zero outside
// the output grid), the B operand is the filter rearranged per phase (pre-split
// image, bulk copies), and the epilogue writes dx in NCHW.  Every dx element
// is produced by exactly one accumulator, so col2im needs no scatter, no
// atomics and no column-matrix buffer.
#include "conv_common.cuh"

namespace cb200 {

constexpr int kMaxPhases = 16;   // phases handled by one launch

struct Phase {
    int a, b;           // residue of h and w
    int da, db;         // dy row/col offset: oh = hh + da - i
    int r0, q0;         // first filter tap of the phase
    int Ri, Rj;         // taps per axis
    int Hg, Wg;         // pixels of the phase per axis
    int M, Kd;          // GEMM rows (N*Hg*Wg) and reduction length (K*Ri*Rj)
    int k_stages, tile_begin;
    size_t img_off;     // floats into the image workspace
    FastDiv f_hw, f_w, f_rr, f_r;
};

struct DgradFilterGen {   // B[c, (k, i, j)] = W[k, c, r0 + s*i, q0 + s*j]
    const float* w;
    int C, R, S, r0, q0;
    FastDiv f_rr, f_r;
    __device__ float operator()(int c, int kk) const
    {
        uint32_t k, rem, i, j;
        f_rr.divmod(uint32_t(kk), k, rem);
        f_r.divmod(rem, i, j);
        const int r = r0 + S * int(i), q = q0 + S * int(j);
        return __ldg(w + ((size_t(k) * C + c) * R + r) * R + q);
    }
};

template <int BN>
struct ConvDgradProb {
    static constexpr bool kBBulk = true;
    static constexpr Map kAMap = Map::RowFast;
    static constexpr Map kBMap = Map::RowFast;   // unused (bulk)

    const float* dy;
    const float* bimg;
    float* dx;
    int C, H, W, K, S, P, Q;
    int PQ, HW;
    int n_tiles, num_phases, total_tiles;
    Phase ph[kMaxPhases];

    __device__ int num_tiles() const { return total_tiles; }
    __device__ Tile tile(int t) const
    {
        int g = 0;
        while (g + 1 < num_phases && t >= ph[g + 1].tile_begin) ++g;
        const int local = t - ph[g].tile_begin;
        Tile r;
        r.n0 = (local % n_tiles) * BN;
        r.m0 = (local / n_tiles) * kBM;
        r.ks0 = 0;
        r.ks1 = ph[g].k_stages;
        r.grp = g;
        return r;
    }

    struct AState {
        int base;       // offset of dy[n][0][oh0][ow0]
        int oh0, ow0;   // dy position of tap (0, 0)
        int g;
    };
    __device__ AState a_setup(const Tile& tl, int tid) const
    {
        const Phase& f = ph[tl.grp];
        AState s;
        s.g = tl.grp;
        const int m = tl.m0 + tid;
        if (m < f.M) {
            uint32_t n, rem, hh, ww;
            f.f_hw.divmod(uint32_t(m), n, rem);
            f.f_w.divmod(rem, hh, ww);
            s.oh0 = int(hh) + f.da;
            s.ow0 = int(ww) + f.db;
            s.base = int(n) * K * PQ + s.oh0 * Q + s.ow0;
        } else {
            s.oh0 = -(1 << 24);
            s.ow0 = 0;
            s.base = 0;
        }
        return s;
    }

    __device__ void load_a(const AState& s, const Tile& tl, int ks, int tid, float (&v)[32]) const
    {
        const Phase& f = ph[tl.grp];
        const int kk = ks * kBK + (tid & 31);
        int koff = 0, kij = -(0x7FFF << 16);   // past the reduction: oh lands far past P
        if (kk < f.Kd) {
            uint32_t k, rem, i, j;
            f.f_rr.divmod(uint32_t(kk), k, rem);
            f.f_r.divmod(rem, i, j);
            koff = int(k) * PQ - int(i) * Q - int(j);
            kij = int((i << 16) | j);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int off = __shfl_sync(0xffffffffu, koff, e);
            const int ij = __shfl_sync(0xffffffffu, kij, e);
            const int oh = s.oh0 - (ij >> 16);
            const int ow = s.ow0 - (ij & 0xFFFF);
            v[e] = (unsigned(oh) < unsigned(P) && unsigned(ow) < unsigned(Q)) ? __ldg(dy + (s.base + off)) : 0.f;
        }
    }

    struct BState {};
    __device__ BState b_setup(const Tile&, int) const { return {}; }
    __device__ void load_b(const BState&, const Tile&, int, int, int, float (&)[32]) const {}
    __device__ const float* b_image(const Tile& tl, int ks) const
    {
        const Phase& f = ph[tl.grp];
        return bimg + f.img_off + (size_t(tl.n0 / BN) * f.k_stages + ks) * 2 * size_t(BN) * kBK;
    }

    struct EState {
        float* xpix;   // dx[n][0][h][w]; channel stride HW
        bool valid;
    };
    __device__ EState e_setup(const Tile& tl, int row) const
    {
        const Phase& f = ph[tl.grp];
        EState e;
        const int m = tl.m0 + row;
        e.valid = m < f.M;
        uint32_t n = 0, rem = 0, hh = 0, ww = 0;
        if (e.valid) {
            f.f_hw.divmod(uint32_t(m), n, rem);
            f.f_w.divmod(rem, hh, ww);
        }
        e.xpix = dx + size_t(n) * C * HW + size_t(f.a + S * int(hh)) * W + (f.b + S * int(ww));
        return e;
    }

    __device__ void store(const EState& e, const Tile& tl, int, int c, const uint32_t (&r)[32]) const
    {
        if (!e.valid) return;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int ch = tl.n0 + c + i;
            if (ch < C) e.xpix[size_t(ch) * HW] = __uint_as_float(r[i]);
        }
    }
};

// Phase geometry for residues (a, b).
static Phase make_phase(const ConvDims& d, int a, int b)
{
    Phase f{};
    const int s = d.S;
    f.a = a;
    f.b = b;
    f.r0 = (a + d.pad) % s;
    f.q0 = (b + d.pad) % s;
    f.da = (a + d.pad - f.r0) / s;
    f.db = (b + d.pad - f.q0) / s;
    f.Ri = f.r0 < d.R ? (d.R - f.r0 + s - 1) / s : 0;
    f.Rj = f.q0 < d.R ? (d.R - f.q0 + s - 1) / s : 0;
    f.Hg = a < d.H ? (d.H - a + s - 1) / s : 0;
    f.Wg = b < d.W ? (d.W - b + s - 1) / s : 0;
    f.M = d.N * f.Hg * f.Wg;
    f.Kd = d.K * f.Ri * f.Rj;
    f.k_stages = (f.Kd + kBK - 1) / kBK;
    if (f.Hg > 0 && f.Wg > 0) {
        f.f_hw = FastDiv(uint32_t(f.Hg * f.Wg));
        f.f_w = FastDiv(uint32_t(f.Wg));
    }
    if (f.Ri > 0 && f.Rj > 0) {
        f.f_rr = FastDiv(uint32_t(f.Ri * f.Rj));
        f.f_r = FastDiv(uint32_t(f.Rj));
    }
    return f;
}

size_t conv_dgrad_ws(const ConvDims& d)
{
    int n_tiles;
    const int bn = pick_conv_bn(d.C, &n_tiles);
    size_t total = 0;
    for (int a = 0; a < d.S; ++a)
        for (int b = 0; b < d.S; ++b) {
            Phase f = make_phase(d, a, b);
            if (f.M > 0 && f.Kd > 0) total += bimage_floats(d.C, f.Kd, bn);
        }
    return total * sizeof(float);
}

template <int BN>
static cudaError_t run_dgrad(const ConvDims& d, const float* w, const float* dy, float* dx, void* ws,
                             cudaStream_t st)
{
    // Phases whose pixels see no filter tap have dx == 0 there.
    bool any_empty = false;
    for (int a = 0; a < d.S; ++a)
        for (int b = 0; b < d.S; ++b) {
            Phase f = make_phase(d, a, b);
            if (f.M > 0 && f.Kd == 0) any_empty = true;
        }
    if (any_empty) {
        cudaError_t e = cudaMemsetAsync(dx, 0, size_t(d.N) * d.C * d.H * d.W * sizeof(float), st);
        if (e != cudaSuccess) return e;
    }

    ConvDgradProb<BN> p;
    p.dy = dy;
    p.bimg = static_cast<const float*>(ws);
    p.dx = dx;
    p.C = d.C; p.H = d.H; p.W = d.W; p.K = d.K; p.S = d.S; p.P = d.P; p.Q = d.Q;
    p.PQ = d.P * d.Q;
    p.HW = d.H * d.W;
    p.n_tiles = (d.C + BN - 1) / BN;
    p.num_phases = 0;
    p.total_tiles = 0;
    size_t img_off = 0;
    for (int a = 0; a < d.S; ++a)
        for (int b = 0; b < d.S; ++b) {
            Phase f = make_phase(d, a, b);
            if (f.M == 0 || f.Kd == 0) continue;
            f.img_off = img_off;
            f.tile_begin = p.total_tiles;
            DgradFilterGen gen{w, d.C, d.R, d.S, f.r0, f.q0, FastDiv(uint32_t(f.Ri * f.Rj)), FastDiv(uint32_t(f.Rj))};
            cudaError_t e = build_bimage(gen, d.C, f.Kd, BN, static_cast<float*>(ws) + img_off, st);
            if (e != cudaSuccess) return e;
            img_off += bimage_floats(d.C, f.Kd, BN);
            p.total_tiles += ((f.M + kBM - 1) / kBM) * p.n_tiles;
            p.ph[p.num_phases++] = f;
            if (p.num_phases == kMaxPhases) {
                e = launch_tc_gemm<ConvDgradProb<BN>, BN>(p, p.total_tiles, device_error_word(), st);
                if (e != cudaSuccess) return e;
                p.num_phases = 0;
                p.total_tiles = 0;
            }
        }
    if (p.num_phases > 0) return launch_tc_gemm<ConvDgradProb<BN>, BN>(p, p.total_tiles, device_error_word(), st);
    return cudaSuccess;
}

cudaError_t launch_conv_dgrad(const ConvDims& d, const float* w, const float* dy, float* dx, void* ws,
                              cudaStream_t st)
{
    int n_tiles;
    switch (pick_conv_bn(d.C, &n_tiles)) {
    case 32: return run_dgrad<32>(d, w, dy, dx, ws, st);
    case 64: return run_dgrad<64>(d, w, dy, dx, ws, st);
    case 128: return run_dgrad<128>(d, w, dy, dx, ws, st);
    case 192: return run_dgrad<192>(d, w, dy, dx, ws, st);
    default: return run_dgrad<256>(d, w, dy, dx, ws, st);
    }
}

}  // namespace cb200
