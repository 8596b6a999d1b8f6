// conv_fwd.cu -- forward convolution of the page "DirectCompute Neural Network
// Engine", section "Convolution: The im2col Approach" (forward steps 1-3), as
// one implicit GEMM on the tcgen05 tensor cores:
//
//   D[pixel m, filter k] = sum_crs col[crs, m] * Wmat[k, crs]
//   y[n, k, oh, ow]      = D[(n, oh, ow), k] + b[k]
//
// Step 1 (im2col) is the A-operand gather: each producer thread owns one
// output pixel and reads its patch straight from x, 32 patch entries per
// pipeline stage, zero in the padding -- the column matrix is never stored.
// Step 2 (filters x columns) is the MMA; the filters are laid out once per
// call as pre-split hi/lo tiles (conv_common.cuh) and fed by bulk copies.
// Step 3 (conv_reshape + bias) is the epilogue: one thread per pixel writes
// its outC values into NCHW, a warp covering 32 consecutive pixels.
#include "conv_common.cuh"

namespace cb200 {

struct FwdFilterGen {   // B[k, crs] = Wmat[k][crs]
    const float* w;
    int CRS;
    __device__ float operator()(int row, int k) const { return __ldg(w + size_t(row) * CRS + k); }
};

template <int BN>
struct ConvFwdProb {
    static constexpr bool kBBulk = true;
    static constexpr Map kAMap = Map::RowFast;
    static constexpr Map kBMap = Map::RowFast;   // unused (bulk)

    const float* x;
    const float* bimg;
    const float* bias;
    float* y;
    int C, H, W, K, R, S, pad, P, Q;
    int NPQ, PQ, CRS, HW;
    FastDiv f_pq, f_q, f_rr, f_r;
    int m_tiles, n_tiles, k_stages;

    __device__ int num_tiles() const { return m_tiles * n_tiles; }
    __device__ Tile tile(int t) const
    {
        Tile r;
        r.n0 = (t % n_tiles) * BN;
        r.m0 = (t / n_tiles) * kBM;
        r.ks0 = 0;
        r.ks1 = k_stages;
        r.grp = t % n_tiles;
        return r;
    }

    struct AState {
        int base;        // offset of x[n][0][ih0][iw0]
        int ih0, iw0;    // top-left input position of the patch
    };
    __device__ AState a_setup(const Tile& tl, int tid) const
    {
        AState s;
        const int m = tl.m0 + tid;
        if (m < NPQ) {
            uint32_t n, pq, oh, ow;
            f_pq.divmod(uint32_t(m), n, pq);
            f_q.divmod(pq, oh, ow);
            s.ih0 = int(oh) * S - pad;
            s.iw0 = int(ow) * S - pad;
            s.base = int(n) * C * HW + s.ih0 * W + s.iw0;
        } else {
            s.ih0 = -(1 << 24);   // no patch position is ever inside the image
            s.iw0 = 0;
            s.base = 0;
        }
        return s;
    }

    __device__ void load_a(const AState& s, const Tile&, int ks, int tid, float (&v)[32]) const
    {
        // Lane l decodes patch entry k = ks*32 + l; the warp shares the table.
        const int k = ks * kBK + (tid & 31);
        int koff = 0, krs = 0x7FFF0000;   // past CRS: row offset huge -> never inside
        if (k < CRS) {
            uint32_t c, rem, r, q;
            f_rr.divmod(uint32_t(k), c, rem);
            f_r.divmod(rem, r, q);
            koff = int(c) * HW + int(r) * W + int(q);
            krs = int((r << 16) | q);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int off = __shfl_sync(0xffffffffu, koff, i);
            const int rs = __shfl_sync(0xffffffffu, krs, i);
            const int h = s.ih0 + (rs >> 16);
            const int w = s.iw0 + (rs & 0xFFFF);
            v[i] = (unsigned(h) < unsigned(H) && unsigned(w) < unsigned(W)) ? __ldg(x + (s.base + off)) : 0.f;
        }
    }

    struct BState {};
    __device__ BState b_setup(const Tile&, int) const { return {}; }
    __device__ void load_b(const BState&, const Tile&, int, int, int, float (&)[32]) const {}
    __device__ const float* b_image(const Tile& tl, int ks) const
    {
        return bimg + (size_t(tl.grp) * k_stages + ks) * 2 * size_t(BN) * kBK;
    }

    struct EState {
        float* ypix;   // y[n][0][oh][ow]; channel stride PQ
        bool valid;
    };
    __device__ EState e_setup(const Tile& tl, int row) const
    {
        EState e;
        const int m = tl.m0 + row;
        e.valid = m < NPQ;
        uint32_t n = 0, pq = 0;
        if (e.valid) f_pq.divmod(uint32_t(m), n, pq);
        e.ypix = y + size_t(n) * K * PQ + pq;
        return e;
    }

    __device__ void store(const EState& e, const Tile& tl, int, int c, const uint32_t (&r)[32]) const
    {
        if (!e.valid) return;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int k = tl.n0 + c + i;
            if (k < K) e.ypix[size_t(k) * PQ] = __uint_as_float(r[i]) + (bias ? __ldg(bias + k) : 0.f);
        }
    }
};

size_t conv_fwd_ws(const ConvDims& d)
{
    int n_tiles;
    const int bn = pick_conv_bn(d.K, &n_tiles);
    return bimage_floats(d.K, d.C * d.R * d.R, bn) * sizeof(float);
}

template <int BN>
static cudaError_t run_fwd(const ConvDims& d, const float* x, const float* w, const float* b, float* y, void* ws,
                           cudaStream_t st)
{
    ConvFwdProb<BN> p;
    p.x = x;
    p.bimg = static_cast<const float*>(ws);
    p.bias = b;
    p.y = y;
    p.C = d.C; p.H = d.H; p.W = d.W; p.K = d.K; p.R = d.R; p.S = d.S; p.pad = d.pad; p.P = d.P; p.Q = d.Q;
    p.PQ = d.P * d.Q;
    p.NPQ = d.N * p.PQ;
    p.CRS = d.C * d.R * d.R;
    p.HW = d.H * d.W;
    p.f_pq = FastDiv(p.PQ);
    p.f_q = FastDiv(d.Q);
    p.f_rr = FastDiv(d.R * d.R);
    p.f_r = FastDiv(d.R);
    p.m_tiles = (p.NPQ + kBM - 1) / kBM;
    p.n_tiles = (d.K + BN - 1) / BN;
    p.k_stages = (p.CRS + kBK - 1) / kBK;
    cudaError_t e = build_bimage(FwdFilterGen{w, p.CRS}, d.K, p.CRS, BN, static_cast<float*>(ws), st);
    if (e != cudaSuccess) return e;
    return launch_tc_gemm<ConvFwdProb<BN>, BN>(p, p.m_tiles * p.n_tiles, device_error_word(), st);
}

cudaError_t launch_conv_fwd(const ConvDims& d, const float* x, const float* w, const float* b, float* y, void* ws,
                            cudaStream_t st)
{
    int n_tiles;
    switch (pick_conv_bn(d.K, &n_tiles)) {
    case 32: return run_fwd<32>(d, x, w, b, y, ws, st);
    case 64: return run_fwd<64>(d, x, w, b, y, ws, st);
    case 128: return run_fwd<128>(d, x, w, b, y, ws, st);
    case 192: return run_fwd<192>(d, x, w, b, y, ws, st);
    default: return run_fwd<256>(d, x, w, b, y, ws, st);
    }
}

}  // namespace cb200
