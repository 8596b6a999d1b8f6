// conv_window.cuh -- the convolution-window GEMM problems shared by the
// translation units that launch them (page "DirectCompute Neural Network
// Engine", section "Convolution: The im2col Approach"): the window gather
// geometry, the output geometry with its epilogue store (conv_reshape + bias
// [+ ReLU] for the forward, the stride-phase scatter of the input gradient),
// the register-gather problem and the flat-kernel problem.  The K orders and
// the forward / input-gradient GEMM forms are described in conv_gather.cu.
#pragma once
#include "conv_common.cuh"
#include "gemm_flat.cuh"

namespace cb200 {

struct GatherGeom {
    const float* in;         // gathered tensor [Nb][Ci][Hi][Wi]
    const float* mask;       // null, or a tensor shaped like `in`: each gathered value is multiplied by
                             // (mask > 0) as it is loaded (nn_relu_grad fused into the input gradient)
    int Ci, Hi, Wi, HiWi, CiHiWi;
    int Gp, Gq, M;           // row grid per image and rows in all (Nb * Gp * Gq)
    int sp;                  // window stride on the input
    int o;                   // window origin offset: h = p*sp + o + tap_r
    int T;                   // taps per axis
    int mode;                // K order: 0 chunk of one tap, 1 tap group (Ci <= 16), 2 generic
    int Cp, lcp;             // padded channels (modes 0/1) and log2 Cp (mode 1)
    int K;                   // reduction length: T*T*Cp (modes 0/1), T*T*Ci (mode 2)
    FastDiv f_gpq, f_gq;     // row decode
    FastDiv f_cchunks;       // Cp / 32 (mode 0)
    FastDiv f_tt, f_t;       // T*T and T
};

// K order of a gather over a tensor with `ci` channels (see top of file).
static inline void k_order(int ci, int* mode, int* cp, int* lcp)
{
    if (ci % 32 == 0 || (ci > 16 && ci < 32)) {
        *mode = 0;
        *cp = (ci + 31) / 32 * 32;
        *lcp = 0;
    } else if (ci < 32) {
        int l = 0;
        while ((1 << l) < ci) ++l;
        *mode = 1;
        *cp = 1 << l;
        *lcp = l;
    } else {
        *mode = 2;
        *cp = ci;
        *lcp = 0;
    }
}

struct OutGeom {
    float* out;              // [Nb][Co][Ho][Wo]
    const float* bias;       // [Co] or null
    int relu;                // forward only: max(0, .) after the bias (nn_relu fused into the epilogue)
    int Co, Ho, Wo, HoWo;
    int so;                  // output phase stride (1: plain NCHW)
    int oo;                  // phase offset: row p's phase block starts at output row p * so - oo (0 <= oo < so)
    int ncols;               // Co * so * so
    int vec;                 // 1: so = 2 or 4, oo = 0, Wo % so == 0, out 16-byte aligned: each (ch, a) row of
                             //    so phases is one float2 / float4 store
                             // 2: so = 4, oo = 2, Wo even, out 8-byte aligned: two float2 stores per (ch, a)
};

template <int BN>
struct ConvGatherProb {
    static constexpr bool kBBulk = true;
    int terms = 3;                                // tensor-core products per K step: 3 (3xTF32) or 1 (TF32)
    // A stages in tensor memory up to 128 columns (two accumulators still fit).
    // Wider tiles keep A in shared memory: with A in tensor memory they would
    // keep a single accumulator, and measured 5-20% slower on the AlexNet layers.
    static constexpr bool kATmem = BN <= 128;
    static constexpr int kGroups = 2;
    static constexpr Map kAMap = Map::RowFast;
    static constexpr Map kBMap = Map::RowFast;   // unused (bulk)

    GatherGeom g;
    OutGeom o;
    const float* bimg;
    int m_tiles, n_tiles, k_stages;
    // Tail split (see plan_tail): units [0, full_units) are whole tiles; each
    // later tile is cut along K into tail_split pieces whose partial sums go
    // to part_buf [piece][kBM][BN] and are added by tail_reduce_kernel.
    int full_units = 0, tail_split = 1;
    float* part_buf = nullptr;

    __device__ int num_tiles() const { return full_units + (m_tiles * n_tiles - full_units) * tail_split; }
    __device__ Tile whole_tile(int t) const
    {
        Tile r;
        r.n0 = (t % n_tiles) * BN;
        r.m0 = (t / n_tiles) * kBM;
        r.ks0 = 0;
        r.ks1 = k_stages;
        r.grp = t % n_tiles;
        return r;
    }
    __device__ Tile tile(int t) const
    {
        if (t < full_units) return whole_tile(t);
        const int u = t - full_units;
        const int j = u % tail_split;
        Tile r = whole_tile(full_units + u / tail_split);
        r.ks0 = int((long long)j * k_stages / tail_split);
        r.ks1 = int((long long)(j + 1) * k_stages / tail_split);
        r.part = u;
        return r;
    }

    struct AState {
        int base;      // offset of in[n][0][h0][w0]
        int h0, w0;    // window origin of this row
    };
    __device__ AState a_setup(const Tile& tl, int tid) const
    {
        AState s;
        const int m = tl.m0 + tid;
        if (m < g.M) {
            uint32_t n, pq, p, q;
            g.f_gpq.divmod(uint32_t(m), n, pq);
            g.f_gq.divmod(pq, p, q);
            s.h0 = int(p) * g.sp + g.o;
            s.w0 = int(q) * g.sp + g.o;
            s.base = int(n) * g.CiHiWi + s.h0 * g.Wi + s.w0;
        } else {
            s.h0 = -(1 << 24);   // no window position is ever inside
            s.w0 = 0;
            s.base = 0;
        }
        return s;
    }

    // Mode 1: 32 / CP taps per stage, CP channels each.
    template <int LCP>
    __device__ __forceinline__ void load_taps(const AState& s, int ks, float (&v)[32]) const
    {
        constexpr int CP = 1 << LCP, TPS = 32 >> LCP;
        const int TT = g.T * g.T;
#pragma unroll
        for (int t = 0; t < TPS; ++t) {
            const int tap = ks * TPS + t;
            uint32_t tr, tq;
            g.f_t.divmod(uint32_t(tap), tr, tq);
            const int h = s.h0 + int(tr);
            const int w = s.w0 + int(tq);
            const bool ok = tap < TT && unsigned(h) < unsigned(g.Hi) && unsigned(w) < unsigned(g.Wi);
            const int off = s.base + int(tr) * g.Wi + int(tq);
            const float* p = g.in + off;
            if (g.mask == nullptr) {
#pragma unroll
                for (int c = 0; c < CP; ++c) v[t * CP + c] = ldg_keep_if(p + c * g.HiWi, ok && c < g.Ci);
            } else {
                const float* mp = g.mask + off;
#pragma unroll
                for (int c = 0; c < CP; ++c)
                    v[t * CP + c] = ldg_keep_if(p + c * g.HiWi, ok && c < g.Ci) *
                                    relu_gate(ldg_keep_if(mp + c * g.HiWi, ok && c < g.Ci));
            }
        }
    }

    __device__ void load_a(const AState& s, const Tile&, int ks, int tid, float (&v)[32]) const
    {
        if (g.mode == 0) {
            // One tap, 32 consecutive channels.
            uint32_t tap, chunk, tr, tq;
            g.f_cchunks.divmod(uint32_t(ks), tap, chunk);
            g.f_t.divmod(tap, tr, tq);
            const int h = s.h0 + int(tr);
            const int w = s.w0 + int(tq);
            const bool ok = unsigned(h) < unsigned(g.Hi) && unsigned(w) < unsigned(g.Wi);
            const int cleft = g.Ci - int(chunk) * 32;   // channels of this chunk that exist
            const int off = s.base + int(chunk) * 32 * g.HiWi + int(tr) * g.Wi + int(tq);
            const float* p = g.in + off;
            if (g.mask == nullptr && cleft >= 32) {
                // a whole chunk: one predicate for all 32 loads
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = ldg_keep_if(p + i * g.HiWi, ok);
            } else if (g.mask == nullptr) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = ldg_keep_if(p + i * g.HiWi, ok && i < cleft);
            } else {
                const float* mp = g.mask + off;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = ldg_keep_if(p + i * g.HiWi, ok && i < cleft) *
                           relu_gate(ldg_keep_if(mp + i * g.HiWi, ok && i < cleft));
            }
        } else if (g.mode == 1) {
            switch (g.lcp) {
            case 0: load_taps<0>(s, ks, v); break;
            case 1: load_taps<1>(s, ks, v); break;
            case 2: load_taps<2>(s, ks, v); break;
            case 3: load_taps<3>(s, ks, v); break;
            default: load_taps<4>(s, ks, v); break;
            }
        } else {
            // Generic order: lane l decodes k = ks*32 + l, the warp shares it.
            const int k = ks * kBK + (tid & 31);
            int koff = 0, krs = 0x7FFF0000;   // past K: the tap lands far outside
            if (k < g.K) {
                uint32_t c, rem, r, q;
                g.f_tt.divmod(uint32_t(k), c, rem);
                g.f_t.divmod(rem, r, q);
                koff = int(c) * g.HiWi + int(r) * g.Wi + int(q);
                krs = int((r << 16) | q);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int off = __shfl_sync(0xffffffffu, koff, i);
                const int rs = __shfl_sync(0xffffffffu, krs, i);
                const int h = s.h0 + (rs >> 16);
                const int w = s.w0 + (rs & 0xFFFF);
                const bool in = unsigned(h) < unsigned(g.Hi) && unsigned(w) < unsigned(g.Wi);
                v[i] = ldg_keep_if(g.in + (s.base + off), in);
                if (g.mask != nullptr) v[i] *= relu_gate(ldg_keep_if(g.mask + (s.base + off), in));
            }
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
        float* opix;   // out[n][0][h][w], (h, w) = (p*so - oo, q*so - oo): may lie before the row/image
        bool valid;
        int hrem, wrem;   // rows/cols of the output left below/right of this pixel's phase block
        int hmin, wmin;   // phases a < hmin (b < wmin) fall above (left of) the output: -h, -w
    };
    __device__ EState e_setup(const Tile& tl, int row) const
    {
        EState e;
        const int m = tl.m0 + row;
        e.valid = m < g.M;
        uint32_t n = 0, pq = 0, p = 0, q = 0;
        if (e.valid) {
            g.f_gpq.divmod(uint32_t(m), n, pq);
            g.f_gq.divmod(pq, p, q);
        }
        const int h = int(p) * o.so - o.oo, w = int(q) * o.so - o.oo;
        e.hrem = o.Ho - h;
        e.wrem = o.Wo - w;
        e.hmin = -h;
        e.wmin = -w;
        e.opix = o.out + (ptrdiff_t(n) * o.Co * o.HoWo + ptrdiff_t(h) * o.Wo + w);
        return e;
    }

    // epilogue of split trailing tile b, once its pieces are summed
    __device__ void reduce_store(int b, int row, int c0, const uint32_t (&r)[32]) const;

    __device__ void store(const EState& e, const Tile& tl, int row, int c0, const uint32_t (&r)[32]) const
    {
        if (tl.part >= 0) {
            float4* d = reinterpret_cast<float4*>(part_buf + (size_t(tl.part) * kBM + row) * BN + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                d[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                   __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
            return;
        }
        if (o.so == 1) {
            // the 32 columns' biases: lane i loads column c0 + i once and the
            // warp shares them (every epilogue lane calls store, valid row or not)
            const int chl = tl.n0 + c0 + int(threadIdx.x & 31);
            const float bl = (o.bias && chl < o.Co) ? __ldg(o.bias + chl) : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float bias = __shfl_sync(0xffffffffu, bl, i);
                const int ch = tl.n0 + c0 + i;
                if (e.valid && ch < o.Co) {
                    const float v = __uint_as_float(r[i]) + bias;
                    e.opix[size_t(ch) * o.HoWo] = o.relu && !(v > 0.f) ? 0.f : v;
                }
            }
            return;
        }
        if (!e.valid) return;
        if (o.vec == 2) {
            // so = 4, oo = 2: the four phases b of one (ch, a) are output
            // columns w .. w + 3 with w = 4q - 2 (even): two 8-byte-aligned
            // pairs, the first left of the image when q = 0, the second right
            // of it when w + 2 = Wo
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const int col = tl.n0 + c0 + i;
                const int ch = col >> 4, a = (col >> 2) & 3;
                if (ch < o.Co && a < e.hrem && a >= e.hmin) {
                    float* rowp = e.opix + (size_t(ch) * o.HoWo + a * o.Wo);
                    if (e.wmin <= 0)
                        *reinterpret_cast<float2*>(rowp) = make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                    if (e.wrem > 2)
                        *reinterpret_cast<float2*>(rowp + 2) =
                            make_float2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                }
            }
        } else if (o.vec) {
            // columns (ch, a, b) with b fastest: the so phases b of one (ch, a)
            // are so adjacent columns and so adjacent floats of output row
            // h + a (oo = 0 and w = so * q is a multiple of so, so wrem >= so)
            if (o.so == 4) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int col = tl.n0 + c0 + i;
                    const int ch = col >> 4, a = (col >> 2) & 3;
                    if (ch < o.Co && a < e.hrem)
                        *reinterpret_cast<float4*>(e.opix + size_t(ch) * o.HoWo + a * o.Wo) =
                            make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                                        __uint_as_float(r[i + 3]));
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const int col = tl.n0 + c0 + i;
                    const int ch = col >> 2, a = (col >> 1) & 1;
                    if (ch < o.Co && a < e.hrem)
                        *reinterpret_cast<float2*>(e.opix + size_t(ch) * o.HoWo + a * o.Wo) =
                            make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                }
            }
        } else {
            const int ss = o.so * o.so;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int col = tl.n0 + c0 + i;
                const int ch = col / ss, ab = col - ch * ss;
                const int a = ab / o.so, b = ab - a * o.so;
                if (ch < o.Co && a < e.hrem && b < e.wrem && a >= e.hmin && b >= e.wmin)
                    e.opix[size_t(ch) * o.HoWo + a * o.Wo + b] = __uint_as_float(r[i]);
            }
        }
    }
};

template <int BN>
__device__ void ConvGatherProb<BN>::reduce_store(int b, int row, int c0, const uint32_t (&r)[32]) const
{
    const Tile tl = whole_tile(full_units + b);
    store(e_setup(tl, row), tl, row, c0, r);
}

// The forward of a space-to-depth convolution on the flat kernel
// (gemm_flat.cuh): a stride-1 window over the channel-blocked space-to-depth
// copy, at most 64 columns (one column tile), the A operand read by the
// tensor core straight from the TMA box.  Rows of a tile are 128
// consecutive flat positions v = p * Wt + q of one image; those with q >= Gq
// (or past the image's last row) are computed and dropped.
template <int BN>
struct ConvFlatProb {
    int terms = 3;   // tensor-core products per K step: 3 (3xTF32) or 1 (TF32)
    FlatGeom fg;
    OutGeom o;
    const float* bimg;   // build_bimage16 image, K order 3 (16-channel chunk, tap, channel), taps padded to 2 * spc
    int n_tiles, k_stages;

    __device__ int num_tiles() const { return fg.Nb * fg.tpi * n_tiles; }
    __device__ const float* b_image(int nt, int ks) const
    {
        return bimg + (size_t(nt) * k_stages + ks) * 4 * size_t(BN) * 16;   // two taps of 2 * BN rows
    }
    using EState = typename ConvGatherProb<64>::EState;
    __device__ EState e_setup(int t, int row) const
    {
        const int m = t / n_tiles;
        const int n = m / fg.tpi;
        const int v = (m % fg.tpi) * kBM + row;
        uint32_t p = 0, q = 0;
        fg.f_wt.divmod(uint32_t(v), p, q);
        EState e;
        e.valid = v < fg.vpi && int(q) < fg.Gq;
        if (!e.valid) p = q = 0;
        const int h = int(p) * o.so - o.oo, w = int(q) * o.so - o.oo;
        e.hrem = o.Ho - h;
        e.wrem = o.Wo - w;
        e.hmin = -h;
        e.wmin = -w;
        e.opix = o.out + (ptrdiff_t(n) * o.Co * o.HoWo + ptrdiff_t(h) * o.Wo + w);
        return e;
    }
    // columns n0 + c0 .. + 31 of row `row`; those past the tile's own columns
    // (BN not a multiple of 32) lie past the output's columns and are dropped
    // by the store, since a flat GEMM has a single column tile
    __device__ void store(const EState& e, int n0, int row, int c0, const uint32_t (&r)[32]) const
    {
        ConvGatherProb<64> helper;
        helper.o = o;
        helper.part_buf = nullptr;
        Tile tl;
        tl.n0 = n0;
        tl.m0 = 0;
        tl.ks0 = tl.ks1 = 0;
        tl.grp = 0;
        tl.part = -1;
        helper.store(e, tl, row, c0, r);
    }
};

// Flat-kernel launch (conv_flat.cu): one column tile of bn (16, 32, 48 or 64)
// columns over the geometry fg, B image img (build_bimage16 layout, K order 3).
cudaError_t dispatch_flat(int bn, const FlatGeom& fg, const OutGeom& o, const float* img, cudaStream_t st);

}  // namespace cb200
