// gemm_patch.cuh -- implicit-GEMM convolution whose A operand (the column
// matrix of the page's im2col step) is built from input patches staged in
// shared memory.
//
// A tile is 128 consecutive output positions of ONE image (tiles never straddle
// images; the last tile of an image is partial).  For each chunk of channels
// the tile reads, from the gathered tensor, every input row any tap of the tile
// touches -- full-width rows, one contiguous run per channel -- into shared
// memory with coalesced loads.  The taps of that chunk are then gathered from
// shared memory: per element one shared load instead of one global load, and a
// global request count lower by about the number of taps.
//
// Roles (480 threads, one CTA per SM, persistent over tiles):
//   warps 0-3, 4-7   two converter groups.  A converter thread owns one output
//                    position (one A row): per stage it reads its 32 K values
//                    from the patch, splits them into 3xTF32 hi/lo and writes
//                    both into the stage's tensor-memory columns; the group's
//                    first thread bulk-copies the stage's pre-split B tiles.
//   warp 8           patch loader: fills a ring of two patch buffers one
//                    chunk ahead, one bulk copy per channel run.
//   warps 9, 10      MMA issuers (lane 0 of each; warp 9 also allocates tensor
//                    memory): tcgen05.mma with A from tensor memory and B from
//                    shared memory.
//   warps 11-14      epilogue: adds the two issuers' accumulators and hands
//                    the rows to the problem's store.
//
// Two issuers, because one thread cannot issue tcgen05.mma fast enough to keep
// the tensor core busy on tiles this narrow (N <= 128): measured on GB300, a
// single thread issues about one MMA per 25 ns whatever N is, while an
// M=128, N=64, K=8 tf32 MMA takes the pipe about 16 ns, and every stage
// handshake (barrier wait + commit) stalls the issuing thread further.  With
// two threads feeding separate accumulators the pipe stays near its peak.
//
// The K stages of a tile are split by parity of the CTA-wide stage counter c:
// stage c is filled by converter group c % 2 into slot c % S (S even, so the
// slot has the same parity) and consumed by issuer c % 2 into that issuer's
// accumulator; the epilogue adds accumulator 0 and accumulator 1 (always in
// that order, so results do not depend on timing).  Each slot therefore has
// exactly one filler group and one consumer, each visiting it in stage order,
// so every parity wait is at most one phase ahead of its barrier.  Every
// converter warp waits on every chunk's "patch loaded" barrier and signals its
// "patch read" barrier.  All waits are bounded (ptx.cuh).
#pragma once
#include <atomic>
#include <cuda.h>   // CUtensorMap (the type only; encoding is done on the host through the runtime's driver entry point)

#include "gemm_tc.cuh"

namespace cb200 {

struct PatchGeom {
    const float* in;   // gathered tensor [Nb][Ci][Hi][Wi]
    int Nb, Ci, Hi, Wi, HiWi, CiHiWi;
    long long total;   // Nb*Ci*Hi*Wi (copies never read past it)
    int Gp, Gq, GpGq;  // output grid of one image
    int tpi;           // tiles per image
    int sp, o, T;      // window: h = p*sp + o + tap_r
    int mode;          // 0: 32-channel chunks, stage = one tap; 1: Ci <= 16, stage = 32/Cp taps
    int Cp, lcp;       // mode 1: channels padded to Cp = 2^lcp
    int nch;           // channel chunks per tile (mode 1: 1)
    int spc;           // stages per chunk
    // Tensor-map form with at most 16 channels in the last chunk: its stages
    // take two taps of 16 channels each (half), spch = ceil(T*T / 2) of them
    // instead of spc (otherwise half = 0, spch = spc).
    int half, spch;
    int pc;            // channels one patch holds (mode 0: 32, mode 1: Ci)
    FastDiv f_gq, f_t;
    __host__ __device__ int stages_of(int cc) const { return cc == nch - 1 ? spch : spc; }
    // K stages of chunks [cc0, cc1), cc0 < cc1
    __host__ __device__ int stages_range(int cc0, int cc1) const
    {
        return (cc1 - cc0) * spc - (cc1 == nch ? spc - spch : 0);
    }
    // Tensor-map form (mode 0 only): the gathered tensor re-laid as
    // [Nb][Ci/32][Hi][Wi][32] (channels innermost, zero-padded to 32) and one
    // 4-D TMA box per (tile, chunk): rows [p_lo*sp + o, + rowsT), columns
    // [o, o + Wt), 32 channels -- pixel-major, 128 bytes per pixel, 128-byte
    // swizzled, and zero wherever the window leaves the image.
    int Wt, rowsT, Cb;
    uint32_t tbytes;   // shared-memory bytes of one box buffer (multiple of 1024)
    uint32_t tbox;     // bytes one box delivers
    alignas(64) CUtensorMap tmap;
};

// Floats between consecutive channels of a staged patch holding `run`
// floats per channel: at least run + 6 (room for a 16-byte-aligned copy of
// the run, rounded out on both sides) and congruent to Hi*Wi modulo 4, so
// every channel's run starts at the same offset (0..3) within its block.
__host__ __device__ inline int patch_cstride(int run, int HiWi)
{
    int cps = run + 6;
    cps += ((HiWi - cps) % 4 + 4) % 4;
    return cps;
}

// Largest patch (floats) any tile of this geometry stages.
inline int max_patch_floats(const PatchGeom& g)
{
    int best = 0;
    for (int ti = 0; ti < g.tpi; ++ti) {
        const int first = ti * kBM;
        const int last = (first + kBM < g.GpGq ? first + kBM : g.GpGq) - 1;
        const int p_lo = first / g.Gq, p_hi = last / g.Gq;
        int h_lo = p_lo * g.sp + g.o, h_hi = p_hi * g.sp + g.o + g.T - 1;
        if (h_lo < 0) h_lo = 0;
        if (h_hi > g.Hi - 1) h_hi = g.Hi - 1;
        const int rows = h_hi >= h_lo ? h_hi - h_lo + 1 : 0;
        const int f = patch_cstride(rows * g.Wi, g.HiWi) * g.pc;
        if (f > best) best = f;
    }
    return best;
}

// Mode 1 (Ci <= 16): 32 / CP whole taps per stage, CP (padded) channels each.
template <int LCP>
__device__ __forceinline__ void patch_taps(const PatchGeom& g, const float* pbuf, int j, int hp0, int wp0, bool pvalid,
                                           int h_lo, int cstride, float (&v)[32])
{
    constexpr int CP = 1 << LCP, TPS = 32 >> LCP;
    const int TT = g.T * g.T;
#pragma unroll
    for (int t = 0; t < TPS; ++t) {
        const int tap = j * TPS + t;
        uint32_t tr, tq;
        g.f_t.divmod(uint32_t(tap), tr, tq);
        const int h = hp0 + int(tr), w = wp0 + int(tq);
        const bool ok = pvalid && tap < TT && unsigned(h) < unsigned(g.Hi) && unsigned(w) < unsigned(g.Wi);
        const float* p = pbuf + ((h - h_lo) * g.Wi + w);
#pragma unroll
        for (int c = 0; c < CP; ++c) v[t * CP + c] = (ok && c < g.Ci) ? p[c * cstride] : 0.f;
    }
}

// DB2 asks for two accumulator buffers per issuer even where that leaves only
// four A stages (64-wide tiles): worth it when tiles have few K stages, so that
// the epilogue of one tile would otherwise stall the next tile's MMAs.
//
// STACK (tiles at most 64 wide, 3xTF32): per 8-deep K step two MMAs instead of
// three.  The stage's B tiles lie back to back in shared memory (hi rows, then
// lo rows), so one MMA with N = 2*BN multiplies A_hi by both: hi*hi into the
// accumulator's first BN columns, hi*lo into the next BN; a second MMA (N = BN)
// adds lo*hi to the first BN.  The epilogue adds the two halves.  Each A column
// block is then read from tensor memory twice per K step instead of three times.
template <int BN, bool DB2 = false, bool STACK = false>
struct PatchCfg {
    static_assert(BN <= 128, "the patch kernel keeps an accumulator per issuer and at least four A stages in "
                             "tensor memory");
    static_assert(!DB2 || BN <= 64, "two buffers per issuer and four A stages need tiles at most 64 wide");
    static_assert(!STACK || BN <= 64, "stacked B tiles need 2*BN <= 128 accumulator columns");
    static constexpr int kThreads = 480;
    static constexpr int kAccW = STACK ? 2 * BN : BN;   // accumulator columns per issuer and buffer
    // accumulator buffers per issuer: two (the epilogue of tile i overlaps the
    // main loop of tile i+1) when six A stages still fit beside them (or DB2
    // and four still fit), else one
    static constexpr int kDBuf = ((DB2 && 512 - 4 * kAccW >= 4 * 64) || (512 - 4 * kAccW) / 64 >= 6) ? 2 : 1;
    static constexpr int kTmemStages0 = (512 - 2 * kDBuf * kAccW) / 64;
    static constexpr int kStages = (kTmemStages0 > 6 ? 6 : kTmemStages0) & ~1;   // even: slot parity = issuer
    static_assert(kStages >= 4, "too few A stages fit in tensor memory");
    static constexpr uint32_t kBTile = BN * kBK * 4;
    static constexpr uint32_t kStage = 2 * kBTile;
    static constexpr uint32_t kACol = uint32_t(2 * kDBuf * kAccW);   // accumulators: [buffer][issuer]
    static constexpr size_t kCtlBytes = 512;
    static constexpr size_t kMaxSmem = 227 * 1024;
    // two patch buffers share what the B stages leave
    static constexpr size_t kPatchBytes =
        ((kMaxSmem - 1024 - kCtlBytes - size_t(kStages) * kStage) / 2) & ~size_t(15);
    static constexpr int kPatchFloats = int(kPatchBytes / 4);
    static constexpr size_t kSmemBytes = 1024 + size_t(kStages) * kStage + 2 * kPatchBytes + kCtlBytes;
    static constexpr uint32_t kIdesc = idesc_tf32(kBM, BN);
    static constexpr uint32_t kIdesc2 = idesc_tf32(kBM, STACK ? 2 * BN : BN);   // the stacked hi*[hi; lo] MMA
};

// Dynamic shared memory of the tensor-map form: alignment slack, B stages, two
// box buffers of `tbytes` each, control block.
template <int BN, bool DB2 = false, bool STACK = false>
constexpr size_t patch_tma_smem(uint32_t tbytes)
{
    using C = PatchCfg<BN, DB2, STACK>;
    return 1024 + size_t(C::kStages) * C::kStage + 2 * size_t(tbytes) + C::kCtlBytes;
}

// One work unit of the patch kernel (see the problem interface below).
struct PatchUnit {
    int tt;         // whole tile
    int cc0, cc1;   // channel chunks [cc0, cc1)
    int part;       // >= 0: partial-tile slot of a K piece of a split trailing tile
};

struct PatchCtl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t accf[2];
    uint64_t acce[2];
    uint64_t pfull[2];     // patch buffer holds its chunk (loader arrival)
    uint64_t pempty[2];    // every converter warp is done with the buffer (8 arrivals)
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort_flag;
};

// The problem supplies the B image location and the epilogue (same interface
// as ConvGatherProb: b_image, EState, e_setup, store).  Work units: unit(t)
// gives the whole tile tt it belongs to (decoded as n_tile = tt % n_tiles,
// image, tile in image), its chunk range [cc0, cc1) and, for one K piece of a
// split trailing tile, the slot of its partial tile (part >= 0).  Units can
// differ in stage count, so every role keeps the CTA-wide stage counter as a
// running sum.
//
// TMA selects how a chunk's patch arrives: per-channel bulk copies of the
// NCHW tensor (channel-major patch, any channel count), or one 4-D tensor-map
// box of the channel-blocked copy (pixel-major swizzled patch, mode 0): there
// a converter thread reads its 32 channels with eight conflict-free 16-byte
// loads and needs no bounds tests, since the box is zero outside the image.
template <class Prob, int BN, bool TMA, bool DB2, int TERMS, bool STACK>
__global__ void __launch_bounds__(PatchCfg<BN, DB2, STACK>::kThreads, 1) tc_patch_kernel(const __grid_constant__ Prob prob, int* err_word)
{
    static_assert(!STACK || TERMS == 3, "stacking pairs the hi and lo B tiles of 3xTF32");
    using Cfg = PatchCfg<BN, DB2, STACK>;
    constexpr int AW = Cfg::kAccW;
    constexpr int S = Cfg::kStages;
    constexpr int DB = Cfg::kDBuf;
    const PatchGeom& g = prob.pg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const size_t pbytes = TMA ? size_t(g.tbytes) : Cfg::kPatchBytes;
    float* patch[2] = {reinterpret_cast<float*>(smem + size_t(S) * Cfg::kStage),
                       reinterpret_cast<float*>(smem + size_t(S) * Cfg::kStage + pbytes)};
    PatchCtl* ctl = reinterpret_cast<PatchCtl*>(smem + size_t(S) * Cfg::kStage + 2 * pbytes);
    volatile int* abort_flag = &ctl->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t smem_base = smem_u32(smem);
    auto b_hi = [&](int s) { return smem_base + uint32_t(s) * Cfg::kStage; };
    auto b_lo = [&](int s) { return b_hi(s) + Cfg::kBTile; };
    auto a_col = [&](int s) { return Cfg::kACol + uint32_t(s) * 64u; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], 5);   // 4 converter warps + the B bulk copy
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->accf[b], 2);   // one commit per issuer
            mbar_init(&ctl->acce[b], 4);
            mbar_init(&ctl->pfull[b], 1);
            mbar_init(&ctl->pempty[b], 8);
            mbar_init(&ctl->drain[b], 1);
        }
        ctl->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(&ctl->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    // set-up above overlaps the previous kernel when launched with PDL
    griddep_wait();
    griddep_launch();

    const int num_tiles = prob.num_tiles();
    // TERMS == 3: hi*hi + hi*lo + lo*hi (fp32-faithful); TERMS == 1: hi*hi only
    constexpr bool three = TERMS == 3;
    constexpr uint32_t b_bytes = (three ? 2u : 1u) * Cfg::kBTile;
    auto fail = [&]() {
        ctl->abort_flag = 1;
        atomicOr(err_word, kDevErrTimeout);
    };

    // Patch geometry of tile t: image, tile in image, first/last output
    // position, and the clamped input-row range every tap of the tile touches.
    struct TileGeo {
        int n, first, last, h_lo, rows, p_lo;
    };
    auto tile_geo = [&](int t) {
        TileGeo q;
        const int mt = t / prob.n_tiles;
        q.n = mt / g.tpi;
        q.first = (mt % g.tpi) * kBM;
        q.last = (q.first + kBM < g.GpGq ? q.first + kBM : g.GpGq) - 1;
        q.p_lo = q.first / g.Gq;
        int h_lo = q.p_lo * g.sp + g.o;
        int h_hi = (q.last / g.Gq) * g.sp + g.o + g.T - 1;
        if (h_lo < 0) h_lo = 0;
        if (h_hi > g.Hi - 1) h_hi = g.Hi - 1;
        q.h_lo = h_lo;
        q.rows = h_hi >= h_lo ? h_hi - h_lo + 1 : 0;
        return q;
    };

    if (warp < 8) {
        // ---------------- converter groups ----------------
        const int grp = warp >> 2;
        const int tid = threadIdx.x - 128 * grp;   // 0..127: the A row this thread owns
        uint32_t u = 0;                            // chunk counter of this CTA
        uint32_t cst = 0;                          // stage counter of this CTA
        int last_issued = -1;
        bool ok = true;
        const uint32_t tbase = tmem_base + (uint32_t((warp & 3) * 32) << 16);
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const PatchUnit un = prob.unit(t);
            const TileGeo q = tile_geo(un.tt);
            const int cstride = patch_cstride(q.rows * g.Wi, g.HiWi);   // floats per channel in the patch
            const int pix = q.first + tid;
            const bool pvalid = pix <= q.last;
            uint32_t pp = 0, pq = 0;
            // tensor-map form: a row past the tile's last position reads the
            // last position's pixels (any in-box address will do: the
            // epilogue drops the row)
            if (pvalid || TMA) g.f_gq.divmod(uint32_t(pvalid ? pix : q.last), pp, pq);
            const int hp0 = int(pp) * g.sp + g.o;  // input row of tap 0
            const int wp0 = int(pq) * g.sp + g.o;  // input column of tap 0
            const int tpix0 = (int(pp) - q.p_lo) * g.sp * g.Wt + int(pq) * g.sp;   // box pixel of tap 0
            for (int cc = un.cc0; cc < un.cc1 && ok; ++cc, ++u) {
                const int pb = int(u & 1u);
                // every channel run of this chunk starts s0 floats into its block
                const long long x0 = (long long)q.n * g.CiHiWi + (long long)(cc * 32) * g.HiWi + (long long)q.h_lo * g.Wi;
                const float* pbuf = patch[pb] + (TMA ? 0 : int(x0 & 3));
                if (!mbar_wait_warp(&ctl->pfull[pb], (u >> 1) & 1u, abort_flag)) { ok = false; break; }
                const uint32_t c_first = cst;   // CTA-wide counter of the chunk's first stage
                const int nst = g.stages_of(cc);
                cst += uint32_t(nst);
                const bool halfc = TMA && g.half && cc == g.nch - 1;
                const int j0 = int((uint32_t(grp) + 2u - (c_first & 1u)) & 1u);   // first stage of this group
                for (int j = j0; j < nst; j += 2) {
                    const uint32_t c = c_first + uint32_t(j);
                    const int slot = int(c % uint32_t(S));
                    const uint32_t phase = (c / uint32_t(S)) & 1u;
                    const int ks = cc * g.spc + j;
                    float va[32];
                    if (halfc) {
                        // taps 2j and 2j + 1, channels 0..15 of the chunk each
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int tap = 2 * j + h;
                            if (tap < g.T * g.T) {
                                uint32_t tr, tq;
                                g.f_t.divmod(uint32_t(tap), tr, tq);
                                const int P = tpix0 + int(tr) * g.Wt + int(tq);
                                const uint8_t* rowp = reinterpret_cast<const uint8_t*>(pbuf) + size_t(P) * 128;
#pragma unroll
                                for (int c4 = 0; c4 < 4; ++c4) {
                                    const float4 v = *reinterpret_cast<const float4*>(rowp + ((c4 ^ (P & 7)) << 4));
                                    va[16 * h + 4 * c4] = v.x;
                                    va[16 * h + 4 * c4 + 1] = v.y;
                                    va[16 * h + 4 * c4 + 2] = v.z;
                                    va[16 * h + 4 * c4 + 3] = v.w;
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i) va[16 * h + i] = 0.f;
                            }
                        }
                    } else if constexpr (TMA) {
                        uint32_t tr, tq;
                        g.f_t.divmod(uint32_t(j), tr, tq);
                        const int P = tpix0 + int(tr) * g.Wt + int(tq);
                        const uint8_t* rowp = reinterpret_cast<const uint8_t*>(pbuf) + size_t(P) * 128;
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 v = *reinterpret_cast<const float4*>(rowp + ((c4 ^ (P & 7)) << 4));
                            va[4 * c4] = v.x;
                            va[4 * c4 + 1] = v.y;
                            va[4 * c4 + 2] = v.z;
                            va[4 * c4 + 3] = v.w;
                        }
                    } else if (g.mode == 0) {
                        uint32_t tr, tq;
                        g.f_t.divmod(uint32_t(j), tr, tq);
                        const int h = hp0 + int(tr), w = wp0 + int(tq);
                        const bool okp = pvalid && unsigned(h) < unsigned(g.Hi) && unsigned(w) < unsigned(g.Wi);
                        const int climit = okp ? g.Ci - cc * 32 : 0;
                        const float* pp0 = pbuf + ((h - q.h_lo) * g.Wi + w);
#pragma unroll
                        for (int i = 0; i < 32; ++i) va[i] = i < climit ? pp0[i * cstride] : 0.f;
                    } else {
                        switch (g.lcp) {
                        case 0: patch_taps<0>(g, pbuf, j, hp0, wp0, pvalid, q.h_lo, cstride, va); break;
                        case 1: patch_taps<1>(g, pbuf, j, hp0, wp0, pvalid, q.h_lo, cstride, va); break;
                        case 2: patch_taps<2>(g, pbuf, j, hp0, wp0, pvalid, q.h_lo, cstride, va); break;
                        case 3: patch_taps<3>(g, pbuf, j, hp0, wp0, pvalid, q.h_lo, cstride, va); break;
                        default: patch_taps<4>(g, pbuf, j, hp0, wp0, pvalid, q.h_lo, cstride, va); break;
                        }
                    }
                    if (!mbar_wait_warp(&ctl->empty[slot], phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (tid == 0) {
                        mbar_arrive_expect_tx(&ctl->full[slot], b_bytes);
                        bulk_g2s(smem + (b_hi(slot) - smem_base), prob.b_image_t(un.tt, ks), b_bytes,
                                 &ctl->full[slot]);
                        last_issued = int(c);
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h4 = 0; h4 < 4; ++h4) {
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) split_tf32(va[8 * h4 + i], hi[i], lo[i]);
                        tmem_st8(tbase + a_col(slot) + 8 * h4, hi);
                        if (three) tmem_st8(tbase + a_col(slot) + 32 + 8 * h4, lo);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->full[slot]);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->pempty[pb]);   // this warp is done reading the buffer
            }
        }
        if (!ok) {
            fail();
            if (tid == 0 && last_issued >= 0) {
                for (int c = last_issued; c >= 0 && c > last_issued - S; c -= 2) {
                    uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->full[c % S], uint32_t(c / S) & 1u) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 8) {
        // ---------------- patch loader ----------------
        uint32_t u = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const PatchUnit un = prob.unit(t);
            const TileGeo q = tile_geo(un.tt);
            const int cstride = patch_cstride(q.rows * g.Wi, g.HiWi);
            for (int cc = un.cc0; cc < un.cc1 && ok; ++cc, ++u) {
                const int pb = int(u & 1u);
                // chunk u - 2 (same buffer) must be fully read
                if (u >= 2 && !mbar_wait_warp(&ctl->pempty[pb], ((u >> 1) - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if constexpr (TMA) {
                    // one box: 32 channels x Wt columns x rowsT rows of image n
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&ctl->pfull[pb], g.tbox);
                        tma_load_4d(patch[pb], &prob.pg.tmap, 0, g.o, q.p_lo * g.sp + g.o, q.n * g.Cb + cc,
                                    &ctl->pfull[pb]);
                    }
                    __syncwarp();
                    continue;
                }
                // lane c copies channel cc*32 + c: its run of rows*Wi floats, widened
                // to 16-byte boundaries, with one bulk copy into block c of the buffer;
                // a tail that would reach past the tensor's last 16-byte boundary
                // (at most 3 floats) is copied with plain loads instead
                const int c = lane;
                const int run = q.rows * g.Wi;
                const bool has = c < g.pc && cc * 32 + c < g.Ci && run > 0;
                const long long x = (long long)q.n * g.CiHiWi + (long long)(cc * 32 + c) * g.HiWi +
                                    (long long)q.h_lo * g.Wi;   // run start (floats into the tensor)
                const long long x0 = x - (long long)c * g.HiWi;   // start of channel cc*32's run
                const int sh = int(x0 & 3);                        // common offset of every run in its block
                const long long a0 = x & ~3LL;                     // 16-byte-aligned copy start
                long long a1 = (x + run + 3) & ~3LL;               // 16-byte-aligned copy end
                const long long lim = g.total & ~3LL;
                if (a1 > lim) a1 = lim;
                const uint32_t bytes = has && a1 > a0 ? uint32_t((a1 - a0) * 4) : 0u;
                // destination: element x of the run lands at block c + sh
                const int dst_f = c * cstride + sh - int(x - a0);
                uint32_t total_bytes = bytes;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) total_bytes += __shfl_xor_sync(0xffffffffu, total_bytes, o);
                if (has) {
                    // tail past the last aligned boundary of the tensor
                    for (long long e = (a1 > x ? a1 : x); e < x + run; ++e)
                        patch[pb][dst_f + int(e - a0)] = __ldg(g.in + e);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(&ctl->pfull[pb], total_bytes);
                __syncwarp();
                if (bytes) bulk_g2s(patch[pb] + dst_f, g.in + a0, bytes, &ctl->pfull[pb]);
            }
        }
        if (!ok) fail();
    } else if (warp == 9 || warp == 10) {
        // ---------------- MMA issuers ----------------
        const uint32_t me = uint32_t(warp - 9);
        if (lane == 0) {
            int local = 0;
            bool ok = true;
            bool issued_any = false;
            uint32_t c0 = 0;   // CTA-wide counter of the unit's first stage
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
                const PatchUnit un = prob.unit(t);
                const uint32_t k_stages = uint32_t(g.stages_range(un.cc0, un.cc1));
                const int buf = local % DB;
                const uint32_t acc_phase = uint32_t(local / DB) & 1u;
                if (!mbar_wait(&ctl->acce[buf], acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t((2 * buf + int(me)) * AW);
                uint32_t accumulate = 0;
                for (uint32_t ks = me ^ (c0 & 1u); ks < k_stages; ks += 2) {
                    const uint32_t c = c0 + ks;
                    const int slot = int(c % uint32_t(S));
                    if (!mbar_wait(&ctl->full[slot], (c / uint32_t(S)) & 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 8; ++kk) {
                        const uint64_t bh = sdesc_k_sw128(b_hi(slot) + kk * 32);
                        const uint64_t bl = sdesc_k_sw128(b_lo(slot) + kk * 32);
                        const uint32_t ah = tmem_base + a_col(slot) + uint32_t(kk * 8);
                        const uint32_t al = ah + 32;
                        if (STACK) {
                            // columns [0, BN): hi*hi (+ lo*hi below); [BN, 2BN): hi*lo
                            mma_tf32_ts(d_tmem, ah, bh, Cfg::kIdesc2, accumulate);
                            mma_tf32_ts(d_tmem, al, bh, Cfg::kIdesc, 1);
                        } else if (three) {
                            mma_tf32_ts(d_tmem, al, bh, Cfg::kIdesc, accumulate);
                            mma_tf32_ts(d_tmem, ah, bl, Cfg::kIdesc, 1);
                            mma_tf32_ts(d_tmem, ah, bh, Cfg::kIdesc, 1);
                        } else {
                            mma_tf32_ts(d_tmem, ah, bh, Cfg::kIdesc, accumulate);
                        }
                        accumulate = 1;
                    }
                    issued_any = true;
                    mma_commit(&ctl->empty[slot]);
                }
                if (!ok) break;
                c0 += k_stages;
                // arrives once this issuer's MMAs of the tile are done (at once
                // if it had none: a one-stage tile)
                mma_commit(&ctl->accf[buf]);
            }
            if (!ok) {
                fail();
                if (issued_any) {
                    mma_commit(&ctl->drain[me]);
                    uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->drain[me], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;
        const int row = q * 32 + lane;
        uint32_t c0 = 0;   // CTA-wide counter of the unit's first stage
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
            const PatchUnit un = prob.unit(t);
            const uint32_t k_stages = uint32_t(g.stages_range(un.cc0, un.cc1));
            const int buf = local % DB;
            const uint32_t acc_phase = uint32_t(local / DB) & 1u;
            if (!mbar_wait_warp(&ctl->accf[buf], acc_phase, abort_flag)) { ok = false; break; }
            tc_fence_after();
            // a one-stage unit leaves the other issuer's accumulator untouched
            const bool use0 = k_stages >= 2 || (c0 & 1u) == 0;
            const bool use1 = k_stages >= 2 || (c0 & 1u) == 1;
            c0 += k_stages;
            Tile tile = prob.tile_t(un.tt);
            tile.part = un.part;
            typename Prob::EState es = prob.e_setup_t(un.tt, row);
            const uint32_t lane_base = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(2 * buf * AW);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r0[32], r1[32];
                if constexpr (STACK) {
                    // each issuer's hi*lo half added to its first half, one
                    // issuer at a time (keeps two register blocks live)
                    tmem_ld32x2(lane_base + uint32_t(c), lane_base + uint32_t(BN + c), r0, r1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r0[i] = __float_as_uint(__uint_as_float(r0[i]) + __uint_as_float(r1[i]));
                    uint32_t h[32];
                    tmem_ld32x2(lane_base + uint32_t(AW + c), lane_base + uint32_t(AW + BN + c), r1, h);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r1[i] = __float_as_uint(__uint_as_float(r1[i]) + __uint_as_float(h[i]));
                } else {
                    tmem_ld32x2(lane_base + uint32_t(c), lane_base + uint32_t(AW + c), r0, r1);
                }
                if (c + 32 >= BN) {
                    // the accumulators are free once the last columns are in registers
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->acce[buf]);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r0[i] = __float_as_uint((use0 ? __uint_as_float(r0[i]) : 0.f) +
                                            (use1 ? __uint_as_float(r1[i]) : 0.f));
                prob.store(es, tile, row, c, r0);
            }
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <class Prob, int BN, bool TMA, bool DB2, int TERMS, bool STACK>
cudaError_t launch_tc_patch_terms(const Prob& prob, int num_tiles, int* err_word, cudaStream_t stream)
{
    using Cfg = PatchCfg<BN, DB2, STACK>;
    static std::atomic<bool> attr_set{false};   // set once; racing setters are harmless
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_patch_kernel<Prob, BN, TMA, DB2, TERMS, STACK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kMaxSmem));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (num_tiles <= 0) return cudaSuccess;
    const size_t smem = TMA ? patch_tma_smem<BN, DB2, STACK>(prob.pg.tbytes) : Cfg::kSmemBytes;
    int grid = num_tiles < sm_count() ? num_tiles : sm_count();
    cudaError_t e = launch_pdl(tc_patch_kernel<Prob, BN, TMA, DB2, TERMS, STACK>, dim3(grid), dim3(Cfg::kThreads), smem,
                               stream, prob, err_word);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

// prob.terms (3 or 1) selects the kernel instantiation; 3xTF32 tiles at most
// 64 wide stack their B tiles when `stack` is set.
template <class Prob, int BN, bool TMA, bool DB2>
cudaError_t launch_tc_patch(const Prob& prob, int num_tiles, int* err_word, cudaStream_t stream, bool stack)
{
    if (prob.terms == 1) return launch_tc_patch_terms<Prob, BN, TMA, DB2, 1, false>(prob, num_tiles, err_word, stream);
    if constexpr (BN <= 64)
        if (stack) return launch_tc_patch_terms<Prob, BN, TMA, DB2, 3, true>(prob, num_tiles, err_word, stream);
    return launch_tc_patch_terms<Prob, BN, TMA, DB2, 3, false>(prob, num_tiles, err_word, stream);
}

}  // namespace cb200
