// gemm_flat.cuh -- implicit-GEMM convolution over a stride-1 window whose A
// operand (the column matrix of the page's im2col step) is read by the tensor
// core straight out of a TMA-loaded input box: no register gather and no
// per-tap copy of A.
//
// Flat output grid.  For one image the outputs (p, q), p < Gp, q < Gq, are
// numbered v = p * Wt + q with the row pitch Wt = Gq + T - 1 equal to the
// width of the input box (positions with q >= Gq are padding outputs that
// are computed and dropped).  Input pixel (p + tr, q + tq) of tap (tr, tq)
// then sits at box pixel v - p_lo * Wt + tr * Wt + tq, so for a tile of 128
// consecutive v the rows of tap (tr, tq) are 128 CONSECUTIVE box pixels: the
// A operand of every tap is the same box seen from a different start row.
// One shared-memory descriptor per tap addresses it; nothing is copied.
//
// The box is a 4-D TMA load of a channel-blocked copy of the gathered tensor
// ([n][c/32][h][w][32]): 16 channels x Wt columns x Rb rows, zero outside the
// image, written with the 64-byte swizzle -- exactly a K-major operand with
// 64-byte rows (16 fp32 channels per pixel).  A K stage is two taps of one
// 16-channel chunk (four 8-deep MMA steps, eight MMAs per barrier handshake;
// a chunk's last stage holds one tap when T*T is odd).
//
// 3xTF32 without converting A per tap: the tensor core reads an fp32 operand
// as TF32 by ignoring its 13 low mantissa bits (measured bit-exact against
// explicit truncation), so the raw box IS the hi part of every A value.  The
// lo part, a - trunc(a), is computed once per box by converter warps into a
// second buffer with the same layout and then serves all T*T taps.  B (the
// filters, fixed per call) comes as pre-split stage images by bulk copy, hi
// rows then lo rows, so one MMA with N = 2*BN multiplies A_hi by both
// (hi*hi into the first BN accumulator columns, hi*lo into the next BN) and
// a second, N = BN, adds lo*hi: two MMAs per 8-deep step.
//
// Roles (384 threads, one CTA per SM, persistent over tiles):
//   warp 0       box loader (TMA, one box per 16-channel chunk, two buffers)
//   warp 1       B loader (bulk copy of one stage image per K stage, S slots)
//   warps 2, 3   MMA issuers: stage c of the CTA-wide count goes to issuer
//                c % 2, into its own accumulator (one thread cannot issue
//                narrow MMAs fast enough); warp 2 also owns tensor memory
//   warps 4-7    converters: the lo box of each chunk
//   warps 8-11   epilogue: the accumulators of both issuers added in a fixed
//                order, handed row by row to the problem's store
// Every wait is bounded (ptx.cuh); on give-up the kernel raises its abort
// flag, records the timeout, waits (bounded) for its own copies and MMAs in
// flight, frees tensor memory and returns.
#pragma once
#include <atomic>
#include <cuda.h>   // CUtensorMap (type only)

#include "gemm_tc.cuh"

namespace cb200 {

// cuTensorMapEncodeTiled through the runtime's driver entry point (looked up
// once; null when the driver does not provide it).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled()
{
    // a function-local static's initialiser runs once, thread-safely
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
        return nullptr;
    }();
    return fn;
}


struct FlatGeom {
    int Nb, Ci, Hi, Wi;   // gathered tensor (channel-blocked copy) [Nb][Cb][Hi][Wi][32]
    int Cb;               // 32-channel blocks of the copy
    int nch;              // 16-channel chunks: ceil(Ci / 16)
    int Gp, Gq;           // output grid of one image
    int o;                // window origin: input row p + o + tr, column q + o + tq
    int T, TT;            // taps per axis and per window
    int spc;              // K stages per chunk: ceil(TT / 2), two taps each
    int Wt, Rb;           // box: Wt = Gq + T - 1 columns (the flat row pitch), Rb rows
    int vpi;              // flat positions per image: Gp * Wt
    int tpi;              // tiles per image: ceil(vpi / 128)
    uint32_t box_bytes;   // Rb * Wt * 64
    uint32_t box_stride;  // shared-memory bytes per box buffer (multiple of 1024)
    FastDiv f_wt, f_t, f_tt;
    alignas(64) CUtensorMap tmap;
};

// K stages of one tile: one per (16-channel chunk, pair of taps).
__host__ __device__ inline int flat_kstages(const FlatGeom& g) { return g.nch * g.spc; }

// Box rows so that every tap of every row of a tile stays inside the box: a
// tile starts at most Wt - 1 pixels into its first box row.
inline int flat_box_rows(int Wt, int T) { return (Wt - 1 + kBM + (T - 1) * (Wt + 1) + Wt - 1) / Wt; }

// Shared-memory descriptor of a K-major operand with 64-byte rows (16 fp32)
// and the 64-byte swizzle: 8-row groups 512 bytes apart.  The swizzle is a
// function of the shared-memory address, so the start may be any row.
__device__ __forceinline__ uint64_t sdesc_k_sw64(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                   // leading offset (unused with this swizzle)
    d |= static_cast<uint64_t>(512 >> 4) << 32;            // stride offset: 8-row group
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version for tcgen05
    d |= static_cast<uint64_t>(4) << 61;                   // 64-byte swizzle
    return d;
}

template <int BN>
struct FlatCfg {
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 64, "flat tiles are 16..64 columns (stacked hi|lo B)");
    static constexpr int kThreads = 384;
    static constexpr int kStages = 8;                              // B slots (even: slot parity = issuer)
    static constexpr uint32_t kBTap = 2u * BN * 64u;               // one tap: hi rows + lo rows, 16 fp32 each
    static constexpr uint32_t kBStage = 2u * kBTap;                // two taps
    static constexpr int kBNp = (BN + 31) / 32 * 32;               // epilogue column blocks of 32
    static constexpr uint32_t kRegion = 2u * kBNp;                 // TMEM columns per (buffer, issuer)
    // two accumulator buffers per issuer: the epilogue of tile i overlaps the
    // MMAs of tile i+1
    static_assert(2 * 2 * kRegion <= 512, "accumulators must fit tensor memory");
    static constexpr size_t kCtlBytes = 512;
    static constexpr uint32_t kIdescStack = idesc_tf32(kBM, 2 * BN);
    static constexpr uint32_t kIdesc = idesc_tf32(kBM, BN);
};

template <int BN>
constexpr size_t flat_smem(uint32_t box_stride)
{
    return 1024 + size_t(FlatCfg<BN>::kStages) * FlatCfg<BN>::kBStage + 4 * size_t(box_stride) +
           FlatCfg<BN>::kCtlBytes;
}

struct FlatCtl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t box_full[2];
    uint64_t lo_full[2];
    uint64_t box_empty[2];
    uint64_t accf[2];
    uint64_t acce[2];
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort_flag;
};

// Problem interface: fg (FlatGeom), n_tiles (column tiles), k_stages
// (= nch * spc), b_image(nt, ks) (global address of the stage image),
// EState / e_setup(t, row) for row 0 .. 127 of tile t, and
// store(es, n0, row, c, r).  Tile t: column tile nt = t % n_tiles,
// m = t / n_tiles: image m / tpi, flat positions [(m % tpi) * 128, + 128).
template <class Prob, int BN, int TERMS>
__global__ void __launch_bounds__(FlatCfg<BN>::kThreads, 1)
    tc_flat_kernel(const __grid_constant__ Prob prob, int* err_word)
{
    using Cfg = FlatCfg<BN>;
    constexpr int S = Cfg::kStages;
    constexpr bool three = TERMS == 3;
    const FlatGeom& g = prob.fg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* bstage0 = smem;
    uint8_t* box0 = smem + size_t(S) * Cfg::kBStage;   // raw[0], raw[1], lo[0], lo[1]
    FlatCtl* ctl = reinterpret_cast<FlatCtl*>(box0 + 4 * size_t(g.box_stride));
    volatile int* abort_flag = &ctl->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bstage_base = smem_u32(bstage0);
    const uint32_t box_base = smem_u32(box0);
    auto raw_addr = [&](int b) { return box_base + uint32_t(b) * g.box_stride; };
    auto lo_addr = [&](int b) { return box_base + uint32_t(2 + b) * g.box_stride; };
    // TMEM columns of the accumulator of (buffer, issuer)
    auto region = [&](int buf, int iss) { return uint32_t(buf * 2 + iss) * Cfg::kRegion; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->box_full[b], 1);
            mbar_init(&ctl->lo_full[b], 4);     // the four converter warps
            mbar_init(&ctl->box_empty[b], 2);   // one commit per issuer
            mbar_init(&ctl->accf[b], 2);        // one commit per issuer
            mbar_init(&ctl->acce[b], 4);        // the four epilogue warps
            mbar_init(&ctl->drain[b], 1);
        }
        ctl->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 2) tmem_alloc(&ctl->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    griddep_wait();
    griddep_launch();

    const int num_tiles = prob.num_tiles();
    const int ks_tile = flat_kstages(g);   // K stages per tile
    auto fail = [&]() {
        ctl->abort_flag = 1;
        atomicOr(err_word, kDevErrTimeout);
    };

    if (warp == 0) {
        // ---------------- box loader ----------------
        if (lane == 0) {
            uint32_t u = 0;   // chunk counter of this CTA
            int last = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int m = t / prob.n_tiles;
                const int n = m / g.tpi;
                const int v0 = (m % g.tpi) * kBM;
                const int p_lo = int(g.f_wt.div(uint32_t(v0)));
                for (int cc = 0; cc < g.nch; ++cc, ++u) {
                    const int b = int(u & 1u);
                    if (u >= 2 && !mbar_wait(&ctl->box_empty[b], ((u >> 1) - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ctl->box_full[b], g.box_bytes);
                    tma_load_4d(box0 + size_t(b) * g.box_stride, &prob.fg.tmap, 16 * (cc & 1), g.o, p_lo + g.o,
                                n * g.Cb + (cc >> 1), &ctl->box_full[b]);
                    last = int(u);
                }
            }
            if (!ok) {
                fail();
                for (int c = last; c >= 0 && c > last - 2; --c) {   // boxes in flight land before exit
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->box_full[c & 1], uint32_t(c >> 1) & 1u) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- B loader ----------------
        if (lane == 0) {
            constexpr uint32_t b_bytes = Cfg::kBStage;   // both taps' hi and lo rows
            uint32_t c = 0;
            int last = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int nt = t % prob.n_tiles;
                for (int ks = 0; ks < ks_tile; ++ks, ++c) {
                    const int slot = int(c % uint32_t(S));
                    if (!mbar_wait(&ctl->empty[slot], ((c / uint32_t(S)) & 1u) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ctl->full[slot], b_bytes);
                    bulk_g2s(bstage0 + size_t(slot) * Cfg::kBStage, prob.b_image(nt, ks), b_bytes, &ctl->full[slot]);
                    last = int(c);
                    if (ks + kBPrefetch < ks_tile) prefetch_l2_bulk(prob.b_image(nt, ks + kBPrefetch), b_bytes);
                }
            }
            if (!ok) {
                fail();
                for (int cc = last; cc >= 0 && cc > last - S; --cc) {
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->full[cc % S], uint32_t(cc / S) & 1u) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ---------------- MMA issuers ----------------
        const uint32_t me = uint32_t(warp - 2);
        if (lane == 0) {
            uint32_t c0 = 0;   // CTA-wide stage count at the tile's start
            uint32_t u0 = 0;   // CTA-wide chunk count at the tile's start
            int local = 0;
            bool ok = true, issued_any = false;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
                const int m = t / prob.n_tiles;
                const int v0 = (m % g.tpi) * kBM;
                const int r0 = v0 - int(g.f_wt.div(uint32_t(v0))) * g.Wt;   // first row's pixel in the box
                const int buf = local & 1;
                if (!mbar_wait(&ctl->acce[buf], (uint32_t(local >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + region(buf, int(me));
                uint32_t accumulate = 0;
                for (int cc = 0; cc < g.nch && ok; ++cc) {
                    const uint32_t u = u0 + uint32_t(cc);
                    const int b = int(u & 1u);
                    bool waited = false;
                    const int s_lo = cc * g.spc;
                    for (int s = s_lo + int((me ^ ((c0 + uint32_t(s_lo)) & 1u)) & 1u); s < s_lo + g.spc; s += 2) {
                        if (!waited) {
                            if (!mbar_wait(&ctl->lo_full[b], (u >> 1) & 1u, abort_flag)) { ok = false; break; }
                            waited = true;
                        }
                        const uint32_t c = c0 + uint32_t(s);
                        const int slot = int(c % uint32_t(S));
                        if (!mbar_wait(&ctl->full[slot], (c / uint32_t(S)) & 1u, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const int tap0 = 2 * (s - s_lo);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (tap0 + h >= g.TT) break;   // odd T*T: the chunk's last stage has one tap
                            uint32_t tr, tq;
                            g.f_t.divmod(uint32_t(tap0 + h), tr, tq);
                            const uint32_t arow = uint32_t(r0) + tr * uint32_t(g.Wt) + tq;   // A's first box pixel
                            const uint32_t bsl = bstage_base + uint32_t(slot) * Cfg::kBStage + uint32_t(h) * Cfg::kBTap;
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t aoff = arow * 64u + uint32_t(kk) * 32u;
                                const uint64_t ah = sdesc_k_sw64(raw_addr(b) + aoff);
                                const uint64_t bb = sdesc_k_sw64(bsl + kk * 32);
                                if (three) {
                                    const uint64_t al = sdesc_k_sw64(lo_addr(b) + aoff);
                                    // [0, BN): hi*hi (+ lo*hi below); [BN, 2BN): hi*lo
                                    mma_tf32_ss(d_tmem, ah, bb, Cfg::kIdescStack, accumulate);
                                    mma_tf32_ss(d_tmem, al, bb, Cfg::kIdesc, 1);
                                } else {
                                    mma_tf32_ss(d_tmem, ah, bb, Cfg::kIdesc, accumulate);
                                }
                                accumulate = 1;
                            }
                        }
                        issued_any = true;
                        mma_commit(&ctl->empty[slot]);
                    }
                    if (!ok) break;
                    // this issuer is done with the chunk's boxes once its MMAs complete
                    mma_commit(&ctl->box_empty[b]);
                }
                if (!ok) break;
                c0 += uint32_t(ks_tile);
                u0 += uint32_t(g.nch);
                mma_commit(&ctl->accf[buf]);
            }
            if (!ok) {
                fail();
                if (issued_any) {
                    mma_commit(&ctl->drain[me]);
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->drain[me], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
                }
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ---------------- converters: lo box of each chunk ----------------
        const int tid = threadIdx.x - 128;   // 0..127
        uint32_t u = 0;
        bool ok = true;
        const uint32_t n16 = g.box_bytes / 16u;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            for (int cc = 0; cc < g.nch; ++cc, ++u) {
                const int b = int(u & 1u);
                if (!mbar_wait_warp(&ctl->box_full[b], (u >> 1) & 1u, abort_flag)) { ok = false; break; }
                if (three) {
                    const uint4* src = reinterpret_cast<const uint4*>(box0 + size_t(b) * g.box_stride);
                    uint4* dst = reinterpret_cast<uint4*>(box0 + size_t(2 + b) * g.box_stride);
                    for (uint32_t i = uint32_t(tid); i < n16; i += 128u) {
                        const uint4 v = src[i];
                        uint32_t h, l0, l1, l2, l3;
                        split_tf32(__uint_as_float(v.x), h, l0);
                        split_tf32(__uint_as_float(v.y), h, l1);
                        split_tf32(__uint_as_float(v.z), h, l2);
                        split_tf32(__uint_as_float(v.w), h, l3);
                        dst[i] = make_uint4(l0, l1, l2, l3);
                    }
                    fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->lo_full[b]);
            }
        }
        if (!ok) fail();
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
            const int buf = local & 1;
            if (!mbar_wait_warp(&ctl->accf[buf], uint32_t(local >> 1) & 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const int n0 = (t % prob.n_tiles) * BN;
            typename Prob::EState es = prob.e_setup(t, row);
            const uint32_t lane_off = uint32_t(q * 32) << 16;
            const uint32_t a0 = tmem_base + lane_off + region(buf, 0);
            const uint32_t a1 = tmem_base + lane_off + region(buf, 1);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r0[32], r1[32];
                if constexpr (three) {
                    uint32_t h[32];
                    tmem_ld32x2(a0 + uint32_t(c), a0 + uint32_t(BN + c), r0, h);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r0[i] = __float_as_uint(__uint_as_float(r0[i]) + __uint_as_float(h[i]));
                    tmem_ld32x2(a1 + uint32_t(c), a1 + uint32_t(BN + c), r1, h);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r1[i] = __float_as_uint(__uint_as_float(r1[i]) + __uint_as_float(h[i]));
                } else {
                    tmem_ld32x2(a0 + uint32_t(c), a1 + uint32_t(c), r0, r1);
                }
                if (c + 32 >= BN) {
                    // every accumulator column of the tile is in registers
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->acce[buf]);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) r0[i] = __float_as_uint(__uint_as_float(r0[i]) + __uint_as_float(r1[i]));
                prob.store(es, n0, row, c, r0);
            }
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <class Prob, int BN, int TERMS>
cudaError_t launch_tc_flat_terms(const Prob& prob, int num_tiles, int* err_word, cudaStream_t stream)
{
    using Cfg = FlatCfg<BN>;
    static std::atomic<bool> attr_set{false};   // set once; racing setters are harmless
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_flat_kernel<Prob, BN, TERMS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (num_tiles <= 0) return cudaSuccess;
    const size_t smem = flat_smem<BN>(prob.fg.box_stride);
    const int grid = num_tiles < sm_count() ? num_tiles : sm_count();
    cudaError_t e = launch_pdl(tc_flat_kernel<Prob, BN, TERMS>, dim3(grid), dim3(Cfg::kThreads), smem, stream, prob,
                               err_word);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

// prob.terms (3 or 1) selects the instantiation.
template <class Prob, int BN>
cudaError_t launch_tc_flat(const Prob& prob, int num_tiles, int* err_word, cudaStream_t stream)
{
    return prob.terms == 1 ? launch_tc_flat_terms<Prob, BN, 1>(prob, num_tiles, err_word, stream)
                           : launch_tc_flat_terms<Prob, BN, 3>(prob, num_tiles, err_word, stream);
}

}  // namespace cb200
