// gemm_tma.cuh -- tcgen05 GEMM whose operands arrive by TMA, for the flagged
// matmul when the shape is large enough for wide tiles, any flags.
//
// D (128 x BN tile, fp32, tensor memory) = sum over K of A(128 x K) B(BN x K)^T.
// A stage is 16 deep: one 2-D TMA box per operand ({16 fp32, rows}, 64-byte
// swizzle) lands each tile straight in the K-major layout the tensor core
// reads (64-byte rows, 8-row groups 512 bytes apart) -- no register gather,
// no address arithmetic per element, zero fill past M, N and K.
//
// 3xTF32 without converting hi: the tensor core reads an fp32 operand as TF32
// by ignoring its 13 low mantissa bits (measured bit-exact against explicit
// truncation), so the landed raw tile IS the hi part.  Converter warps compute
// the lo part, a - trunc(a), into a second tile of identical layout (the
// swizzle is a function of the address, so the same offsets serve both).
// Each 8-deep step then issues lo*hi, hi*lo and hi*hi -- or, for tiles at
// most 128 wide, whose B hi and lo rows lie back to back, hi*[hi; lo] as one
// MMA with N = 2*BN plus lo*hi.  One TF32 product (TERMS == 1) of
// K-contiguous operands needs no converter at all: the MMAs read what TMA
// delivered.
//
// An operand stored with its rows contiguous (A stored K x M, B stored K x N:
// AT / BT) lands raw, in [16 k][32 r] boxes with the 128-byte swizzle, in a
// buffer of its stage; the converters transpose each box into the K-major
// tile (hi, and lo in 3xTF32): a lane takes a 4 x 4 block, four 16-byte reads
// down k, four 16-byte writes along r (lane (r4, k4) = (lane % 8,
// (lane / 8) ^ (lane % 4)): at most two lanes of a quarter-warp share a bank
// group on either side).
//
// Roles (320 threads, one CTA per SM, persistent over tiles, n fastest):
//   warp 0       TMA producer (lane 0): one A box and one B box per stage
//   warps 1-4    converters: the stage's lo tiles (3xTF32) and transposes
//   warp 5       MMA issuer (lane 0); allocates tensor memory
//   warps 6-9    epilogue: tcgen05.ld, row-major C with 16-byte stores
// Two accumulator buffers: the epilogue of tile i overlaps tile i+1.  Every
// wait is bounded (ptx.cuh); on give-up the kernel raises its abort flag,
// records the timeout, waits (bounded) for its own copies and MMAs in flight,
// frees tensor memory and returns.
#pragma once
#include <atomic>
#include <cuda.h>   // CUtensorMap (type only)

#include "gemm_flat.cuh"   // sdesc_k_sw64

namespace cb200 {

constexpr int kTmaBK = 16;   // K depth of a stage: one 64-byte swizzle row

template <int BN, int TERMS, bool AT = false, bool BT = false>
struct TmaCfg {
    static_assert(BN == 128 || BN == 256, "TMA-fed tiles are 128 or 256 wide");
    static constexpr bool kThree = TERMS == 3;
    static constexpr bool kStack = kThree && BN <= 128;   // hi|lo B rows back to back: N = 2*BN
    static constexpr bool kConvert = kThree || AT || BT;  // converters have work
    static constexpr int kThreads = 320;
    static constexpr uint32_t kATile = kBM * kTmaBK * 4;   // 8 KB
    static constexpr uint32_t kBTile = BN * kTmaBK * 4;
    static constexpr uint32_t kARaw = AT ? kATile : 0u;    // raw boxes of a rows-contiguous operand
    static constexpr uint32_t kBRaw = BT ? kBTile : 0u;
    // stage: A hi, [A lo], B hi, [B lo], [A raw], [B raw]
    static constexpr uint32_t kStage = (kThree ? 2u : 1u) * (kATile + kBTile) + kARaw + kBRaw;
    static constexpr size_t kCtlBytes = 512;
    static constexpr int kStages0 = int((216u * 1024u) / kStage);
    static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
    static_assert(kStages >= 3, "at least three stages in flight");
    static constexpr int kAccW = kStack ? 2 * BN : BN;   // accumulator columns per buffer
    static_assert(2 * kAccW <= 512, "two accumulator buffers must fit tensor memory");
    static constexpr size_t kSmemBytes = 1024 + size_t(kStages) * kStage + kCtlBytes;
    static constexpr uint32_t kIdesc = idesc_tf32(kBM, BN);
    static constexpr uint32_t kIdescStack = idesc_tf32(kBM, kStack ? 2 * BN : BN);
    // bytes one stage's two TMA boxes deliver
    static constexpr uint32_t kTxBytes = kATile + kBTile;
};

struct TmaGemmArgs {
    // K-contiguous operand: dims {K, rows}, box {16, rows of the tile}, 64-byte swizzle;
    // rows-contiguous operand: dims {rows, K}, box {32, 16}, 128-byte swizzle
    alignas(64) CUtensorMap ta;
    alignas(64) CUtensorMap tb;
    float* C;
    int M, N, K;
    int m_tiles, n_tiles, k_stages;
    int vec_c;   // 16-byte stores allowed along N
};

struct TmaCtl {
    uint64_t tfull[8];   // TMA boxes landed
    uint64_t cfull[8];   // lo tiles written (four converter warps)
    uint64_t empty[8];   // MMAs done with the stage
    uint64_t accf[2];
    uint64_t acce[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int c0, int c1, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t u4_at(const uint4& v, int j)
{
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint4 lo_of(uint4 v)
{
    uint32_t h, l0, l1, l2, l3;
    split_tf32(__uint_as_float(v.x), h, l0);
    split_tf32(__uint_as_float(v.y), h, l1);
    split_tf32(__uint_as_float(v.z), h, l2);
    split_tf32(__uint_as_float(v.w), h, l3);
    return make_uint4(l0, l1, l2, l3);
}

// One raw [16 k][32 r] box (128-byte swizzle) -> rows r0 .. r0+31 of a K-major
// tile with 64-byte rows (64-byte swizzle): the raw values as hi (the tensor
// core drops their low bits), and with LO their a - trunc(a) parts.
template <bool LO>
__device__ __forceinline__ void transpose_box(const uint8_t* raw, uint8_t* hi, uint8_t* lo, int r0, int lane)
{
    const int r4 = lane & 7, k4 = (lane >> 3) ^ (lane & 3);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = 4 * k4 + i;
        v[i] = *reinterpret_cast<const uint4*>(raw + k * 128 + ((r4 ^ (k & 7)) << 4));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = r0 + 4 * r4 + j;
        const uint4 row = make_uint4(u4_at(v[0], j), u4_at(v[1], j), u4_at(v[2], j), u4_at(v[3], j));
        const int off = r * 64 + ((k4 ^ ((r >> 1) & 3)) << 4);
        *reinterpret_cast<uint4*>(hi + off) = row;
        if (LO) *reinterpret_cast<uint4*>(lo + off) = lo_of(row);
    }
}

template <int BN, int TERMS, bool AT, bool BT>
__global__ void __launch_bounds__(TmaCfg<BN, TERMS, AT, BT>::kThreads, 1)
    tc_tma_gemm_kernel(const __grid_constant__ TmaGemmArgs args, int* err_word)
{
    using Cfg = TmaCfg<BN, TERMS, AT, BT>;
    constexpr bool convert = Cfg::kConvert;
    constexpr int S = Cfg::kStages;
    constexpr bool three = Cfg::kThree;
    constexpr bool STACK = Cfg::kStack;
    constexpr int AW = Cfg::kAccW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    TmaCtl* ctl = reinterpret_cast<TmaCtl*>(smem + size_t(S) * Cfg::kStage);
    volatile int* abort_flag = &ctl->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t base = smem_u32(smem);
    // stage layout: [A hi][A lo][B hi][B lo] (3xTF32) or [A hi][B hi]
    auto a_hi = [&](int s) { return base + uint32_t(s) * Cfg::kStage; };
    auto a_lo = [&](int s) { return a_hi(s) + Cfg::kATile; };
    auto b_hi = [&](int s) { return a_hi(s) + (three ? 2u : 1u) * Cfg::kATile; };
    auto b_lo = [&](int s) { return b_hi(s) + Cfg::kBTile; };
    auto a_raw = [&](int s) { return a_hi(s) + (three ? 2u : 1u) * (Cfg::kATile + Cfg::kBTile); };
    auto b_raw = [&](int s) { return a_raw(s) + Cfg::kARaw; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->tfull[s], 1);
            mbar_init(&ctl->cfull[s], 4);   // the four converter warps
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->accf[b], 1);
            mbar_init(&ctl->acce[b], 4);    // the four epilogue warps
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) tmem_alloc(&ctl->tmem_base, 2 * AW);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    griddep_wait();
    griddep_launch();

    const int num_tiles = args.m_tiles * args.n_tiles;
    const int ks_tile = args.k_stages;
    auto fail = [&]() {
        ctl->abort_flag = 1;
        atomicOr(err_word, kDevErrTimeout);
    };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t c = 0;
            int last = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int m0 = (t / args.n_tiles) * kBM;
                const int n0 = (t % args.n_tiles) * BN;
                for (int ks = 0; ks < ks_tile; ++ks, ++c) {
                    const int slot = int(c % uint32_t(S));
                    if (!mbar_wait(&ctl->empty[slot], ((c / uint32_t(S)) & 1u) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ctl->tfull[slot], Cfg::kTxBytes);
                    if constexpr (AT) {
#pragma unroll
                        for (int j = 0; j < kBM / 32; ++j)
                            tma_load_2d(smem + (a_raw(slot) - base) + 2048 * j, &args.ta, m0 + 32 * j, ks * kTmaBK,
                                        &ctl->tfull[slot]);
                    } else {
                        tma_load_2d(smem + (a_hi(slot) - base), &args.ta, ks * kTmaBK, m0, &ctl->tfull[slot]);
                    }
                    if constexpr (BT) {
#pragma unroll
                        for (int j = 0; j < BN / 32; ++j)
                            tma_load_2d(smem + (b_raw(slot) - base) + 2048 * j, &args.tb, n0 + 32 * j, ks * kTmaBK,
                                        &ctl->tfull[slot]);
                    } else {
                        tma_load_2d(smem + (b_hi(slot) - base), &args.tb, ks * kTmaBK, n0, &ctl->tfull[slot]);
                    }
                    last = int(c);
                }
            }
            if (!ok) {
                fail();
                for (int cc = last; cc >= 0 && cc > last - S; --cc) {   // copies in flight land before exit
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->tfull[cc % S], uint32_t(cc / S) & 1u) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < 5) {
        // ---------------- converters: lo tiles, transposes ----------------
        if constexpr (convert) {
            const int tid = threadIdx.x - 32;   // 0..127
            const int cw = warp - 1;            // converter warp 0..3
            uint32_t c = 0;
            bool ok = true;
            constexpr uint32_t nA = Cfg::kATile / 16u, nB = Cfg::kBTile / 16u;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                for (int ks = 0; ks < ks_tile; ++ks, ++c) {
                    const int slot = int(c % uint32_t(S));
                    if (!mbar_wait_warp(&ctl->tfull[slot], (c / uint32_t(S)) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* ah = smem + (a_hi(slot) - base);
                    uint8_t* al = smem + (a_lo(slot) - base);
                    uint8_t* bh = smem + (b_hi(slot) - base);
                    uint8_t* bl = smem + (b_lo(slot) - base);
                    if constexpr (AT) {   // four boxes, one per converter warp
                        transpose_box<three>(smem + (a_raw(slot) - base) + 2048 * cw, ah, al, 32 * cw, lane);
                    } else if constexpr (three) {
#pragma unroll
                        for (uint32_t i = uint32_t(tid); i < nA; i += 128u)
                            reinterpret_cast<uint4*>(al)[i] = lo_of(reinterpret_cast<const uint4*>(ah)[i]);
                    }
                    if constexpr (BT) {
#pragma unroll
                        for (int j = cw; j < BN / 32; j += 4)
                            transpose_box<three>(smem + (b_raw(slot) - base) + 2048 * j, bh, bl, 32 * j, lane);
                    } else if constexpr (three) {
#pragma unroll 4
                        for (uint32_t i = uint32_t(tid); i < nB; i += 128u)
                            reinterpret_cast<uint4*>(bl)[i] = lo_of(reinterpret_cast<const uint4*>(bh)[i]);
                    }
                    fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->cfull[slot]);
                }
            }
            if (!ok) fail();
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            uint32_t c = 0;
            int local = 0;
            bool ok = true, issued_any = false;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
                const int buf = local & 1;
                if (!mbar_wait(&ctl->acce[buf], (uint32_t(local >> 1) & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(buf * AW);
                uint32_t accumulate = 0;
                for (int ks = 0; ks < ks_tile; ++ks, ++c) {
                    const int slot = int(c % uint32_t(S));
                    const uint32_t ph = (c / uint32_t(S)) & 1u;
                    if (!mbar_wait(&ctl->tfull[slot], ph, abort_flag) ||
                        (convert && !mbar_wait(&ctl->cfull[slot], ph, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTmaBK / 8; ++kk) {
                        const uint64_t ah = sdesc_k_sw64(a_hi(slot) + kk * 32);
                        const uint64_t bh = sdesc_k_sw64(b_hi(slot) + kk * 32);
                        if constexpr (STACK) {
                            const uint64_t al = sdesc_k_sw64(a_lo(slot) + kk * 32);
                            // [0, BN): hi*hi (+ lo*hi below); [BN, 2BN): hi*lo
                            mma_tf32_ss(d_tmem, ah, bh, Cfg::kIdescStack, accumulate);
                            mma_tf32_ss(d_tmem, al, bh, Cfg::kIdesc, 1);
                        } else if constexpr (three) {
                            const uint64_t al = sdesc_k_sw64(a_lo(slot) + kk * 32);
                            const uint64_t bl = sdesc_k_sw64(b_lo(slot) + kk * 32);
                            mma_tf32_ss(d_tmem, al, bh, Cfg::kIdesc, accumulate);
                            mma_tf32_ss(d_tmem, ah, bl, Cfg::kIdesc, 1);
                            mma_tf32_ss(d_tmem, ah, bh, Cfg::kIdesc, 1);
                        } else {
                            mma_tf32_ss(d_tmem, ah, bh, Cfg::kIdesc, accumulate);
                        }
                        accumulate = 1;
                    }
                    issued_any = true;
                    mma_commit(&ctl->empty[slot]);
                }
                if (!ok) break;
                mma_commit(&ctl->accf[buf]);
            }
            if (!ok) {
                fail();
                if (issued_any) {
                    mma_commit(&ctl->drain);
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;   // the TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
            const int buf = local & 1;
            if (!mbar_wait_warp(&ctl->accf[buf], uint32_t(local >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int m = (t / args.n_tiles) * kBM + row;
            const int n_base = (t % args.n_tiles) * BN;
            const bool valid = m < args.M;
            float* crow = args.C + size_t(valid ? m : 0) * args.N;
            const uint32_t lane_base = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * AW);
#pragma unroll 1
            for (int cc = 0; cc < BN; cc += 32) {
                uint32_t r[32];
                if constexpr (STACK) {
                    uint32_t h[32];
                    tmem_ld32x2(lane_base + uint32_t(cc), lane_base + uint32_t(BN + cc), r, h);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(h[i]));
                } else {
                    tmem_ld32(lane_base + uint32_t(cc), r);
                }
                const int n0 = n_base + cc;
                if (valid) {
                    if (args.vec_c && n0 + 32 <= args.N) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(crow + n0 + i) =
                                make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                            __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (n0 + i < args.N) crow[n0 + i] = __uint_as_float(r[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->acce[buf]);
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 2 * AW);
    }
}

template <int BN, int TERMS, bool AT, bool BT>
cudaError_t launch_tma_gemm_terms(const TmaGemmArgs& args, int* err_word, cudaStream_t stream)
{
    using Cfg = TmaCfg<BN, TERMS, AT, BT>;
    static std::atomic<bool> attr_set{false};   // set once; racing setters are harmless
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_tma_gemm_kernel<BN, TERMS, AT, BT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int tiles = args.m_tiles * args.n_tiles;
    if (tiles <= 0) return cudaSuccess;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    cudaError_t e = launch_pdl(tc_tma_gemm_kernel<BN, TERMS, AT, BT>, dim3(grid), dim3(Cfg::kThreads),
                               Cfg::kSmemBytes, stream, args, err_word);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

}  // namespace cb200
