// gemm_tc.cuh -- persistent, warp-specialised tcgen05 GEMM in fp32-faithful
// 3xTF32 mode, shared by the flagged matmul and the three convolution GEMMs.
//
// D (128 x BN tile, fp32, in tensor memory) = sum over K of A (rows x K) * B (cols x K)^T
//
// Each operand value a is split in registers into hi = tf32(a) and
// lo = tf32(a - hi); every 8-deep K step issues three tcgen05.mma.kind::tf32:
// hi*hi, hi*lo and lo*hi (the lo*lo term is below fp32 resolution).  The
// tensor core accumulates in fp32.
//
// Warp roles (one CTA per SM, persistent over output tiles):
//   warps 0 .. 4G-1   G producer groups of 4 warps.  Pipeline stages are dealt
//                     round-robin to the groups, so G stages' worth of global
//                     loads are in flight at once.  For its stage a group
//                     gathers the 128 x 32 slice of A and -- unless the problem
//                     ships B as a pre-split image (one cp.async.bulk by the
//                     group's first thread) -- the BN x 32 slice of B, splits
//                     every value into hi/lo and stores both into the stage's
//                     tiles (128-byte swizzled, K-major)
//   warp 4G           allocates tensor memory; lane 0 issues the MMAs
//   warp 4G+1         (tiles at most 64 wide, A in shared memory) lane 0 is a
//                     second MMA issuer: one thread cannot issue tcgen05.mma
//                     fast enough to keep the tensor core busy on such narrow
//                     tiles (about one MMA per 25 ns whatever N is, plus the
//                     stage handshakes).  Stage c of the CTA-wide stage count
//                     is then consumed by issuer c % 2 into its own
//                     accumulator (S even, so slot c % S has the parity of its
//                     producer group and of its issuer) and the epilogue adds
//                     the two accumulators in a fixed order.
//   last 4 warps      epilogue: tcgen05.ld the accumulator, hand rows to the
//                     problem's store (bias, NCHW reshape, split-K partials ...)
// Two accumulators per issuer (2 x BN TMEM columns) let the epilogue of tile i
// overlap the main loop of tile i+1.
//
// Stacked B tiles (two issuers, 3xTF32): a stage's hi and lo B tiles lie back
// to back in shared memory, so one MMA with N = 2*BN multiplies A_hi by both
// (hi*hi into the accumulator's first BN columns, hi*lo into the next BN) and
// a second MMA (N = BN) adds lo*hi: two MMAs per 8-deep step instead of three,
// and A is read from shared memory twice instead of three times.  On these
// narrow tiles the shared-memory operand traffic (producer stores + MMA reads)
// is what bounds the stage rate.  The epilogue adds the halves.
//
// Every wait is bounded (ptx.cuh); on give-up the kernel raises its abort
// flag, records kDevErrTimeout in the device error word, waits for what it
// already launched asynchronously, frees its tensor memory and returns.
// withhold_stage (a test hook, -1 in normal use): CTA 0's producers do not
// arrive on the "full" barrier of that CTA-wide stage, so the MMA issuer's
// bounded wait runs out and the kernel takes the path above.
//
// Cluster split (problems with kClusterSplit, prob.csplit > 1): when a GEMM
// has too few output tiles to occupy the SMs, each tile's K range is cut into
// csplit pieces run by the CTAs of one thread-block cluster (one piece, and
// so one unit, per CTA).  A piece's epilogue writes its partial tile into the
// CTA's own shared memory (the pipeline stages are idle by then); after a
// cluster barrier every CTA adds, for its 128 / csplit rows of the tile, the
// partials of all pieces in rank order through distributed shared memory and
// hands the sums to prob.reduce_store.  Deterministic, no global workspace.
#pragma once
#include <atomic>
#include <cooperative_groups.h>

#include "ptx.cuh"

namespace cb200 {

constexpr int kBM = 128;       // UMMA M: rows of a tile (TMEM lanes)
constexpr int kBK = 32;        // K depth of one pipeline stage (one 128-byte swizzle row)
constexpr size_t kSmemBudget = 200 * 1024;
constexpr int kBPrefetch = 4;  // stages ahead at which a bulk-fed B block is prefetched into L2

template <int G, int NI>
struct Roles {
    static constexpr int kWarpMma = 4 * G;               // first issuer warp
    static constexpr int kWarpEpi = 4 * G + NI;          // first epilogue warp
    static constexpr int kThreads = (4 * G + NI + 4) * 32;
};


struct Tile {
    int m0, n0;     // first row of A / of B (output row / column)
    int ks0, ks1;   // K stages [ks0, ks1)
    int grp;        // problem-defined: sub-problem (stride phase) or split index
    int part = -1;  // >= 0: this unit is one K piece of a split tile (its partial-sum slot)
};

// Tile configuration.  With ATMEM the A operand does not use shared memory:
// producers write its hi/lo halves into tensor memory (64 columns per stage)
// and the MMA reads A from there; shared memory then holds only B stages.
template <int BN, bool ATMEM = false>
struct TileCfg {
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");
    static constexpr uint32_t kATile = ATMEM ? 0 : kBM * kBK * 4;   // smem bytes of one hi (or lo) A tile
    static constexpr uint32_t kBTile = BN * kBK * 4;
    static constexpr uint32_t kStage = 2 * kATile + 2 * kBTile;
    // accumulators: two (epilogue of tile i overlaps tile i+1) unless tensor
    // memory is needed for A stages
    static constexpr int kDBuf = (ATMEM && BN > 128) ? 1 : 2;
    static constexpr int kIssuers = (!ATMEM && BN <= 64) ? 2 : 1;
    static constexpr int kSmemStages = int(kSmemBudget / kStage);
    static constexpr int kTmemStages = ATMEM ? (512 - kDBuf * BN) / 64 : 8;
    static constexpr int kStages0 = kSmemStages < kTmemStages ? kSmemStages : kTmemStages;
    static constexpr int kStages1 = kStages0 > (ATMEM ? 8 : 6) ? (ATMEM ? 8 : 6) : kStages0;
    static constexpr int kStages = kIssuers == 2 ? (kStages1 & ~1) : kStages1;   // two issuers: S even
    static_assert(kIssuers == 1 || kStages >= 2, "two issuers need an even number of stages");
    static constexpr uint32_t kACol = uint32_t(kDBuf * BN);   // first TMEM column of the A stages
    // accumulators: [buffer][issuer], each 2*BN wide when B tiles are stacked
    // (two issuers, 3xTF32: the allocation covers that case for both modes)
    static constexpr int kAccCols = kIssuers * kDBuf * BN * (kIssuers == 2 ? 2 : 1);
    static constexpr uint32_t kTmemCols =
        ATMEM ? 512 : (kAccCols <= 64) ? 64 : (kAccCols <= 128) ? 128 : (kAccCols <= 256) ? 256 : 512;
    static constexpr size_t kSmemBytes = size_t(kStages) * kStage + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr uint32_t kIdesc = idesc_tf32(kBM, BN);
    static constexpr uint32_t kIdescStack = idesc_tf32(kBM, kIssuers == 2 ? 2 * BN : BN);   // the hi*[hi; lo] MMA
};

template <class Prob>
struct UsesClusterSplit {
    template <class P>
    static constexpr bool test(decltype(P::kClusterSplit)*) { return P::kClusterSplit; }
    template <class P>
    static constexpr bool test(...) { return false; }
    static constexpr bool value = test<Prob>(nullptr);
};

// Row pitch (floats) of a cluster-split partial tile in shared memory: 16
// bytes past a multiple of 128, so eight consecutive rows' 16-byte stores hit
// eight different bank groups.
template <int BN>
__host__ __device__ constexpr int part_pitch() { return BN + 4; }

template <class Prob>
struct UsesTmemA {
    template <class P>
    static constexpr bool test(decltype(P::kATmem)*) { return P::kATmem; }
    template <class P>
    static constexpr bool test(...) { return false; }
    static constexpr bool value = test<Prob>(nullptr);
};

// Producer groups actually used: never more than the pipeline has stages.
// A group waits on a slot's "empty" barrier by phase parity, which is only
// sound while no waiter runs more than one phase ahead of the barrier; with
// G <= S the stage a group fills next is at most S ahead of one it already
// saw consumed.
template <class Prob, int BN>
struct Groups {
    static constexpr int kS = TileCfg<BN, UsesTmemA<Prob>::value>::kStages;
    static constexpr int value = Prob::kGroups < kS ? Prob::kGroups : kS;
};

// Producer-side layout of a gathered 32-value slice (per thread):
//   RowFast:   thread t owns row t of a 128-row block; v[i] is k = ks*32 + i.
//   ChunkFast: thread t owns 16-byte chunk (t % 8) of rows (t / 8) + 16 p,
//              p = 0..7; v[4p + e] is k = ks*32 + 4 (t % 8) + e.
//   QuadRow:   thread t owns rows 4 (t / 4) + j, j = 0..3, and K values
//              8 (t % 4) + kk, kk = 0..7: v[4 kk + j] is (row 4 (t / 4) + j,
//              k = ks*32 + 8 (t % 4) + kk).  For an operand stored with the
//              ROWS contiguous: one 16-byte load covers four rows of one k.
enum class Map { RowFast, ChunkFast, QuadRow };

template <Map M>
__device__ __forceinline__ void store_slice(uint32_t hi_tile, uint32_t lo_tile, int row_base, int rows, int tid,
                                            const float (&v)[32], bool with_lo = true)
{
    if constexpr (M == Map::RowFast) {
        int row = row_base + tid;
        if (row - row_base < rows) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                store_split_chunk(hi_tile, lo_tile, row, c, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3],
                                  with_lo);
        }
    } else if constexpr (M == Map::ChunkFast) {
        int chunk = tid & 7;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            int r = (tid >> 3) + 16 * p;
            if (r < rows)
                store_split_chunk(hi_tile, lo_tile, row_base + r, chunk, v[4 * p], v[4 * p + 1], v[4 * p + 2],
                                  v[4 * p + 3], with_lo);
        }
    } else {
        // Thread t writes chunks 2 (t % 4) and 2 (t % 4) + 1 of its four rows,
        // odd quads of lanes the two chunks in the other order: a quarter-warp
        // then covers all eight 16-byte bank groups of the swizzled rows.
        const int kg = tid & 3, rq = tid >> 2;
        const bool swap = (rq & 1) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = 4 * rq + j;
            if (r < rows) {
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    float a[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float first = v[4 * (4 * s + e) + j], second = v[4 * (4 * (1 - s) + e) + j];
                        a[e] = swap ? second : first;
                    }
                    const int h = swap ? 1 - s : s;
                    store_split_chunk(hi_tile, lo_tile, row_base + r, 2 * kg + h, a[0], a[1], a[2], a[3], with_lo);
                }
            }
        }
    }
}

struct SharedCtl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t accf[2];
    uint64_t acce[2];
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort_flag;
};

template <class Prob, int BN>
struct EngineRoles {
    using Cfg = TileCfg<BN, UsesTmemA<Prob>::value>;
    using R = Roles<Groups<Prob, BN>::value, Cfg::kIssuers>;
};

// The cluster split's reduction (see the top of the file), run by every thread
// of every CTA of the cluster once its unit is done.  Not inlined: the main
// kernel keeps its register allocation (inlined, it spilled the wide tiles).
template <class Prob, int BN>
__device__ __noinline__ void cluster_split_reduce(const Prob& prob, const uint8_t* smem, bool good)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();   // every piece's partial tile is in its CTA's shared memory
    const int pieces = prob.csplit;
    const int rank = int(cluster.block_rank());
    const Tile tile = prob.tile(int(blockIdx.x));
    const int rows = kBM / pieces;
    constexpr int kC4 = BN / 4;
    const float* part = reinterpret_cast<const float*>(smem);
    for (int i = int(threadIdx.x); i < rows * kC4; i += int(blockDim.x)) {
        const int row = rank * rows + i / kC4;
        const int c = 4 * (i % kC4);
        const int off = row * part_pitch<BN>() + c;
        float4 acc = *reinterpret_cast<const float4*>(cluster.map_shared_rank(part, 0) + off);
        for (int j = 1; j < pieces; ++j) {
            const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(part, j) + off);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (good) prob.reduce_store(tile, row, c, acc);
    }
    cluster.sync();   // each CTA's shared memory stays alive until its peers have read it
}

template <class Prob, int BN, int TERMS>
__global__ void __launch_bounds__(EngineRoles<Prob, BN>::R::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ Prob prob, int* err_word, int withhold_stage)
{
    constexpr bool ATMEM = UsesTmemA<Prob>::value;
    using Cfg = TileCfg<BN, ATMEM>;
    constexpr int S = Cfg::kStages;
    constexpr int G = Groups<Prob, BN>::value;
    constexpr int DB = Cfg::kDBuf;
    constexpr int NI = Cfg::kIssuers;
    static_assert(G >= 1 && G <= S, "producer groups must not outnumber pipeline stages");
    static_assert(NI == 1 || G == 2, "two issuers pair with two producer groups (stage parity)");
    constexpr int kWarpMma = Roles<G, NI>::kWarpMma;
    constexpr int kWarpEpi = Roles<G, NI>::kWarpEpi;
    constexpr int kBPasses = BN > 128 ? 2 : 1;
    constexpr bool CS = UsesClusterSplit<Prob>::value;
    static_assert(!CS || size_t(kBM) * part_pitch<BN>() * 4 <= size_t(S) * Cfg::kStage,
                  "a cluster-split partial tile must fit the pipeline stages");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + size_t(S) * Cfg::kStage);
    volatile int* abort_flag = &ctl->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t smem_base = smem_u32(smem);
    auto a_hi = [&](int s) { return smem_base + uint32_t(s) * Cfg::kStage; };
    auto a_lo = [&](int s) { return a_hi(s) + Cfg::kATile; };
    auto b_hi = [&](int s) { return a_hi(s) + 2 * Cfg::kATile; };
    auto b_lo = [&](int s) { return b_hi(s) + Cfg::kBTile; };
    auto a_col = [&](int s) { return Cfg::kACol + uint32_t(s) * 64u; };   // ATMEM: hi at +0, lo at +32

    if (threadIdx.x == 0) {
        const uint32_t full_count = 4 + (Prob::kBBulk ? 1 : 0);
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], full_count);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < DB; ++b) {
            mbar_init(&ctl->accf[b], NI);   // one commit per issuer
            mbar_init(&ctl->acce[b], 4);
        }
        for (int i = 0; i < NI; ++i) mbar_init(&ctl->drain[i], 1);
        ctl->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kWarpMma) tmem_alloc(&ctl->tmem_base, Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    // set-up above overlaps the previous kernel when launched with PDL
    griddep_wait();
    griddep_launch();

    const int num_tiles = prob.num_tiles();
    // TERMS == 3: hi*hi + hi*lo + lo*hi (fp32-faithful); TERMS == 1: hi*hi only
    // (one TF32 product: no lo halves are stored, copied or multiplied).  A
    // template parameter, so that the 3xTF32 kernel carries no trace of the
    // other mode (a runtime switch measured 7% slower).
    constexpr bool three = TERMS == 3;
    constexpr bool STACK = three && NI == 2 && !ATMEM;   // stacked hi|lo B tiles (see the top of the file)
    constexpr int AW = STACK ? 2 * BN : BN;              // accumulator columns per (buffer, issuer)
    constexpr uint32_t b_bytes = (three ? 2u : 1u) * Cfg::kBTile;
    auto fail = [&]() {
        ctl->abort_flag = 1;
        atomicOr(err_word, kDevErrTimeout);
    };

    if (warp < 4 * G) {
        // ---------------- producer groups ----------------
        const int g = warp >> 2;
        const int tid = threadIdx.x - 128 * g;   // 0..127 inside the group
        uint32_t cnt = 0;                        // stages of this CTA so far (all groups agree)
        int last_issued = -1;                    // last stage this group bulk-copied
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const Tile tile = prob.tile(t);
            const int nks = tile.ks1 - tile.ks0;
            const int first = int((uint32_t(g) + uint32_t(G) - cnt % uint32_t(G)) % uint32_t(G));
            if (first < nks) {
                typename Prob::AState ast = prob.a_setup(tile, tid);
                typename Prob::BState bst = prob.b_setup(tile, tid);
                // Everything for stage i except the A gather (already in va).
                auto produce = [&](int i, float (&va)[32]) -> bool {
                    const uint32_t c = cnt + uint32_t(i);
                    const int slot = int(c % uint32_t(S));
                    const uint32_t phase = (c / uint32_t(S)) & 1u;
                    const int ks = tile.ks0 + i;
                    float vb[kBPasses][32];
                    if constexpr (!Prob::kBBulk) {
#pragma unroll
                        for (int pass = 0; pass < kBPasses; ++pass) prob.load_b(bst, tile, ks, pass, tid, vb[pass]);
                        // Every gathered value lands in its register here, before
                        // the wait for the slot: all of the stage's loads are then
                        // in flight together.  Without this the TF32 build (fewer
                        // stores to schedule against) let loads trail into the
                        // stores and ran 2.8x slower on B stored K x N.
#pragma unroll
                        for (int pass = 0; pass < kBPasses; ++pass)
#pragma unroll
                            for (int i = 0; i < 32; ++i) asm volatile("" : "+f"(vb[pass][i]));
#pragma unroll
                        for (int i = 0; i < 32; ++i) asm volatile("" : "+f"(va[i]));
                    }
                    if (!mbar_wait_warp(&ctl->empty[slot], phase ^ 1u, abort_flag)) return false;
                    if constexpr (Prob::kBBulk) {
                        if (tid == 0) {
                            mbar_arrive_expect_tx(&ctl->full[slot], b_bytes);
                            bulk_g2s(smem + (b_hi(slot) - smem_base), prob.b_image(tile, ks), b_bytes,
                                     &ctl->full[slot]);
                            last_issued = int(c);
                            // the B image may stream from HBM (the filter gradient's dy
                            // image is larger than L2): pull a later stage's block into L2
                            // now, so that its copy finds it there
                            if (ks + kBPrefetch < tile.ks1)
                                prefetch_l2_bulk(prob.b_image(tile, ks + kBPrefetch), b_bytes);
                        }
                    }
                    if constexpr (ATMEM) {
                        // Thread = row 32 * (warp % 4) + lane = tid: write its split
                        // row into the stage's hi and lo column blocks.
                        static_assert(Prob::kAMap == Map::RowFast, "tensor-memory A needs one row per thread");
                        tc_fence_after();
                        const uint32_t tbase = tmem_base + (uint32_t((warp & 3) * 32) << 16) + a_col(slot);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            uint32_t hi[8], lo[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) split_tf32(va[8 * h + i], hi[i], lo[i]);
                            tmem_st8(tbase + 8 * h, hi);
                            if (three) tmem_st8(tbase + 32 + 8 * h, lo);
                        }
                        tmem_wait_st();
                        tc_fence_before();
                    } else {
                        store_slice<Prob::kAMap>(a_hi(slot), a_lo(slot), 0, kBM, tid, va, three);
                    }
                    if constexpr (!Prob::kBBulk) {
#pragma unroll
                        for (int pass = 0; pass < kBPasses; ++pass) {
                            const int rows = BN - 128 * pass < 128 ? BN - 128 * pass : 128;
                            store_slice<Prob::kBMap>(b_hi(slot), b_lo(slot), 128 * pass, rows, tid, vb[pass],
                                                     three);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && !(blockIdx.x == 0 && int(c) == withhold_stage)) mbar_arrive(&ctl->full[slot]);
                    return true;
                };
                if constexpr (Prob::kBBulk) {
                    // A gathers run one owned stage ahead: while stage i is
                    // split and stored, the loads of stage i + G are in flight
                    // (two register buffers, used in turn).
                    float v0[32], v1[32];
                    prob.load_a(ast, tile, tile.ks0 + first, tid, v0);
                    for (int i = first; i < nks; i += 2 * G) {
                        if (i + G < nks) prob.load_a(ast, tile, tile.ks0 + i + G, tid, v1);
                        if (!produce(i, v0)) { ok = false; break; }
                        if (i + G >= nks) break;
                        if (i + 2 * G < nks) prob.load_a(ast, tile, tile.ks0 + i + 2 * G, tid, v0);
                        if (!produce(i + G, v1)) { ok = false; break; }
                    }
                } else {
                    for (int i = first; i < nks; i += G) {
                        float va[32];
                        prob.load_a(ast, tile, tile.ks0 + i, tid, va);
                        if (!produce(i, va)) { ok = false; break; }
                    }
                }
            }
            cnt += uint32_t(nks);
        }
        if (!ok) {
            fail();
            if (Prob::kBBulk && tid == 0 && last_issued >= 0) {
                // Bulk copies already issued may still be landing in stages the
                // MMA will not consume; wait (bounded) for each before exit.
                for (int c = last_issued; c >= 0 && c > last_issued - S; c -= G) {
                    uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->full[c % S], uint32_t(c / S) & 1u) &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp < kWarpEpi) {
        // ---------------- MMA issuer(s) ----------------
        const uint32_t me = uint32_t(warp - kWarpMma);
        if (lane == 0) {
            uint32_t cnt = 0;   // CTA-wide stage counter (as the producers count)
            int local = 0;
            bool ok = true;
            bool issued_any = false;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
                const Tile tile = prob.tile(t);
                const int nks = tile.ks1 - tile.ks0;
                const int acc = local % DB;
                const uint32_t acc_phase = uint32_t(local / DB) & 1u;
                if (!mbar_wait(&ctl->acce[acc], acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t((acc * NI + int(me)) * AW);
                uint32_t accumulate = 0;
                const int i0 = NI == 1 ? 0 : int(me ^ (cnt & 1u));   // this issuer's first stage of the tile
                for (int i = i0; i < nks; i += NI) {
                    const uint32_t c = cnt + uint32_t(i);
                    const int stage = int(c % uint32_t(S));
                    const uint32_t phase = (c / uint32_t(S)) & 1u;
                    if (!mbar_wait(&ctl->full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 8; ++kk) {
                        const uint64_t bh = sdesc_k_sw128(b_hi(stage) + kk * 32);
                        const uint64_t bl = sdesc_k_sw128(b_lo(stage) + kk * 32);
                        if constexpr (ATMEM) {
                            const uint32_t ah = tmem_base + a_col(stage) + uint32_t(kk * 8);
                            const uint32_t al = ah + 32;
                            if (three) {
                                mma_tf32_ts(d_tmem, al, bh, Cfg::kIdesc, accumulate);
                                mma_tf32_ts(d_tmem, ah, bl, Cfg::kIdesc, 1);
                                mma_tf32_ts(d_tmem, ah, bh, Cfg::kIdesc, 1);
                            } else {
                                mma_tf32_ts(d_tmem, ah, bh, Cfg::kIdesc, accumulate);
                            }
                            accumulate = 1;
                        } else {
                            const uint64_t ah = sdesc_k_sw128(a_hi(stage) + kk * 32);
                            const uint64_t al = sdesc_k_sw128(a_lo(stage) + kk * 32);
                            if constexpr (STACK) {
                                // [0, BN): hi*hi (+ lo*hi below); [BN, 2BN): hi*lo
                                mma_tf32_ss(d_tmem, ah, bh, Cfg::kIdescStack, accumulate);
                                mma_tf32_ss(d_tmem, al, bh, Cfg::kIdesc, 1);
                            } else if (three) {
                                mma_tf32_ss(d_tmem, al, bh, Cfg::kIdesc, accumulate);
                                mma_tf32_ss(d_tmem, ah, bl, Cfg::kIdesc, 1);
                                mma_tf32_ss(d_tmem, ah, bh, Cfg::kIdesc, 1);
                            } else {
                                mma_tf32_ss(d_tmem, ah, bh, Cfg::kIdesc, accumulate);
                            }
                            accumulate = 1;
                        }
                    }
                    issued_any = true;
                    mma_commit(&ctl->empty[stage]);
                }
                if (!ok) break;
                cnt += uint32_t(nks);
                // arrives once this issuer's MMAs of the tile are done (at once if it had none)
                mma_commit(&ctl->accf[acc]);
            }
            if (!ok) {
                fail();
                if (issued_any) {
                    // Let the MMAs in flight finish before the memory goes away.
                    mma_commit(&ctl->drain[me]);
                    uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&ctl->drain[me], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;               // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;        // accumulator row of this thread
        // a cluster-split piece keeps its partial row in shared memory
        auto emit = [&](const typename Prob::EState& es, const Tile& tl, int c, const uint32_t (&r)[32]) {
            if constexpr (CS) {
                if (tl.part >= 0) {
                    float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(smem) + row * part_pitch<BN>() + c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                           __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                    return;
                }
            }
            prob.store(es, tl, row, c, r);
        };
        uint32_t cnt = 0;                     // CTA-wide stage counter at the tile's start
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
            const Tile tile = prob.tile(t);
            const int nks = tile.ks1 - tile.ks0;
            const int acc = local % DB;
            const uint32_t acc_phase = uint32_t(local / DB) & 1u;
            if (!mbar_wait_warp(&ctl->accf[acc], acc_phase, abort_flag)) { ok = false; break; }
            tc_fence_after();
            typename Prob::EState es = prob.e_setup(tile, row);
            const uint32_t lane_base = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * NI * AW);
            if constexpr (NI == 1) {
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + uint32_t(c), r);
                    emit(es, tile, c, r);
                }
            } else {
                // an issuer with no stage in the tile left its accumulator untouched
                const bool use0 = nks >= 2 || (nks == 1 && (cnt & 1u) == 0);
                const bool use1 = nks >= 2 || (nks == 1 && (cnt & 1u) == 1);
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r0[32], r1[32];
                    if constexpr (STACK) {
                        // each issuer's hi*lo half added to its first half
                        uint32_t h[32];
                        tmem_ld32x2(lane_base + uint32_t(c), lane_base + uint32_t(BN + c), r0, h);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r0[i] = __float_as_uint(__uint_as_float(r0[i]) + __uint_as_float(h[i]));
                        tmem_ld32x2(lane_base + uint32_t(AW + c), lane_base + uint32_t(AW + BN + c), r1, h);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r1[i] = __float_as_uint(__uint_as_float(r1[i]) + __uint_as_float(h[i]));
                    } else {
                        tmem_ld32x2(lane_base + uint32_t(c), lane_base + uint32_t(AW + c), r0, r1);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r0[i] = __float_as_uint((use0 ? __uint_as_float(r0[i]) : 0.f) +
                                                (use1 ? __uint_as_float(r1[i]) : 0.f));
                    emit(es, tile, c, r0);
                }
            }
            cnt += uint32_t(nks);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->acce[acc]);
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }

    // one unit per CTA when split: blockIdx.x is this CTA's piece
    if constexpr (CS) {
        if (prob.csplit > 1) cluster_split_reduce<Prob, BN>(prob, smem, *abort_flag == 0);
    }
}

// Largest number of clusters of `cs` CTAs of this kernel that the device runs
// at once (0 when it cannot launch them).  Cached per instantiation.
template <class Prob, int BN, int TERMS>
int max_active_clusters(int cs)
{
    using Cfg = TileCfg<BN, UsesTmemA<Prob>::value>;
    static std::atomic<int> cache[9];   // 0: not asked yet, -1: none fit (calls from several threads may race)
    if (cs < 1 || cs > 8) return 0;
    const int hit = cache[cs].load(std::memory_order_relaxed);
    if (hit != 0) return hit > 0 ? hit : 0;
    int n = 0;
    if (cudaFuncSetAttribute(tc_gemm_kernel<Prob, BN, TERMS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(Cfg::kSmemBytes)) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(cs));
        cfg.blockDim = dim3(EngineRoles<Prob, BN>::R::kThreads);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(cs);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<Prob, BN, TERMS>, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    cache[cs].store(n > 0 ? n : -1, std::memory_order_relaxed);
    return n > 0 ? n : 0;
}

// Host-side launch: persistent grid of min(tiles, SMs) CTAs.
template <class Prob, int BN, int TERMS>
cudaError_t launch_tc_gemm_terms(const Prob& prob, int num_tiles, int* err_word, cudaStream_t stream)
{
    using Cfg = TileCfg<BN, UsesTmemA<Prob>::value>;
    constexpr int kThreads = EngineRoles<Prob, BN>::R::kThreads;
    static std::atomic<bool> attr_set{false};   // per process; the attribute is per function
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<Prob, BN, TERMS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (num_tiles <= 0) return cudaSuccess;
    int grid = num_tiles < sm_count() ? num_tiles : sm_count();
    int cluster = 1;
    if constexpr (UsesClusterSplit<Prob>::value) {
        if (prob.csplit > 1) {   // one unit per CTA, clusters of csplit CTAs
            grid = num_tiles;
            cluster = prob.csplit;
        }
    }
    const int withhold = int(take_withhold_stage());
    cudaError_t e = launch_pdl_cluster(tc_gemm_kernel<Prob, BN, TERMS>, dim3(grid), dim3(kThreads), Cfg::kSmemBytes,
                                       stream, cluster, prob, err_word, withhold);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

// prob.terms (3 or 1) selects the kernel instantiation.
template <class Prob, int BN>
cudaError_t launch_tc_gemm(const Prob& prob, int num_tiles, int* err_word, cudaStream_t stream)
{
    return prob.terms == 1 ? launch_tc_gemm_terms<Prob, BN, 1>(prob, num_tiles, err_word, stream)
                           : launch_tc_gemm_terms<Prob, BN, 3>(prob, num_tiles, err_word, stream);
}

// ---------------------------------------------------------------------------
// Fast unsigned division by a runtime constant (Granlund-Montgomery):
// q = floor(n / d) for 0 <= n < 2^31, d >= 1.
struct FastDiv {
    uint32_t d, m, s;
    FastDiv() = default;
    __host__ explicit FastDiv(uint32_t divisor) : d(divisor)
    {
        uint32_t l = 0;
        while ((uint64_t(1) << l) < divisor) ++l;
        s = l;
        m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - divisor)) / divisor + 1);
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const
    {
        uint32_t t = __umulhi(n, m);
        return (t + n) >> s;   // exact for n < 2^31: t + n < 2^32
    }
    __device__ __forceinline__ void divmod(uint32_t n, uint32_t& q, uint32_t& r) const
    {
        q = div(n);
        r = n - q * d;
    }
};

}  // namespace cb200
