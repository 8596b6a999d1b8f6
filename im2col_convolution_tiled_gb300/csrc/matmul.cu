// matmul.cu -- the flagged matmul of the page "DirectCompute Neural Network
// Engine", section "Optimizations" -> "Transpose via Flags": C = op(A) op(B),
// row-major, flags bit 0 = A stored K x M, bit 1 = B stored N x K.
//
// Mapped onto the tcgen05 GEMM with A rows = rows of C and B rows = columns of
// C.  The gathers keep a warp's loads contiguous: a K-contiguous operand is
// read 16 bytes per thread along K (ChunkFast); A stored K x M 16 bytes per
// thread along M, four rows of one k (QuadRow); B stored K x N 4 bytes per
// thread along N (RowFast).  Either way the producer writes K-major swizzled
// hi/lo tiles, so all four flag combinations feed the same MMA.
//
// Tile width and K split are planned together (plan_matmul below): where the
// widest tiles leave SMs idle, each tile's K range is cut over a thread-block
// cluster (the engine's cluster split): csplit CTAs each run one K piece and
// the pieces are added in a fixed order through distributed shared memory.
#include "gemm_tc.cuh"
#include "gemm_tma.cuh"   // kTmaBK

namespace cb200 {

template <unsigned FLAGS, int BN>
struct MatmulProb {
    static constexpr bool kBBulk = false;
    static constexpr bool kClusterSplit = true;
    int terms = 3;    // tensor-core products per K step: 3 (3xTF32) or 1 (TF32)
    int csplit = 1;   // K pieces per tile, one per CTA of a cluster (1: whole tiles; a power of two)
    int lcsplit = 0;  // log2(csplit)
    static constexpr int kGroups = 2;
    static constexpr Map kAMap = (FLAGS & 1u) ? Map::QuadRow : Map::ChunkFast;
    // B stored K x N stays one row per thread: measured faster than QuadRow
    // for it (flag 0: 0.69 vs 0.61 of the roofline on 9216 x 9216 x 4096)
    static constexpr Map kBMap = (FLAGS & 2u) ? Map::ChunkFast : Map::RowFast;

    const float* A;
    const float* B;
    float* C;
    int M, K, N;
    // Fused epilogue (matmul_fused): c + bias[n], then max(0, .), then
    // c * (gate[m][n] > 0) -- each an fp32 operation, as add_bias, relu_fwd
    // and relu_bwd compute them; off when epi == 0.
    const float* bias = nullptr;
    const float* gate = nullptr;
    int relu = 0, epi = 0;
    int vec_bias = 0, vec_gate = 0;   // 16-byte loads allowed (bias aligned; gate aligned with N % 4 == 0)

    __device__ __forceinline__ float epilogue(float v, int m, int n) const
    {
        if (bias) v = __fadd_rn(v, __ldg(bias + n));
        if (relu) v = v > 0.f ? v : 0.f;
        if (gate) v = __fmul_rn(v, __ldg(gate + size_t(m) * N + n) > 0.f ? 1.f : 0.f);
        return v;
    }
    int m_tiles, n_tiles, k_stages;
    int vec_a, vec_b, vec_c;   // 16-byte accesses allowed along K (A, B) / along N (C)
    int vec_am;                // 16-byte accesses allowed along M (A stored K x M)

    __device__ int num_tiles() const { return m_tiles * n_tiles * csplit; }

    // Unit t: tile t / csplit, K piece t % csplit (the CTA's rank in its
    // cluster when csplit > 1).
    __device__ Tile tile(int t) const
    {
        const int tt = t >> lcsplit, j = t & (csplit - 1);
        Tile r;
        r.n0 = (tt % n_tiles) * BN;
        r.m0 = (tt / n_tiles) * kBM;
        r.ks0 = (j * k_stages) >> lcsplit;
        r.ks1 = ((j + 1) * k_stages) >> lcsplit;
        r.grp = 0;
        r.part = csplit > 1 ? j : -1;
        return r;
    }

    // Four consecutive-k values of a K-contiguous row (zero past K).
    __device__ __forceinline__ static void load4_k(const float* row, int k, int K, bool vec, float* v)
    {
        if (vec && k + 3 < K) {
            float4 f = __ldg(reinterpret_cast<const float4*>(row + k));
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = (k + e < K) ? __ldg(row + k + e) : 0.f;
        }
    }

    // QuadRow gather of an operand stored K x R (rows contiguous): rows
    // r0 + 4 (tid / 4) + j, K values k0 + 8 (tid % 4) + kk (zero past R or K).
    __device__ __forceinline__ static void load_quad(const float* X, int R, int K, bool vec, int r0, int k0, int tid,
                                                     float (&v)[32])
    {
        const int r = r0 + 4 * (tid >> 2);
        const int kb = k0 + 8 * (tid & 3);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int k = kb + kk;
            const float* src = X + size_t(k) * R + r;
            if (k < K && vec && r + 3 < R) {
                const float4 f = __ldg(reinterpret_cast<const float4*>(src));
                v[4 * kk] = f.x; v[4 * kk + 1] = f.y; v[4 * kk + 2] = f.z; v[4 * kk + 3] = f.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[4 * kk + j] = (k < K && r + j < R) ? __ldg(src + j) : 0.f;
            }
        }
    }

    struct AState {};
    __device__ AState a_setup(const Tile&, int) const { return {}; }

    __device__ void load_a(const AState&, const Tile& tl, int ks, int tid, float (&v)[32]) const
    {
        const int k0 = ks * kBK;
        if constexpr (FLAGS & 1u) {   // A stored K x M: (m, k) at k*M + m
            load_quad(A, M, K, vec_am != 0, tl.m0, k0, tid, v);
        } else {                      // A stored M x K: (m, k) at m*K + k
            const int kc = k0 + 4 * (tid & 7);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const int m = tl.m0 + (tid >> 3) + 16 * p;
                if (m < M) {
                    load4_k(A + size_t(m) * K, kc, K, vec_a, &v[4 * p]);
                } else {
                    v[4 * p] = v[4 * p + 1] = v[4 * p + 2] = v[4 * p + 3] = 0.f;
                }
            }
        }
    }

    struct BState {};
    __device__ BState b_setup(const Tile&, int) const { return {}; }

    __device__ void load_b(const BState&, const Tile& tl, int ks, int pass, int tid, float (&v)[32]) const
    {
        const int k0 = ks * kBK;
        if constexpr (FLAGS & 2u) {   // B stored N x K: (n, k) at n*K + k
            const int kc = k0 + 4 * (tid & 7);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const int n = tl.n0 + 128 * pass + (tid >> 3) + 16 * p;
                if (n < N) {
                    load4_k(B + size_t(n) * K, kc, K, vec_b, &v[4 * p]);
                } else {
                    v[4 * p] = v[4 * p + 1] = v[4 * p + 2] = v[4 * p + 3] = 0.f;
                }
            }
        } else {                      // B stored K x N: (n, k) at k*N + n
            // every thread loads a column, also past a narrower tile's BN
            // (the stores drop those): measured faster on small and mid-size
            // shapes than predicating the loads off, slower only on the
            // largest (4096^3: 0.69 vs 0.63 ms)
            const int n = tl.n0 + 128 * pass + tid;
            const bool nv = n < N;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int k = k0 + i;
                v[i] = (nv && k < K) ? __ldg(B + size_t(k) * N + n) : 0.f;
            }
        }
    }

    struct EState {
        float* crow;
        bool valid;
    };
    __device__ EState e_setup(const Tile& tl, int row) const
    {
        const int m = tl.m0 + row;
        EState e;
        e.valid = m < M;
        e.crow = C + size_t(e.valid ? m : 0) * N;
        return e;
    }

    // Cluster split: the sum of all pieces for columns n0 + c .. + 3 of one row.
    __device__ void reduce_store(const Tile& tl, int row, int c, float4 v) const
    {
        const int m = tl.m0 + row;
        const int n = tl.n0 + c;
        if (m >= M || n >= N) return;
        if (epi) {
            v.x = epilogue(v.x, m, n);
            if (n + 1 < N) v.y = epilogue(v.y, m, n + 1);
            if (n + 2 < N) v.z = epilogue(v.z, m, n + 2);
            if (n + 3 < N) v.w = epilogue(v.w, m, n + 3);
        }
        float* dst = C + size_t(m) * N + n;
        if (vec_c && n + 3 < N) {
            *reinterpret_cast<float4*>(dst) = v;
        } else {
            dst[0] = v.x;
            if (n + 1 < N) dst[1] = v.y;
            if (n + 2 < N) dst[2] = v.z;
            if (n + 3 < N) dst[3] = v.w;
        }
    }

    __device__ void store(const EState& e, const Tile& tl, int row, int c, const uint32_t (&r)[32]) const
    {
        if (!e.valid) return;
        const int n0 = tl.n0 + c;
        if (epi) {
            // eight columns at a time: their bias and gate values are loaded
            // together (16-byte loads where aligned), then applied in order
            const int m = tl.m0 + row;
            const float* grow = gate ? gate + size_t(m) * N : nullptr;
            const bool full = n0 + 32 <= N;
            uint32_t q[32];
#pragma unroll
            for (int g8 = 0; g8 < 32; g8 += 8) {
                float bv[8], gv[8];
                const int n = n0 + g8;
                if (bias) {
                    if (full && vec_bias) {
                        const float4 u = __ldg(reinterpret_cast<const float4*>(bias + n));
                        const float4 w = __ldg(reinterpret_cast<const float4*>(bias + n + 4));
                        bv[0] = u.x; bv[1] = u.y; bv[2] = u.z; bv[3] = u.w;
                        bv[4] = w.x; bv[5] = w.y; bv[6] = w.z; bv[7] = w.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) bv[i] = n + i < N ? __ldg(bias + n + i) : 0.f;
                    }
                }
                if (grow) {
                    if (full && vec_gate) {
                        const float4 u = __ldg(reinterpret_cast<const float4*>(grow + n));
                        const float4 w = __ldg(reinterpret_cast<const float4*>(grow + n + 4));
                        gv[0] = u.x; gv[1] = u.y; gv[2] = u.z; gv[3] = u.w;
                        gv[4] = w.x; gv[5] = w.y; gv[6] = w.z; gv[7] = w.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) gv[i] = n + i < N ? __ldg(grow + n + i) : 0.f;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float v = __uint_as_float(r[g8 + i]);
                    if (bias) v = __fadd_rn(v, bv[i]);
                    if (relu) v = v > 0.f ? v : 0.f;
                    if (grow) v = __fmul_rn(v, gv[i] > 0.f ? 1.f : 0.f);
                    q[g8 + i] = __float_as_uint(v);
                }
            }
            store_row(e, n0, q);
            return;
        }
        store_row(e, n0, r);
    }

    __device__ __forceinline__ void store_row(const EState& e, int n0, const uint32_t (&r)[32]) const
    {
        if (vec_c && n0 + 32 <= N) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(e.crow + n0 + i) =
                    make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                                __uint_as_float(r[i + 3]));
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (n0 + i < N) e.crow[n0 + i] = __uint_as_float(r[i]);
        }
    }
};

// Tiling plan: tile width BN and K pieces per tile (cluster split).
//
// The producers gather each stage through registers at a nearly fixed cost
// per operand row loaded (measured on GB300: about 7 cycles per 32-value row,
// against which the MMAs of a stage rarely bound it), so a stage costs about
// (A rows + B rows) -- min(M, 128) for A; min(N, BN) for B stored N x K, but
// 128 per pass for B stored K x N, whose loader reads a column per thread
// whatever the tile's width.  Wide tiles therefore do more work per producer
// cycle, and where they leave SMs idle the cluster split fills them.  The plan
// minimises rounds x (stages per unit + a fixed cost) x (cost of a stage) over
// BN in {256, 128, 64} (32 when N <= 32) and 1, 2, 4 or 8 pieces per tile, and,
// where the operands qualify, the TMA-fed kernel's whole tiles 128 or 256 wide.
struct MatmulPlan {
    int bn, cs;
    bool tma;   // operands by TMA (gemm_tma.cuh; whole tiles, cs == 1)
};

// Stage costs, measured on GB300 in cycles x 10 per 32 deep (steady-state
// stage times of large shapes at 2070 MHz):
// * register gather: a nearly fixed cost per operand row a producer loads,
//   7.2 cycles in 3xTF32, 5.4 in TF32 (no lo tiles to store);
// * TMA-fed: 2390 / 2040 cycles (3xTF32, 256 / 128 columns), 1100 / 1190
//   (TF32) -- the tensor core and the shared-memory port set it -- plus 3.2
//   cycles per row of an operand stored rows-contiguous, which the converters
//   transpose through shared memory (landing, reading and rewriting it).
constexpr long long kGatherRow10[2] = {72, 54};   // [3xTF32, TF32]
// ... scaled per flag combination (percent), measured at 256 columns on
// 9216 x 9216 x 4096 against the 384-row model: how each operand is gathered
// (A: 16 bytes along K or four rows of one k; B: a column per thread or 16
// bytes along K) shows in the stage time.
constexpr long long kGatherFlagPct[2][4] = {{89, 99, 107, 109}, {101, 99, 100, 123}};
constexpr long long kTransposeRow10 = 32;
inline long long tma_stage10(int bn, bool tf32)
{
    if (tf32) return bn == 256 ? 11000 : 11900;
    return bn == 256 ? 23900 : 20400;
}

constexpr int kTileFixedStages = 1;    // a whole tile's epilogue and hand-over
constexpr int kClusterFixedStages = 3; // a split tile's partials, cluster barriers and reduction

template <unsigned FLAGS, int BN>
static int mm_clusters(int cs)
{
    return math_terms() == 1 ? max_active_clusters<MatmulProb<FLAGS, BN>, BN, 1>(cs)
                             : max_active_clusters<MatmulProb<FLAGS, BN>, BN, 3>(cs);
}

template <unsigned FLAGS>
static int clusters_for(int bn, int cs)
{
    switch (bn) {
    case 256: return mm_clusters<FLAGS, 256>(cs);
    case 128: return mm_clusters<FLAGS, 128>(cs);
    case 64: return mm_clusters<FLAGS, 64>(cs);
    default: return mm_clusters<FLAGS, 32>(cs);
    }
}

// tma_ok: the shape and operands qualify for the TMA-fed kernel (tma_fed).
template <unsigned FLAGS>
static MatmulPlan plan_matmul(int M, int K, int N, bool tma_ok)
{
    const int P = sm_count();
    const bool tf32 = math_terms() == 1;
    const long long mt = (M + kBM - 1) / kBM;
    const int ks = (K + kBK - 1) / kBK;
    const int bn_max = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;
    const int bn_min = bn_max < 64 ? bn_max : 64;
    MatmulPlan best{bn_max, 1, false};
    long long best_cost = -1, best_units = 0;
    const int engine = matmul_engine_override();   // test hook: -1 plan, 0 gather, 1 TMA where eligible
    if (engine == 0) tma_ok = false;
    // the TMA-fed kernel: whole tiles 128 or 256 wide on a persistent grid,
    // whose boxes (128 rows of A, bn rows of B) the tensors can fill
    if (tma_ok && M >= kBM) {
        for (int bn = bn_max; bn >= 128; bn /= 2) {
            if (N < bn) continue;
            const long long tiles = mt * ((N + bn - 1) / bn);
            const long long trows = ((FLAGS & 1u) ? kBM : 0) + ((FLAGS & 2u) ? 0 : bn);   // transposed rows
            const long long cost = ((tiles + P - 1) / P) * (ks + kTileFixedStages) *
                                   (tma_stage10(bn, tf32) + trows * kTransposeRow10);
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                best_units = tiles;
                best = MatmulPlan{bn, 1, true};
            }
        }
    }
    for (int bn = bn_max; bn >= bn_min; bn /= 2) {
        const long long tiles = mt * ((N + bn - 1) / bn);
        const long long rows_a = M < kBM ? M : kBM;
        const long long rows_b = (FLAGS & 2u) ? (N < bn ? N : bn) : 128LL * ((bn + 127) / 128);
        if (engine == 1 && best.tma) break;   // forced TMA: the register plans are not candidates
        for (int cs = 1; cs <= 8; cs *= 2) {
            if (cs > 1 && ks < 2 * cs) break;
            const int slots = cs == 1 ? P : clusters_for<FLAGS>(bn, cs);
            if (slots <= 0) continue;
            const long long rounds = (tiles + slots - 1) / slots;
            const long long per = (ks + cs - 1) / cs + (cs == 1 ? kTileFixedStages : kClusterFixedStages);
            const long long cost =
                rounds * per * (rows_a + rows_b) * kGatherRow10[tf32 ? 1 : 0] * kGatherFlagPct[tf32 ? 1 : 0][FLAGS] / 100;
            // on a tie the plan with more CTAs wins: they share the same work
            // (small shapes are latency-bound)
            const long long units = tiles * cs;
            if (best_cost < 0 || cost < best_cost || (cost == best_cost && units > best_units)) {
                best_cost = cost;
                best_units = units;
                best = MatmulPlan{bn, cs, false};
            }
        }
    }
    return best;
}

template <unsigned FLAGS, int BN>
static cudaError_t run_matmul(int M, int K, int N, int cs, const float* A, const float* B, float* C,
                              const MatmulEpi& ep, cudaStream_t st)
{
    MatmulProb<FLAGS, BN> p;
    p.terms = math_terms();
    p.bias = ep.bias;
    p.gate = ep.gate;
    p.relu = ep.relu ? 1 : 0;
    p.epi = (ep.bias || ep.gate || ep.relu) ? 1 : 0;
    p.vec_bias = ep.bias && aligned16(ep.bias);
    p.vec_gate = ep.gate && (N % 4 == 0) && aligned16(ep.gate);
    p.A = A;
    p.B = B;
    p.C = C;
    p.M = M;
    p.K = K;
    p.N = N;
    p.m_tiles = (M + kBM - 1) / kBM;
    p.n_tiles = (N + BN - 1) / BN;
    p.k_stages = (K + kBK - 1) / kBK;
    p.vec_a = (K % 4 == 0) && aligned16(A);
    p.vec_b = (K % 4 == 0) && aligned16(B);
    p.vec_c = (N % 4 == 0) && aligned16(C);
    p.vec_am = (M % 4 == 0) && aligned16(A);
    p.csplit = cs;
    while ((1 << p.lcsplit) < p.csplit) ++p.lcsplit;
    return launch_tc_gemm<MatmulProb<FLAGS, BN>, BN>(p, p.m_tiles * p.n_tiles * p.csplit, device_error_word(), st);
}

// TMA-fed path (gemm_tma.cuh): every operand's row pitch a multiple of 16
// bytes (K % 4 == 0 for a K-contiguous operand, M or N % 4 == 0 for a
// rows-contiguous one), 16-byte aligned operands, no fused epilogue; the plan
// then offers it whole tiles 128 or 256 wide that M and N fill (M >= 128,
// N >= the tile width).  Everything else runs on the register-gather engine.
static bool tma_ok(unsigned flags, int M, int N, int K, const float* A, const float* B, const MatmulEpi& ep)
{
    const bool pitch_a = (flags & 1u) ? M % 4 == 0 : K % 4 == 0;
    const bool pitch_b = (flags & 2u) ? K % 4 == 0 : N % 4 == 0;
    return pitch_a && pitch_b && N > 64 && aligned16(A) && aligned16(B) && !ep.bias && !ep.gate && !ep.relu;
}

template <unsigned FLAGS>
static cudaError_t run_flags(int M, int K, int N, const float* A, const float* B, float* C, const MatmulEpi& ep,
                             cudaStream_t st)
{
    const MatmulPlan pl = plan_matmul<FLAGS>(M, K, N, tma_ok(FLAGS, M, N, K, A, B, ep));
    if (pl.tma) return launch_matmul_tma(FLAGS, pl.bn, M, K, N, A, B, C, st);
    switch (pl.bn) {
    case 256: return run_matmul<FLAGS, 256>(M, K, N, pl.cs, A, B, C, ep, st);
    case 128: return run_matmul<FLAGS, 128>(M, K, N, pl.cs, A, B, C, ep, st);
    case 64: return run_matmul<FLAGS, 64>(M, K, N, pl.cs, A, B, C, ep, st);
    default: return run_matmul<FLAGS, 32>(M, K, N, pl.cs, A, B, C, ep, st);
    }
}

void matmul_tiling(int M, int K, int N, unsigned flags, const float* A, const float* B, int* bn, int* csplit,
                   int* tma)
{
    MatmulPlan pl;
    const bool ok = tma_ok(flags, M, N, K, A, B, MatmulEpi{});
    switch (flags) {
    case 0: pl = plan_matmul<0>(M, K, N, ok); break;
    case 1: pl = plan_matmul<1>(M, K, N, ok); break;
    case 2: pl = plan_matmul<2>(M, K, N, ok); break;
    default: pl = plan_matmul<3>(M, K, N, ok); break;
    }
    *bn = pl.bn;
    *csplit = pl.cs;
    *tma = pl.tma ? 1 : 0;
}

cudaError_t launch_matmul(int M, int K, int N, unsigned flags, const float* A, const float* B, float* C,
                          cudaStream_t st, const MatmulEpi& ep)
{
    switch (flags) {
    case 0: return run_flags<0>(M, K, N, A, B, C, ep, st);
    case 1: return run_flags<1>(M, K, N, A, B, C, ep, st);
    case 2: return run_flags<2>(M, K, N, A, B, C, ep, st);
    default: return run_flags<3>(M, K, N, A, B, C, ep, st);
    }
}

}  // namespace cb200
