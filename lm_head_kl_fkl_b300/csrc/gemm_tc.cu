// Persistent 2-SM tcgen05 GEMM for sm_103a and the epilogues of every
// tensor-core pass of the library (loss forward, dz, fp32 tiles for dh and dW,
// the kept-logits forward, the KL + CE mixture, the teacher top-K passes), plus a
// one-thread kernel that exercises the bounded pipeline wait.
//
//   C[m, n] = sum_k A(m, k) B(n, k)      bf16 operands, fp32 accumulator in TMEM
//
// CTAs run in pairs (a cluster of 2).  A pair owns one 256 x BN output tile at a
// time: CTA rank r holds rows [128 r, 128 r + 128) of A and columns
// [r BN/2, (r+1) BN/2) of B in its own shared memory, and the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = BN, K = 16), which reads both CTAs'
// operands and leaves rows [128 r, 128 r + 128) of the tile in CTA r's TMEM.
// Per SM this halves the B operand's L2->SMEM traffic and shared-memory reads
// against a one-SM 128 x BN tile, and leaves room for a deeper TMA ring.
//
// Wide tiles (NSUB = 2, EPI_F32 only): a pair owns 256 x 512 outputs as two
// N = 256 sub-tiles that share every A k-block, so each CTA loads 16 KB of A and
// 32 KB of B per 64-deep k-block for twice the MMA work of a 256-wide tile: 25 %
// less L2->SMEM traffic per FLOP.  The 512-column accumulator fills TMEM, so it
// is single-buffered (the epilogue does not overlap the next tile's MMAs); this
// pays where the k-loop is long against the epilogue (dh).
//
// On the last, ragged column tile (of either kind) the MMA's N shrinks to the
// valid columns rounded up to 64, and both CTAs load their halves of that
// narrower B, so no tensor work goes to padding.
//
// Roles, in each CTA of the pair (192 threads, one CTA per SM):
//   warp 0      one lane issues the CTA's TMA loads of A and B k-blocks into a
//               STAGES-deep ring (128-byte swizzle); both CTAs' copies complete
//               on the even CTA's `full` barrier, which the even CTA arms with
//               the byte count of the pair;
//   warp 1      allocates 512 TMEM columns (two 256-column accumulators, or one
//               512-column accumulator for wide tiles) for the pair; in
//               the even CTA one lane issues the MMAs, commits `empty` (stage
//               reusable) and `tfull` (accumulator complete) to both CTAs.  This
//               one thread paces the 256-wide tiles, so their k-blocks go out in
//               pairs, eight MMAs per asm block, with the next stages' barriers
//               tested without blocking inside the same block;
//   warps 2-5   the epilogue: each warp drains its 32 TMEM lanes (= 32 output
//               rows) with tcgen05.ld and reports the buffer free on the even
//               CTA's `tempty` barrier, so the next tile's MMAs overlap it.
//
// Epilogues
//   EPI_LSE  logits of a row pair-tile x 256 vocabulary columns: online base-2
//            max / sum of 2^(z log2e / T) per row plus the teacher gather
//            sum_k p_k z_{idx_k}; one (max, sum, gather) triple per row and tile.
//   EPI_DZ   the same logits recomputed: dz = coef * (2^(z log2e/T - lse log2e) - s)
//            in bf16, staged per warp in swizzled shared memory and TMA-stored.
//   EPI_F32  plain fp32 tile, TMA-stored or TMA reduce-added (dh partials, dW).
//   EPI_LSE_MIX / EPI_DZ_MIX  the same for the KL + hard-label cross-entropy
//            mixture: also a temperature-1 running max / sum and the logit at the
//            row's label; dz gains (1 - alpha)/T (q_1 - onehot(label)) per row.
//   EPI_TMAX each row's kTopPerTile largest logits over the tile, with their
//            ids (teacher top-K; the first of them is the tile max).
//   EPI_CAND for the rows flagged by topk_rows_kernel (a tile with kTopPerTile or
//            more logits >= the row's threshold), every logit >= the threshold,
//            appended to the row's candidate list with an atomic counter; logits
//            equal to the threshold go to a separate list of at most K ids.  The
//            whole launch returns at once when no row is flagged.
//   EPI_LSE_Y  EPI_LSE for a forward whose backward follows at once: a first
//            pass over the tile finds each row's tile max (and gathers the
//            teacher logits), a second sums 2^(y) and keeps y = z log2e / T - max
//            in fp16 (staged like EPI_DZ, TMA-stored), so that dz can later be
//            formed from y without recomputing the tile.  Relative to the tile
//            max, y is exact to 2^-11 of |y| where q is largest.
//
// Operand majorness (template): K-major tiles arrive as one TMA box {64, rows};
// MN-major tiles as boxes {64 (MN), 64 (K)} side by side, 8 KB apart.  When A is
// the dz buffer (p.a_panel), it is read through a 3-D map of its 64-column panels
// {64, rows, panel}: a K-major k-block is one box {64, 128, 1} (dh), an MN-major one
// a single box {64, 64, 2} covering both panels of the CTA's 128 rows (dW); the
// staged epilogues of dz and of the kept logits store into the same panels.
#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "ptx.cuh"

namespace fkl {

template <int BN, int NSUB, int B_MN, int EPI>
struct PairCfg {
    static constexpr int BNH = BN / 2;                     // B columns of one sub-tile held by one CTA
    static constexpr int TW = BN * NSUB;                   // output columns of a pair tile
    static constexpr int NBUF = NSUB == 1 ? 2 : 1;         // TMEM accumulator buffers
    static constexpr uint32_t A_BYTES = kBM * kBK * 2;     // 128 rows x 64 k, bf16
    static constexpr int B_BOXES = B_MN ? (BNH + 63) / 64 : 1;
    static constexpr uint32_t B_SUB_BYTES = B_MN ? B_BOXES * 8192u : static_cast<uint32_t>(BNH) * 128u;
    static constexpr uint32_t B_BYTES = NSUB * B_SUB_BYTES;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t STAGING_BYTES = epi_staged(EPI) ? 4u * 2u * 4096u : 0u;  // 2 x 4 KB per epilogue warp
    static constexpr uint32_t RING_BUDGET = 196608u + (epi_staged(EPI) ? 0u : 32768u);
    static constexpr int STAGES = (RING_BUDGET / STAGE_BYTES) > 8 ? 8 : (RING_BUDGET / STAGE_BYTES);
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr size_t SMEM = size_t(STAGES) * STAGE_BYTES + STAGING_BYTES + BAR_BYTES + 1024;
};

__device__ __forceinline__ void decode_unit(int u, const GemmParams& p, int& m, int& n, int& s) {
    const int mn = p.m_tiles * p.n_tiles;
    s = u / mn;
    const int r = u - s * mn;
    if (p.m_fastest) {
        m = r % p.m_tiles;
        n = r / p.m_tiles;
    } else {
        n = r % p.n_tiles;
        m = r / p.n_tiles;
    }
}

__device__ __forceinline__ int kb_begin(const GemmParams& p, int s) {
    return static_cast<int>((static_cast<long long>(s) * p.kb_total) / p.splits);
}

// Sorted-teacher cursor of one row: first position whose id is >= v0.
struct TeacherCursor {
    const int* ids;
    const float* probs;
    int K, pos, next_id;
    float next_p;

    __device__ __forceinline__ void seek(const int* sidx, const float* sp, int row, bool row_ok, int k,
                                         int v0) {
        K = k;
        ids = sidx + static_cast<size_t>(row_ok ? row : 0) * k;
        probs = sp + static_cast<size_t>(row_ok ? row : 0) * k;
        next_id = INT_MAX;
        next_p = 0.f;
        pos = k;
        if (!row_ok) return;
        int lo = 0, hi = k;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(ids + mid) < v0) lo = mid + 1; else hi = mid;
        }
        pos = lo;
        if (pos < K) {
            next_id = __ldg(ids + pos);
            next_p = __ldg(probs + pos);
        }
    }
    __device__ __forceinline__ void advance() {
        if (++pos < K) {
            next_id = __ldg(ids + pos);
            next_p = __ldg(probs + pos);
        } else {
            next_id = INT_MAX;
        }
    }
};

// Lane 0 waits, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Width of sub-tile j of column tile n: BN, except on the ragged last column
// tile, where the MMA's N shrinks to the valid columns rounded up to 64 (0 if none
// are left), so that no MMA work goes to padding (d = 2880 on 256-wide tiles would
// otherwise waste 6.7 %).  Accumulator columns beyond the width keep stale values;
// every epilogue reads only columns below Ncols, which the width covers.
template <int BN, int NSUB>
__device__ __forceinline__ int sub_width(const GemmParams& p, int n, int j) {
    const int rest = p.Ncols - n * BN * NSUB - j * BN;
    if (rest >= BN) return BN;
    return rest <= 0 ? 0 : (rest + 63) & ~63;
}

template <int BN, int NSUB, int A_MN, int B_MN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
    using C = PairCfg<BN, NSUB, B_MN, EPI>;
    constexpr int STAGES = C::STAGES;
    constexpr int TW = C::TW;
    constexpr int NBUF = C::NBUF;
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tile width");
    static_assert(NSUB == 1 || (NSUB == 2 && BN == 256 && EPI == EPI_F32), "wide tiles: 2 x 256, fp32 epilogue");
    static_assert((EPI != EPI_DZ && EPI != EPI_DZ_MIX && EPI != EPI_LSE_Y) || BN % 64 == 0,
                  "dz / logit boxes are 64 columns");
    static_assert(B_MN || BN / 2 <= 256, "K-major B box height");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t staging0 = base + STAGES * C::STAGE_BYTES;
    const uint32_t bar0 = staging0 + C::STAGING_BYTES;
    uint8_t* gbar = gbase + (bar0 - base);
    const uint32_t full0 = bar0, empty0 = bar0 + 8u * STAGES, tfull0 = bar0 + 16u * STAGES,
                   tempty0 = tfull0 + 16u, drain_bar = tempty0 + 16u;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(gbar + 16 * STAGES + 40);
    volatile int* s_abort = reinterpret_cast<volatile int*>(gbar + 16 * STAGES + 44);

    if constexpr (EPI == EPI_CAND) {
        if (*p.any_flag == 0) return;  // every CTA reads the same word: all leave, nothing was set up
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            mbar_init(tempty0 + 8u * a, 8);  // 4 epilogue warps in each CTA of the pair
        }
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (epi_staged(EPI)) tma_prefetch_desc(&tmOut);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(s_tmem), 512);
        tmem_relinquish_pair();
    }
    // barriers of both CTAs initialised and TMEM allocated before any peer traffic
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int units = p.m_tiles * p.n_tiles * p.splits;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t full_leader = mapa_shared(full0, 0);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int u = pair; u < units && ok; u += npairs) {
                int m, n, s;
                decode_unit(u, p, m, n, s);
                const int kb0 = kb_begin(p, s), kb1 = kb_begin(p, s + 1);
                const int arow = m * 2 * kBM + static_cast<int>(rank) * kBM;
                int bcol[NSUB];  // first B column of this CTA's half of each sub-tile
#pragma unroll
                for (int j = 0; j < NSUB; ++j) {
                    const int w = sub_width<BN, NSUB>(p, n, j);
                    bcol[j] = n * TW + j * BN + static_cast<int>(rank) * (w == BN ? BN / 2 : w / 2);
                }
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * C::STAGE_BYTES, sb = sa + C::A_BYTES;
                    const uint32_t fb = full_leader + 8u * stage;
                    if (leader) mbar_arrive_expect_tx(full0 + 8u * stage, 2u * C::STAGE_BYTES);
                    if (A_MN == 0) {
                        if (p.a_panel) tma_load_3d_pair(sa, &tmA, fb, 0, arow, kb);
                        else tma_load_2d_pair(sa, &tmA, fb, kb * kBK, arow);
                    } else if (p.a_panel) {
                        // the two 64-column panels of the CTA's 128 A rows in one box {64, 64, 2}:
                        // each TMA instruction costs the producer about 100 cycles, whatever its size
                        tma_load_3d_pair(sa, &tmA, fb, 0, kb * kBK, arow >> 6);
                    } else {
                        tma_load_2d_pair(sa, &tmA, fb, arow, kb * kBK);
                        tma_load_2d_pair(sa + 8192u, &tmA, fb, arow + 64, kb * kBK);
                    }
#pragma unroll
                    for (int j = 0; j < NSUB; ++j) {
                        const uint32_t sbj = sb + j * C::B_SUB_BYTES;
                        if (B_MN == 0) {
                            tma_load_2d_pair(sbj, &tmB, fb, kb * kBK, bcol[j]);
                        } else {
#pragma unroll
                            for (int b = 0; b < C::B_BOXES; ++b)
                                tma_load_2d_pair(sbj + 8192u * b, &tmB, fb, bcol[j] + 64 * b, kb * kBK);
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && leader) {  // let the pair's copies already in flight land
                const long long first = issued > STAGES ? issued - STAGES : 0;
                for (long long i = first; i < issued; ++i)
                    mbar_wait_drain(full0 + 8u * static_cast<uint32_t>(i % STAGES),
                                    static_cast<uint32_t>((i / STAGES) & 1));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && leader) {
            int stage = 0, tc = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = pair; u < units && ok; u += npairs, ++tc) {
                int m, n, s;
                decode_unit(u, p, m, n, s);
                const int kb0 = kb_begin(p, s), kb1 = kb_begin(p, s + 1);
                const int acc = tc % NBUF;
                const uint32_t aph = (tc / NBUF) & 1;
                int width[NSUB];
                bool full = true;
#pragma unroll
                for (int j = 0; j < NSUB; ++j) {
                    width[j] = sub_width<BN, NSUB>(p, n, j);
                    full = full && width[j] == BN;
                }
                if (!mbar_wait(tempty0 + 8u * acc, aph ^ 1u, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * 256);
                // Full tiles (all but the ragged last column tile) issue with the
                // compile-time instruction descriptor and no width tests.
                auto kloop = [&](auto full_tag) {
                    constexpr bool FULL = decltype(full_tag)::value;
                    uint32_t idesc[NSUB];
#pragma unroll
                    for (int j = 0; j < NSUB; ++j)
                        idesc[j] = FULL ? umma_idesc_bf16(2 * kBM, BN, A_MN, B_MN)
                                        : umma_idesc_bf16(2 * kBM, width[j] > 0 ? width[j] : BN, A_MN, B_MN);
                    if constexpr (FULL && NSUB == 1) {
                        // k-blocks go in pairs, each pair from one asm block
                        // (umma_2kblocks_pair; an odd last one from umma_kblock_pair)
                        // that also tests, without blocking, whether the stages after
                        // it have landed: when they have, the next pair starts without
                        // a barrier round trip.  The descriptors of stage s are those
                        // of stage 0 plus s * STAGE_BYTES / 16 (the address field is
                        // linear below 256 KB).
                        static_assert(STAGES >= 4, "two stages issued and two tested are distinct");
                        const uint64_t ad0 = A_MN ? smem_desc_sw128(base, 8192u, 1024u)
                                                  : smem_desc_sw128(base, 16u, 1024u);
                        const uint64_t bd0 = B_MN ? smem_desc_sw128(base + C::A_BYTES, 8192u, 1024u)
                                                  : smem_desc_sw128(base + C::A_BYTES, 16u, 1024u);
                        constexpr uint32_t KA = A_MN ? 2048u / 16u : 32u / 16u;
                        constexpr uint32_t KB = B_MN ? 2048u / 16u : 32u / 16u;
                        constexpr uint64_t kStageDesc = C::STAGE_BYTES >> 4;
                        auto next = [](int st, uint32_t ph, int& nst, uint32_t& nph) {
                            nst = st + 1 == STAGES ? 0 : st + 1;
                            nph = st + 1 == STAGES ? ph ^ 1u : ph;
                        };
                        bool landed = false;  // the stages this iteration uses are known to have landed
                        int kb = kb0;
                        for (; kb + 1 < kb1; kb += 2) {
                            int s1, s2, s3;
                            uint32_t p1, p2, p3;
                            next(stage, phase, s1, p1);
                            next(s1, p1, s2, p2);
                            next(s2, p2, s3, p3);
                            if (!landed && (!mbar_wait(full0 + 8u * stage, phase, s_abort, p.status) ||
                                            !mbar_wait(full0 + 8u * s1, p1, s_abort, p.status))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t o0 = static_cast<uint64_t>(stage) * kStageDesc;
                            const uint64_t o1 = static_cast<uint64_t>(s1) * kStageDesc;
                            landed = umma_2kblocks_pair<KA, KB>(dt, ad0 + o0, bd0 + o0, ad0 + o1, bd0 + o1, idesc[0],
                                                                kb > kb0 ? 1u : 0u, empty0 + 8u * stage,
                                                                empty0 + 8u * s1, full0 + 8u * s2, p2,
                                                                full0 + 8u * s3, p3) != 0;
                            stage = s2;
                            phase = p2;
                        }
                        if (ok && kb < kb1) {
                            int s1;
                            uint32_t p1;
                            next(stage, phase, s1, p1);
                            if (!landed && !mbar_wait(full0 + 8u * stage, phase, s_abort, p.status)) {
                                ok = false;
                                return;
                            }
                            tc_fence_after();
                            const uint64_t o0 = static_cast<uint64_t>(stage) * kStageDesc;
                            umma_kblock_pair<KA, KB>(dt, ad0 + o0, bd0 + o0, idesc[0], kb > kb0 ? 1u : 0u,
                                                     empty0 + 8u * stage, full0 + 8u * s1, p1);
                            stage = s1;
                            phase = p1;
                        }
                    } else {
                        for (int kb = kb0; kb < kb1; ++kb) {
                            if (!mbar_wait(full0 + 8u * stage, phase, s_abort, p.status)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t sa = base + stage * C::STAGE_BYTES, sb = sa + C::A_BYTES;
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk) {
                                const uint64_t ad = A_MN ? smem_desc_sw128(sa + 2048u * kk, 8192u, 1024u)
                                                         : smem_desc_sw128(sa + 32u * kk, 16u, 1024u);
#pragma unroll
                                for (int j = 0; j < NSUB; ++j) {
                                    if (!FULL && width[j] == 0) continue;
                                    const uint32_t sbj = sb + j * C::B_SUB_BYTES;
                                    const uint64_t bd = B_MN ? smem_desc_sw128(sbj + 2048u * kk, 8192u, 1024u)
                                                             : smem_desc_sw128(sbj + 32u * kk, 16u, 1024u);
                                    umma_bf16_pair(dt + static_cast<uint32_t>(j * BN), ad, bd, idesc[j],
                                                   (kb > kb0 || kk > 0) ? 1u : 0u);
                                }
                            }
                            umma_commit_pair(empty0 + 8u * stage);
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                };
                if (full) kloop(std::true_type{});
                else kloop(std::false_type{});
                if (!ok) break;
                umma_commit_pair(tfull0 + 8u * acc);
            }
            if (!ok) {  // no MMA may still be running when TMEM is released
                umma_commit_pair(drain_bar);
                mbar_wait_drain(drain_bar, 0);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t tempty_leader = mapa_shared(tempty0, 0);
        uint32_t box = 0;
        int tc = 0;
        for (int u = pair; u < units; u += npairs, ++tc) {
            int m, n, s;
            decode_unit(u, p, m, n, s);
            const int acc = tc % NBUF;
            const uint32_t aph = (tc / NBUF) & 1;
            const int wrow = m * 2 * kBM + static_cast<int>(rank) * kBM + q * 32;  // first row of this warp
            const int row = wrow + lane;
            const bool row_ok = row < p.M;
            const uint32_t tt = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(acc * 256);

            if constexpr (EPI == EPI_LSE || EPI == EPI_LSE_MIX) {
                constexpr bool MIX = EPI == EPI_LSE_MIX;
                const int v0 = n * BN;
                TeacherCursor cur;
                cur.seek(p.sidx, p.sp, row, row_ok, p.K, v0);
                int ylab = -1;
                if constexpr (MIX) ylab = row_ok ? __ldg(p.label + row) : -1;
                if (!warp_wait(tfull0 + 8u * acc, aph, s_abort, p.status)) break;
                tc_fence_after();
                float mrun = -INFINITY, lrun = 0.f, g = 0.f;
                float m1run = -INFINITY, l1run = 0.f, gy = 0.f;  // temperature-1 terms (MIX only)
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int col0 = v0 + c * 32;
                    if (col0 >= p.Ncols) break;
                    float z[32];
                    __syncwarp();
                    tmem_ld32(tt + c * 32, z);
                    while (cur.next_id < col0 + 32) {
                        g += cur.next_p * select32(z, cur.next_id - col0);
                        cur.advance();
                    }
                    if constexpr (MIX) {
                        if (ylab >= col0 && ylab < col0 + 32) gy = select32(z, ylab - col0);
                    }
                    const int nv = p.Ncols - col0;
                    // the max of the raw logits (scale2 > 0: max(z) scale2 = max(z scale2), bit
                    // for bit), then 2^(z scale2 - max) with one FMA per logit; columns beyond
                    // Ncols (last tile only) are -inf
                    if (nv < 32) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) z[j] = (j < nv) ? z[j] : -INFINITY;
                    }
                    float cm0 = z[0], cm1 = z[1];
#pragma unroll
                    for (int j = 2; j < 32; j += 2) {
                        cm0 = fmaxf(cm0, z[j]);
                        cm1 = fmaxf(cm1, z[j + 1]);
                    }
                    const float zmax = fmaxf(cm0, cm1);
                    const float mnew = fmaxf(mrun, zmax * p.scale2);
                    const float nm = -mnew;
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        s0 += ex2_approx(fmaf(z[j], p.scale2, nm));
                        s1 += ex2_approx(fmaf(z[j + 1], p.scale2, nm));
                        s2 += ex2_approx(fmaf(z[j + 2], p.scale2, nm));
                        s3 += ex2_approx(fmaf(z[j + 3], p.scale2, nm));
                    }
                    lrun = lrun * ex2_approx(mrun - mnew) + ((s0 + s1) + (s2 + s3));
                    mrun = mnew;
                    if constexpr (MIX) {  // the same online sum at temperature 1, on z log2e
                        constexpr float kL2e = 1.4426950408889634f;
                        const float m1new = fmaxf(m1run, zmax * kL2e);
                        const float nm1 = -m1new;
                        float t0 = 0.f, t1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            t0 += ex2_approx(fmaf(z[j], kL2e, nm1));
                            t1 += ex2_approx(fmaf(z[j + 1], kL2e, nm1));
                        }
                        l1run = l1run * ex2_approx(m1run - m1new) + (t0 + t1);
                        m1run = m1new;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
                if (row_ok) {
                    const size_t o = static_cast<size_t>(n) * p.part_stride + row;
                    p.part_m[o] = mrun;
                    p.part_l[o] = lrun;
                    p.part_g[o] = g;
                    if constexpr (MIX) {
                        p.part_m1[o] = m1run;
                        p.part_l1[o] = l1run;
                        p.part_gy[o] = gy;
                    }
                }
            } else if constexpr (EPI == EPI_LSE_Y) {
                const int v0 = n * BN;
                TeacherCursor cur;
                cur.seek(p.sidx, p.sp, row, row_ok, p.K, v0);
                if (!warp_wait(tfull0 + 8u * acc, aph, s_abort, p.status)) break;
                tc_fence_after();
                // pass 1: the row's max over this tile and the teacher gather
                float mt = -INFINITY, g = 0.f;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int col0 = v0 + c * 32;
                    if (col0 >= p.Ncols) break;
                    float z[32];
                    __syncwarp();
                    tmem_ld32(tt + c * 32, z);
                    while (cur.next_id < col0 + 32) {
                        g += cur.next_p * select32(z, cur.next_id - col0);
                        cur.advance();
                    }
                    const int nv = p.Ncols - col0;
                    if (nv < 32) {  // the last tile: columns beyond Ncols are -inf
#pragma unroll
                        for (int j = 0; j < 32; ++j) z[j] = (j < nv) ? z[j] : -INFINITY;
                    }
                    float cm0 = z[0], cm1 = z[1];
#pragma unroll
                    for (int j = 2; j < 32; j += 2) {
                        cm0 = fmaxf(cm0, z[j]);
                        cm1 = fmaxf(cm1, z[j + 1]);
                    }
                    mt = fmaxf(mt, fmaxf(cm0, cm1));
                }
                mt *= p.scale2;  // scale2 > 0: the max of the scaled logits
                // pass 2: sum of 2^(y) and y = z scale2 - mt kept in fp16, 64 columns per TMA box
                float l0 = 0.f, l1 = 0.f;
#pragma unroll 1
                for (int c2 = 0; c2 < BN / 64; ++c2) {
                    const int col0 = v0 + c2 * 64;
                    if (col0 >= p.Ncols) break;
                    const uint32_t buf = staging0 + static_cast<uint32_t>(q * 2 + (box & 1)) * 4096u;
                    if (lane == 0) bulk_wait_read_le1();
                    __syncwarp();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int cc = col0 + hh * 32;
                        float z[32];
                        __syncwarp();
                        tmem_ld32(tt + c2 * 64 + hh * 32, z);
                        const int nv = p.Ncols - cc;
                        const float nmt = -mt;
                        if (nv >= 32) {
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                z[j] = fmaf(z[j], p.scale2, nmt);
                                z[j + 1] = fmaf(z[j + 1], p.scale2, nmt);
                                l0 += ex2_approx(z[j]);
                                l1 += ex2_approx(z[j + 1]);
                            }
                        } else {  // the last tile: columns beyond Ncols add nothing
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                z[j] = fmaf(z[j], p.scale2, nmt);
                                z[j + 1] = fmaf(z[j + 1], p.scale2, nmt);
                                l0 += (j < nv) ? ex2_approx(z[j]) : 0.f;
                                l1 += (j + 1 < nv) ? ex2_approx(z[j + 1]) : 0.f;
                            }
                        }
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) w[j] = pack_f16x2(z[2 * j], z[2 * j + 1]);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            st_shared_v4(buf + lane * 128u + ((static_cast<uint32_t>(hh * 4 + k) ^ (lane & 7u)) << 4),
                                         w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0 && wrow < p.M) {
                        tma_store_3d(&tmOut, buf, 0, wrow, col0 >> 6);
                        bulk_commit();
                    }
                    ++box;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
                if (row_ok) {
                    const size_t o = static_cast<size_t>(n) * p.part_stride + row;
                    p.part_m[o] = mt;
                    p.part_l[o] = l0 + l1;
                    p.part_g[o] = g;
                }
            } else if constexpr (EPI == EPI_TMAX) {
                if (!warp_wait(tfull0 + 8u * acc, aph, s_abort, p.status)) break;
                tc_fence_after();
                const int v0 = n * BN;
                // the row's kTopPerTile largest logits over the tile, descending; equal
                // ones keep the smaller id (columns arrive in increasing order)
                float tv[kTopPerTile];
                int ti[kTopPerTile];
#pragma unroll
                for (int e = 0; e < kTopPerTile; ++e) {
                    tv[e] = -INFINITY;
                    ti[e] = INT_MAX;
                }
                // insert x (id xi) into the descending list, below the kept values >= x
                auto insert = [&](float x, int xi) {
                    bool gt[kTopPerTile];
#pragma unroll
                    for (int e = 0; e < kTopPerTile; ++e) gt[e] = x > tv[e];
#pragma unroll
                    for (int e = kTopPerTile - 1; e > 0; --e) {  // shift down below x's place
                        tv[e] = gt[e - 1] ? tv[e - 1] : (gt[e] ? x : tv[e]);
                        ti[e] = gt[e - 1] ? ti[e - 1] : (gt[e] ? xi : ti[e]);
                    }
                    tv[0] = gt[0] ? x : tv[0];
                    ti[0] = gt[0] ? xi : ti[0];
                };
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int col0 = v0 + c * 32;
                    if (col0 >= p.Ncols) break;
                    float z[32];
                    __syncwarp();
                    tmem_ld32(tt + c * 32, z);
                    const int nv = p.Ncols - col0;
                    if (c == 0) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) insert((j < nv) ? z[j] : -INFINITY, col0 + j);
                    } else {
                        // only the values above the current eighth can enter: each lane walks
                        // its own mask in column order (most values of later chunks fail)
                        uint32_t above = 0;
#pragma unroll
                        for (int j = 0; j < 32; ++j) above |= (j < nv && z[j] > tv[kTopPerTile - 1]) ? (1u << j) : 0u;
                        while (above) {
                            const int j = __ffs(above) - 1;
                            above &= above - 1;
                            const float x = select32(z, j);
                            if (x > tv[kTopPerTile - 1]) insert(x, col0 + j);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
                if (row_ok) {
                    const size_t o = static_cast<size_t>(n) * p.part_stride + row;
                    p.part_m[o] = tv[0];
                    float4* vo = reinterpret_cast<float4*>(p.top_v) + o * (kTopPerTile / 4);
                    int4* io = reinterpret_cast<int4*>(p.top_i) + o * (kTopPerTile / 4);
#pragma unroll
                    for (int q4 = 0; q4 < kTopPerTile / 4; ++q4) {
                        vo[q4] = make_float4(tv[4 * q4], tv[4 * q4 + 1], tv[4 * q4 + 2], tv[4 * q4 + 3]);
                        io[q4] = make_int4(ti[4 * q4], ti[4 * q4 + 1], ti[4 * q4 + 2], ti[4 * q4 + 3]);
                    }
                }
            } else if constexpr (EPI == EPI_CAND) {
                const float th = (row_ok && p.row_flag[row]) ? p.theta[row] : INFINITY;
                if (!warp_wait(tfull0 + 8u * acc, aph, s_abort, p.status)) break;
                tc_fence_after();
                const int v0 = n * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int col0 = v0 + c * 32;
                    if (col0 >= p.Ncols) break;
                    float z[32];
                    __syncwarp();
                    tmem_ld32(tt + c * 32, z);
                    const int nv = p.Ncols - col0;
                    uint32_t hit = 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) hit |= (j < nv && z[j] >= th) ? (1u << j) : 0u;
                    while (hit) {  // rare: about K logits per row pass the threshold over the whole vocabulary
                        const int j = __ffs(hit) - 1;
                        hit &= hit - 1;
                        const float v = select32(z, j);
                        if (v > th) {
                            const int slot = atomicAdd(p.cnt_gt + row, 1);
                            if (slot < p.cand_cap) {
                                p.cand_v[static_cast<size_t>(row) * p.cand_cap + slot] = v;
                                p.cand_i[static_cast<size_t>(row) * p.cand_cap + slot] = col0 + j;
                            }
                        } else {
                            const int slot = atomicAdd(p.cnt_eq + row, 1);
                            if (slot < p.K) p.tie_i[static_cast<size_t>(row) * p.K + slot] = col0 + j;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
            } else if constexpr (EPI == EPI_DZ || EPI == EPI_DZ_MIX) {
                constexpr bool MIX = EPI == EPI_DZ_MIX;
                const int v0 = n * BN;
                TeacherCursor cur;
                cur.seek(p.sidx, p.sp, row, row_ok, p.K, v0);
                float lse2 = 0.f, coef = 0.f;
                float lse1_2 = 0.f, cT = 0.f, c1 = 0.f;  // MIX: dz = cT (q_T - s) + c1 (q_1 - onehot)
                int ylab = -1;
                if (row_ok) {
                    lse2 = p.lse[row] * 1.4426950408889634f;
                    const int nvalid = *p.n_valid;
                    if (p.valid[row] && nvalid > 0)
                        coef = p.T * (p.grad ? *p.grad : 1.f) / static_cast<float>(nvalid);
                    if constexpr (MIX) {
                        lse1_2 = p.lse1[row] * 1.4426950408889634f;
                        cT = coef * p.alpha;
                        c1 = coef * (1.f - p.alpha) / p.T;
                        ylab = __ldg(p.label + row);
                    }
                }
                // coef 2^(z scale2 - lse2) = sign(coef) 2^(z scale2 - lse2 + log2|coef|): one FMA
                // and one exponential per logit, the sign applied to the packed bf16 (coef = 0
                // gives 2^-inf = 0)
                const float bias = log2f(fabsf(coef)) - lse2, acoef = fabsf(coef);
                const uint32_t sgn = coef < 0.f ? 0x80008000u : 0u;
                if (!warp_wait(tfull0 + 8u * acc, aph, s_abort, p.status)) break;
                tc_fence_after();
#pragma unroll 1
                for (int c2 = 0; c2 < BN / 64; ++c2) {
                    const int col0 = v0 + c2 * 64;
                    if (col0 >= p.Ncols) break;
                    const uint32_t buf = staging0 + static_cast<uint32_t>(q * 2 + (box & 1)) * 4096u;
                    if (lane == 0) bulk_wait_read_le1();
                    __syncwarp();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int cc = col0 + hh * 32;
                        float z[32];
                        __syncwarp();
                        tmem_ld32(tt + c2 * 64 + hh * 32, z);
                        const int nv = p.Ncols - cc;
                        uint32_t w[16];
                        if constexpr (!MIX) {
                            if (nv >= 32) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) z[j] = ex2_approx(fmaf(z[j], p.scale2, bias));
                            } else {  // the last tile: columns beyond Ncols are 0
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    z[j] = (j < nv) ? ex2_approx(fmaf(z[j], p.scale2, bias)) : 0.f;
                            }
                            while (cur.next_id < cc + 32) {
                                const int off = cur.next_id - cc;
                                const float ps = acoef * cur.next_p;
#pragma unroll
                                for (int j = 0; j < 32; ++j) z[j] -= (j == off) ? ps : 0.f;
                                cur.advance();
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(z[2 * j], z[2 * j + 1]) ^ sgn;
                        } else {
                            constexpr float kL2e = 1.4426950408889634f;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                z[j] = (j < nv) ? cT * ex2_approx(z[j] * p.scale2 - lse2) +
                                                      c1 * ex2_approx(z[j] * kL2e - lse1_2)
                                                : 0.f;
                            while (cur.next_id < cc + 32) {
                                const int off = cur.next_id - cc;
#pragma unroll
                                for (int j = 0; j < 32; ++j) z[j] -= (j == off) ? cT * cur.next_p : 0.f;
                                cur.advance();
                            }
                            const int yoff = ylab - cc;
#pragma unroll
                            for (int j = 0; j < 32; ++j) z[j] -= (j == yoff) ? c1 : 0.f;
#pragma unroll
                            for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(z[2 * j], z[2 * j + 1]);
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            st_shared_v4(buf + lane * 128u + ((static_cast<uint32_t>(hh * 4 + k) ^ (lane & 7u)) << 4),
                                         w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0 && wrow < p.M) {
                        tma_store_3d(&tmOut, buf, 0, wrow, col0 >> 6);
                        bulk_commit();
                    }
                    ++box;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
            } else {
                if (!warp_wait(tfull0 + 8u * acc, aph, s_abort, p.status)) break;
                tc_fence_after();
                const int out_row = s * p.split_row_stride + wrow;
                const bool rows_ok = wrow < p.M;
#pragma unroll 1
                for (int c = 0; c < TW / 32; ++c) {
                    const int col0 = n * TW + c * 32;
                    if (col0 >= p.Ncols) break;
                    const uint32_t buf = staging0 + static_cast<uint32_t>(q * 2 + (box & 1)) * 4096u;
                    if (lane == 0) bulk_wait_read_le1();
                    __syncwarp();
                    float z[32];
                    tmem_ld32(tt + c * 32, z);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        st_shared_v4(buf + lane * 128u + ((static_cast<uint32_t>(k) ^ (lane & 7u)) << 4),
                                     __float_as_uint(z[4 * k]), __float_as_uint(z[4 * k + 1]),
                                     __float_as_uint(z[4 * k + 2]), __float_as_uint(z[4 * k + 3]));
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0 && rows_ok) {
                        if (p.reduce) tma_reduce_add_2d(&tmOut, buf, col0, out_row);
                        else tma_store_2d(&tmOut, buf, col0, out_row);
                        bulk_commit();
                    }
                    ++box;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
            }
        }
        if (epi_staged(EPI) && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // Neither CTA may leave while its peer can still touch its shared memory or TMEM.
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

// ---------------------------------------------------------------- bounded-wait self-test
// One thread waits on an mbarrier that nothing arrives on, with the pipeline's
// bounded wait and a short limit: the wait gives up, records FKL_ERR_TIMEOUT in
// the status word and the kernel returns (no copy or MMA is in flight).
__global__ void wait_timeout_kernel(int* status, uint64_t limit_ns) {
    __shared__ alignas(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    mbar_wait_for(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

cudaError_t launch_wait_timeout(int* status, uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- host dispatch
template <int BN, int NSUB, int A_MN, int B_MN, int EPI>
static cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmOut,
                              const GemmParams& p, int max_pairs, cudaStream_t stream) {
    constexpr size_t smem = PairCfg<BN, NSUB, B_MN, EPI>::SMEM;
    static_assert(smem <= 232448, "shared memory per CTA");
    // Per device: the shared-memory attribute is set and the resident pair count
    // queried on the first launch of this instantiation there.
    constexpr int kMaxDevices = 256;
    static std::mutex mu;
    static int pairs_resident[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int resident;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (pairs_resident[dev] == 0) {
            auto kern = gemm_kernel<BN, NSUB, A_MN, B_MN, EPI>;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * max_pairs);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (e != cudaSuccess || clusters <= 0) {
                cudaGetLastError();
                clusters = max_pairs;
            }
            pairs_resident[dev] = clusters < max_pairs ? clusters : max_pairs;
        }
        resident = pairs_resident[dev];
    }
    const long long units = static_cast<long long>(p.m_tiles) * p.n_tiles * p.splits;
    const int pairs = static_cast<int>(units < resident ? units : resident);
    gemm_kernel<BN, NSUB, A_MN, B_MN, EPI><<<2 * pairs, kThreads, smem, stream>>>(tmA, tmB, tmOut, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm(int bn, int a_mn, int b_mn, int epi, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const CUtensorMap& tmOut, const GemmParams& p,
                        int max_pairs, cudaStream_t stream) {
    if (epi == EPI_LSE) {
        if (bn == 256 && a_mn == 0 && b_mn == 0)
            return launch_one<256, 1, 0, 0, EPI_LSE>(tmA, tmB, tmOut, p, max_pairs, stream);
        return cudaErrorInvalidValue;
    }
    if (epi == EPI_DZ) {
        if (bn == 256 && a_mn == 0 && b_mn == 0)
            return launch_one<256, 1, 0, 0, EPI_DZ>(tmA, tmB, tmOut, p, max_pairs, stream);
        return cudaErrorInvalidValue;
    }
    if (epi == EPI_LSE_MIX) {
        if (bn == 256 && a_mn == 0 && b_mn == 0)
            return launch_one<256, 1, 0, 0, EPI_LSE_MIX>(tmA, tmB, tmOut, p, max_pairs, stream);
        return cudaErrorInvalidValue;
    }
    if (epi == EPI_DZ_MIX) {
        if (bn == 256 && a_mn == 0 && b_mn == 0)
            return launch_one<256, 1, 0, 0, EPI_DZ_MIX>(tmA, tmB, tmOut, p, max_pairs, stream);
        return cudaErrorInvalidValue;
    }
    if (epi == EPI_TMAX) {
        if (bn == 256 && a_mn == 0 && b_mn == 0)
            return launch_one<256, 1, 0, 0, EPI_TMAX>(tmA, tmB, tmOut, p, max_pairs, stream);
        return cudaErrorInvalidValue;
    }
    if (epi == EPI_CAND) {
        if (bn == 256 && a_mn == 0 && b_mn == 0)
            return launch_one<256, 1, 0, 0, EPI_CAND>(tmA, tmB, tmOut, p, max_pairs, stream);
        return cudaErrorInvalidValue;
    }
    if (epi == EPI_LSE_Y) {
        if (bn == 256 && a_mn == 0 && b_mn == 0)
            return launch_one<256, 1, 0, 0, EPI_LSE_Y>(tmA, tmB, tmOut, p, max_pairs, stream);
        return cudaErrorInvalidValue;
    }
#define FKL_F32_CASE(BN_, NS_, A_, B_)                                                      \
    if (bn == BN_ * NS_ && a_mn == A_ && b_mn == B_)                                        \
        return launch_one<BN_, NS_, A_, B_, EPI_F32>(tmA, tmB, tmOut, p, max_pairs, stream);
    FKL_F32_CASE(256, 2, 0, 0) FKL_F32_CASE(256, 2, 0, 1) FKL_F32_CASE(256, 2, 1, 0) FKL_F32_CASE(256, 2, 1, 1)
    FKL_F32_CASE(256, 1, 0, 0) FKL_F32_CASE(256, 1, 0, 1) FKL_F32_CASE(256, 1, 1, 0) FKL_F32_CASE(256, 1, 1, 1)
    FKL_F32_CASE(192, 1, 0, 0) FKL_F32_CASE(192, 1, 0, 1) FKL_F32_CASE(192, 1, 1, 0) FKL_F32_CASE(192, 1, 1, 1)
    FKL_F32_CASE(128, 1, 0, 0) FKL_F32_CASE(128, 1, 0, 1) FKL_F32_CASE(128, 1, 1, 0) FKL_F32_CASE(128, 1, 1, 1)
#undef FKL_F32_CASE
    return cudaErrorInvalidValue;
}

}  // namespace fkl
