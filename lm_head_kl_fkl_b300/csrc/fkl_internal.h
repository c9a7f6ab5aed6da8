// Internal declarations shared by the host scheduler and the kernels of libfkl.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fkl.h"

namespace fkl {

constexpr int kBM = 128;          // rows of a tile held by one CTA (its TMEM lanes)
constexpr int kPairRows = 256;    // rows of the tile a CTA pair computes
constexpr int kBK = 64;           // K elements per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kVocabTile = 256;   // vocabulary columns per tile in the logit GEMMs
constexpr int kThreads = 192;     // warp 0: TMA producer, warp 1: MMA issuer, warps 2-5: epilogue
constexpr int kPlanSMs = 148;     // SM count the workspace plan is sized for (B300)
constexpr int kMaxK = 256;        // teacher entries per token
constexpr int kTopPerTile = 8;    // teacher top-K: largest logits kept per row and vocabulary tile

// Kernel kinds, for the launch counter and the profiling hooks.
enum KernelKind {
    KK_COUNT_VALID = 0,
    KK_TEACHER_PREP,
    KK_FWD_LSE,      // tcgen05 GEMM z = h W^T + online logsumexp / teacher gather epilogue
    KK_FWD_FINALIZE,
    KK_LOSS_REDUCE,
    KK_BWD_DZ,       // tcgen05 GEMM recompute of z + dz epilogue (bf16, TMA store)
    KK_BWD_DH,       // tcgen05 GEMM dh partials = dz W (split over V)
    KK_DH_REDUCE,
    KK_BWD_DW,       // tcgen05 GEMM dW (+)= dz^T h (TMA store / reduce-add)
    KK_SELFTEST,
    KK_FB_GEMM_LSE_Y,  // tcgen05 GEMM z = h W^T, logsumexp / gather epilogue that also keeps the logits
    KK_FB_DZ,          // dz from the kept logits (elementwise)
    KK_TK_GEMM_TMAX,   // teacher top-K: tcgen05 GEMM, per row the eight largest logits of each vocabulary tile
    KK_TK_ROWS,        // teacher top-K: per-row threshold, candidates and selection (one warp per row)
    KK_TK_GEMM_CAND,   // teacher top-K: tcgen05 GEMM again for flagged rows (returns at once if none)
    KK_TK_SELECT,      // teacher top-K: selection for the rows the second tensor-core pass completed
    KK_SELFTEST_WAIT,  // bounded-wait self-test
    KK_SCALE_GRADS,    // dh, dW times an upstream gradient
    KK_TRANSPOSE_H,    // h of a chunk transposed: the dW GEMM's K-major operand
    KK_TK_FLAGS,       // teacher top-K: the call's second-pass flag from the sub-chunks' flags
    KK_NUM
};

enum Epilogue {
    EPI_LSE = 0, EPI_DZ = 1, EPI_F32 = 2, EPI_LSE_Y = 3, EPI_TMAX = 4, EPI_CAND = 5,
    EPI_LSE_MIX = 6,  // EPI_LSE plus the hard-label terms of the KL + cross-entropy mixture
    EPI_DZ_MIX = 7    // EPI_DZ of the mixture
};

// Epilogues that stage a tile in shared memory for a TMA store (the others write
// a few values per row with plain stores).
constexpr bool epi_staged(int epi) {
    return epi == EPI_DZ || epi == EPI_F32 || epi == EPI_LSE_Y || epi == EPI_DZ_MIX;
}

// Parameters of one persistent GEMM launch.  The unit space is
// m_tiles (of 256 rows) x n_tiles (of BN columns) x splits; unit u maps to (m, n, s) with s slowest and either
// m (m_fastest = 1) or n fastest; split s covers k-blocks
// [s * kb_total / splits, (s + 1) * kb_total / splits).
struct GemmParams {
    int m_tiles, n_tiles, splits, kb_total, m_fastest;
    int M;             // valid rows of the output (rows beyond are not written)
    int a_panel;       // 1: A is the dz panel buffer, a 3-D map {64 columns, rows, panel} (MN-major: boxes of 2 panels)
    int Ncols;         // valid columns (V for the logit GEMMs, d for dh / dW)
    int* status;       // device status word
    // EPI_LSE / EPI_DZ
    float scale2;      // log2(e) / T
    const int* sidx;   // [M][K] teacher ids sorted ascending (chunk-local rows)
    const float* sp;   // [M][K] teacher probabilities in the same order
    int K;
    float* part_m;     // EPI_LSE(_Y): [n_tiles][part_stride] running (EPI_LSE_Y: tile) max, base 2
    float* part_l;     //          [n_tiles][part_stride] sum of 2^(y - max)
    float* part_g;     //          [n_tiles][part_stride] sum_k p_k z_{idx_k}
    int part_stride;
    const float* lse;      // EPI_DZ: [M] natural-log lse of z/T
    const uint8_t* valid;  // EPI_DZ: [M]
    const int* n_valid;    // EPI_DZ: device scalar
    const float* grad;     // EPI_DZ: device scalar or nullptr (1.0)
    float T;
    // EPI_F32
    int split_row_stride;  // output row offset per split (dh partials), 0 otherwise
    int reduce;            // 1: TMA reduce-add into the output, 0: TMA store
    // EPI_TMAX writes part_m ([n_tiles][part_stride], tile max of the raw logits)
    // and the tile's four largest logits and ids:
    float* top_v;          // [n_tiles][part_stride][kTopPerTile]
    int* top_i;            // [n_tiles][part_stride][kTopPerTile]
    // EPI_CAND:
    const int* any_flag;   // device word: non-zero if some row is flagged
    const uint8_t* row_flag;  // [M] rows whose candidates the gather could not complete
    const float* theta;    // [M] per-row threshold
    int* cnt_gt;           // [M] logits > theta seen so far
    int* cnt_eq;           // [M] logits == theta seen so far
    float* cand_v;         // [M][cand_cap] values of the logits > theta
    int* cand_i;           // [M][cand_cap] their vocabulary ids
    int cand_cap;
    int* tie_i;            // [M][K] ids of the first K logits == theta
    // EPI_LSE_MIX / EPI_DZ_MIX (KL + cross-entropy mixture)
    const int* label;      // [M] hard label per row
    float alpha;           // weight of the KL term
    float* part_m1;        // EPI_LSE_MIX: [n_tiles][part_stride] running max of z log2e
    float* part_l1;        //              sum of 2^(z log2e - max)
    float* part_gy;        //              z at the label (0 in tiles without it)
    const float* lse1;     // EPI_DZ_MIX: [M] natural-log lse of z (temperature 1)
};

// Launch helpers implemented in gemm_tc.cu.  Return cudaSuccess or the launch error.
// Launches on at most `max_pairs` CTA pairs (clusters of 2), fewer if the unit
// space is smaller or fewer pairs can be resident.
cudaError_t launch_gemm(int bn, int a_mn, int b_mn, int epi, const CUtensorMap& tmA,
                        const CUtensorMap& tmB, const CUtensorMap& tmOut, const GemmParams& p,
                        int max_pairs, cudaStream_t stream);
cudaError_t launch_wait_timeout(int* status, uint64_t limit_ns, cudaStream_t stream);

// Small kernels implemented in aux_kernels.cu.
void launch_count_valid(const float* tlogit, const uint8_t* mask, int64_t N, int K, int* n_valid,
                        int grid, cudaStream_t s);
void launch_teacher_prep(const int32_t* idx, const float* tlogit, const uint8_t* mask, int64_t row0,
                         int rows, int K, int64_t V, float T, int* sidx, float* sp, float* H,
                         uint8_t* valid, int* status, cudaStream_t s);
void launch_fwd_finalize(const float* pm, const float* pl, const float* pg, int stride, int ntiles,
                         int rows, const float* H, const uint8_t* valid, float T, float* lse,
                         float* rowloss, cudaStream_t s);
void launch_fwd_finalize_mix(const float* pm, const float* pl, const float* pg, const float* pm1, const float* pl1,
                             const float* pgy, int stride, int ntiles, int rows, const float* H,
                             const uint8_t* valid, const int* label, int64_t V, float T, float alpha, float* lse,
                             float* lse1, float* rowloss, int* status, cudaStream_t s);
void launch_loss_reduce(const float* rowloss, int64_t N, const int* n_valid, float T, float* loss,
                        cudaStream_t s);
void launch_dh_reduce(const float* part, int splits, size_t split_elems, int rows, int d, void* dh,
                      cudaStream_t s);
void launch_topk_rows(const float* part_m, const float* top_v, const int* top_i, int part_stride, int ntiles,
                      int rows, int K, int sub_rows, float* theta, int* cnt_gt, int* cnt_eq, uint8_t* row_flag,
                      int* sub_flag, int32_t* idx_out, float* logit_out, cudaStream_t s);
void launch_topk_select(const float* cand_v, const int* cand_i, int cap, const int* cnt_gt, const int* cnt_eq,
                        const int* tie_i, const float* theta, const uint8_t* row_flag, int rows, int K,
                        int32_t* idx_out, float* logit_out, cudaStream_t s);
void launch_or_flags(const int* flags, int n, int* out, cudaStream_t s);
void launch_scale_grads(void* dh, size_t n_dh, float* dW, size_t n_dw, const float* g, int grid, cudaStream_t s);
void launch_dz_from_logits(void* yz, int64_t pstride, int64_t V, const float* part_m, int part_stride,
                           const float* lse, const uint8_t* valid, const int* n_valid, const float* grad,
                           float T, const int* sidx, const float* sp, int K, int rows, float* yk, cudaStream_t s);
void launch_transpose_h(const void* h, int rows, int d, void* hT, int64_t ld, cudaStream_t s);

}  // namespace fkl
