// CUDA-core kernels around the tensor-core GEMMs: teacher preparation, the
// per-row merge of the forward partials, the deterministic loss reduction, the
// split-K reduction of dh and the count of valid rows.
#include <climits>
#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fkl_internal.h"

namespace fkl {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// N_valid = #{i : mask_i != 0 and some teacher logit of row i is finite}.  One warp per row.
__global__ void count_valid_kernel(const float* __restrict__ t, const uint8_t* __restrict__ mask,
                                   int64_t N, int K, int* __restrict__ n_valid) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    int count = 0;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < N;
         r += warps) {
        if (mask && mask[r] == 0) continue;  // warp-uniform
        bool fin = false;
        for (int k = lane; k < K; k += 32) fin |= isfinite(t[r * K + k]);
        if (__any_sync(0xffffffffu, fin)) ++count;
    }
    __shared__ int s_cnt;
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    if (lane == 0 && count) atomicAdd(&s_cnt, count);
    __syncthreads();
    if (threadIdx.x == 0 && s_cnt) atomicAdd(n_valid, s_cnt);
}

// Ascending bitonic sort of 32 E keys held by one warp, key i = lane + 32 j in
// v[j] of lane `lane`: compare-exchanges at a distance below 32 go through warp
// shuffles, the others stay inside a lane's registers.
template <int E>
__device__ __forceinline__ void warp_bitonic_sort(unsigned long long (&v)[E], int lane) {
    constexpr int P = 32 * E;
#pragma unroll
    for (int size = 2; size <= P; size <<= 1) {
#pragma unroll
        for (int str = size >> 1; str > 0; str >>= 1) {
            if (str >= 32) {
                const int js = str >> 5;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    if (j & js) continue;
                    const bool asc = ((32 * j) & size) == 0;  // size >= 64: the lane does not matter
                    const unsigned long long a = v[j], b = v[j | js];
                    const bool sw = (a > b) == asc;
                    v[j] = sw ? b : a;
                    v[j | js] = sw ? a : b;
                }
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[j], str);
                    const bool asc = ((lane + 32 * j) & size) == 0;
                    const bool keep_min = ((lane & str) == 0) == asc;
                    v[j] = keep_min ? (o < v[j] ? o : v[j]) : (o > v[j] ? o : v[j]);
                }
            }
        }
    }
}

// Per row of a chunk (one warp per row): p = softmax(t/T) over the K cached
// entries, H = sum p log p, validity, and (id, p) sorted by id (equal ids by their
// position in the cache).  Ids outside [0, V) raise FKL_ERR_INDEX and are replaced by
// INT_MAX, which no tile reaches.  E = ceil(K / 32) rounded up to a power of two:
// each lane holds E entries, entry k = lane + 32 j in slot j.
template <int E>
__global__ void teacher_prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ t,
                                    const uint8_t* __restrict__ mask, int64_t row0, int rows, int K,
                                    int64_t V, float T, int* __restrict__ sidx, float* __restrict__ sp,
                                    float* __restrict__ H, uint8_t* __restrict__ valid,
                                    int* __restrict__ status) {
    __shared__ float s_e[4][32 * E];  // p by original position
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 4 + w;
    if (r >= rows) return;
    const int64_t gr = row0 + r;
    const int32_t* ir = idx + gr * K;
    const float* tr = t + gr * K;
    int ix[E];
    float u[E];
    float mx = -INFINITY;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int k = lane + 32 * j;
        ix[j] = INT_MAX;
        u[j] = -INFINITY;
        if (k < K) {
            int id = ir[k];
            if (id < 0 || static_cast<int64_t>(id) >= V) {
                bad = true;
                id = INT_MAX;
            }
            ix[j] = id;
            const float tv = tr[k];
            u[j] = isfinite(tv) ? tv / T : -INFINITY;  // non-finite logits carry no mass
            mx = fmaxf(mx, u[j]);
        }
    }
    if (bad) atomicCAS(status, 0, static_cast<int>(FKL_ERR_INDEX));
    mx = warp_max(mx);
    const bool has_mass = mx > -INFINITY;
    float e[E];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        e[j] = (has_mass && u[j] > -INFINITY) ? expf(u[j] - mx) : 0.f;
        s += e[j];
    }
    s = warp_sum(s);
    float hs = 0.f;
    unsigned long long key[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int k = lane + 32 * j;
        e[j] = has_mass ? e[j] / s : 0.f;
        if (e[j] > 0.f) hs += e[j] * logf(e[j]);
        s_e[w][k] = e[j];
        // ascending by id, equal ids by position; slots beyond K sort last
        key[j] = k < K ? (static_cast<unsigned long long>(static_cast<uint32_t>(ix[j])) << 32) | static_cast<uint32_t>(k)
                       : ~0ull;
    }
    hs = warp_sum(hs);
    warp_bitonic_sort<E>(key, lane);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int k = lane + 32 * j;
        if (k < K) {
            sidx[static_cast<size_t>(r) * K + k] = static_cast<int>(key[j] >> 32);
            sp[static_cast<size_t>(r) * K + k] = s_e[w][static_cast<uint32_t>(key[j])];
        }
    }
    if (lane == 0) {
        H[r] = hs;
        valid[r] = static_cast<uint8_t>((mask == nullptr || mask[gr] != 0) && has_mass);
    }
}

// lse_i and KL_i of one chunk from the per-tile partials.  A block takes 8 rows;
// 32 threads share a row, thread group g merging the tiles n = g + 32 t (for a fixed
// tile, the 8 rows are one 32-byte sector) into four independent running pairs by
// t mod 4 (so that four loads and merges are in flight), then the four in order,
// then the 32 groups pairwise in a fixed tree.  The order depends only on the tile
// index, so a row's lse is the same whatever chunk it is in.
constexpr int kFinRows = 8, kFinGroups = 32;

__device__ __forceinline__ void merge_ml(float& M, float& L, float m, float l) {
    if (l == 0.f) return;  // an empty part (no tile merged into it)
    if (m > M) {
        L = L * exp2f(M - m) + l;
        M = m;
    } else {
        L += l * exp2f(m - M);
    }
}

// A row's (max, sum, gather) over this thread's tiles n = grp + kFinGroups t, merged
// into four independent pairs by t mod 4 and then in that order (the row's 32 groups
// are merged afterwards by merge_groups).  The grouping depends only on n.
struct MLG {
    float M, L, G;
};
__device__ __forceinline__ MLG merge_tiles(const float* __restrict__ pm, const float* __restrict__ pl,
                                           const float* __restrict__ pg, int stride, int ntiles, int grp, int r) {
    float Ma[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY}, La[4] = {0.f, 0.f, 0.f, 0.f};
    float Ga[4] = {0.f, 0.f, 0.f, 0.f};
    int n = grp;
    for (; n + 3 * kFinGroups < ntiles; n += 4 * kFinGroups) {
        float m[4], l[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const size_t o = static_cast<size_t>(n + a * kFinGroups) * stride + r;
            m[a] = pm[o];
            l[a] = pl[o];
            Ga[a] += pg[o];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) merge_ml(Ma[a], La[a], m[a], l[a]);
    }
    for (int a = 0; n < ntiles; n += kFinGroups, ++a) {
        const size_t o = static_cast<size_t>(n) * stride + r;
        Ga[a] += pg[o];
        merge_ml(Ma[a], La[a], pm[o], pl[o]);
    }
    MLG v{-INFINITY, 0.f, 0.f};
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        v.G += Ga[a];
        merge_ml(v.M, v.L, Ma[a], La[a]);
    }
    return v;
}

// The row's 32 groups merged pairwise in a fixed tree through shared memory; every
// thread of the block calls it (it synchronises), group 0 ends with the row's total.
__device__ __forceinline__ void merge_groups(MLG& v, float (*sm)[kFinRows], float (*sl)[kFinRows],
                                             float (*sg)[kFinRows], int grp, int rl) {
    sm[grp][rl] = v.M;
    sl[grp][rl] = v.L;
    sg[grp][rl] = v.G;
#pragma unroll
    for (int half = kFinGroups / 2; half > 0; half >>= 1) {
        __syncthreads();
        if (grp < half) {
            v.G += sg[grp + half][rl];
            merge_ml(v.M, v.L, sm[grp + half][rl], sl[grp + half][rl]);
            sm[grp][rl] = v.M;
            sl[grp][rl] = v.L;
            sg[grp][rl] = v.G;
        }
    }
}

__global__ void fwd_finalize_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                                    const float* __restrict__ pg, int stride, int ntiles, int rows,
                                    const float* __restrict__ H, const uint8_t* __restrict__ valid,
                                    float T, float* __restrict__ lse, float* __restrict__ rowloss) {
    __shared__ float s_m[kFinGroups][kFinRows], s_l[kFinGroups][kFinRows], s_g[kFinGroups][kFinRows];
    const int rl = threadIdx.x % kFinRows, grp = threadIdx.x / kFinRows;
    const int r = blockIdx.x * kFinRows + rl;
    MLG v{-INFINITY, 0.f, 0.f};
    if (r < rows) v = merge_tiles(pm, pl, pg, stride, ntiles, grp, r);
    merge_groups(v, s_m, s_l, s_g, grp, rl);
    if (grp != 0 || r >= rows) return;
    const float lse_r = (v.M + log2f(v.L)) * 0.69314718055994531f;
    lse[r] = lse_r;
    rowloss[r] = valid[r] ? (H[r] - v.G / T + lse_r) : 0.f;
}

// The same for the KL + hard-label cross-entropy mixture: also lse1_i (temperature
// 1) and CE_i = lse1_i - z_{i,label_i}; rowloss_i = alpha KL_i + (1 - alpha) CE_i / T^2,
// so that loss_reduce's T^2 / N_valid gives alpha T^2 KL + (1 - alpha) CE averaged
// over the valid rows.  A valid row's label outside [0, V) records FKL_ERR_INDEX.
__global__ void fwd_finalize_mix_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                                        const float* __restrict__ pg, const float* __restrict__ pm1,
                                        const float* __restrict__ pl1, const float* __restrict__ pgy, int stride,
                                        int ntiles, int rows, const float* __restrict__ H,
                                        const uint8_t* __restrict__ valid, const int* __restrict__ label,
                                        int64_t V, float T, float alpha, float* __restrict__ lse,
                                        float* __restrict__ lse1, float* __restrict__ rowloss,
                                        int* __restrict__ status) {
    __shared__ float s_v[3][kFinGroups][kFinRows];
    const int rl = threadIdx.x % kFinRows, grp = threadIdx.x / kFinRows;
    const int r = blockIdx.x * kFinRows + rl;
    MLG v{-INFINITY, 0.f, 0.f}, v1{-INFINITY, 0.f, 0.f};  // temperature T with the teacher gather; 1 with the label
    if (r < rows) {
        v = merge_tiles(pm, pl, pg, stride, ntiles, grp, r);
        v1 = merge_tiles(pm1, pl1, pgy, stride, ntiles, grp, r);
    }
    merge_groups(v, s_v[0], s_v[1], s_v[2], grp, rl);
    __syncthreads();
    merge_groups(v1, s_v[0], s_v[1], s_v[2], grp, rl);
    if (grp != 0 || r >= rows) return;
    const float M = v.M, L = v.L, G = v.G, M1 = v1.M, L1 = v1.L, GY = v1.G;
    constexpr float kLn2 = 0.69314718055994531f;
    const float lse_r = (M + log2f(L)) * kLn2;
    const float lse1_r = (M1 + log2f(L1)) * kLn2;
    lse[r] = lse_r;
    lse1[r] = lse1_r;
    const int y = label[r];
    if (valid[r] && (y < 0 || static_cast<int64_t>(y) >= V)) atomicCAS(status, 0, static_cast<int>(FKL_ERR_INDEX));
    rowloss[r] = valid[r] ? alpha * (H[r] - G / T + lse_r) + (1.f - alpha) * (lse1_r - GY) / (T * T) : 0.f;
}

// loss = T^2 * sum_i rowloss_i / N_valid, summed in fp64 in a fixed order by one block.
__global__ void loss_reduce_kernel(const float* __restrict__ rowloss, int64_t N,
                                   const int* __restrict__ n_valid, float T, float* __restrict__ loss) {
    __shared__ double s_part[1024];
    double acc = 0.0;
    for (int64_t i = threadIdx.x; i < N; i += blockDim.x) acc += static_cast<double>(rowloss[i]);
    s_part[threadIdx.x] = acc;
    __syncthreads();
    for (int w = blockDim.x >> 1; w > 0; w >>= 1) {
        if (static_cast<int>(threadIdx.x) < w) s_part[threadIdx.x] += s_part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int nv = *n_valid;
        loss[0] = nv > 0 ? static_cast<float>(static_cast<double>(T) * T * s_part[0] / nv) : 0.f;
    }
}

// dh[r][j] = bf16(sum_s part[s][r][j]) for the rows of one chunk.
__global__ void dh_reduce_kernel(const float4* __restrict__ part, int splits, size_t split_elems4,
                                 size_t n4, uint2* __restrict__ dh) {
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float4 a = part[i];
        for (int s = 1; s < splits; ++s) {
            const float4 b = part[s * split_elems4 + i];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&lo);
        o.y = *reinterpret_cast<uint32_t*>(&hi);
        dh[i] = o;
    }
}

// dz of one chunk from the logits its forward kept: y = z log2e/T - m_tile (fp16,
// m_tile = part_m[tile][row], base 2), dz = coef (2^(y + m_tile - lse log2e) - s) in
// bf16, written over y in place, in three launches:
//  1. teacher_y_kernel (a warp per row): y + m_tile at the row's teacher ids, kept in
//     yk [rows][K] before they are overwritten;
//  2. dz_panels_kernel (a block per 64 rows x kDzPanels panels): coef 2^(y + m_tile -
//     lse log2e) over the panels, each a contiguous 64 x 128-byte run;
//  3. teacher_dz_kernel (a warp per row): the teacher entries (each run of equal ids
//     once, its p summed) rewritten with s subtracted, from yk.
// Element (r, v) of the panel layout is yz[(v / 64) pstride + 64 r + v % 64].
struct DzRow {
    float lse2, coef;
};
__device__ __forceinline__ DzRow dz_row(const float* lse, const uint8_t* valid, const int* n_valid,
                                        const float* grad, float T, int r) {
    constexpr float kLog2eF = 1.4426950408889634f;
    const int nv = *n_valid;
    DzRow d;
    d.lse2 = lse[r] * kLog2eF;
    d.coef = (valid[r] && nv > 0) ? T * (grad ? *grad : 1.f) / static_cast<float>(nv) : 0.f;
    return d;
}

__global__ void teacher_y_kernel(const uint16_t* __restrict__ yz, int64_t pstride, int64_t V,
                                 const float* __restrict__ part_m, int stride, const int* __restrict__ sidx, int K,
                                 int rows, float* __restrict__ yk) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= rows) return;
    for (int k = lane; k < K; k += 32) {
        const int v = sidx[static_cast<size_t>(r) * K + k];
        float y = 0.f;
        if (v < V)
            y = __half2float(__ushort_as_half(yz[(v >> 6) * pstride + static_cast<int64_t>(r) * 64 + (v & 63)])) +
                part_m[static_cast<size_t>(v >> 8) * stride + r];
        yk[static_cast<size_t>(r) * K + k] = y;
    }
}

constexpr int kDzRows = 64;    // rows per block of dz_panels_kernel
constexpr int kDzPanels = 16;  // panels per block

// 2^x with the special-function unit (relative error ~2^-22, results below 2^-126
// flushed to zero): ample for a bf16 result.
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Eight fp16 y of one row -> eight bf16 dz = sign * 2^(y + shift), shift = m_tile +
// log2|coef| - lse log2e (-inf for a row whose coef is 0); columns >= V (only in the
// last panel) get 0.
__device__ __forceinline__ uint4 dz_from_y8(uint4 in, float shift, uint32_t sgn, int64_t v, int64_t V) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        const __nv_bfloat162 ab = __floats2bfloat162_rn(ex2_fast(y.x + shift), ex2_fast(y.y + shift));
        o[j] = *reinterpret_cast<const uint32_t*>(&ab) ^ sgn;
    }
    if (v + 8 > V) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (v + 2 * j >= V) o[j] &= 0xffff0000u;
            if (v + 2 * j + 1 >= V) o[j] &= 0x0000ffffu;
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// A block covers 64 rows x kDzPanels panels; thread t owns columns (t % 8) * 8 .. + 7
// of rows t / 8 and t / 8 + 32 in every panel, so it keeps its two rows' constants in
// registers, and it loads the next panel's 16-byte pieces before converting the
// current ones.
__global__ void __launch_bounds__(256)
    dz_panels_kernel(uint16_t* __restrict__ yz, int64_t pstride, int64_t npan, int64_t V,
                     const float* __restrict__ part_m, int stride, const float* __restrict__ lse,
                     const uint8_t* __restrict__ valid, const int* __restrict__ n_valid, const float* __restrict__ grad,
                     float T, int rows) {
    const int t = threadIdx.x;
    const int r0 = blockIdx.x * kDzRows;
    const int64_t p0 = static_cast<int64_t>(blockIdx.y) * kDzPanels;
    const int64_t p1 = p0 + kDzPanels < npan ? p0 + kDzPanels : npan;
    const int col = (t & 7) * 8;
    int ra[2];
    bool ok[2];
    float bias[2], shift[2] = {0.f, 0.f};
    uint32_t sgn[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        ra[i] = (t >> 3) + 32 * i;
        ok[i] = r0 + ra[i] < rows;
        bias[i] = -INFINITY;
        sgn[i] = 0u;
        if (ok[i]) {
            const DzRow d = dz_row(lse, valid, n_valid, grad, T, r0 + ra[i]);
            bias[i] = log2f(fabsf(d.coef)) - d.lse2;  // -inf when coef is 0
            sgn[i] = d.coef < 0.f ? 0x80008000u : 0u;
        }
    }
    auto piece = [&](int64_t p, int i) {
        return reinterpret_cast<uint4*>(yz + p * pstride + static_cast<int64_t>(r0 + ra[i]) * 64 + col);
    };
    uint4 cur[2], nxt[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        cur[i] = nxt[i] = make_uint4(0u, 0u, 0u, 0u);
        if (ok[i]) cur[i] = *piece(p0, i);
    }
    for (int64_t p = p0; p < p1; ++p) {
        if (p + 1 < p1) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (ok[i]) nxt[i] = *piece(p + 1, i);
        }
        if (p == p0 || (p & 3) == 0) {  // a 256-column tile spans four panels
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (ok[i]) shift[i] = part_m[static_cast<size_t>(p >> 2) * stride + r0 + ra[i]] + bias[i];
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
            if (ok[i]) *piece(p, i) = dz_from_y8(cur[i], shift[i], sgn[i], p * 64 + col, V);
#pragma unroll
        for (int i = 0; i < 2; ++i) cur[i] = nxt[i];
    }
}

__global__ void teacher_dz_kernel(uint16_t* __restrict__ yz, int64_t pstride, int64_t V,
                                  const float* __restrict__ lse, const uint8_t* __restrict__ valid,
                                  const int* __restrict__ n_valid, const float* __restrict__ grad, float T,
                                  const int* __restrict__ sidx, const float* __restrict__ sp, int K, int rows,
                                  const float* __restrict__ yk) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= rows) return;
    const DzRow d = dz_row(lse, valid, n_valid, grad, T, r);
    const int* ids = sidx + static_cast<size_t>(r) * K;
    const float* ps = sp + static_cast<size_t>(r) * K;
    for (int k = lane; k < K; k += 32) {
        const int v = ids[k];
        if (v >= V || (k > 0 && ids[k - 1] == v)) continue;
        float s = ps[k];
        for (int j = k + 1; j < K && ids[j] == v; ++j) s += ps[j];
        const __nv_bfloat16 dz = __float2bfloat16_rn(d.coef * (exp2f(yk[static_cast<size_t>(r) * K + k] - d.lse2) - s));
        yz[(v >> 6) * pstride + static_cast<int64_t>(r) * 64 + (v & 63)] = __bfloat16_as_ushort(dz);
    }
}

void launch_dz_from_logits(void* yz, int64_t pstride, int64_t V, const float* part_m, int part_stride,
                           const float* lse, const uint8_t* valid, const int* n_valid, const float* grad,
                           float T, const int* sidx, const float* sp, int K, int rows, float* yk, cudaStream_t s) {
    uint16_t* y = static_cast<uint16_t*>(yz);
    const int64_t npan = (V + 63) / 64;
    teacher_y_kernel<<<(rows + 7) / 8, 256, 0, s>>>(y, pstride, V, part_m, part_stride, sidx, K, rows, yk);
    const dim3 grid(static_cast<unsigned>((rows + kDzRows - 1) / kDzRows),
                    static_cast<unsigned>((npan + kDzPanels - 1) / kDzPanels));
    dz_panels_kernel<<<grid, 256, 0, s>>>(y, pstride, npan, V, part_m, part_stride, lse, valid, n_valid, grad, T,
                                          rows);
    teacher_dz_kernel<<<(rows + 7) / 8, 256, 0, s>>>(y, pstride, V, lse, valid, n_valid, grad, T, sidx, sp, K, rows,
                                                     yk);
}

// ---------------------------------------------------------------- h transposed
// hT[c][r] = h[r][c] over one chunk's rows (row stride of hT: ld elements, a multiple
// of 8): the dW GEMM reads h as a K-major operand.  64 x 64 tiles through shared
// memory with 16-byte global loads and stores (d is a multiple of 8, so a load of
// eight columns is wholly inside or outside the row).  Rows beyond `rows` are
// written as zeros up to the next multiple of 8 (inside hT, past the GEMM's map).
// The tile's rows are 65 elements apart, so that the eight lanes reading one column
// at rows 8 apart hit eight different banks.
constexpr int kTrStride = 65;

__global__ void __launch_bounds__(256)
    transpose_h_kernel(const uint16_t* __restrict__ h, int rows, int d, uint16_t* __restrict__ hT, int64_t ld) {
    __shared__ uint16_t tile[64 * kTrStride];
    const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int q = t + 256 * i;
        const int row = q >> 3, cc = (q & 7) * 8;  // eight columns of one row
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + row < rows && c0 + cc < d)
            v = *reinterpret_cast<const uint4*>(h + static_cast<size_t>(r0 + row) * d + c0 + cc);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint16_t* dst = tile + row * kTrStride + cc;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            dst[2 * k] = static_cast<uint16_t>(w[k] & 0xffffu);
            dst[2 * k + 1] = static_cast<uint16_t>(w[k] >> 16);
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int q = t + 256 * i;
        const int col = q >> 3, rr = (q & 7) * 8;  // eight rows of one column
        if (c0 + col >= d || r0 + rr >= rows) continue;
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(tile[(rr + 2 * k) * kTrStride + col]) |
                   (static_cast<uint32_t>(tile[(rr + 2 * k + 1) * kTrStride + col]) << 16);
        *reinterpret_cast<uint4*>(hT + static_cast<size_t>(c0 + col) * ld + r0 + rr) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

void launch_transpose_h(const void* h, int rows, int d, void* hT, int64_t ld, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((d + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
    transpose_h_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(h), rows, d, static_cast<uint16_t*>(hT),
                                            ld);
}

// ---------------------------------------------------------------- teacher top-K
// Order-preserving map of a float onto uint32 (a < b  <=>  key(a) < key(b)).
__device__ __forceinline__ uint32_t fkey(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unkey(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Sum over the warp (every lane gets the total).
__device__ __forceinline__ int warp_sum(int c) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
}

// Candidates of one row, (key, id) pairs in shared memory, sorted by key
// descending and id ascending (one ascending sort of (~key, id) as a 64-bit value,
// in registers: E slots per lane, 32 E >= n); the first K are written out.
template <int E>
__device__ __forceinline__ void sort_and_write(const uint32_t* skey, const int* sid, int n, int K, int lane,
                                               int32_t* __restrict__ idx_row, float* __restrict__ logit_row) {
    unsigned long long c[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int i = lane + 32 * j;
        c[j] = i < n ? (static_cast<unsigned long long>(~skey[i]) << 32) | static_cast<uint32_t>(sid[i]) : ~0ull;
    }
    warp_bitonic_sort<E>(c, lane);
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int i = lane + 32 * j;
        if (i < K) {
            idx_row[i] = static_cast<int>(static_cast<uint32_t>(c[j]));
            logit_row[i] = unkey(~static_cast<uint32_t>(c[j] >> 32));
        }
    }
}

// The rare rows with more than 256 candidates: the same in a function of its own,
// so that its 16 slots per lane do not raise the register count of the common path.
__device__ __noinline__ void sort_and_write_16(const uint32_t* skey, const int* sid, int n, int K, int lane,
                                               int32_t* __restrict__ idx_row, float* __restrict__ logit_row) {
    sort_and_write<16>(skey, sid, n, K, lane, idx_row, logit_row);
}

// Teacher top-K of one row per warp, from the first tensor-core pass's per-tile
// top eight (tile maxima part_m [tile][row], kept logits and ids [tile][row][8]):
//  1. theta = the K-th largest of the row's tile maxima (-inf with fewer than K
//     tiles), by a bitwise search over order-preserving keys held in registers
//     (NK per lane), from the highest bit in which the keys differ.  At least K
//     logits of the row are >= theta (each of the K tiles contributes its max), and
//     every logit > theta lies in one of the < K tiles whose max exceeds theta.
//  2. The tiles whose max reaches theta, listed in shared memory from the same
//     registers; their kept logits are read 32 tiles at a time, and every kept
//     logit > theta and up to K logits == theta are compacted, in tile order,
//     into shared memory.
//  3. The candidates (those > theta; when fewer than K, with the first K - n_gt
//     logits == theta, i.e. the smallest ids, appended) sorted by value descending and
//     id ascending; the first K are the row's top K (ties by the smallest ids).
// A tile whose eighth kept logit is still >= theta may hold more candidates than
// were kept; such a row (or one with more than kTopCap candidates or kTopHits
// tiles) is flagged instead -- theta stored, its counters cleared, its sub-chunk's
// flag raised, nothing written -- for the second tensor-core pass and
// topk_select_kernel.
constexpr int kRowsPerBlock = 8;  // one warp per row
constexpr int kTopCap = 384;      // candidates > theta held in shared memory per row
constexpr int kTopHits = 2 * kMaxK;  // tiles reaching theta listed per row

template <int NK>  // tile maxima per lane kept in registers; tiles beyond 32 NK are re-read
__global__ void __launch_bounds__(32 * kRowsPerBlock, 4)
    topk_rows_kernel(const float* __restrict__ part_m, const float* __restrict__ top_v,
                     const int* __restrict__ top_i, int stride, int ntiles, int rows, int K, int sub_rows,
                     float* __restrict__ theta, int* __restrict__ cnt_gt, int* __restrict__ cnt_eq,
                     uint8_t* __restrict__ row_flag, int* __restrict__ sub_flag, int32_t* __restrict__ idx_out,
                     float* __restrict__ logit_out) {
    __shared__ uint32_t s_key[kRowsPerBlock][kTopCap];
    __shared__ int s_id[kRowsPerBlock][kTopCap];
    __shared__ int s_tie[kRowsPerBlock][kMaxK];
    __shared__ int s_hits[kRowsPerBlock][kTopHits];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int* const s_hit = s_hits[w];
    const int r = blockIdx.x * kRowsPerBlock + w;
    if (r >= rows) return;  // whole warps only; no block-wide barrier follows
    const unsigned lt = (1u << lane) - 1u;

    // 1. theta
    uint32_t key[NK];
    uint32_t k_and = ~0u, k_or = 0u;  // over the row's keys: their common leading bits
#pragma unroll
    for (int j = 0; j < NK; ++j) {
        const int n = lane + 32 * j;
        key[j] = 0u;
        if (n < ntiles) {
            key[j] = fkey(part_m[static_cast<size_t>(n) * stride + r]);
            k_and &= key[j];
            k_or |= key[j];
        }
    }
    for (int n = lane + 32 * NK; n < ntiles; n += 32) {
        const uint32_t kk = fkey(part_m[static_cast<size_t>(n) * stride + r]);
        k_and &= kk;
        k_or |= kk;
    }
    k_and = __reduce_and_sync(0xffffffffu, k_and);
    k_or = __reduce_or_sync(0xffffffffu, k_or);
    uint32_t t = 0;  // largest key with at least K tile maxima at or above it
    if (ntiles >= K) {
        // every key shares the bits above the highest one in which two keys differ,
        // and so does theta: the search starts below them
        const uint32_t diff = k_and ^ k_or;
        const int hb = diff ? 31 - __clz(diff) : -1;
        t = hb < 0 ? k_and : hb >= 31 ? 0u : (k_and & ~((2u << hb) - 1u));  // hb < 0: all keys are equal
        for (int b = hb; b >= 0; --b) {
            const uint32_t cand = t | (1u << b);
            int c = 0;
#pragma unroll
            for (int j = 0; j < NK; ++j) c += key[j] >= cand;
            for (int n = lane + 32 * NK; n < ntiles; n += 32)
                c += fkey(part_m[static_cast<size_t>(n) * stride + r]) >= cand;
            if (static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c))) >= K) t = cand;
        }
    }
    const float th = ntiles >= K ? unkey(t) : -INFINITY;
    const uint32_t tkey = fkey(th);

    // 2. the tiles reaching theta, then their kept logits
    int n_hit = 0;
#pragma unroll
    for (int j = 0; j < NK; ++j) {
        const int n = lane + 32 * j;
        const bool hit = n < ntiles && key[j] >= tkey;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit && n_hit + __popc(m & lt) < kTopHits) s_hit[n_hit + __popc(m & lt)] = n;
        n_hit += __popc(m);
    }
    for (int n0 = 32 * NK; n0 < ntiles; n0 += 32) {
        const int n = n0 + lane;
        const bool hit = n < ntiles && fkey(part_m[static_cast<size_t>(n) * stride + r]) >= tkey;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit && n_hit + __popc(m & lt) < kTopHits) s_hit[n_hit + __popc(m & lt)] = n;
        n_hit += __popc(m);
    }
    __syncwarp();
    bool flag = n_hit > kTopHits;
    int n_gt = 0, n_eq = 0;
    for (int i0 = 0; i0 < n_hit && !flag; i0 += 32) {
        const int i = i0 + lane;
        float v[kTopPerTile];
        int id[kTopPerTile];
#pragma unroll
        for (int e = 0; e < kTopPerTile; ++e) {
            v[e] = -INFINITY;
            id[e] = INT_MAX;
        }
        const bool have = i < n_hit;
        if (have) {
            const size_t o = static_cast<size_t>(s_hit[i]) * stride + r;
#pragma unroll
            for (int q4 = 0; q4 < kTopPerTile / 4; ++q4) {
                const float4 a = reinterpret_cast<const float4*>(top_v)[o * (kTopPerTile / 4) + q4];
                const int4 b = reinterpret_cast<const int4*>(top_i)[o * (kTopPerTile / 4) + q4];
                v[4 * q4] = a.x, v[4 * q4 + 1] = a.y, v[4 * q4 + 2] = a.z, v[4 * q4 + 3] = a.w;
                id[4 * q4] = b.x, id[4 * q4 + 1] = b.y, id[4 * q4 + 2] = b.z, id[4 * q4 + 3] = b.w;
            }
        }
        if (__any_sync(0xffffffffu, have && v[kTopPerTile - 1] >= th)) {
            flag = true;
            break;
        }
#pragma unroll
        for (int e = 0; e < kTopPerTile - 1; ++e) {
            const bool gt = have && v[e] > th, eq = have && v[e] == th;
            const unsigned mg = __ballot_sync(0xffffffffu, gt), me = __ballot_sync(0xffffffffu, eq);
            if (gt) {
                const int slot = n_gt + __popc(mg & lt);
                if (slot < kTopCap) {
                    s_key[w][slot] = fkey(v[e]);
                    s_id[w][slot] = id[e];
                }
            }
            if (eq) {
                const int slot = n_eq + __popc(me & lt);
                if (slot < K) s_tie[w][slot] = id[e];
            }
            n_gt += __popc(mg);
            n_eq += __popc(me);
        }
    }
    if (flag || n_gt > kTopCap) {
        if (lane == 0) {
            theta[r] = th;
            cnt_gt[r] = 0;
            cnt_eq[r] = 0;
            row_flag[r] = 1;
            atomicExch(sub_flag + r / sub_rows, 1);
        }
        return;
    }
    if (lane == 0) row_flag[r] = 0;

    // 3. the candidates, completed with ties at theta when fewer than K, sorted
    int n = n_gt;
    if (n_gt < K) {
        __syncwarp();
        for (int i = lane; i < K - n_gt; i += 32) {  // at least K - n_gt ties exist (K tiles reach theta)
            s_key[w][n_gt + i] = tkey;
            s_id[w][n_gt + i] = s_tie[w][i];
        }
        n = K;
    }
    __syncwarp();
    int32_t* const idx_row = idx_out + static_cast<size_t>(r) * K;
    float* const logit_row = logit_out + static_cast<size_t>(r) * K;
    if (n <= 32) sort_and_write<1>(s_key[w], s_id[w], n, K, lane, idx_row, logit_row);
    else if (n <= 64) sort_and_write<2>(s_key[w], s_id[w], n, K, lane, idx_row, logit_row);
    else if (n <= 128) sort_and_write<4>(s_key[w], s_id[w], n, K, lane, idx_row, logit_row);
    else if (n <= 256) sort_and_write<8>(s_key[w], s_id[w], n, K, lane, idx_row, logit_row);
    else sort_and_write_16(s_key[w], s_id[w], n, K, lane, idx_row, logit_row);
}

// Per row (one block of 256): the K largest logits among the candidates, sorted by
// value (descending), equal values by id (ascending).  If at least K candidates
// are above theta, the K-th largest value is found by a bitwise search over the
// order-preserving keys and the boundary ties are resolved by the smallest ids;
// otherwise all of them are taken and the rest is filled with logits equal to
// theta from the tie list.
__global__ void topk_select_kernel(const float* __restrict__ cand_v, const int* __restrict__ cand_i, int cap,
                                   const int* __restrict__ cnt_gt, const int* __restrict__ cnt_eq,
                                   const int* __restrict__ tie_i, const float* __restrict__ theta,
                                   const uint8_t* __restrict__ row_flag, int K, int32_t* __restrict__ idx_out,
                                   float* __restrict__ logit_out) {
    __shared__ uint32_t s_key[kMaxK];
    __shared__ int s_id[kMaxK];
    __shared__ int s_n;
    const int r = blockIdx.x;
    if (!row_flag[r]) return;  // completed by topk_rows_kernel (uniform over the block)
    const float* v = cand_v + static_cast<size_t>(r) * cap;
    const int* id = cand_i + static_cast<size_t>(r) * cap;
    const int n = min(cnt_gt[r], cap);
    for (int k = threadIdx.x; k < kMaxK; k += blockDim.x) {
        s_key[k] = 0u;  // below every real key: sorts last
        s_id[k] = INT_MAX;
    }
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    if (n >= K) {
        uint32_t t = 0;  // key of the K-th largest candidate
        for (int b = 31; b >= 0; --b) {
            const uint32_t cand = t | (1u << b);
            int c = 0;
            for (int i = threadIdx.x; i < n; i += blockDim.x) c += fkey(v[i]) >= cand;
            if (__syncthreads_count(c > 0) == 0) continue;  // cheap exit: nobody reaches cand
            __shared__ int s_cnt;
            if (threadIdx.x == 0) s_cnt = 0;
            __syncthreads();
            if (c) atomicAdd(&s_cnt, c);
            __syncthreads();
            if (s_cnt >= K) t = cand;
            __syncthreads();
        }
        int above = 0;  // candidates strictly above the K-th value
        for (int i = threadIdx.x; i < n; i += blockDim.x) above += fkey(v[i]) > t;
        __shared__ int s_above;
        if (threadIdx.x == 0) s_above = 0;
        __syncthreads();
        if (above) atomicAdd(&s_above, above);
        __syncthreads();
        const int need = K - s_above;  // ties at the K-th value to keep, smallest ids first
        uint32_t cut = 0;              // largest id bound with at most `need` ties below it ...
        for (int b = 30; b >= 0; --b) {
            const uint32_t c2 = cut | (1u << b);
            int c = 0;
            for (int i = threadIdx.x; i < n; i += blockDim.x) c += (fkey(v[i]) == t && static_cast<uint32_t>(id[i]) < c2);
            __shared__ int s_c2;
            if (threadIdx.x == 0) s_c2 = 0;
            __syncthreads();
            if (c) atomicAdd(&s_c2, c);
            __syncthreads();
            if (s_c2 < need) cut = c2;
            __syncthreads();
        }
        // ... so the ties with id <= cut are exactly `need` of them
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t kk = fkey(v[i]);
            if (kk > t || (kk == t && static_cast<uint32_t>(id[i]) <= cut)) {
                const int slot = atomicAdd(&s_n, 1);
                if (slot < kMaxK) {
                    s_key[slot] = kk;
                    s_id[slot] = id[i];
                }
            }
        }
    } else {
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            s_key[i] = fkey(v[i]);
            s_id[i] = id[i];
        }
        const int ne = min(cnt_eq[r], K - n);
        const uint32_t tk = fkey(theta[r]);
        for (int i = threadIdx.x; i < ne; i += blockDim.x) {
            s_key[n + i] = tk;
            s_id[n + i] = tie_i[static_cast<size_t>(r) * K + i];
        }
    }
    __syncthreads();
    // bitonic sort of the kMaxK slots: key descending, id ascending
    for (int size = 2; size <= kMaxK; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < kMaxK; i += blockDim.x) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const bool i_first = s_key[i] > s_key[j] || (s_key[i] == s_key[j] && s_id[i] < s_id[j]);
                    if (i_first != desc) {
                        const uint32_t tk = s_key[i];
                        s_key[i] = s_key[j];
                        s_key[j] = tk;
                        const int ti = s_id[i];
                        s_id[i] = s_id[j];
                        s_id[j] = ti;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        idx_out[static_cast<size_t>(r) * K + k] = s_id[k];
        logit_out[static_cast<size_t>(r) * K + k] = unkey(s_key[k]);
    }
}

void launch_topk_select(const float* cand_v, const int* cand_i, int cap, const int* cnt_gt, const int* cnt_eq,
                        const int* tie_i, const float* theta, const uint8_t* row_flag, int rows, int K,
                        int32_t* idx_out, float* logit_out, cudaStream_t s) {
    topk_select_kernel<<<rows, 256, 0, s>>>(cand_v, cand_i, cap, cnt_gt, cnt_eq, tie_i, theta, row_flag, K, idx_out,
                                            logit_out);
}

void launch_topk_rows(const float* part_m, const float* top_v, const int* top_i, int part_stride, int ntiles,
                      int rows, int K, int sub_rows, float* theta, int* cnt_gt, int* cnt_eq, uint8_t* row_flag,
                      int* sub_flag, int32_t* idx_out, float* logit_out, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
#define FKL_TOPK_ROWS(NK_)                                                                                     \
    topk_rows_kernel<NK_><<<grid, 32 * kRowsPerBlock, 0, s>>>(part_m, top_v, top_i, part_stride, ntiles, rows, K, \
                                                              sub_rows, theta, cnt_gt, cnt_eq, row_flag, sub_flag,  \
                                                              idx_out, logit_out)
    if (ntiles <= 32 * 4) FKL_TOPK_ROWS(4);
    else if (ntiles <= 32 * 8) FKL_TOPK_ROWS(8);
    else if (ntiles <= 32 * 16) FKL_TOPK_ROWS(16);
    else if (ntiles <= 32 * 25) FKL_TOPK_ROWS(25);  // up to V = 204800 (e.g. 201088)
    else FKL_TOPK_ROWS(32);
#undef FKL_TOPK_ROWS
}

// *out |= any of flags[0, n): the teacher top-K call's record that some row took
// the second tensor-core pass.
__global__ void or_flags_kernel(const int* __restrict__ flags, int n, int* __restrict__ out) {
    int f = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) f |= flags[i];
    if (__syncthreads_or(f) && threadIdx.x == 0) *out = 1;
}

void launch_or_flags(const int* flags, int n, int* out, cudaStream_t s) {
    or_flags_kernel<<<1, 256, 0, s>>>(flags, n, out);
}

// dh *= g (bf16, rounded once more to nearest even) and dW *= g (fp32), with the
// upstream gradient g read from the device: the chain rule of a loss whose
// gradients were formed during the forward.
__global__ void scale_grads_kernel(__nv_bfloat162* __restrict__ dh, size_t n_dh2, float4* __restrict__ dW,
                                   size_t n_dw4, const float* __restrict__ g) {
    const float s = *g;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_dw4; i += stride) {
        float4 v = dW[i];
        v.x *= s;
        v.y *= s;
        v.z *= s;
        v.w *= s;
        dW[i] = v;
    }
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_dh2; i += stride) {
        const float2 v = __bfloat1622float2(dh[i]);
        dh[i] = __floats2bfloat162_rn(v.x * s, v.y * s);
    }
}

void launch_scale_grads(void* dh, size_t n_dh, float* dW, size_t n_dw, const float* g, int grid, cudaStream_t s) {
    scale_grads_kernel<<<grid, 256, 0, s>>>(static_cast<__nv_bfloat162*>(dh), n_dh / 2,
                                            reinterpret_cast<float4*>(dW), n_dw / 4, g);
}

void launch_count_valid(const float* tlogit, const uint8_t* mask, int64_t N, int K, int* n_valid,
                        int grid, cudaStream_t s) {
    count_valid_kernel<<<grid, 256, 0, s>>>(tlogit, mask, N, K, n_valid);
}

void launch_teacher_prep(const int32_t* idx, const float* tlogit, const uint8_t* mask, int64_t row0,
                         int rows, int K, int64_t V, float T, int* sidx, float* sp, float* H,
                         uint8_t* valid, int* status, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>((rows + 3) / 4);
    if (K <= 32)
        teacher_prep_kernel<1><<<grid, 128, 0, s>>>(idx, tlogit, mask, row0, rows, K, V, T, sidx, sp, H, valid, status);
    else if (K <= 64)
        teacher_prep_kernel<2><<<grid, 128, 0, s>>>(idx, tlogit, mask, row0, rows, K, V, T, sidx, sp, H, valid, status);
    else if (K <= 128)
        teacher_prep_kernel<4><<<grid, 128, 0, s>>>(idx, tlogit, mask, row0, rows, K, V, T, sidx, sp, H, valid, status);
    else
        teacher_prep_kernel<8><<<grid, 128, 0, s>>>(idx, tlogit, mask, row0, rows, K, V, T, sidx, sp, H, valid, status);
}

void launch_fwd_finalize(const float* pm, const float* pl, const float* pg, int stride, int ntiles,
                         int rows, const float* H, const uint8_t* valid, float T, float* lse,
                         float* rowloss, cudaStream_t s) {
    const int blocks = (rows + kFinRows - 1) / kFinRows;
    fwd_finalize_kernel<<<blocks, kFinRows * kFinGroups, 0, s>>>(pm, pl, pg, stride, ntiles, rows, H, valid, T, lse,
                                                                 rowloss);
}

void launch_fwd_finalize_mix(const float* pm, const float* pl, const float* pg, const float* pm1, const float* pl1,
                             const float* pgy, int stride, int ntiles, int rows, const float* H,
                             const uint8_t* valid, const int* label, int64_t V, float T, float alpha, float* lse,
                             float* lse1, float* rowloss, int* status, cudaStream_t s) {
    const int blocks = (rows + kFinRows - 1) / kFinRows;
    fwd_finalize_mix_kernel<<<blocks, kFinRows * kFinGroups, 0, s>>>(pm, pl, pg, pm1, pl1, pgy, stride, ntiles, rows,
                                                                     H, valid, label, V, T, alpha, lse, lse1, rowloss,
                                                                     status);
}

void launch_loss_reduce(const float* rowloss, int64_t N, const int* n_valid, float T, float* loss,
                        cudaStream_t s) {
    loss_reduce_kernel<<<1, 1024, 0, s>>>(rowloss, N, n_valid, T, loss);
}

void launch_dh_reduce(const float* part, int splits, size_t split_elems, int rows, int d, void* dh,
                      cudaStream_t s) {
    const size_t n4 = static_cast<size_t>(rows) * d / 4;
    int grid = static_cast<int>((n4 + 255) / 256);
    if (grid > 148 * 8) grid = 148 * 8;
    if (grid < 1) grid = 1;
    dh_reduce_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(part), splits, split_elems / 4,
                                         n4, reinterpret_cast<uint2*>(dh));
}

}  // namespace fkl
