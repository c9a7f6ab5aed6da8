// Host side of libfkl.so: argument checks, the sequence-chunk plan, TMA
// descriptors and the launch sequence of the forward and backward passes.
//
// Forward, per chunk of C rows ("Multiverse Computing uzhala distillyatsiyu",
// iitak.ru, paragraph 3: a chunk's student probabilities are reduced into the
// running total and dropped):
//   teacher_prep -> fwd GEMM with the logsumexp / gather epilogue -> finalize
// then one deterministic loss reduction over all rows.
// Backward, per chunk (logits recomputed rather than stored, same paragraph and
// "Wissensdestillation mit deutlich weniger GPU-Speicher", dailytechsnack.ch,
// section "KL-Verlust wird in Bloecken berechnet"):
//   teacher_prep -> dz GEMM (recompute + dz in bf16) -> dh GEMM (split over V)
//   -> dh reduction -> dW GEMM (store for the first chunk, reduce-add after).
// All launches go to the caller's stream; nothing synchronises.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "fkl_internal.h"

namespace fkl {
namespace {

thread_local char g_err[512] = "";

fkl_status fail(fkl_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
fkl_status fail(fkl_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

std::atomic<int64_t> g_launches{0};

// NVTX range for profilers (a no-op unless a tool is attached): one per entry
// point call and one per chunk.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    NvtxRange(const char* what, long long chunk) {
        char buf[64];
        snprintf(buf, sizeof(buf), "%s chunk %lld", what, chunk);
        nvtxRangePushA(buf);
    }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---------------------------------------------------------------- profiling hooks
struct ProfRec {
    int kind;
    double flop;
    cudaEvent_t a, b;
};
// Records and spare events are shared by every calling thread: g_prof_mu guards both.
std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pool_event() {  // caller holds g_prof_mu
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

struct LaunchScope {
    ProfRec rec{};
    cudaStream_t s;
    LaunchScope(int kind, double flop, cudaStream_t st) : s(st) {
        rec.kind = kind;
        rec.flop = flop;
        if (g_prof_on.load()) {
            {
                std::lock_guard<std::mutex> lock(g_prof_mu);
                rec.a = pool_event();
                rec.b = pool_event();
                if (!rec.a || !rec.b) {  // event creation failed: this launch goes untimed
                    if (rec.a) g_event_pool.push_back(rec.a);
                    if (rec.b) g_event_pool.push_back(rec.b);
                    rec.a = rec.b = nullptr;
                }
            }
            if (rec.a && rec.b) cudaEventRecord(rec.a, s);
        }
    }
    ~LaunchScope() {
        ++g_launches;
        if (rec.a && rec.b) {  // profiled at the start of this launch
            cudaEventRecord(rec.b, s);
            std::lock_guard<std::mutex> lock(g_prof_mu);
            g_prof.push_back(rec);
        }
    }
};

const char* const kKindNames[KK_NUM] = {
    "count_valid", "teacher_prep", "fwd_gemm_lse", "fwd_finalize", "loss_reduce",
    "bwd_gemm_dz", "bwd_gemm_dh", "dh_reduce", "bwd_gemm_dw", "selftest_gemm",
    "fb_gemm_lse_keep", "fb_dz_from_logits",
    "tk_gemm_tile_top8", "tk_rows", "tk_gemm_candidates", "tk_select_flagged", "selftest_wait", "scale_grads",
    "transpose_h", "tk_flags",
};

// ---------------------------------------------------------------- device facts
struct DeviceInfo {
    bool ok = false;
    int sms = 0;
    char why[160] = "";
};

DeviceInfo query_device() {
    DeviceInfo di;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        snprintf(di.why, sizeof(di.why), "no CUDA device");
        cudaGetLastError();
        return di;
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) {
        snprintf(di.why, sizeof(di.why), "device %d is sm_%d%d; libfkl is built for sm_103a only", dev,
                 major, minor);
        return di;
    }
    di.ok = true;
    return di;
}

// Facts of the current device, queried once per device ordinal.
const DeviceInfo& device_info() {
    constexpr int kMaxDevices = 256;
    static std::mutex mu;
    static DeviceInfo infos[kMaxDevices];
    static bool have[kMaxDevices] = {};
    static DeviceInfo none;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        std::lock_guard<std::mutex> lock(mu);
        none = DeviceInfo{};
        snprintf(none.why, sizeof(none.why), "no usable CUDA device");
        return none;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        infos[dev] = query_device();
        have[dev] = true;
    }
    return infos[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D tiled tensor map with 128-byte swizzle: dim0 is contiguous.
bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
               uint64_t stride1_bytes, uint32_t box0, uint32_t box1) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {dim0, dim1};
    cuuint64_t strides[1] = {stride1_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D tiled tensor map of the dz panel buffer: {64 columns, rows, panel}, the
// panels `panel_bytes` apart, each a [rows][64] bf16 (or fp16) array; 128-byte
// swizzle.  Every box {64, box_rows, 1} is one contiguous run of box_rows x 128 bytes.
bool make_panel_tmap(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t rows, uint64_t panels,
                     uint64_t panel_bytes, uint32_t box_rows, uint32_t box_panels = 1) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, panels};
    cuuint64_t strides[2] = {128, panel_bytes};
    cuuint32_t box[3] = {64, box_rows, box_panels};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- the plan
constexpr int kDefaultChunk = 4096;
constexpr int kMaxChunk = 1 << 20;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Plan {
    int64_t N, V, npan, n_chunks;  // npan: 64-column panels of the dz buffer
    int d, K, Cc, nt_v, bn_dh, nt_dh, bn_dw, nt_dw, splits;
    size_t o_sidx, o_sp, o_H, o_valid, o_rowloss, o_yk, o_big, o_part_dh, o_hT, total;
    size_t fwd_total;  // bytes the forward alone touches (a prefix of the workspace)
};

// Column tile of the dh and dW GEMMs (their N is d): the double-buffered width
// that wastes the fewest padded columns.
int pick_bn(int d) {
    const int cands[3] = {256, 192, 128};
    int best = 256;
    int64_t best_waste = INT64_MAX;
    for (int c : cands) {
        const int64_t waste = cdiv(d, c) * c - d;
        if (waste < best_waste) {
            best_waste = waste;
            best = c;
        }
    }
    return best;
}

// From d = 384 on the operand traffic decides instead.  dh (k-loop over a V
// split, tens of thousands deep) takes wide 512-column tiles, which move the
// least operand data per FLOP.  dW (k-loop over one chunk's rows, a few thousand
// deep, then a 256 x BN fp32 reduce-add) keeps 256-column double-buffered
// tiles, so that its epilogue overlaps the next tile's MMAs.
int pick_bn_dh(int d) { return d >= 384 ? 512 : pick_bn(d); }
int pick_bn_dw(int d) { return d >= 384 ? 256 : pick_bn(d); }

int bn_override(const char* name, int fallback) {
    if (const char* e = getenv(name)) {  // tile-width override for tuning sweeps
        const int v = atoi(e);
        if (v == 512 || v == 256 || v == 192 || v == 128) return v;
    }
    return fallback;
}

// Split count of the dh GEMM over V: the smallest S whose units (pair tiles x S)
// fill the CTA pairs' waves best (each extra split costs C * d * 4 bytes).
int pick_splits(int m_tiles, int n_tiles, int64_t kb_total) {
    const int pairs = kPlanSMs / 2;
    auto eff = [&](int s) {
        const int64_t units = int64_t(m_tiles) * n_tiles * s;
        const int64_t waves = cdiv(units, pairs);
        return double(units) / double(waves * pairs);
    };
    int best = 1;
    for (int s = 2; s <= 8; ++s) {
        if (s > kb_total / 2) break;
        if (eff(s) > eff(best) + 0.02) best = s;
    }
    return best;
}

const char* check_sizes(int64_t N, int d, int64_t V, int K, int chunk) {
    if (N < 1) return "N must be >= 1";
    if (d < 8 || d % 8 != 0) return "d must be a positive multiple of 8";
    if (d > 65536) return "d above 65536 is not supported";
    if (V < 1 || V > (int64_t(1) << 30)) return "V must be in [1, 2^30]";
    if (K < 1 || K > kMaxK) return "K must be in [1, 256]";
    if (K > V) return "K must not exceed V";
    if (chunk < 0 || chunk % kBM != 0 || chunk > kMaxChunk)
        return "chunk must be 0 (default) or a positive multiple of 128 up to 2^20";
    if (N > (int64_t(1) << 40)) return "N too large";
    return nullptr;
}

bool make_plan(int64_t N, int d, int64_t V, int K, int chunk, Plan& P) {
    if (check_sizes(N, d, V, K, chunk)) return false;
    P.N = N;
    P.d = d;
    P.V = V;
    P.K = K;
    const int64_t want = chunk > 0 ? chunk : kDefaultChunk;
    P.Cc = static_cast<int>(std::min<int64_t>(want, cdiv(N, kBM) * kBM));
    P.n_chunks = cdiv(N, P.Cc);
    P.nt_v = static_cast<int>(cdiv(V, kVocabTile));
    P.bn_dh = bn_override("FKL_BN_DH", pick_bn_dh(d));
    P.bn_dw = bn_override("FKL_BN_DW", pick_bn_dw(d));
    P.nt_dh = static_cast<int>(cdiv(d, P.bn_dh));
    P.nt_dw = static_cast<int>(cdiv(d, P.bn_dw));
    P.splits = pick_splits(static_cast<int>(cdiv(P.Cc, kPairRows)), P.nt_dh, cdiv(V, kBK));
    P.npan = cdiv(V, 64);
    size_t off = 256;  // header: status word, N_valid
    P.o_sidx = off;
    off += align256(size_t(P.Cc) * K * 4);
    P.o_sp = off;
    off += align256(size_t(P.Cc) * K * 4);
    P.o_H = off;
    off += align256(size_t(P.Cc) * 4);
    P.o_valid = off;
    off += align256(size_t(P.Cc));
    P.o_rowloss = off;
    off += align256(size_t(N) * 4);
    P.o_big = off;
    const size_t part_fwd = 3 * align256(size_t(P.nt_v) * P.Cc * 4);
    const size_t dz = align256(size_t(P.Cc) * P.npan * 64 * 2);
    const size_t part_dh = align256(size_t(P.splits) * P.Cc * d * 4);
    P.o_part_dh = P.o_big + dz;
    // fkl_forward keeps its partials at o_big; fkl_backward puts dz there and
    // the dh partials after it; fkl_forward_backward needs dz and the forward
    // partials at once, so its partials share the dh partials' place.  The
    // chunk's h transposed (for the dW GEMM) comes last.
    P.o_hT = P.o_big + dz + std::max(part_fwd, part_dh);
    P.o_yk = P.o_hT + align256(size_t(P.Cc) * d * 2);  // the one-call path: kept logits at the teacher ids
    P.total = P.o_yk + align256(size_t(P.Cc) * K * 4);
    P.fwd_total = P.o_big + part_fwd;
    // the KL + cross-entropy mixture's forward keeps six partial arrays, not three
    P.total = std::max(P.total, P.o_big + 2 * part_fwd);
    return true;
}

// ---------------------------------------------------------------- teacher top-K plan
// Rows per chunk of the first tensor-core pass and the per-row selection (enough
// warps for the selection to hide its memory latency), and per sub-chunk of the
// second pass, whose candidate lists are sized for the worst case of every row.
constexpr int kDefaultTopkChunk = 4096;
constexpr int kTopkSubChunk = 1024;

struct TopkPlan {
    int64_t N, V, n_chunks;
    int d, K, Cc, Cs, n_sub, nt_v, cap;
    size_t o_part, o_topv, o_topi, o_theta, o_gt, o_eq, o_flag, o_sflag, o_cv, o_ci, o_tie, total;
};

bool make_topk_plan(int64_t N, int d, int64_t V, int K, int chunk, TopkPlan& P) {
    if (check_sizes(N, d, V, K, chunk)) return false;
    P.N = N;
    P.d = d;
    P.V = V;
    P.K = K;
    const int64_t want = chunk > 0 ? chunk : kDefaultTopkChunk;
    P.Cc = static_cast<int>(std::min<int64_t>(want, cdiv(N, kBM) * kBM));
    P.n_chunks = cdiv(N, P.Cc);
    P.Cs = std::min(P.Cc, kTopkSubChunk);
    P.n_sub = static_cast<int>(cdiv(P.Cc, P.Cs));
    P.nt_v = static_cast<int>(cdiv(V, kVocabTile));
    // logits above the threshold lie in fewer than K vocabulary tiles (or the
    // threshold is -inf and there are fewer than K tiles in all)
    P.cap = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(V, int64_t(std::max(K - 1, 1)) * kVocabTile)));
    size_t off = 256;
    P.o_part = off;
    off += align256(size_t(P.nt_v) * P.Cc * 4);
    P.o_topv = off;
    off += align256(size_t(P.nt_v) * P.Cc * kTopPerTile * 4);
    P.o_topi = off;
    off += align256(size_t(P.nt_v) * P.Cc * kTopPerTile * 4);
    P.o_flag = off;
    off += align256(size_t(P.Cc));
    P.o_theta = off;
    off += align256(size_t(P.Cc) * 4);
    P.o_gt = off;
    off += align256(size_t(P.Cc) * 4);
    P.o_eq = off;
    off += align256(size_t(P.Cc) * 4);
    P.o_sflag = off;  // one word per sub-chunk: some row of it needs the second pass
    off += align256(size_t(P.n_sub) * 4);
    P.o_cv = off;  // candidate and tie lists: one sub-chunk's rows
    off += align256(size_t(P.Cs) * P.cap * 4);
    P.o_ci = off;
    off += align256(size_t(P.Cs) * P.cap * 4);
    P.o_tie = off;
    off += align256(size_t(P.Cs) * K * 4);
    P.total = off;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

const char* check_common(const void* h, const void* W, const int32_t* idx, const float* tlogit, int64_t N,
                         int d, int64_t V, int K, float T, int chunk, const void* ws) {
    if (!h || !W || !idx || !tlogit || !ws) return "null input or workspace pointer";
    if (const char* e = check_sizes(N, d, V, K, chunk)) return e;
    if (!(T > 0.f) || !std::isfinite(T)) return "T must be positive and finite";
    if (!aligned16(h) || !aligned16(W) || !aligned16(ws)) return "h, W and ws must be 16-byte aligned";
    return nullptr;
}

#define FKL_CUDA_TRY(expr)                                                                        \
    do {                                                                                          \
        cudaError_t e_ = (expr);                                                                  \
        if (e_ != cudaSuccess) return fail(FKL_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
    } while (0)

fkl_status device_ready() {
    const DeviceInfo& di = device_info();
    if (!di.ok) return fail(FKL_ERR_UNSUPPORTED, "%s", di.why);
    if (!encode_fn()) return fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    return FKL_OK;
}

fkl_status run_gemm(int kind, int bn, int a_mn, int b_mn, int epi, const CUtensorMap& a, const CUtensorMap& b,
                    const CUtensorMap& o, const GemmParams& p, double flop, cudaStream_t s) {
    cudaError_t e;
    {
        LaunchScope ls(kind, flop, s);
        e = launch_gemm(bn, a_mn, b_mn, epi, a, b, o, p, device_info().sms / 2, s);
    }
    if (e != cudaSuccess) return fail(FKL_ERR_CUDA, "%s launch: %s", kKindNames[kind], cudaGetErrorString(e));
    return FKL_OK;
}

#define FKL_TMAP(m, ...)                                                          \
    do {                                                                          \
        if (!make_tmap(&(m), __VA_ARGS__))                                        \
            return fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed for " #m);   \
    } while (0)

// Panel map of the chunk's dz (or kept-logit) buffer with boxes of box_rows rows.
#define FKL_PANEL_TMAP(m, dt, base, box_rows, ...)                                                  \
    do {                                                                                            \
        if (!make_panel_tmap(&(m), dt, base, uint64_t(rows), uint64_t(P.npan), uint64_t(P.Cc) * 128, \
                             box_rows, ##__VA_ARGS__))                                              \
            return fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed for " #m);                     \
    } while (0)

#define FKL_SMALL(kind, call)                                                                     \
    do {                                                                                          \
        {                                                                                         \
            LaunchScope ls_((kind), 0.0, s);                                                      \
            call;                                                                                 \
        }                                                                                         \
        cudaError_t e_ = cudaGetLastError();                                                      \
        if (e_ != cudaSuccess)                                                                    \
            return fail(FKL_ERR_CUDA, "%s launch: %s", kKindNames[kind], cudaGetErrorString(e_)); \
    } while (0)

constexpr float kLog2e = 1.4426950408889634f;
constexpr auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
constexpr auto F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
constexpr auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

// dh and dW of chunk c from its dz (bf16 in the workspace, 64-column panels of
// [rows][64]) and its h transposed (hT, [d][Cc] bf16):
//   dh partials [split][rows][d] = dz[:, split's V range] W[split's V range, :],
//   their fixed-order sum in bf16 into dh_chunk, and
//   dW (+)= dz^T h_chunk (TMA store for chunk 0, reduce-add after; one owner per
//   output tile, chunks in stream order).
fkl_status grads_from_dz(const Plan& P, int64_t c, int rows, const CUtensorMap& tmDz_k, const CUtensorMap& tmDz_mn,
                         const CUtensorMap& tmHT_k, const CUtensorMap& tmW_mn,
                         const CUtensorMap& tmPart, const CUtensorMap& tmDW, float* part, void* dh_chunk, int* status,
                         cudaStream_t s) {
    const int d = P.d;
    const double flop = 2.0 * rows * double(d) * double(P.V);
    GemmParams q{};
    q.m_tiles = static_cast<int>(cdiv(rows, kPairRows));
    q.n_tiles = P.nt_dh;
    q.splits = P.splits;
    q.kb_total = static_cast<int>(cdiv(P.V, kBK));
    q.m_fastest = 0;  // pairs in flight cover every d tile of a few row tiles: dz is read once
    q.M = rows;
    q.a_panel = 1;
    q.Ncols = d;
    q.status = status;
    q.split_row_stride = P.Cc;
    q.reduce = 0;
    if (fkl_status st = run_gemm(KK_BWD_DH, P.bn_dh, 0, 1, EPI_F32, tmDz_k, tmW_mn, tmPart, q, flop, s)) return st;
    FKL_SMALL(KK_DH_REDUCE, launch_dh_reduce(part, P.splits, size_t(P.Cc) * d, rows, d, dh_chunk, s));

    GemmParams r{};
    r.m_tiles = static_cast<int>(cdiv(P.V, kPairRows));
    r.n_tiles = P.nt_dw;
    r.splits = 1;
    r.kb_total = static_cast<int>(cdiv(rows, kBK));
    r.m_fastest = 0;
    r.M = static_cast<int>(P.V);
    r.a_panel = 1;
    r.Ncols = d;
    r.status = status;
    r.reduce = c > 0 ? 1 : 0;
    return run_gemm(KK_BWD_DW, P.bn_dw, 1, 0, EPI_F32, tmDz_mn, tmHT_k, tmDW, r, flop, s);
}

// The forward's launch sequence on a workspace of at least P.fwd_total bytes
// (sizes and pointers already checked).  Only the 256-byte header needs to start
// at zero; it is cleared here.  Every other region is written before it is read.
// Extra inputs / outputs of the KL + hard-label cross-entropy mixture (null: plain KL).
struct Mix {
    const int32_t* label;  // [N] hard labels
    float alpha;           // weight of the KL term
    float* lse1;           // forward: [N] output, lse of z at temperature 1
    const float* lse1_in;  // backward: the forward's lse1
};

fkl_status forward_enqueue(const Plan& P, const void* h, const void* W, const int32_t* idx,
                           const float* tlogit, const uint8_t* mask, float T, float* loss, float* lse,
                           void* ws, cudaStream_t s, const Mix* mix = nullptr) {
    const int64_t N = P.N, V = P.V;
    const int d = P.d, K = P.K;
    char* w = static_cast<char*>(ws);
    int* status = reinterpret_cast<int*>(w);
    int* n_valid = status + 1;
    int* sidx = reinterpret_cast<int*>(w + P.o_sidx);
    float* sp = reinterpret_cast<float*>(w + P.o_sp);
    float* H = reinterpret_cast<float*>(w + P.o_H);
    uint8_t* valid = reinterpret_cast<uint8_t*>(w + P.o_valid);
    float* rowloss = reinterpret_cast<float*>(w + P.o_rowloss);
    const size_t pstride = align256(size_t(P.nt_v) * P.Cc * 4);
    float* pm = reinterpret_cast<float*>(w + P.o_big);
    float* pl = reinterpret_cast<float*>(w + P.o_big + pstride);
    float* pg = reinterpret_cast<float*>(w + P.o_big + 2 * pstride);
    float* pm1 = reinterpret_cast<float*>(w + P.o_big + 3 * pstride);  // mixture only
    float* pl1 = reinterpret_cast<float*>(w + P.o_big + 4 * pstride);
    float* pgy = reinterpret_cast<float*>(w + P.o_big + 5 * pstride);

    FKL_CUDA_TRY(cudaMemsetAsync(w, 0, 256, s));
    const int sms = device_info().sms;
    FKL_SMALL(KK_COUNT_VALID, launch_count_valid(tlogit, mask, N, K, n_valid, sms * 4, s));

    CUtensorMap tmW;  // B of the logit GEMM: each CTA of a pair loads 128 of the tile's 256 vocab rows
    FKL_TMAP(tmW, BF16, W, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, kVocabTile / 2);
    for (int64_t c = 0; c < P.n_chunks; ++c) {
        NvtxRange nvtx_chunk("forward", static_cast<long long>(c));
        const int64_t row0 = c * P.Cc;
        const int rows = static_cast<int>(std::min<int64_t>(P.Cc, N - row0));
        FKL_SMALL(KK_TEACHER_PREP,
                  launch_teacher_prep(idx, tlogit, mask, row0, rows, K, V, T, sidx, sp, H, valid, status, s));
        CUtensorMap tmH;
        FKL_TMAP(tmH, BF16, static_cast<const char*>(h) + size_t(row0) * d * 2, uint64_t(d), uint64_t(rows),
                 uint64_t(d) * 2, 64, 128);
        GemmParams p{};
        p.m_tiles = static_cast<int>(cdiv(rows, kPairRows));
        p.n_tiles = P.nt_v;
        p.splits = 1;
        p.kb_total = static_cast<int>(cdiv(d, kBK));
        p.m_fastest = 1;
        p.M = rows;
        p.Ncols = static_cast<int>(V);
        p.status = status;
        p.scale2 = kLog2e / T;
        p.sidx = sidx;
        p.sp = sp;
        p.K = K;
        p.part_m = pm;
        p.part_l = pl;
        p.part_g = pg;
        p.part_stride = P.Cc;
        if (mix) {
            p.T = T;  // the temperature-1 sum rescales z log2e / T by T
            p.label = mix->label + row0;
            p.part_m1 = pm1;
            p.part_l1 = pl1;
            p.part_gy = pgy;
        }
        if (fkl_status st = run_gemm(KK_FWD_LSE, 256, 0, 0, mix ? EPI_LSE_MIX : EPI_LSE, tmH, tmW, tmW, p,
                                     2.0 * rows * double(d) * double(V), s))
            return st;
        if (mix)
            FKL_SMALL(KK_FWD_FINALIZE,
                      launch_fwd_finalize_mix(pm, pl, pg, pm1, pl1, pgy, P.Cc, P.nt_v, rows, H, valid,
                                              mix->label + row0, V, T, mix->alpha, lse + row0, mix->lse1 + row0,
                                              rowloss + row0, status, s));
        else
            FKL_SMALL(KK_FWD_FINALIZE, launch_fwd_finalize(pm, pl, pg, P.Cc, P.nt_v, rows, H, valid, T, lse + row0,
                                                           rowloss + row0, s));
    }
    FKL_SMALL(KK_LOSS_REDUCE, launch_loss_reduce(rowloss, N, n_valid, T, loss, s));
    return FKL_OK;
}
// The backward's launch sequence on a checked plan and workspace.
fkl_status backward_enqueue(const Plan& P, const void* h, const void* W, const int32_t* idx, const float* tlogit,
                            const uint8_t* mask, float T, const float* lse, const float* grad_loss, void* dh,
                            float* dW, void* ws, cudaStream_t s, const Mix* mix = nullptr) {
    const int64_t N = P.N, V = P.V;
    const int d = P.d, K = P.K;
    char* w = static_cast<char*>(ws);
    int* status = reinterpret_cast<int*>(w);
    int* n_valid = status + 1;
    int* sidx = reinterpret_cast<int*>(w + P.o_sidx);
    float* sp = reinterpret_cast<float*>(w + P.o_sp);
    float* H = reinterpret_cast<float*>(w + P.o_H);
    uint8_t* valid = reinterpret_cast<uint8_t*>(w + P.o_valid);
    void* dz = w + P.o_big;
    float* part = reinterpret_cast<float*>(w + P.o_part_dh);
    void* hT = w + P.o_hT;

    FKL_CUDA_TRY(cudaMemsetAsync(w, 0, 256, s));
    const int sms = device_info().sms;
    FKL_SMALL(KK_COUNT_VALID, launch_count_valid(tlogit, mask, N, K, n_valid, sms * 4, s));

    CUtensorMap tmW_k, tmW_mn, tmDW;
    FKL_TMAP(tmW_k, BF16, W, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, kVocabTile / 2);
    FKL_TMAP(tmW_mn, BF16, W, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, 64);
    FKL_TMAP(tmDW, F32, dW, uint64_t(d), uint64_t(V), uint64_t(d) * 4, 32, 32);
    for (int64_t c = 0; c < P.n_chunks; ++c) {
        NvtxRange nvtx_chunk("backward", static_cast<long long>(c));
        const int64_t row0 = c * P.Cc;
        const int rows = static_cast<int>(std::min<int64_t>(P.Cc, N - row0));
        const double flop = 2.0 * rows * double(d) * double(V);
        FKL_SMALL(KK_TEACHER_PREP,
                  launch_teacher_prep(idx, tlogit, mask, row0, rows, K, V, T, sidx, sp, H, valid, status, s));
        const char* hc = static_cast<const char*>(h) + size_t(row0) * d * 2;
        CUtensorMap tmH_k, tmHT_k, tmDz_st, tmDz_k, tmDz_mn, tmPart;
        FKL_TMAP(tmH_k, BF16, hc, uint64_t(d), uint64_t(rows), uint64_t(d) * 2, 64, 128);
        // the dW GEMM's B operand: each CTA of a pair loads half of a (sub-)tile's columns of d
        FKL_TMAP(tmHT_k, BF16, hT, uint64_t(rows), uint64_t(d), uint64_t(P.Cc) * 2, 64,
                 uint32_t(std::min(P.bn_dw, 256) / 2));
        FKL_PANEL_TMAP(tmDz_st, BF16, dz, 32);
        FKL_PANEL_TMAP(tmDz_k, BF16, dz, 128);
        FKL_PANEL_TMAP(tmDz_mn, BF16, dz, 64, 2);  // dW's A: the two panels of a CTA's 128 rows in one box
        FKL_TMAP(tmPart, F32, part, uint64_t(d), uint64_t(P.splits) * P.Cc, uint64_t(d) * 4, 32, 32);
        FKL_SMALL(KK_TRANSPOSE_H, launch_transpose_h(hc, rows, d, hT, P.Cc, s));

        // dz = T g (q - s) / N_valid for this chunk's rows, bf16 [rows][V]
        GemmParams p{};
        p.m_tiles = static_cast<int>(cdiv(rows, kPairRows));
        p.n_tiles = P.nt_v;
        p.splits = 1;
        p.kb_total = static_cast<int>(cdiv(d, kBK));
        p.m_fastest = 1;
        p.M = rows;
        p.Ncols = static_cast<int>(V);
        p.status = status;
        p.scale2 = kLog2e / T;
        p.sidx = sidx;
        p.sp = sp;
        p.K = K;
        p.lse = lse + row0;
        p.valid = valid;
        p.n_valid = n_valid;
        p.grad = grad_loss;
        p.T = T;
        if (mix) {
            p.label = mix->label + row0;
            p.alpha = mix->alpha;
            p.lse1 = mix->lse1_in + row0;
        }
        if (fkl_status st = run_gemm(KK_BWD_DZ, 256, 0, 0, mix ? EPI_DZ_MIX : EPI_DZ, tmH_k, tmW_k, tmDz_st, p,
                                     flop, s))
            return st;

        if (fkl_status st = grads_from_dz(P, c, rows, tmDz_k, tmDz_mn, tmHT_k, tmW_mn, tmPart, tmDW, part,
                                          static_cast<char*>(dh) + size_t(row0) * d * 2, status, s))
            return st;
    }
    return FKL_OK;
}

}  // namespace
}  // namespace fkl

using namespace fkl;

extern "C" {

size_t fkl_workspace_size(int64_t N, int d, int64_t V, int K, int chunk) {
    Plan P;
    return make_plan(N, d, V, K, chunk, P) ? P.total : 0;
}

const char* fkl_status_string(fkl_status st) {
    switch (st) {
        case FKL_OK: return "ok";
        case FKL_ERR_INVALID_ARG: return "invalid argument";
        case FKL_ERR_WORKSPACE: return "workspace too small";
        case FKL_ERR_INDEX: return "teacher index outside [0, V)";
        case FKL_ERR_CUDA: return "CUDA error";
        case FKL_ERR_UNSUPPORTED: return "unsupported device or size";
        case FKL_ERR_TIMEOUT: return "device pipeline wait timed out";
    }
    return "unknown status";
}

const char* fkl_last_error(void) { return g_err; }

fkl_status fkl_forward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                       const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T, int chunk,
                       float* loss, float* lse, void* ws, size_t ws_bytes, void* stream) {
    g_err[0] = 0;
    NvtxRange nvtx_call("fkl_forward");
    if (const char* e = check_common(h, W, idx, tlogit, N, d, V, K, T, chunk, ws))
        return fail(FKL_ERR_INVALID_ARG, "%s", e);
    if (!loss || !lse) return fail(FKL_ERR_INVALID_ARG, "null loss or lse pointer");
    Plan P;
    make_plan(N, d, V, K, chunk, P);
    if (ws_bytes < P.total)
        return fail(FKL_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, P.total);
    if (fkl_status st = device_ready()) return st;
    return forward_enqueue(P, h, W, idx, tlogit, mask, T, loss, lse, ws, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- forward without allocation
// Scratch of fkl_forward_noalloc: a fixed array in the library's own device
// image, present on every GPU that loads the library until the process exits.
// Shared by every call; only its 256-byte header must start at zero, and the
// forward clears it itself.
static __device__ __align__(256) unsigned char g_fwd_scratch[FKL_NOALLOC_SCRATCH_BYTES];

// Device address of g_fwd_scratch on the current device.  In host code
// `g_fwd_scratch` names a host-side stand-in, never the device memory, so kernels
// are only ever given this looked-up address.  The first call on a device looks
// it up (and must come before any stream capture); the lookup is repeated on every
// later call whose stream is not capturing (it is cheap), so that a context that
// was destroyed and rebuilt (cudaDeviceReset) never leaves a stale address behind.
static fkl_status noalloc_scratch(cudaStream_t s, void** out) {
    constexpr int kMaxDevices = 256;
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FKL_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(FKL_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        cs = cudaStreamCaptureStatusActive;  // cannot tell: treat as capturing
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cs == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fwd_scratch);
        if (e != cudaSuccess || !p)
            return fail(FKL_ERR_CUDA, "cudaGetSymbolAddress of the forward scratch on device %d: %s", dev,
                        cudaGetErrorString(e));
        addr[dev] = p;
    } else if (!addr[dev]) {
        return fail(FKL_ERR_UNSUPPORTED,
                    "the first fkl_forward_noalloc call on device %d came during stream capture: make one call "
                    "outside capture first, so that the scratch's address can be looked up",
                    dev);
    }
    *out = addr[dev];
    return FKL_OK;
}

fkl_status fkl_forward_noalloc(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                               const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T, int chunk,
                               float* loss, float* lse, int* status, void* stream) {
    g_err[0] = 0;
    NvtxRange nvtx_call("fkl_forward_noalloc");
    const char* e = check_sizes(N, d, V, K, chunk);
    if (!e && (!h || !W || !idx || !tlogit)) e = "null input pointer";
    if (!e && (!(T > 0.f) || !std::isfinite(T))) e = "T must be positive and finite";
    if (!e && (!aligned16(h) || !aligned16(W))) e = "h and W must be 16-byte aligned";
    if (e) return fail(FKL_ERR_INVALID_ARG, "%s", e);
    if (!loss || !lse) return fail(FKL_ERR_INVALID_ARG, "null loss or lse pointer");
    Plan P;
    make_plan(N, d, V, K, chunk, P);
    if (P.fwd_total > FKL_NOALLOC_SCRATCH_BYTES) {
        Plan Pmin;  // the smallest chunk: if even that does not fit, the 4 bytes per row are the limit
        make_plan(N, d, V, K, kBM, Pmin);
        if (Pmin.fwd_total > FKL_NOALLOC_SCRATCH_BYTES)
            return fail(FKL_ERR_WORKSPACE,
                        "the forward needs %zu bytes of scratch for N=%lld, V=%lld, K=%d even at the smallest "
                        "chunk (128), of which %lld grow with N (4 per row); the built-in scratch holds %zu: "
                        "pass fewer rows per call, or use fkl_forward with a caller workspace",
                        Pmin.fwd_total, static_cast<long long>(N), static_cast<long long>(V), K,
                        static_cast<long long>(N) * 4, static_cast<size_t>(FKL_NOALLOC_SCRATCH_BYTES));
        return fail(FKL_ERR_WORKSPACE,
                    "the forward needs %zu bytes of scratch for N=%lld, V=%lld, K=%d, chunk=%d; the built-in "
                    "scratch holds %zu: pass a smaller chunk, or use fkl_forward with a caller workspace",
                    P.fwd_total, static_cast<long long>(N), static_cast<long long>(V), K, P.Cc,
                    static_cast<size_t>(FKL_NOALLOC_SCRATCH_BYTES));
    }
    if (fkl_status st = device_ready()) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* scratch = nullptr;
    if (fkl_status st = noalloc_scratch(s, &scratch)) return st;
    if (fkl_status st = forward_enqueue(P, h, W, idx, tlogit, mask, T, loss, lse, scratch, s)) return st;
    if (status) FKL_CUDA_TRY(cudaMemcpyAsync(status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, s));
    return FKL_OK;
}

fkl_status fkl_backward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                        const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T, int chunk,
                        const float* lse, const float* grad_loss, void* dh, float* dW, void* ws,
                        size_t ws_bytes, void* stream) {
    g_err[0] = 0;
    NvtxRange nvtx_call("fkl_backward");
    if (const char* e = check_common(h, W, idx, tlogit, N, d, V, K, T, chunk, ws))
        return fail(FKL_ERR_INVALID_ARG, "%s", e);
    if (!lse || !dh || !dW) return fail(FKL_ERR_INVALID_ARG, "null lse, dh or dW pointer");
    if (!aligned16(dh) || !aligned16(dW)) return fail(FKL_ERR_INVALID_ARG, "dh and dW must be 16-byte aligned");
    Plan P;
    make_plan(N, d, V, K, chunk, P);
    if (ws_bytes < P.total)
        return fail(FKL_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, P.total);
    if (fkl_status st = device_ready()) return st;
    return backward_enqueue(P, h, W, idx, tlogit, mask, T, lse, grad_loss, dh, dW, ws,
                            static_cast<cudaStream_t>(stream));
}

fkl_status fkl_mix_forward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                           const uint8_t* mask, const int32_t* label, int64_t N, int d, int64_t V, int K, float T,
                           float alpha, int chunk, float* loss, float* lse, float* lse1, void* ws, size_t ws_bytes,
                           void* stream) {
    g_err[0] = 0;
    NvtxRange nvtx_call("fkl_mix_forward");
    if (const char* e = check_common(h, W, idx, tlogit, N, d, V, K, T, chunk, ws))
        return fail(FKL_ERR_INVALID_ARG, "%s", e);
    if (!loss || !lse || !lse1 || !label) return fail(FKL_ERR_INVALID_ARG, "null loss, lse, lse1 or label pointer");
    if (!(alpha >= 0.f && alpha <= 1.f)) return fail(FKL_ERR_INVALID_ARG, "alpha must be in [0, 1]");
    Plan P;
    make_plan(N, d, V, K, chunk, P);
    if (ws_bytes < P.total)
        return fail(FKL_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, P.total);
    if (fkl_status st = device_ready()) return st;
    const Mix mix{label, alpha, lse1, nullptr};
    return forward_enqueue(P, h, W, idx, tlogit, mask, T, loss, lse, ws, static_cast<cudaStream_t>(stream), &mix);
}

fkl_status fkl_mix_backward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                            const uint8_t* mask, const int32_t* label, int64_t N, int d, int64_t V, int K, float T,
                            float alpha, int chunk, const float* lse, const float* lse1, const float* grad_loss,
                            void* dh, float* dW, void* ws, size_t ws_bytes, void* stream) {
    g_err[0] = 0;
    NvtxRange nvtx_call("fkl_mix_backward");
    if (const char* e = check_common(h, W, idx, tlogit, N, d, V, K, T, chunk, ws))
        return fail(FKL_ERR_INVALID_ARG, "%s", e);
    if (!lse || !lse1 || !label || !dh || !dW) return fail(FKL_ERR_INVALID_ARG, "null lse, lse1, label, dh or dW");
    if (!aligned16(dh) || !aligned16(dW)) return fail(FKL_ERR_INVALID_ARG, "dh and dW must be 16-byte aligned");
    if (!(alpha >= 0.f && alpha <= 1.f)) return fail(FKL_ERR_INVALID_ARG, "alpha must be in [0, 1]");
    Plan P;
    make_plan(N, d, V, K, chunk, P);
    if (ws_bytes < P.total)
        return fail(FKL_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, P.total);
    if (fkl_status st = device_ready()) return st;
    const Mix mix{label, alpha, nullptr, lse1};
    return backward_enqueue(P, h, W, idx, tlogit, mask, T, lse, grad_loss, dh, dW, ws,
                            static_cast<cudaStream_t>(stream), &mix);
}

fkl_status fkl_forward_backward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                                const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T, int chunk,
                                const float* grad_loss, float* loss, float* lse, void* dh, float* dW, void* ws,
                                size_t ws_bytes, void* stream) {
    g_err[0] = 0;
    NvtxRange nvtx_call("fkl_forward_backward");
    if (const char* e = check_common(h, W, idx, tlogit, N, d, V, K, T, chunk, ws))
        return fail(FKL_ERR_INVALID_ARG, "%s", e);
    if (!loss || !lse || !dh || !dW) return fail(FKL_ERR_INVALID_ARG, "null loss, lse, dh or dW pointer");
    if (!aligned16(dh) || !aligned16(dW)) return fail(FKL_ERR_INVALID_ARG, "dh and dW must be 16-byte aligned");
    Plan P;
    make_plan(N, d, V, K, chunk, P);
    if (ws_bytes < P.total)
        return fail(FKL_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, P.total);
    if (fkl_status st = device_ready()) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(ws);
    int* status = reinterpret_cast<int*>(w);
    int* n_valid = status + 1;
    int* sidx = reinterpret_cast<int*>(w + P.o_sidx);
    float* sp = reinterpret_cast<float*>(w + P.o_sp);
    float* H = reinterpret_cast<float*>(w + P.o_H);
    uint8_t* valid = reinterpret_cast<uint8_t*>(w + P.o_valid);
    float* rowloss = reinterpret_cast<float*>(w + P.o_rowloss);
    void* yz = w + P.o_big;  // kept logits (fp16), then dz (bf16) in place
    float* part = reinterpret_cast<float*>(w + P.o_part_dh);
    void* hT = w + P.o_hT;
    const size_t pstride = align256(size_t(P.nt_v) * P.Cc * 4);
    float* pm = reinterpret_cast<float*>(w + P.o_part_dh);  // forward partials share the dh partials' place
    float* pl = reinterpret_cast<float*>(w + P.o_part_dh + pstride);
    float* pg = reinterpret_cast<float*>(w + P.o_part_dh + 2 * pstride);

    FKL_CUDA_TRY(cudaMemsetAsync(w, 0, 256, s));
    const int sms = device_info().sms;
    FKL_SMALL(KK_COUNT_VALID, launch_count_valid(tlogit, mask, N, K, n_valid, sms * 4, s));

    CUtensorMap tmW_k, tmW_mn, tmDW;
    FKL_TMAP(tmW_k, BF16, W, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, kVocabTile / 2);
    FKL_TMAP(tmW_mn, BF16, W, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, 64);
    FKL_TMAP(tmDW, F32, dW, uint64_t(d), uint64_t(V), uint64_t(d) * 4, 32, 32);
    for (int64_t c = 0; c < P.n_chunks; ++c) {
        NvtxRange nvtx_chunk("forward_backward", static_cast<long long>(c));
        const int64_t row0 = c * P.Cc;
        const int rows = static_cast<int>(std::min<int64_t>(P.Cc, N - row0));
        FKL_SMALL(KK_TEACHER_PREP,
                  launch_teacher_prep(idx, tlogit, mask, row0, rows, K, V, T, sidx, sp, H, valid, status, s));
        const char* hc = static_cast<const char*>(h) + size_t(row0) * d * 2;
        CUtensorMap tmH_k, tmHT_k, tmY_st, tmDz_k, tmDz_mn, tmPart;
        FKL_TMAP(tmH_k, BF16, hc, uint64_t(d), uint64_t(rows), uint64_t(d) * 2, 64, 128);
        // the dW GEMM's B operand: each CTA of a pair loads half of a (sub-)tile's columns of d
        FKL_TMAP(tmHT_k, BF16, hT, uint64_t(rows), uint64_t(d), uint64_t(P.Cc) * 2, 64,
                 uint32_t(std::min(P.bn_dw, 256) / 2));
        FKL_PANEL_TMAP(tmY_st, F16, yz, 32);
        FKL_PANEL_TMAP(tmDz_k, BF16, yz, 128);
        FKL_PANEL_TMAP(tmDz_mn, BF16, yz, 64, 2);
        FKL_TMAP(tmPart, F32, part, uint64_t(d), uint64_t(P.splits) * P.Cc, uint64_t(d) * 4, 32, 32);
        FKL_SMALL(KK_TRANSPOSE_H, launch_transpose_h(hc, rows, d, hT, P.Cc, s));

        // logits of the chunk: lse / gather partials, and y = z log2e/T - tile max kept in fp16
        GemmParams p{};
        p.m_tiles = static_cast<int>(cdiv(rows, kPairRows));
        p.n_tiles = P.nt_v;
        p.splits = 1;
        p.kb_total = static_cast<int>(cdiv(d, kBK));
        p.m_fastest = 1;
        p.M = rows;
        p.Ncols = static_cast<int>(V);
        p.status = status;
        p.scale2 = kLog2e / T;
        p.sidx = sidx;
        p.sp = sp;
        p.K = K;
        p.part_m = pm;
        p.part_l = pl;
        p.part_g = pg;
        p.part_stride = P.Cc;
        if (fkl_status st = run_gemm(KK_FB_GEMM_LSE_Y, 256, 0, 0, EPI_LSE_Y, tmH_k, tmW_k, tmY_st, p,
                                     2.0 * rows * double(d) * double(V), s))
            return st;
        FKL_SMALL(KK_FWD_FINALIZE,
                  launch_fwd_finalize(pm, pl, pg, P.Cc, P.nt_v, rows, H, valid, T, lse + row0, rowloss + row0, s));
        // dz from the kept logits, in place (no second pass over the tensor cores)
        FKL_SMALL(KK_FB_DZ, launch_dz_from_logits(yz, int64_t(P.Cc) * 64, V, pm, P.Cc, lse + row0, valid, n_valid,
                                                  grad_loss, T, sidx, sp, K, rows,
                                                  reinterpret_cast<float*>(w + P.o_yk), s));
        if (fkl_status st = grads_from_dz(P, c, rows, tmDz_k, tmDz_mn, tmHT_k, tmW_mn, tmPart, tmDW, part,
                                          static_cast<char*>(dh) + size_t(row0) * d * 2, status, s))
            return st;
    }
    FKL_SMALL(KK_LOSS_REDUCE, launch_loss_reduce(rowloss, N, n_valid, T, loss, s));
    return FKL_OK;
}

size_t fkl_topk_workspace_size(int64_t N, int d, int64_t V, int K, int chunk) {
    TopkPlan P;
    return make_topk_plan(N, d, V, K, chunk, P) ? P.total : 0;
}

fkl_status fkl_teacher_topk(const void* h, const void* W, int64_t N, int d, int64_t V, int K, int chunk,
                            int32_t* idx, float* logit, void* ws, size_t ws_bytes, void* stream) {
    g_err[0] = 0;
    NvtxRange nvtx_call("fkl_teacher_topk");
    if (!h || !W || !idx || !logit || !ws) return fail(FKL_ERR_INVALID_ARG, "null pointer");
    if (const char* e = check_sizes(N, d, V, K, chunk)) return fail(FKL_ERR_INVALID_ARG, "%s", e);
    if (!aligned16(h) || !aligned16(W) || !aligned16(ws))
        return fail(FKL_ERR_INVALID_ARG, "h, W and ws must be 16-byte aligned");
    TopkPlan P;
    make_topk_plan(N, d, V, K, chunk, P);
    if (ws_bytes < P.total)
        return fail(FKL_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, P.total);
    if (fkl_status st = device_ready()) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(ws);
    int* status = reinterpret_cast<int*>(w);
    int* any_flag = status + 1;  // some row of the call needed the second pass (diagnostic)
    float* part = reinterpret_cast<float*>(w + P.o_part);
    float* top_v = reinterpret_cast<float*>(w + P.o_topv);
    int* top_i = reinterpret_cast<int*>(w + P.o_topi);
    uint8_t* row_flag = reinterpret_cast<uint8_t*>(w + P.o_flag);
    float* theta = reinterpret_cast<float*>(w + P.o_theta);
    int* cnt_gt = reinterpret_cast<int*>(w + P.o_gt);
    int* cnt_eq = reinterpret_cast<int*>(w + P.o_eq);
    int* sub_flag = reinterpret_cast<int*>(w + P.o_sflag);
    float* cand_v = reinterpret_cast<float*>(w + P.o_cv);
    int* cand_i = reinterpret_cast<int*>(w + P.o_ci);
    int* tie_i = reinterpret_cast<int*>(w + P.o_tie);
    FKL_CUDA_TRY(cudaMemsetAsync(w, 0, 256, s));

    CUtensorMap tmW;
    FKL_TMAP(tmW, BF16, W, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, kVocabTile / 2);
    for (int64_t c = 0; c < P.n_chunks; ++c) {
        NvtxRange nvtx_chunk("teacher_topk", static_cast<long long>(c));
        const int64_t row0 = c * P.Cc;
        const int rows = static_cast<int>(std::min<int64_t>(P.Cc, N - row0));
        const double flop = 2.0 * rows * double(d) * double(V);
        const char* hc = static_cast<const char*>(h) + size_t(row0) * d * 2;
        CUtensorMap tmH;
        FKL_TMAP(tmH, BF16, hc, uint64_t(d), uint64_t(rows), uint64_t(d) * 2, 64, 128);
        GemmParams p{};
        p.m_tiles = static_cast<int>(cdiv(rows, kPairRows));
        p.n_tiles = P.nt_v;
        p.splits = 1;
        p.kb_total = static_cast<int>(cdiv(d, kBK));
        p.m_fastest = 1;
        p.M = rows;
        p.Ncols = static_cast<int>(V);
        p.status = status;
        p.part_m = part;
        p.top_v = top_v;
        p.top_i = top_i;
        p.part_stride = P.Cc;
        p.K = K;
        FKL_CUDA_TRY(cudaMemsetAsync(sub_flag, 0, size_t(P.n_sub) * 4, s));
        if (fkl_status st = run_gemm(KK_TK_GEMM_TMAX, 256, 0, 0, EPI_TMAX, tmH, tmW, tmW, p, flop, s)) return st;
        // theta, candidates and selection per row; rows it cannot complete are flagged
        FKL_SMALL(KK_TK_ROWS, launch_topk_rows(part, top_v, top_i, P.Cc, P.nt_v, rows, K, P.Cs, theta, cnt_gt,
                                               cnt_eq, row_flag, sub_flag, idx + size_t(row0) * K,
                                               logit + size_t(row0) * K, s));
        // the second tensor-core pass and the selection of its rows, per sub-chunk
        // with a flagged row (a launch returns at once when its sub-chunk has none)
        for (int r0 = 0; r0 < rows; r0 += P.Cs) {
            const int srows = std::min(P.Cs, rows - r0);
            const int sc = r0 / P.Cs;
            CUtensorMap tmHs;
            FKL_TMAP(tmHs, BF16, hc + size_t(r0) * d * 2, uint64_t(d), uint64_t(srows), uint64_t(d) * 2, 64, 128);
            GemmParams q{};
            q.m_tiles = static_cast<int>(cdiv(srows, kPairRows));
            q.n_tiles = P.nt_v;
            q.splits = 1;
            q.kb_total = static_cast<int>(cdiv(d, kBK));
            q.m_fastest = 1;
            q.M = srows;
            q.Ncols = static_cast<int>(V);
            q.status = status;
            q.K = K;
            q.any_flag = sub_flag + sc;
            q.row_flag = row_flag + r0;
            q.theta = theta + r0;
            q.cnt_gt = cnt_gt + r0;
            q.cnt_eq = cnt_eq + r0;
            q.cand_v = cand_v;
            q.cand_i = cand_i;
            q.cand_cap = P.cap;
            q.tie_i = tie_i;
            // (its FLOP are not counted: the launch usually returns at once)
            if (fkl_status st = run_gemm(KK_TK_GEMM_CAND, 256, 0, 0, EPI_CAND, tmHs, tmW, tmW, q, 0.0, s)) return st;
            FKL_SMALL(KK_TK_SELECT,
                      launch_topk_select(cand_v, cand_i, P.cap, cnt_gt + r0, cnt_eq + r0, tie_i, theta + r0,
                                         row_flag + r0, srows, K, idx + size_t(row0 + r0) * K,
                                         logit + size_t(row0 + r0) * K, s));
        }
        FKL_SMALL(KK_TK_FLAGS, launch_or_flags(sub_flag, P.n_sub, any_flag, s));
    }
    return FKL_OK;
}

fkl_status fkl_scale_grads(void* dh, float* dW, int64_t N, int d, int64_t V, const float* grad, void* stream) {
    g_err[0] = 0;
    if (!dh || !dW || !grad) return fail(FKL_ERR_INVALID_ARG, "null dh, dW or grad pointer");
    if (N < 1 || V < 1 || d < 8 || d % 8 != 0) return fail(FKL_ERR_INVALID_ARG, "N, V >= 1 and d a multiple of 8");
    if (!aligned16(dh) || !aligned16(dW)) return fail(FKL_ERR_INVALID_ARG, "dh and dW must be 16-byte aligned");
    if (fkl_status st = device_ready()) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FKL_SMALL(KK_SCALE_GRADS, launch_scale_grads(dh, size_t(N) * d, dW, size_t(V) * d, grad,
                                                 device_info().sms * 8, s));
    return FKL_OK;
}

fkl_status fkl_get_status(const void* ws, void* stream) {
    g_err[0] = 0;
    if (!ws) return fail(FKL_ERR_INVALID_ARG, "null workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FKL_CUDA_TRY(cudaStreamSynchronize(s));
    int st = 0;
    FKL_CUDA_TRY(cudaMemcpy(&st, ws, sizeof(int), cudaMemcpyDeviceToHost));
    return static_cast<fkl_status>(st);
}

void fkl_profile_enable(int on) { g_prof_on.store(on != 0); }

void fkl_profile_reset(void) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    for (auto& r : g_prof) {
        g_event_pool.push_back(r.a);
        g_event_pool.push_back(r.b);
    }
    g_prof.clear();
}

int fkl_profile_read(double* ms, int64_t* launches, double* flop, int n) {
    for (int k = 0; k < n && k < KK_NUM; ++k) {
        if (ms) ms[k] = 0;
        if (launches) launches[k] = 0;
        if (flop) flop[k] = 0;
    }
    std::lock_guard<std::mutex> lock(g_prof_mu);
    for (auto& r : g_prof) {
        if (r.kind >= n) continue;
        float t = 0.f;
        cudaEventSynchronize(r.b);
        cudaEventElapsedTime(&t, r.a, r.b);
        if (ms) ms[r.kind] += t;
        if (launches) launches[r.kind] += 1;
        if (flop) flop[r.kind] += r.flop;
    }
    return KK_NUM;
}

const char* fkl_kernel_name(int kind) { return (kind >= 0 && kind < KK_NUM) ? kKindNames[kind] : ""; }

int64_t fkl_launch_count(void) { return g_launches.load(); }

fkl_status fkl_selftest_wait_timeout(void* ws, int64_t limit_ns, void* stream) {
    g_err[0] = 0;
    if (!ws || !aligned16(ws)) return fail(FKL_ERR_INVALID_ARG, "ws must be a 16-byte aligned device pointer");
    if (limit_ns < 1000 || limit_ns > 2000000000) return fail(FKL_ERR_INVALID_ARG, "limit_ns must be in [1e3, 2e9]");
    if (fkl_status st = device_ready()) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FKL_CUDA_TRY(cudaMemsetAsync(ws, 0, 256, s));
    cudaError_t e;
    {
        LaunchScope ls(KK_SELFTEST_WAIT, 0.0, s);
        e = launch_wait_timeout(static_cast<int*>(ws), static_cast<uint64_t>(limit_ns), s);
    }
    if (e != cudaSuccess) return fail(FKL_ERR_CUDA, "selftest_wait launch: %s", cudaGetErrorString(e));
    return FKL_OK;
}

fkl_status fkl_selftest_gemm(const void* A, const void* B, float* C, int M, int N, int K, int a_mn, int b_mn,
                             int bn, void* ws, void* stream) {
    g_err[0] = 0;
    if (!A || !B || !C || !ws) return fail(FKL_ERR_INVALID_ARG, "null pointer");
    if (M < 1 || N < 1 || K < 1 || M % 8 || N % 8 || K % 8)
        return fail(FKL_ERR_INVALID_ARG, "M, N, K must be positive multiples of 8");
    if ((a_mn | b_mn) & ~1) return fail(FKL_ERR_INVALID_ARG, "a_mn and b_mn must be 0 or 1");
    if (bn != 512 && bn != 256 && bn != 192 && bn != 128)
        return fail(FKL_ERR_INVALID_ARG, "bn must be 512, 256, 192 or 128");
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(ws))
        return fail(FKL_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (fkl_status st = device_ready()) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FKL_CUDA_TRY(cudaMemsetAsync(ws, 0, 256, s));
    CUtensorMap ta, tb, tc;
    if (a_mn == 0) FKL_TMAP(ta, BF16, A, uint64_t(K), uint64_t(M), uint64_t(K) * 2, 64, 128);
    else FKL_TMAP(ta, BF16, A, uint64_t(M), uint64_t(K), uint64_t(M) * 2, 64, 64);
    if (b_mn == 0) FKL_TMAP(tb, BF16, B, uint64_t(K), uint64_t(N), uint64_t(K) * 2, 64, uint32_t(std::min(bn, 256) / 2));
    else FKL_TMAP(tb, BF16, B, uint64_t(N), uint64_t(K), uint64_t(N) * 2, 64, 64);
    FKL_TMAP(tc, F32, C, uint64_t(N), uint64_t(M), uint64_t(N) * 4, 32, 32);
    GemmParams p{};
    p.m_tiles = static_cast<int>(cdiv(M, kPairRows));
    p.n_tiles = static_cast<int>(cdiv(N, bn));
    p.splits = 1;
    p.kb_total = static_cast<int>(cdiv(K, kBK));
    p.m_fastest = 1;
    p.M = M;
    p.Ncols = N;
    p.status = static_cast<int*>(ws);
    return run_gemm(KK_SELFTEST, bn, a_mn, b_mn, EPI_F32, ta, tb, tc, p, 2.0 * M * double(N) * K, s);
}

}  // extern "C"
