/*
 * fkl.h -- C ABI of libfkl.so: the fused chunked top-K forward-KL distillation
 * loss over an LM head, on one B300 (sm_103a).
 *
 * The operation.  Student hidden states h[N,d] (bf16) meet the LM-head weight
 * W[V,d] (bf16); z = h W^T is formed tile by tile on the tensor cores and never
 * stored.  Each token carries an offline teacher cache of K (index, logit)
 * pairs: the top-100 of the teacher per position in "Effektivnaya distillyatsiya
 * znaniy" (malakhovai.ru, paragraph 2) and "Wissensdestillation mit deutlich
 * weniger GPU-Speicher" (dailytechsnack.ch, section "Teacher-Ausgaben einmalig
 * zwischenspeichern").  With temperature T ("Distillyatsiya i szhatie modeley",
 * ml-book.com, section "Kak eto rabotaet: myagkie metki i temperatura"):
 *
 *   p_ik  = softmax_k(t_ik / T)                (renormalised over the K cached ids)
 *   lse_i = logsumexp_v (z_iv / T)             (over the FULL vocabulary V)
 *   KL_i  = sum_k p_ik (log p_ik - z_{i,idx_ik}/T + lse_i)      (0 log 0 = 0)
 *   loss  = T^2 * sum_{valid i} KL_i / N_valid                  (0 if N_valid = 0)
 *   dz_iv = g * valid_i * T * (exp(z_iv/T - lse_i) - s_iv) / N_valid,
 *           s_iv = sum_{k: idx_ik = v} p_ik,   g = upstream gradient
 *   dh = dz W,  dW = dz^T h
 *
 * A token is valid when mask_i != 0 and at least one of its teacher logits is
 * finite.  The sequence is processed in chunks of rows: logits of a chunk are
 * reduced and discarded, and recomputed in the backward pass ("Multiverse
 * Computing uzhala distillyatsiyu", iitak.ru, paragraph 3; dailytechsnack.ch,
 * section "KL-Verlust wird in Bloecken berechnet": the output projection feeds
 * the loss directly).  Workspace grows linearly in N.
 *
 * Conventions shared by every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory and keeps no state between calls (the one
 *    exception, fkl_forward_noalloc, brings fixed scratch of its own).
 *  - Layouts are dense row-major: h [N][d] bf16, W [V][d] bf16, idx [N][K]
 *    int32, tlogit [N][K] fp32, mask [N] uint8 (NULL = every row valid),
 *    lse [N] fp32, dh [N][d] bf16, dW [V][d] fp32.
 *  - Preconditions checked on the host (FKL_ERR_INVALID_ARG, before any launch):
 *    non-NULL required pointers; 1 <= N <= 2^40; 8 <= d <= 65536, d % 8 == 0;
 *    1 <= V <= 2^30 (V % 8 == 0 is NOT required); 1 <= K <= 256, K <= V; T > 0
 *    and finite; chunk == 0 (library default) or a positive multiple of 128 up
 *    to 2^20; h, W, dh, dW and the workspace 16-byte aligned.  Teacher ids within a row must be distinct
 *    (not checked; repeated ids are summed into s).
 *  - Calls enqueue on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    and return without synchronising.  Errors found on the device (a teacher
 *    id outside [0, V), a pipeline wait that timed out) are written to a status
 *    word at the start of the workspace; read it with fkl_get_status.
 *  - `ws` must hold at least fkl_workspace_size(N, d, V, K, chunk) bytes
 *    (FKL_ERR_WORKSPACE otherwise).  The same workspace may serve the forward
 *    and the backward call; its contents between calls carry no meaning except
 *    the status word.
 *  - Host threads: calls from several threads at once, on their own streams,
 *    are safe as long as no workspace or output is shared between calls whose
 *    work overlaps on the GPU (per-device set-up is done once, under a lock).
 */
#ifndef FKL_H
#define FKL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FKL_OK = 0,
    FKL_ERR_INVALID_ARG = 1,  /* a precondition above failed (host-side, nothing launched) */
    FKL_ERR_WORKSPACE = 2,    /* ws_bytes below fkl_workspace_size */
    FKL_ERR_INDEX = 3,        /* a teacher id outside [0, V); outputs are undefined */
    FKL_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed; see fkl_last_error */
    FKL_ERR_UNSUPPORTED = 5,  /* no sm_103a device, or a size beyond the kernels' limits */
    FKL_ERR_TIMEOUT = 6       /* a bounded pipeline wait gave up on the device */
} fkl_status;

/* Bytes of device workspace needed by fkl_forward, fkl_backward,
 * fkl_forward_backward, fkl_mix_forward and fkl_mix_backward for these sizes
 * (chunk as passed to them).  Pure host arithmetic; 0 if the sizes are invalid.
 * It is O(chunk * V + N): one bf16 dz chunk buffer, split-K partials of dh for
 * one chunk, the chunk's h transposed, the sorted teacher cache of one chunk and
 * 4 bytes per token (1.82 GB at N = 131072, d = 2880, V = 201088, K = 100,
 * default chunk).  The environment variables FKL_BN_DH and FKL_BN_DW (512, 256,
 * 192 or 128; other values are ignored) override the column-tile width of the dh
 * and dW GEMMs for tuning sweeps; the dh width sets the split count and so this
 * size, which is read at each call (a workspace sized under another setting is
 * refused with FKL_ERR_WORKSPACE if too small). */
size_t fkl_workspace_size(int64_t N, int d, int64_t V, int K, int chunk);

/* Forward: writes loss (one fp32, device) and lse[N] (fp32, natural-log
 * logsumexp of z/T for every row, masked rows included). */
fkl_status fkl_forward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                       const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T,
                       int chunk, float* loss, float* lse,
                       void* ws, size_t ws_bytes, void* stream);

/* Forward for callers that cannot allocate device memory: the same launch
 * sequence and results as fkl_forward, with the workspace replaced by scratch
 * that the library carries itself.  The pages have no counterpart to this entry
 * point; it exists for callers that own no device allocator of their own (a
 * plain C host program, or a plug-in running inside a runtime that has already
 * reserved the GPU's memory for its own pool) and for step loops that must not
 * call cudaMalloc/cudaFree, which can synchronise the device and can fail under
 * memory pressure.
 *
 *  - Scratch: a fixed array of FKL_NOALLOC_SCRATCH_BYTES (64 MiB) in the
 *    library's device image.  Every GPU that loads the library holds it until
 *    the process exits.  This call allocates nothing: no cudaMalloc, cudaFree or
 *    allocating library routine.
 *  - Size limit: the forward needs 256 + 8*C*K + 5*C + 4*N + 12*C*ceil(V/256)
 *    bytes (each term rounded up to 256) for chunk C (0 = 4096, capped at N
 *    rounded up to 128); beyond FKL_NOALLOC_SCRATCH_BYTES the call returns
 *    FKL_ERR_WORKSPACE before any launch, with the sizes in fkl_last_error.  At
 *    V = 201088, K = 100 and C = 4096 that is about 42 MB + 4*N.  The 4*N
 *    bytes do not depend on the chunk: from about 16 million rows on no chunk
 *    fits, and the message names N as the limit.
 *  - Set-up: the first call on each device looks up the scratch's device
 *    address (with that device current).  Make that first call before any
 *    stream capture.  Later calls whose stream is not capturing look the
 *    address up again (a cheap query), so that it stays right after the
 *    device's context has been destroyed and rebuilt (cudaDeviceReset).
 *  - Sharing: every call on a device uses the same scratch, which keeps the
 *    previous call's contents (the call clears what must start at zero).  Calls
 *    whose work overlaps on the GPU -- on different streams, or from different
 *    host threads -- race on it: order them on one stream or with events.
 *  - Device-side errors (a teacher id outside [0, V), a pipeline wait that
 *    timed out) are copied, when the call's work finishes, into *status (one
 *    int32 in device memory, caller-owned; NULL = not reported): FKL_OK or the
 *    fkl_status code.
 * Other arguments, preconditions and outputs are those of fkl_forward. */
#define FKL_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
fkl_status fkl_forward_noalloc(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                               const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T,
                               int chunk, float* loss, float* lse, int* status, void* stream);

/* Backward: recomputes every logit tile and writes dh [N][d] (bf16, overwritten)
 * and dW [V][d] (fp32, overwritten).  `lse` is the forward's output for the same
 * inputs.  `grad_loss` points to one fp32 upstream gradient on the device
 * (NULL = 1.0).  dW is accumulated chunk by chunk in a fixed order, so repeated
 * calls give bit-identical results. */
fkl_status fkl_backward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                        const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T,
                        int chunk, const float* lse, const float* grad_loss,
                        void* dh, float* dW,
                        void* ws, size_t ws_bytes, void* stream);

/* KL + hard-label cross-entropy mixture.  "Distillyatsiya i szhatie modeley"
 * (ml-book.com, section "Kak eto rabotaet: myagkie metki i temperatura") has the
 * student's loss mix the KL between the softened distributions with the ordinary
 * cross-entropy on the true labels, the T^2 factor keeping the KL gradients in
 * scale; the weighting formula itself is lost from the page and is read as the
 * usual convex mix:
 *   loss  = alpha T^2 mean KL_i + (1 - alpha) mean CE_i     (means over valid rows)
 *   CE_i  = lse1_i - z_{i,label_i},  lse1_i = logsumexp_v z_iv  (temperature 1)
 *   dz_iv = g valid_i [alpha T (q_iv - s_iv) + (1 - alpha)(q1_iv - [v = label_i])] / N_valid,
 *           q1 = exp(z - lse1)
 * label [N] int32, in [0, V) for every valid row (FKL_ERR_INDEX in the status
 * word otherwise); 0 <= alpha <= 1 (alpha = 1 is the plain loss of fkl_forward /
 * fkl_backward).  lse1 [N] fp32 is written by the forward and read by the
 * backward.  Everything else as in fkl_forward / fkl_backward, with the same
 * workspace.  Costs one more exponential per logit in each pass. */
fkl_status fkl_mix_forward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                           const uint8_t* mask, const int32_t* label, int64_t N, int d, int64_t V, int K,
                           float T, float alpha, int chunk, float* loss, float* lse, float* lse1,
                           void* ws, size_t ws_bytes, void* stream);
fkl_status fkl_mix_backward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                            const uint8_t* mask, const int32_t* label, int64_t N, int d, int64_t V, int K,
                            float T, float alpha, int chunk, const float* lse, const float* lse1,
                            const float* grad_loss, void* dh, float* dW,
                            void* ws, size_t ws_bytes, void* stream);

/* Forward and backward in one call, for a training step that needs the loss
 * gradient at once (the upstream gradient is known before the call; grad_loss
 * NULL = 1.0).  Writes what fkl_forward followed by fkl_backward write: loss,
 * lse [N], dh [N][d] (bf16) and dW [V][d] (fp32, overwritten).  Each chunk's
 * logits are kept between the chunk's loss pass and its gradient pass, in the
 * workspace's dz buffer, as fp16 y = z log2(e)/T minus the row's max over each
 * 256-column vocabulary tile; dz is then formed from y in place.  The tensor
 * cores therefore compute 6 N d V FLOP instead of 8 N d V, with the same
 * workspace (fkl_workspace_size).  This is the forward-chunked alternative the
 * pages weigh against recomputation ("Effektivnaya distillyatsiya znaniy",
 * malakhovai.ru, the table of dense / forward-chunked / fused variants), here
 * with per-chunk rather than per-sequence storage.  lse and loss equal
 * fkl_forward's up to float rounding (the per-tile max / sum order differs); dz,
 * hence dh and dW, differ from the recomputed ones by the fp16 rounding of y
 * (relative 2^-11 of |y|, smallest where q is largest). */
fkl_status fkl_forward_backward(const void* h, const void* W, const int32_t* idx, const float* tlogit,
                                const uint8_t* mask, int64_t N, int d, int64_t V, int K, float T,
                                int chunk, const float* grad_loss, float* loss, float* lse,
                                void* dh, float* dW,
                                void* ws, size_t ws_bytes, void* stream);

/* ---- teacher top-K cache producer ------------------------------------------
 * The offline step before the loss: z = h W^T for the TEACHER's hidden states h
 * [N][d] (bf16) and LM head W [V][d] (bf16), and per row the K largest logits:
 * idx [N][K] (int32) and logit [N][K] (fp32, the fp32-accumulated z), sorted by
 * logit descending, equal logits by id ascending -- the cache of the teacher's
 * top-100 per position of "Effektivnaya distillyatsiya znaniy" (malakhovai.ru,
 * paragraph 2) and "Wissensdestillation mit deutlich weniger GPU-Speicher"
 * (dailytechsnack.ch, section "Teacher-Ausgaben einmalig zwischenspeichern"),
 * in the layout fkl_forward reads (its `idx` and `tlogit`).
 * One tensor-core pass per chunk of rows keeps each row's eight largest logits
 * per 256-column vocabulary tile.  theta = the K-th largest of the tile maxima
 * is a lower bound of the row's K-th largest logit, and every logit >= theta
 * lies in a tile whose max reaches it, so the candidates are gathered from the
 * per-tile lists -- completely, unless some such tile holds eight or more logits
 * >= theta; those rows (rare: eight of the row's top logits in one tile) get a
 * second tensor-core pass over their 1024-row sub-chunk that keeps all their
 * logits >= theta.  Selection and sorting of the K largest run one warp per row
 * (a block per row for the rows of the second pass).  Where more than K logits
 * tie at theta itself, which of them are kept is unspecified for the rows of the
 * second pass (the others keep the smallest ids).  The full N x V logits are
 * never stored.  Conventions as above (device pointers, caller-owned,
 * stream-ordered, status word at the start of ws); chunk = 0 means 4096 rows.
 * The workspace is O(chunk * V / 4 + min(chunk, 1024) * min(V, 256 K)) bytes:
 * 427 MB at V = 201088, K = 100. */
size_t fkl_topk_workspace_size(int64_t N, int d, int64_t V, int K, int chunk);
fkl_status fkl_teacher_topk(const void* h, const void* W, int64_t N, int d, int64_t V, int K, int chunk,
                            int32_t* idx, float* logit, void* ws, size_t ws_bytes, void* stream);

/* dh [N][d] (bf16) *= g and dW [V][d] (fp32) *= g, g = *grad (one fp32 on the
 * device): the chain rule for gradients that fkl_forward_backward formed during
 * the forward with grad_loss = 1, once the upstream gradient is known (autograd's
 * backward).  g = 1 leaves both unchanged bit for bit. */
fkl_status fkl_scale_grads(void* dh, float* dW, int64_t N, int d, int64_t V, const float* grad, void* stream);

/* Synchronises `stream` and returns the device status word of `ws` (FKL_OK if
 * no device-side error was recorded since the last call that used `ws`). */
fkl_status fkl_get_status(const void* ws, void* stream);

/* Static description of a status code. */
const char* fkl_status_string(fkl_status status);

/* Message of the last host-side error in the calling thread ("" if none). */
const char* fkl_last_error(void);

/* ---- measurement hooks (not part of the loss) ----------------------------
 * When enabled, every kernel launch of this library is bracketed by two CUDA
 * events recorded on the launching stream.  fkl_profile_read synchronises the
 * recorded events and reports, per kernel kind k < n, the summed device time in
 * ms, the number of launches and the algorithmic FLOP those launches performed
 * (tensor-core kernels only; 0 otherwise); it returns the number of kinds.
 * fkl_profile_reset forgets the records.  Safe to call from several host
 * threads; a launch is timed if profiling was on when it started. */
void fkl_profile_enable(int on);
void fkl_profile_reset(void);
int fkl_profile_read(double* ms, int64_t* launches, double* flop, int n);
const char* fkl_kernel_name(int kind);
/* Kernels launched by this library since it was loaded. */
int64_t fkl_launch_count(void);

/* ---- self-test entry (not part of the loss) -------------------------------
 * C[M][N] (fp32, row-major) = sum_k A(m,k) B(n,k) on the same tcgen05/TMA
 * pipeline the loss kernels use.  a_mn = 0: A is [M][K] row-major (K-major);
 * a_mn = 1: A is stored [K][M] (M-major).  b_mn = 0: B is [N][K]; b_mn = 1: B
 * is stored [K][N].  bn selects the N tile: 256, 192 or 128 (double-buffered
 * accumulators), or 512 (two 256-wide sub-tiles sharing A, single-buffered).
 * M, N, K >= 1 and multiples of 8.  `ws` (>= 256 bytes, device) receives the status word.  Used
 * to check the operand descriptors in isolation. */
fkl_status fkl_selftest_gemm(const void* A, const void* B, float* C, int M, int N, int K,
                             int a_mn, int b_mn, int bn, void* ws, void* stream);

/* ---- bounded-wait self-test (not part of the loss) -------------------------
 * Every pipeline wait of the kernels gives up after a time limit, records
 * FKL_ERR_TIMEOUT in the status word and lets the kernel return, so that a
 * defect ends in an error instead of a hung GPU.  This entry runs that same wait
 * in a one-thread kernel on a barrier nothing ever arrives on, with limit_ns
 * (1e3 .. 2e9) instead of the pipelines' 2 s: afterwards fkl_get_status(ws)
 * reports FKL_ERR_TIMEOUT and the context stays usable.  `ws`: >= 256 bytes of
 * device memory; its status word is cleared first. */
fkl_status fkl_selftest_wait_timeout(void* ws, int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FKL_H */
