// Thin wrappers over the sm_100-family PTX used by the loss kernels: mbarriers,
// TMA (cp.async.bulk.tensor), tcgen05 (UMMA issue, TMEM allocation and loads)
// and a few scalar helpers.  Every wait is bounded by the global timer so that a
// broken pipeline ends in an error status instead of a hung GPU.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fkl_internal.h"

namespace fkl {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait before giving up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(int* status, int code) {
    atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of parity `parity` to complete.  Returns false (and
// raises the CTA's abort flag and the device status) after limit_ns, or at
// once if another role of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int* status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                set_status(status, FKL_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
    return mbar_wait_for(bar, parity, abort_flag, status, kWaitLimitNs);
}

// Time-bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* m, uint32_t src, int x, int y) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most one committed bulk group is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_le1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 D,
// M x N tile, operand majorness (0 = K-major, 1 = MN-major).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.  lbo / sbo in bytes:
// K-major operands use sbo = 1024 (8 rows x 128 B) and an ignored lbo;
// MN-major operands use lbo = byte distance between 64-element MN blocks and
// sbo = 1024 (8 K-rows x 128 B).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // SWIZZLE_128B
    return d;
}

// ---------------------------------------------------------------- CTA pairs (cluster of 2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on an mbarrier that may live in the peer CTA (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar_cluster,
                                                 int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}
// The same for a 3-D tensor map (the panel layout of dz: {64 columns, rows, panel}).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar_cluster,
                                                 int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
// TMEM allocation shared by the pair: one warp of each CTA executes these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[tmem of both CTAs] (+)= A * B^T over the pair's operands (M = 256), issued by the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// When the MMAs issued so far complete, arrive once on the mbarrier at this
// shared-memory offset in BOTH CTAs of the pair.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    const uint16_t both = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(both)
        : "memory");
}

// One 64-deep k-block of a 256-column pair tile: four K = 16 MMAs whose operand
// descriptors advance by KA / KB (the descriptor units of 16 k-elements), then the
// commit that frees the stage in both CTAs.  Before them, a non-blocking test of
// the next stage's `full` barrier; its result is read only after the commit, so
// its shared-memory latency overlaps the MMA issue instead of preceding the next
// k-block.  Returns 1 if the next stage had already landed.
template <uint32_t KA, uint32_t KB>
__device__ __forceinline__ uint32_t umma_kblock_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                     uint32_t idesc, uint32_t accumulate, uint32_t empty_bar,
                                                     uint32_t next_full_bar, uint32_t next_parity) {
    uint32_t ready;
    const uint16_t both = 0x3;
    asm volatile(
        "{\n\t.reg .pred acc, one, landed;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 landed, [%7], %8;\n\t"
        "setp.ne.b32 acc, %5, 0;\n\t"
        "setp.ne.b32 one, %10, 0;\n\t"
        "add.s64 a1, %2, %11;\n\tadd.s64 b1, %3, %14;\n\t"
        "add.s64 a2, %2, %12;\n\tadd.s64 b2, %3, %15;\n\t"
        "add.s64 a3, %2, %13;\n\tadd.s64 b3, %3, %16;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%1], %2, %3, %4, acc;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%1], a1, b1, %4, one;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%1], a2, b2, %4, one;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%1], a3, b3, %4, one;\n\t"
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%6], %9;\n\t"
        "selp.u32 %0, 1, 0, landed;\n\t}"
        : "=r"(ready)
        : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(empty_bar),
          "r"(next_full_bar), "r"(next_parity), "h"(both), "r"(1u), "n"(KA), "n"(2 * KA), "n"(3 * KA),
          "n"(KB), "n"(2 * KB), "n"(3 * KB)
        : "memory");
    return ready;
}

// Two consecutive k-blocks (stages s0 and s1) as above: eight MMAs, one commit
// freeing each stage, and non-blocking tests of the two stages after them.
// Returns 1 if both of those had landed.  Halves the issuing thread's fixed cost
// (loop, fence, barrier test) per MMA against umma_kblock_pair.
template <uint32_t KA, uint32_t KB>
__device__ __forceinline__ uint32_t umma_2kblocks_pair(uint32_t d_tmem, uint64_t a0_desc, uint64_t b0_desc,
                                                       uint64_t a1_desc, uint64_t b1_desc, uint32_t idesc,
                                                       uint32_t accumulate, uint32_t empty0_bar,
                                                       uint32_t empty1_bar, uint32_t full2_bar,
                                                       uint32_t parity2, uint32_t full3_bar, uint32_t parity3) {
    uint32_t ready;
    const uint16_t both = 0x3;
    asm volatile(
        "{\n\t.reg .pred acc, one, l2, l3;\n\t"
        ".reg .b64 a01, a02, a03, b01, b02, b03, a11, a12, a13, b11, b12, b13;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 l2, [%10], %11;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 l3, [%12], %13;\n\t"
        "setp.ne.b32 acc, %7, 0;\n\t"
        "setp.ne.b32 one, %15, 0;\n\t"
        "add.s64 a01, %1, %16;\n\tadd.s64 b01, %2, %19;\n\t"
        "add.s64 a02, %1, %17;\n\tadd.s64 b02, %2, %20;\n\t"
        "add.s64 a03, %1, %18;\n\tadd.s64 b03, %2, %21;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], %1, %2, %6, acc;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], a01, b01, %6, one;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], a02, b02, %6, one;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], a03, b03, %6, one;\n\t"
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%8], %14;\n\t"
        "add.s64 a11, %3, %16;\n\tadd.s64 b11, %4, %19;\n\t"
        "add.s64 a12, %3, %17;\n\tadd.s64 b12, %4, %20;\n\t"
        "add.s64 a13, %3, %18;\n\tadd.s64 b13, %4, %21;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], %3, %4, %6, one;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], a11, b11, %6, one;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], a12, b12, %6, one;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%5], a13, b13, %6, one;\n\t"
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%9], %14;\n\t"
        "and.pred l2, l2, l3;\n\t"
        "selp.u32 %0, 1, 0, l2;\n\t}"
        : "=r"(ready)
        : "l"(a0_desc), "l"(b0_desc), "l"(a1_desc), "l"(b1_desc), "r"(d_tmem), "r"(idesc), "r"(accumulate),
          "r"(empty0_bar), "r"(empty1_bar), "r"(full2_bar), "r"(parity2), "r"(full3_bar), "r"(parity3),
          "h"(both), "r"(1u), "n"(KA), "n"(2 * KA), "n"(3 * KA), "n"(KB), "n"(2 * KB), "n"(3 * KB)
        : "memory");
    return ready;
}

// ---------------------------------------------------------------- scalar helpers
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// z[off] for a run-time off in [0, 32) without local memory: a 5-level select tree.
__device__ __forceinline__ float select32(const float (&z)[32], int off) {
    float a[16], b[8], c[4], e[2];
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = (off & 16) ? z[j + 16] : z[j];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = (off & 8) ? a[j + 8] : a[j];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = (off & 4) ? b[j + 4] : b[j];
#pragma unroll
    for (int j = 0; j < 2; ++j) e[j] = (off & 2) ? c[j + 2] : c[j];
    return (off & 1) ? e[1] : e[0];
}

}  // namespace fkl
