// sm103_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100a/sm_103a)
// features the kernels use: mbarriers with bounded waits, TMA tiled and bulk
// copies, and the 5th-generation tensor core (tcgen05: TMEM allocation, MMA,
// commit, TMEM loads/stores, fences).  Each wrapper is one PTX instruction
// (or a short fixed sequence) with its operands spelled out; no library code.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace attn {

// ---------------------------------------------------------------- status word
// The status word is four ints of device memory, 8-byte aligned:
//   status[0]  bit 0: a bounded wait ran out;
//   status[1]  site code of the first wait that ran out (for diagnosis);
//   status[2..3]  address of a host-visible flag (mapped, page-locked host memory), written
//              once per device when the library sets the device up; a wait that runs out
//              also sets that flag, so the host learns of it without synchronising.
enum : int { kStatusTimeout = 1 };

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Limits of every in-kernel wait: about two seconds of wall time, and an
// absolute cap on polls.  A wait that runs out raises the CTA's abort flag and
// the device status word and returns false; callers then unwind.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitLimitPolls = 1u << 28;

struct WaitCtx {
    volatile int *abort_flag;  // shared memory, one per CTA; null for drain waits
    int *status;               // device status word (global, four ints; see above)
};

// A wait with a null abort flag (used to drain copies in flight while unwinding)
// ignores the CTA's abort state and stops only at its own limits.  Inlined, not
// called: kernels that reconfigure registers per warpgroup (setmaxnreg) cannot
// contain calls.
static __device__ __forceinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, WaitCtx w, int site) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < kWaitLimitPolls; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (w.abort_flag && *w.abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    }
    if (w.abort_flag) *w.abort_flag = 1;
    if (atomicOr(&w.status[0], kStatusTimeout) == 0) atomicExch(&w.status[1], site);
    // the host-visible copy: a plain store (no atomics on host memory), then a system fence
    volatile int *host_flag = *reinterpret_cast<int *const volatile *>(w.status + 2);
    if (host_flag) {
        *host_flag = kStatusTimeout;
        __threadfence_system();
    }
    return false;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, WaitCtx w, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, w, site);
}

// ---------------------------------------------------------------- e4m3
// Four e4m3 codes (byte 0 lowest) -> two f16x2 words: lo = codes 0, 1 and hi = codes 2, 3, the lower
// code in the lower half.  Exact: every e4m3 value is an f16 value.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
// Tiled 3-D load of one box into shared memory, completion counted in bytes
// on `bar`.  Coordinates are element indices, innermost first.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                            int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Tiled 3-D store of one box from shared memory (bulk-group completion).  Parts of the box past the
// tensor's extent are not written.  The coordinates must not be negative.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *smem_src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk group of this thread has completed (its writes performed).
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation: executed by one whole warp; the base address is written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 async op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]  (kind::f16: bf16/fp16 operands, fp32 accumulate)
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Products issued in groups from one asm statement.  A thread that issues its MMAs one asm
// statement at a time, with each operand buffer chosen at run time (a ring slot), keeps the
// tensor core at about 107 cycles per 128x128x16 product; a group in one statement issues at
// the full rate (64 cycles).  The operand descriptors advance by constants inside the
// statement (two temporaries), which keeps the issuing thread's registers few.  In every
// group the first product accumulates into D only if acc != 0, the others always.
//
// K-major operands with a 128-byte swizzle stored as 64-column boxes of box16 x 16 bytes:
// k-steps 0-3 lie 32 bytes apart in the first box, 4-7 likewise in the second.
#define ATTN_SS_STEP(ao, bo)                         \
    "add.s64 ra, %1, " #ao ";\n\t"                   \
    "add.s64 rb, %2, " #bo ";\n\t"                   \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, q;\n\t"
__device__ __forceinline__ void tc_mma_ss_k4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 ra, rb;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        ATTN_SS_STEP(2, 2) ATTN_SS_STEP(4, 4) ATTN_SS_STEP(6, 6) "}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_mma_ss_k2(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 ra, rb;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        ATTN_SS_STEP(2, 2) "}" ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Eight k-steps over two 16 KB boxes (k-steps 4-7 start 16384 bytes = 1024 descriptor units on).
__device__ __forceinline__ void tc_mma_ss_k8_box16k(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                                    uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 ra, rb;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        ATTN_SS_STEP(2, 2) ATTN_SS_STEP(4, 4) ATTN_SS_STEP(6, 6)
        ATTN_SS_STEP(1024, 1024) ATTN_SS_STEP(1026, 1026) ATTN_SS_STEP(1028, 1028) ATTN_SS_STEP(1030, 1030) "}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
#undef ATTN_SS_STEP
// K = d/16 k-steps of a product over K-major 128-byte-swizzled tiles held as 64-column boxes
// of 16 KB (128 rows): groups of four per box, then the remainder.
template <int K>
__device__ __forceinline__ void tc_mma_ss_ksteps(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                                 uint32_t acc) {
    static_assert(K >= 1 && K <= 8, "k-steps of a 128-column tile");
    if constexpr (K == 8) {
        tc_mma_ss_k8_box16k(d_tmem, a, b, idesc, acc);
    } else if constexpr (K >= 4) {
        tc_mma_ss_k4(d_tmem, a, b, idesc, acc);
        constexpr uint64_t box = 16384 >> 4;  // the next box, in descriptor units
        if constexpr (K - 4 >= 2) tc_mma_ss_k2(d_tmem, a + box, b + box, idesc, 1u);
        if constexpr ((K - 4) % 2 == 1) tc_mma_ss(d_tmem, a + box + 2 * ((K - 4) / 2), b + box + 2 * ((K - 4) / 2), idesc, 1u);
    } else {
        if constexpr (K >= 2) tc_mma_ss_k2(d_tmem, a, b, idesc, acc);
        if constexpr (K % 2 == 1) tc_mma_ss(d_tmem, a + 2 * (K / 2), b + 2 * (K / 2), idesc, K >= 2 ? 1u : acc);
    }
}

// Eight k-steps of 16 of a product with A from TMEM (bf16 pairs: 8 columns per k-step, the
// columns of step kk at a_tmem + acol(kk)) and B MN-major in shared memory (2048 bytes, 128
// descriptor units, per k-step).  acol(kk) = 8 kk when cols_gap is 0, else 8 (kk % 4) +
// 64 (kk / 4) (two 64-column halves, as the backward's P^T / dS^T tiles are laid out).
#define ATTN_TS_STEP(ac, bo)                         \
    "add.u32 ta, %1, " #ac ";\n\t"                   \
    "add.s64 rb, %2, " #bo ";\n\t"                   \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %3, q;\n\t"
__device__ __forceinline__ void tc_mma_ts_k8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b32 ta;\n\t.reg .b64 rb;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        ATTN_TS_STEP(8, 128) ATTN_TS_STEP(16, 256) ATTN_TS_STEP(24, 384) ATTN_TS_STEP(32, 512)
        ATTN_TS_STEP(40, 640) ATTN_TS_STEP(48, 768) ATTN_TS_STEP(56, 896) "}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Four k-steps (64 keys) of the same form: A columns 0, 8, 16, 24 from a_tmem.
__device__ __forceinline__ void tc_mma_ts_k4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b32 ta;\n\t.reg .b64 rb;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        ATTN_TS_STEP(8, 128) ATTN_TS_STEP(16, 256) ATTN_TS_STEP(24, 384) "}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_mma_ts_k8_halves(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                    uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b32 ta;\n\t.reg .b64 rb;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        ATTN_TS_STEP(8, 128) ATTN_TS_STEP(16, 256) ATTN_TS_STEP(24, 384) ATTN_TS_STEP(64, 512)
        ATTN_TS_STEP(72, 640) ATTN_TS_STEP(80, 768) ATTN_TS_STEP(88, 896) "}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
#undef ATTN_TS_STEP

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//   bits  0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 version (1), 61-63 layout (2 = 128B swizzle).
// K-major tiles: rows of 128 B, 8-row atoms of 1024 B -> SBO = 1024, LBO unused.
// MN-major tiles: 64 contiguous MN elements per 128-B row, 8 K rows per atom ->
//   SBO = stride between 8-row K groups, LBO = stride between 64-element MN groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// A descriptor advanced by `bytes` along its buffer.  The start-address field (bits 0-13,
// address >> 4) cannot carry into the next field: shared memory ends below 256 KB.  Building
// a buffer's descriptor once and advancing it by constants keeps the MMA-issuing thread's
// instruction stream to one add per operand (a descriptor rebuilt per MMA made the issue of a
// 128x128x16 product take about 100 cycles instead of its 64).
__device__ __forceinline__ uint64_t sdesc_advance(uint64_t desc, uint32_t bytes) {
    return desc + (uint64_t)(bytes >> 4);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   15 A major (0 = K), 16 B major (1 = MN), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with f16 A and B (format code 0 in bits 7-9 and 10-12).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// 32 lanes x 32 columns of 32-bit TMEM -> 32 registers per thread (thread i = lane i,
// register j = column j).  The loaded values are valid only after tmem_wait_ld(...).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 32 lanes x 16 columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
        :
        : "memory");
}

// Waits for all prior tcgen05.ld of this thread; the "+r" operands tie the
// registers to the wait so no use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
          "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
          "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
          "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}
// 16 registers -> 32 lanes x 16 columns of TMEM.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- register reconfiguration
// Per-warpgroup register limits (all four warps of the warpgroup execute it).  The block's
// register pool is its launch allocation (threads x registers at launch); the callers keep
// the sum of the new per-warpgroup limits within it.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- math
// 2^x on the special-function unit (approximate, flush-to-zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input FMNMX).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed pairs of fp32 (one 64-bit register holds {lo, hi}): one instruction does two lanes' worth.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace attn
