// Inline-PTX primitives for sm_103a: mbarriers, TMA (cp.async.bulk.tensor),
// 5th-generation tensor core instructions (tcgen05.*) and TMEM access.
// Written from the PTX ISA descriptions of these instructions; no library
// headers beyond the CUtensorMap type are used.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace fp8bs {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits until the phase with the given parity has completed.  Gives up after
// `limit_ns` nanoseconds of global time and returns false; never spins forever.
// Polls with the non-blocking test (a suspended try_wait was measured to wake
// several hundred cycles after the phase completes, which the MMA pipeline
// cannot hide; keeping several tests in flight, or sleeping between tests,
// measured slower); the timer is read only every 1024 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
#pragma unroll 1
    for (int i = 0; i < 1024; ++i)
        if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 1024; ++i)
            if (mbar_test_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Waits until the phase with the given parity has completed, sleeping in
// mbarrier.try_wait (the thread is suspended until the phase completes or
// the hint runs out) instead of spinning.  For waits off the critical path:
// spinning warps take issue slots and shared-memory bandwidth from the warps
// that feed the tensor core, but a suspended thread wakes a few hundred
// cycles after the phase completes.  Gives up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
            : "memory");
        if (ok) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Release store / acquire load of a shared-memory word (CTA scope): a flag
// one thread publishes after its own waits, for another thread to poll.
__device__ __forceinline__ void st_release_shared(uint32_t *p, uint32_t v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_shared(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

// Waits until the shared word *p (advanced with st_release_shared) reaches at
// least `target`; gives up after `limit_ns` nanoseconds and returns false.
__device__ __forceinline__ bool wait_counter(const uint32_t *p, uint32_t target, uint64_t limit_ns) {
#pragma unroll 1
    for (int i = 0; i < 1024; ++i)
        if ((int32_t)(ld_acquire_shared(p) - target) >= 0) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 1024; ++i)
            if ((int32_t)(ld_acquire_shared(p) - target) >= 0) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// 4-byte asynchronous global -> shared copy; with valid == false nothing is
// read and the destination is zero-filled.
__device__ __forceinline__ void cp_async_4(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}

// 16-byte asynchronous global -> shared copy (both addresses 16-byte
// aligned); with valid == false nothing is read and the destination is
// zero-filled.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

// 16-byte asynchronous global -> shared copy with an L2 eviction-priority
// hint (a createpolicy value); both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async_16_hint(void *dst, const void *src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Waits until at most N of this thread's most recent cp.async groups are
// still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Arrives on `bar` once all of this thread's earlier cp.async copies have
// landed (the barrier's expected count must include this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load global -> shared; completion is signalled on `bar` as
// transaction bytes.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                            int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Same, with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                                 int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled store shared -> global (bulk-group completion).  Rows and
// columns outside the tensor are not written; c0 must be >= 0 and a multiple
// of 16 bytes' worth of elements.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until this thread's bulk groups, all but the newest N, have finished
// reading their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until this thread's bulk groups, all but the newest N, are complete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA store) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05
// TMEM allocation: executed by all 32 threads of one warp.  The allocated
// base address (lane 0, first column) is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
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

// D[tmem] (+)= A[smem] * B[smem]^T for FP8 E4M3 x E4M3 -> FP32, issued by one
// thread.  `accumulate` == 0 overwrites D.
__device__ __forceinline__ void umma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled variant (scale_vec::1X, one UE8M0 scale per row per 32-wide K
// slice, i.e. per instruction): D (+)= sum_k A[m,k] 2^(ea[m]-127) B[n,k]
// 2^(eb[n]-127).  Where the tensor core reads the scales (M = 128; found with
// an in-bounds probe that filled the scale columns with position codes):
//   ea[m]: byte sfa_id (instruction descriptor) of TMEM lane m, column
//          sfa_tmem + m / 32;
//   eb[n]: byte sfb_id of lane 32 q + n % 32, column sfb_tmem + n / 32, where
//          q = m / 32 is the lane quarter of the output row being computed,
//          so B's scales must be present in all four lane quarters.
__device__ __forceinline__ void umma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Warp-collective TMEM -> register loads: thread i of the warp reads lane
// (taddr.lane + i); register j holds column (taddr.col + j).
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Warp-collective register -> TMEM stores (32x32b shape): thread i of the
// warp writes lane (taddr.lane + i); register j goes to column (taddr.col + j).
// The warp may only address its own lane quarter, 32 * (warp % 4).
__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// Waits until this thread's earlier tcgen05.st have been performed.
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile stored as rows
// of 128 bytes with the 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B): 8-row groups are 1024 bytes apart.  The tile
// base must be 1024-byte aligned; advancing along K inside the 128-byte row
// is done by adding (bytes >> 4) to the start-address field.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // [0,14)  start address >> 4
    d |= (uint64_t)1 << 16;                     // [16,30) leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;           // [32,46) stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                     // [46,48) descriptor version 1 (tcgen05)
    d |= (uint64_t)2 << 61;                     // [61,64) swizzle mode: 128-byte
    return d;
}

// Instruction descriptor, kind::f8f6f4: D fp32, A and B E4M3, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
    return (1u << 4)                          // [4,6)   D format: f32
           | (0u << 7) | (0u << 10)           // [7,10) A, [10,13) B: E4M3
           | ((uint32_t)(n >> 3) << 17)       // [17,23) N >> 3
           | ((uint32_t)(m >> 4) << 24);      // [24,29) M >> 4
}

// Instruction descriptor, kind::mxf8f6f4 (block-scaled): A and B E4M3,
// K-major, UE8M0 scale factors; D is fp32.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int m, int n, uint32_t sfa_id, uint32_t sfb_id) {
    return (sfb_id << 4)                      // [4,6)   B scale-factor byte id
           | (0u << 7) | (0u << 10)           // A, B: E4M3
           | ((uint32_t)(n >> 3) << 17)       // [17,23) N >> 3
           | (1u << 23)                       // [23]    scale type UE8M0
           | ((uint32_t)(m >> 4) << 24)       // [24,29) M >> 4
           | (sfa_id << 29);                  // [29,31) A scale-factor byte id
}

// Waits for this thread's outstanding tcgen05.ld and, through the "+f"
// operands, makes the 32 given accumulators inputs of the wait: the compiler
// must finish the arithmetic that produces them before it, so that work
// overlaps the load in flight instead of queueing behind its completion.
__device__ __forceinline__ void tmem_ld_wait_after(float (&a)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(a[0]), "+f"(a[1]), "+f"(a[2]), "+f"(a[3]), "+f"(a[4]), "+f"(a[5]), "+f"(a[6]), "+f"(a[7]),
                   "+f"(a[8]), "+f"(a[9]), "+f"(a[10]), "+f"(a[11]), "+f"(a[12]), "+f"(a[13]), "+f"(a[14]),
                   "+f"(a[15]), "+f"(a[16]), "+f"(a[17]), "+f"(a[18]), "+f"(a[19]), "+f"(a[20]), "+f"(a[21]),
                   "+f"(a[22]), "+f"(a[23]), "+f"(a[24]), "+f"(a[25]), "+f"(a[26]), "+f"(a[27]), "+f"(a[28]),
                   "+f"(a[29]), "+f"(a[30]), "+f"(a[31])
                 :
                 : "memory");
}

// acc[j] = fma(v[j], sc, acc[j]) for 32 fp32 values, as 16 packed
// fma.rn.f32x2 (each lane an IEEE fma.rn.f32, so the result is bit-identical
// to fmaf): half the issue slots of 32 scalar FMAs.
__device__ __forceinline__ void fma32_packed(float (&acc)[32], const uint32_t (&v)[32], float sc) {
    uint64_t s;
    asm("mov.b64 %0, {%1, %1};" : "=l"(s) : "f"(sc));
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        uint64_t a, x;
        asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc[2 * j]), "f"(acc[2 * j + 1]));
        asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(v[2 * j]), "r"(v[2 * j + 1]));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x), "l"(s));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[2 * j]), "=f"(acc[2 * j + 1]) : "l"(a));
    }
}

// acc[j] = fma(v[j], RN(sa * sbv[j]), acc[j]) for 32 fp32 values: a scale
// per column (sbv: 32 floats in shared memory, 16-byte aligned, the same
// address in every lane).  Each scale product is rounded once, as the
// single-scale form rounds sa * sb.
__device__ __forceinline__ void fma32_packed_cols(float (&acc)[32], const uint32_t (&v)[32], float sa,
                                                  const float *sbv) {
    uint64_t s;
    asm("mov.b64 %0, {%1, %1};" : "=l"(s) : "f"(sa));
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const float4 b = *reinterpret_cast<const float4 *>(sbv + 4 * g);
        uint64_t p[2];
        asm("mov.b64 %0, {%1, %2};" : "=l"(p[0]) : "f"(b.x), "f"(b.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(p[1]) : "f"(b.z), "f"(b.w));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 4 * g + 2 * h;
            uint64_t a, x;
            asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(p[h]) : "l"(s));
            asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc[j]), "f"(acc[j + 1]));
            asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(v[j]), "r"(v[j + 1]));
            asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x), "l"(p[h]));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[j]), "=f"(acc[j + 1]) : "l"(a));
        }
    }
}

// Per-warpgroup register reallocation (all four warps of the warpgroup
// execute it).  The sum over warpgroups must stay within the registers the
// CTA was launched with.
template <int N>
__device__ __forceinline__ void regs_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ----------------------------------------------------------------- programmatic dependent launch
// In a kernel launched with programmatic stream serialization: blocks until
// the grids this one depends on have completed and their memory is visible
// (a no-op otherwise).  Must precede every global access to data they wrote.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream, if launched with programmatic stream
// serialization, start its CTAs (up to their griddep_wait) before this grid
// has finished.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

// Named barrier over `count` threads (multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also returns, to every participating thread, the OR of
// their `pred` values: a decision (say, to give up after a wait ran out)
// that all of them take alike, so none is left waiting at a later barrier.
__device__ __forceinline__ bool named_bar_red_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

}  // namespace fp8bs
