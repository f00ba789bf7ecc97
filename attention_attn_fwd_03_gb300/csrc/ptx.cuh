// ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers, TMA tensor copies, tcgen05 (tensor-memory allocation, MMA,
// commit, TMEM loads/stores, fences) and a few scalar instructions.
//
// Every wait in this library is bounded: attn::wait_bar() gives up after
// kWaitLimitNs of wall time (or as soon as the CTA's abort flag or the
// device status word is set), records ATTN_ERR_TIMEOUT in the status word
// and returns false, so a logic error ends a kernel instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace attn {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr unsigned kStatusTimeout = 5u;                      // == ATTN_ERR_TIMEOUT
constexpr unsigned kStatusDeviceData = 6u;                   // == ATTN_ERR_DEVICE_DATA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool bar_try_wait(uint64_t* bar, uint32_t parity) {
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

// As bar_try_wait, but the thread may sleep in hardware for up to
// `suspend_ns` while the phase is incomplete instead of returning at once,
// so waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool bar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// True when some kernel of the device has recorded a timeout in the status
// word (the only bit that makes other kernels stop: ATTN_ERR_DEVICE_DATA
// reports bad caller data, which every kernel clamps, and cancels nothing).
__device__ __forceinline__ bool timeout_recorded(const unsigned* status) {
    return (*(const volatile unsigned*)status & (1u << kStatusTimeout)) != 0u;
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (after flagging the CTA and the device status word) on timeout, or
// when another role of the CTA, or another CTA, has already given up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* status) {
    if (bar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (bar_try_wait_sleep(bar, parity, 20000u)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (timeout_recorded(status)) {
                *abort_flag = 1;
                return false;
            }
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(status, 1u << kStatusTimeout);
                return false;
            }
        }
    }
}

// Programmatic dependent launch: a grid launched with programmatic stream
// serialisation may start while its predecessor runs; griddep_wait blocks
// until the predecessor grid has completed and its writes are visible, and
// griddep_launch_dependents lets the next such grid be scheduled early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait that ignores the abort flag (used only to drain in-flight async work
// before the CTA releases its shared and tensor memory); bounded in time.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned* status) {
    const unsigned long long t0 = globaltimer();
    while (!bar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(status, 1u << kStatusTimeout);
            return;
        }
    }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// 3-D tiled store shared -> global (rows outside the tensor are clipped).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Element-wise add of a shared-memory box into the tensor (f32 maps: an
// atomic per-element reduction done by the bulk-copy engine).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Generic-proxy shared-memory writes -> visible to the async proxy (TMA).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), 16-bit inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem desc), 16-bit inputs.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 8-bit (e4m3) inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four tcgen05.mma of one GEMM in a single asm block (one predicate set-up,
// no address arithmetic between them): step k uses descriptors a + OA_k and
// b + OB_k (descriptor units: 16 bytes), or for a tensor-memory A operand the
// column a + OA_k; the first step accumulates iff `accumulate`.
template <int OA1, int OA2, int OA3, int OB1, int OB2, int OB3, bool F8>
__device__ __forceinline__ void mma4_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    if (F8)
        asm volatile(
            "{\n\t.reg .pred p0, p1;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
            "add.s64 a1, %1, %5;\n\tadd.s64 a2, %1, %6;\n\tadd.s64 a3, %1, %7;\n\t"
            "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a2, b2, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a3, b3, %3, p1;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p0, p1;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
            "add.s64 a1, %1, %5;\n\tadd.s64 a2, %1, %6;\n\tadd.s64 a3, %1, %7;\n\t"
            "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, p1;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
}

template <int OA1, int OA2, int OA3, int OB1, int OB2, int OB3, bool F8>
__device__ __forceinline__ void mma4_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    if (F8)
        asm volatile(
            "{\n\t.reg .pred p0, p1;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
            "add.u32 a1, %1, %5;\n\tadd.u32 a2, %1, %6;\n\tadd.u32 a3, %1, %7;\n\t"
            "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a1], b1, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a2], b2, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a3], b3, %3, p1;\n\t}" ::"r"(d),
            "r"(a), "l"(b), "r"(idesc), "r"(accumulate), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p0, p1;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
            "add.u32 a1, %1, %5;\n\tadd.u32 a2, %1, %6;\n\tadd.u32 a3, %1, %7;\n\t"
            "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, p1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, p1;\n\t}" ::"r"(d),
            "r"(a), "l"(b), "r"(idesc), "r"(accumulate), "n"(OA1), "n"(OA2), "n"(OA3), "n"(OB1), "n"(OB2), "n"(OB3)
            : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// 1024-byte swizzle atoms (8 rows x 128 B) start on 1024-byte boundaries.
//   lbo: byte distance between atoms along the leading (MN for MN-major)
//        dimension; sbo: byte distance between consecutive 8-row groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;  // descriptor version used by tcgen05
    d |= (uint64_t)2u << 61;  // swizzle mode: 128 B
    return d;
}

// Instruction descriptor: fp32 accumulator, dense, M x N tile.
//   ab_fmt: 1 = bf16 for kind::f16; 0 = e4m3 for kind::f8f6f4.
__host__ __device__ constexpr uint32_t idesc_make(int M, int N, uint32_t ab_fmt, bool a_mn_major,
                                                  bool b_mn_major) {
    return (1u << 4)                           // D format: f32
           | (ab_fmt << 7) | (ab_fmt << 10)    // A and B formats
           | ((a_mn_major ? 1u : 0u) << 15)    // A major-ness
           | ((b_mn_major ? 1u : 0u) << 16)    // B major-ness
           | ((uint32_t)(N >> 3) << 17)        // N / 8
           | ((uint32_t)(M >> 4) << 24);       // M / 16
}

// ---- TMEM loads / stores (32 data-path lanes x 32-bit, one lane per thread)

#define ATTN_REG8(a, b) "=r"(a[b + 0]), "=r"(a[b + 1]), "=r"(a[b + 2]), "=r"(a[b + 3]), \
                        "=r"(a[b + 4]), "=r"(a[b + 5]), "=r"(a[b + 6]), "=r"(a[b + 7])
#define ATTN_IREG8(a, b) "r"(a[b + 0]), "r"(a[b + 1]), "r"(a[b + 2]), "r"(a[b + 3]), \
                         "r"(a[b + 4]), "r"(a[b + 5]), "r"(a[b + 6]), "r"(a[b + 7])

// 32 consecutive columns of this thread's lane -> r[0..31].  The values are
// valid only after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : ATTN_REG8(r, 0), ATTN_REG8(r, 8), ATTN_REG8(r, 16), ATTN_REG8(r, 24)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Ties registers filled by tmem_ld32 to the preceding tmem_ld_wait(): every
// later use of r[0..n) is ordered after it.
template <int N>
__device__ __forceinline__ void reg_after_wait(uint32_t* r) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        ATTN_IREG8(r, 0), ATTN_IREG8(r, 8), ATTN_IREG8(r, 16), ATTN_IREG8(r, 24)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        ATTN_IREG8(r, 0), ATTN_IREG8(r, 8)
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#undef ATTN_REG8
#undef ATTN_IREG8

// ---------------------------------------------------------------- scalar helpers

// 2^x (PTX ex2.approx: -inf -> +0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) (PTX lg2.approx).
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed pairs of fp32 in one 64-bit register (element 0 in the low half).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// a * b + c on both halves (round to nearest).
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Two fp32 -> packed bf16x2, `lo` in the low half (round to nearest even).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 -> four e4m3fn bytes (nearest, saturating), x0 in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace attn
