// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA, tcgen05 (TMEM / UMMA).
//
// Each wrapper is one instruction (or a fixed short sequence) of the PTX ISA;
// the kernels compose them. Every wait is bounded: on expiry it raises a
// CTA-wide abort flag and the ORTHROS_DEV_TIMEOUT status bit, so that all roles
// of a kernel drain instead of spinning forever.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "internal.cuh"

namespace orthros {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
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

// Raises the transaction count the current phase waits for, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
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

// About 2 s at 2 GHz: far longer than any legitimate wait in these kernels.
constexpr long long kWaitLimitCycles = 4000000000LL;

// Waits for the phase with the given parity to complete. Returns false (and
// raises *abort plus the status bit) if the limit runs out or another thread
// of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          uint32_t *status, long long limit = kWaitLimitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            set_status(status, ORTHROS_DEV_TIMEOUT);
            return false;
        }
    }
}

// Warp-converged form of mbar_wait for waits that every lane of a warp makes:
// all lanes poll together and leave together, so the warp never splits into
// lanes that were woken and lanes still suspended in try_wait (a split warp
// reconverges only when the slowest lane's wait returns). Returns the same
// value in every lane.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort,
                                               uint32_t *status) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const long long t0 = clock64();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (__any_sync(0xffffffffu, *abort != 0)) return false;
        if (__any_sync(0xffffffffu, clock64() - t0 > kWaitLimitCycles)) {
            if ((threadIdx.x & 31) == 0) {
                *abort = 1;
                set_status(status, ORTHROS_DEV_TIMEOUT);
            }
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag: used while draining (waiting for
// copies or MMAs this thread already issued) so that nothing is left in flight
// when the CTA releases its shared and tensor memory.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity, uint32_t *status) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) {
            set_status(status, ORTHROS_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ----------------------------------------------------------------------------
// proxy fences
// ----------------------------------------------------------------------------
// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tensor core) once ordered by a barrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// TMA (tiled bulk tensor copies, global -> shared, mbarrier completion)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                            int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                            int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// shared -> global tiled store (bulk-group completion); the source must not be
// overwritten before bulk_wait_read().
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *smem_src, int c0, int c1, int c2,
                                             int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of this thread has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core (cta_group::1)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrives (once) on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T  (kind::f16: fp16 or bf16 operands, fp32 accumulate)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle, sm_100 layout version 1.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  version (1)
//   bits 61-63  layout: 2 = SWIZZLE_128B
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16 (dense): D fp32; a_fmt/b_fmt 0 = f16,
// 1 = bf16; a_mn/b_mn: operand is MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t a_fmt, uint32_t b_fmt, uint32_t a_mn, uint32_t b_mn,
                                                 uint32_t M, uint32_t N) {
    return (1u << 4)             // D format: f32
           | (a_fmt << 7)        // A format
           | (b_fmt << 10)       // B format
           | (a_mn << 15)        // A major
           | (b_mn << 16)        // B major
           | ((N >> 3) << 17)    // N / 8
           | ((M >> 4) << 24);   // M / 16
}

// 32 lanes x 32 bits, 32 consecutive columns: thread t of the warp receives
// lane (warp's lane quarter + t), columns [taddr.col, taddr.col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// One 32-bit column: thread t of the warp writes / reads lane (warp's lane quarter + t).
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
    uint32_t v;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr));
    return v;
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// fp32 reduction into global memory (no return value).
__device__ __forceinline__ void red_add_f32(float *addr, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// ----------------------------------------------------------------------------
// math
// ----------------------------------------------------------------------------
// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed pairs of floats (sm_100 and later: one instruction for two fp32
// fused multiply-adds or adds, each rounded as its scalar form).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
// (d0, d1) = (x0, x1) * b + c, b and c given as packed pairs
__device__ __forceinline__ void fma_f32x2(float x0, float x1, uint64_t b, uint64_t c, float &d0, float &d1) {
    asm("{\n\t.reg .b64 xv, r;\n\tmov.b64 xv, {%2, %3};\n\tfma.rn.f32x2 r, xv, %4, %5;\n\tmov.b64 {%0, %1}, r;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(x0), "f"(x1), "l"(b), "l"(c));
}
// (a0, a1) += (p0, p1)
__device__ __forceinline__ void add_f32x2(float &a0, float &a1, float p0, float p1) {
    asm("{\n\t.reg .b64 av, pv;\n\tmov.b64 av, {%0, %1};\n\tmov.b64 pv, {%2, %3};\n\tadd.rn.f32x2 av, av, pv;\n\t"
        "mov.b64 {%0, %1}, av;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(p0), "f"(p1));
}

// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1), one packed instruction
__device__ __forceinline__ void fma2(float a0, float a1, float b0, float b1, float c0, float c1, float &d0,
                                     float &d1) {
    asm("{\n\t.reg .b64 av, bv, cv, r;\n\tmov.b64 av, {%2, %3};\n\tmov.b64 bv, {%4, %5};\n\t"
        "mov.b64 cv, {%6, %7};\n\tfma.rn.f32x2 r, av, bv, cv;\n\tmov.b64 {%0, %1}, r;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
// (d0, d1) = (a0, a1) * (b0, b1), one packed instruction
__device__ __forceinline__ void mul2(float a0, float a1, float b0, float b1, float &d0, float &d1) {
    asm("{\n\t.reg .b64 av, bv, r;\n\tmov.b64 av, {%2, %3};\n\tmov.b64 bv, {%4, %5};\n\t"
        "mul.rn.f32x2 r, av, bv;\n\tmov.b64 {%0, %1}, r;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// 2^x with the hardware approximation (ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^a for a pair of values on the FMA and integer pipes instead of the
// special-function unit. Method (classical range reduction): j = a rounded to
// the nearest integer (adding 1.5 * 2^23 leaves j in the low mantissa bits of
// the sum), f = a - j in [-1/2, 1/2], 2^f from a cubic in Horner form, and j
// added to the exponent field of the result. The cubic's coefficients are a
// near-minimax fit of 2^f on [-1/2, 1/2] in relative error (Lawson's
// iteratively reweighted least squares): 7.5e-5 at most, 26 times below the
// bf16 rounding that P goes through. Inputs are first raised to -127 (NaN
// kept): -inf and everything at or below -127 give exactly +0 (the integer sum
// turns negative there and is clamped to zero), inputs between -127 and -126 a
// subnormal, and a NaN input gives NaN.
__device__ __forceinline__ void exp2_fma_x2(float a0, float a1, float &p0, float &p1) {
    uint32_t r0, r1;
    asm("{\n\t"
        ".reg .b64 av, tv, rv, fv, pv, kv;\n\t"
        ".reg .b32 k, t0, t1, q0, q1, x0, x1;\n\t"
        ".reg .pred n0, n1;\n\t"
        "max.NaN.f32 x0, %2, 0fC2FE0000;\n\t"  // -127
        "max.NaN.f32 x1, %3, 0fC2FE0000;\n\t"
        "mov.b64 av, {x0, x1};\n\t"
        "mov.b32 k, 0f4B400000;\n\t"  // 1.5 * 2^23
        "mov.b64 kv, {k, k};\n\t"
        "add.rn.f32x2 tv, av, kv;\n\t"
        "sub.rn.f32x2 rv, tv, kv;\n\t"  // j
        "sub.rn.f32x2 fv, av, rv;\n\t"  // f, exact
        "mov.b32 k, 0f3D61FBB0;\n\t"    // c3 = 0.05517167
        "mov.b64 pv, {k, k};\n\t"
        "mov.b32 k, 0f3E786F0E;\n\t"    // c2 = 0.24261114
        "mov.b64 kv, {k, k};\n\t"
        "fma.rn.f32x2 pv, pv, fv, kv;\n\t"
        "mov.b32 k, 0f3F31798D;\n\t"    // c1 = 0.69326097
        "mov.b64 kv, {k, k};\n\t"
        "fma.rn.f32x2 pv, pv, fv, kv;\n\t"
        "mov.b32 k, 0f3F7FFB49;\n\t"    // c0 = 0.99992806
        "mov.b64 kv, {k, k};\n\t"
        "fma.rn.f32x2 pv, pv, fv, kv;\n\t"
        "mov.b64 {t0, t1}, tv;\n\t"
        "mov.b64 {q0, q1}, pv;\n\t"
        // bits(sum) << 23 is j << 23 modulo 2^32: the exponent field moves by j
        "mad.lo.u32 x0, t0, 8388608, q0;\n\t"
        "mad.lo.u32 x1, t1, 8388608, q1;\n\t"
        "max.s32 x0, x0, 0;\n\t"
        "max.s32 x1, x1, 0;\n\t"
        "testp.notanumber.f32 n0, %2;\n\t"
        "testp.notanumber.f32 n1, %3;\n\t"
        "selp.b32 %0, 2147483647, x0, n0;\n\t"
        "selp.b32 %1, 2147483647, x1, n1;\n\t"
        "}"
        : "=r"(r0), "=r"(r1)
        : "f"(a0), "f"(a1));
    p0 = __uint_as_float(r0);
    p1 = __uint_as_float(r1);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace ptx
}  // namespace orthros
