// Device-side primitives for the sm_103a W8A16 kernels: bounded mbarrier waits,
// TMA tile loads, tcgen05 (TMEM allocation, MMA, loads/stores) and the exact
// E4M3 -> BF16 conversion. Inline PTX only; no CUTLASS/CuTe.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "w8a16_internal.h"

namespace w8a16 {

// ---------------------------------------------------------------- status --
// First failure recorded by any kernel of this translation unit (0 = none).
// A file-scope device variable: one copy per device that loads the library.
struct DeviceStatus {
    unsigned int code;   // W8A16_STATUS_* of the first failure
    unsigned int where;  // blockIdx.x | blockIdx.y << 16 of the CTA that failed
    unsigned int detail; // kernel-specific (barrier, step)
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void record_failure(DeviceStatus* st, unsigned int code,
                                               unsigned int detail) {
    if (atomicCAS(&st->code, 0u, code) == 0u) {
        st->where = blockIdx.x | (blockIdx.y << 16);
        st->detail = detail;
        __threadfence();
    }
}

// ------------------------------------------------------------- mbarriers --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Acquire at cluster scope: for a barrier whose transactions are other CTAs'
// st.async writes (their complete-tx releases at cluster scope, which a
// CTA-scope acquire does not synchronise with).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed. Gives up when the
// CTA's abort flag is raised or the deadline passes (then raises the flag and
// records the failure); returns false in both cases. Every wait in these
// kernels goes through here, so no wait can spin forever. CLUSTER: acquire at
// cluster scope (the split-K receive barriers).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t deadline,
                                          volatile int* abort_flag, DeviceStatus* st,
                                          unsigned int detail) {
    const auto try_wait = [](uint32_t b, uint32_t ph) {
        return CLUSTER ? mbar_try_wait_cluster(b, ph) : mbar_try_wait(b, ph);
    };
    if (try_wait(bar, parity)) return true;
    uint32_t spins = 0;
    while (true) {
        if (try_wait(bar, parity)) return true;
        if ((++spins & 63u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() > deadline) {
                *abort_flag = 1;
                record_failure(st, W8A16_STATUS_WAIT_TIMEOUT, detail);
                return false;
            }
        }
    }
}

// 16-byte asynchronous copy global -> shared through L2 only (the source may have
// been written by the previous grid), and its group bookkeeping.
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A 32-bit load with acquire semantics at GPU scope (pairs with a release by
// another CTA: a fence before an atomic).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A barrier among `count` threads (whole warps) of the CTA on hardware barrier
// `id` (0 is __syncthreads').
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------ programmatic launches --
// Wait for the grids this one depends on (a no-op unless it was launched as a
// programmatic dependent), and allow dependents to be scheduled.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait for the grids this one depends on, then start the time limit of the
// calling role's bounded waits. A role calls this before its first wait on
// anything downstream of the dependency (the activations, the MMAs that read
// them), so the time a programmatic launch spends behind a long predecessor is
// not charged to that limit.
__device__ __forceinline__ uint64_t deadline_after_dependency(uint64_t timeout_ns) {
    grid_dependency_wait();
    return globaltimer_ns() + timeout_ns;
}

// ------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (x = inner coordinate, y) into shared memory,
// completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
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

// --------------------------------------------------------------- tcgen05 --
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

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16 (BF16 inputs, FP32 accumulate).
__device__ __forceinline__ void tc_mma_a_tmem(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i writes lane (base lane + i).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand stored as
// 8-row x 128-byte swizzle atoms (128-byte swizzle), atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version (tcgen05)
    d |= static_cast<uint64_t>(2) << 61;                    // swizzle: 128-byte
    return d;
}

// Instruction descriptor, kind::f16: BF16 A and B, FP32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t m, uint32_t n) {
    return (1u << 4)                // D format: F32
           | (1u << 7)              // A format: BF16
           | (1u << 10)             // B format: BF16
           | ((n >> 3) << 17)       // N / 8
           | ((m >> 4) << 24);      // M / 16
}

// ------------------------------------------------------- packed FP32 pairs --
// sm_100+ executes two FP32 operations per instruction on register pairs; each lane
// is the IEEE operation with round-to-nearest-even, so these give the bits of the
// scalar fmaf / __fmul_rn on each half.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
// a * b + c on both halves
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// a * b on both halves
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------- E4M3 -> BF16 --
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Exact conversion of four E4M3 codes (one 32-bit word, code i in byte i) to
// two BF16x2 words: lo = (code0, code1), hi = (code2, code3), first code in the
// low half.
//
// BF16 and E4M3 both store sign | exponent | mantissa. Moving an E4M3 code's 7
// exponent+mantissa bits up by 4 and its sign up by 8 gives a BF16 pattern whose
// value is the E4M3 value times 2^-120 (exponent bias 127 versus 7); E4M3
// subnormals land on BF16 subnormals with the same mantissa, so the scaling is
// exact there too, and one BF16 multiply by 2^120 (an exact power of two; the
// result is always normal or zero) restores the value. prmt with sign
// replication puts each code in its own 16-bit half as [sign byte | code];
// shifting that left by 4 leaves the sign at bit 15, copies of it at bits
// 14..11 (cleared by the mask) and the payload at bits 10..4.
//
// The NaN codes 0x7F/0xFF would come out as +-480 this way, so words holding
// one are patched to the BF16 NaN 0x7FC0 (a byte is a NaN code exactly when its
// low 7 bits plus one carry into bit 7).
__device__ __forceinline__ uint32_t e4m3_nan_flags(uint32_t w) {
    return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}

__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    constexpr uint32_t k2p120 = 0x7B807B80u;  // BF16x2 (2^120, 2^120)
    const uint32_t p01 = prmt(w, 0, 0x9180);  // [sx(c1) c1 sx(c0) c0]
    const uint32_t p23 = prmt(w, 0, 0xB3A2);  // [sx(c3) c3 sx(c2) c2]
    lo = bf16x2_mul((p01 << 4) & 0x87F087F0u, k2p120);
    hi = bf16x2_mul((p23 << 4) & 0x87F087F0u, k2p120);
}

__device__ __forceinline__ void e4m3x4_patch_nan(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t f = e4m3_nan_flags(w);
    lo |= prmt(f, 0, 0x9988) & 0x7FC07FC0u;   // 0xFFFF per half whose code is NaN
    hi |= prmt(f, 0, 0xBBAA) & 0x7FC07FC0u;
}

// 16 codes -> 8 BF16x2 words, NaN codes patched (rare path, one branch).
__device__ __forceinline__ void e4m3x16_to_bf16x16(const uint4& q, uint32_t (&o)[8]) {
    e4m3x4_to_bf16x4(q.x, o[0], o[1]);
    e4m3x4_to_bf16x4(q.y, o[2], o[3]);
    e4m3x4_to_bf16x4(q.z, o[4], o[5]);
    e4m3x4_to_bf16x4(q.w, o[6], o[7]);
    const uint32_t any = e4m3_nan_flags(q.x) | e4m3_nan_flags(q.y) | e4m3_nan_flags(q.z) |
                         e4m3_nan_flags(q.w);
    if (__builtin_expect(any != 0u, 0)) {
        e4m3x4_patch_nan(q.x, o[0], o[1]);
        e4m3x4_patch_nan(q.y, o[2], o[3]);
        e4m3x4_patch_nan(q.z, o[4], o[5]);
        e4m3x4_patch_nan(q.w, o[6], o[7]);
    }
}

}  // namespace w8a16
