// Cluster split-K and FP8 tensor-core helpers shared by the tensor-core kernels.
#pragma once
#include <cstdint>

#include "w8a16_device.cuh"
#include "w8a16_internal.h"

namespace w8a16 {

// Relaxed arrive: the only state peers touch before the matching wait is the
// receive mbarrier, whose initialisation fence.mbarrier_init already releases to
// the cluster. A release arrive would also wait for this CTA's in-flight weight
// loads, holding the activation producer back by about a microsecond.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// Release arrive, for a CTA whose shared memory peers may write once the barrier
// completes (its loads and MMAs on that memory have all been waited for).
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_async_v4f32(uint32_t remote_addr, uint32_t remote_bar, float a,
                                               float b, float c, float d) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
            remote_addr),
        "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
        : "memory");
}
// Bytes one fold thread pushes per row: its token group's valid tokens, rounded up
// to whole 16-byte groups of 4.
__device__ __forceinline__ uint32_t push_bytes(uint32_t toks_valid, uint32_t first, uint32_t count) {
    const uint32_t v = toks_valid > first ? min(toks_valid - first, count) : 0u;
    return 16u * ((v + 3u) / 4u);
}
template <uint32_t TN, uint32_t TPF>
__device__ __forceinline__ uint32_t red_row_bytes(uint32_t toks_valid) {
    uint32_t b = 0;
#pragma unroll
    for (uint32_t first = 0; first < TN; first += TPF) b += push_bytes(toks_valid, first, TPF);
    return b;
}
__device__ __forceinline__ uint32_t owned_row0(uint32_t r, uint32_t split_k) {
    return r * kTcRows / split_k;
}
// Generic-proxy shared-memory writes become visible to the tensor core's reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Instruction descriptor, kind::f8f6f4: E4M3 A and B, FP32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t m, uint32_t n) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}
// The same product with A (the weight rows) read from TMEM: lane r holds row r, and
// column c of a K=32 slab holds its K bytes 4c..4c+3 (byte j = element 4c+j).
__device__ __forceinline__ void tc_mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

}  // namespace w8a16
