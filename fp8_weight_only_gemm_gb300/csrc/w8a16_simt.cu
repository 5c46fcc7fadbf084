// CUDA-core W8A16 kernel: one warp per weight row, no tensor cores.
//
// It follows the page "metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs"
// in decoding E4M3 through a 256-entry shared-memory table (doc comment of
// `W8A16_M32_SMEM_BYTES`) and in folding the block scale at K-step granularity
// (doc comment of `W8A16_M32_K_BLOCK`). It is the plain GPU formulation of the
// operation: a second, structurally different GPU path that the tensor-core
// variant is cross-checked against, and the planner's choice for calls too small
// to fill a tensor-core tile.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "w8a16_internal.h"

namespace w8a16 {

namespace {

constexpr uint32_t kSimtWarps = 8;    // weight rows per CTA
constexpr uint32_t kSimtTokens = 8;   // A rows per CTA (grid.y tiles the rest)

// E4M3 "FN" value of a code, built from the bit fields: exponent field 0 is
// subnormal (m * 2^-9); otherwise the FP32 pattern with exponent e - 7 + 127 and
// the 3 mantissa bits on top of FP32's mantissa; 0x7F/0xFF are NaN.
__device__ float e4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 0xFu, m = c & 0x7u;
    float v;
    if (e == 0xFu && m == 0x7u)
        v = __int_as_float(0x7FC00000);
    else if (e == 0u)
        v = static_cast<float>(m) * 0x1p-9f;
    else
        v = __int_as_float(static_cast<int>(((e + 120u) << 23) | (m << 20)));
    return (c & 0x80u) ? -v : v;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__global__ void __launch_bounds__(kSimtWarps * 32)
    w8a16_simt_kernel(const __nv_bfloat16* __restrict__ A, uint32_t lda,
                      const uint8_t* __restrict__ W, const float* __restrict__ scale,
                      __nv_bfloat16* __restrict__ C, uint32_t ldc, uint32_t M, uint32_t N,
                      uint32_t K) {
    __shared__ float lut[256];
    for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) lut[i] = e4m3_value(i);
    // Under a programmatic launch, wait for the previous grid before touching
    // memory it may write (a no-op otherwise), and let the next one be scheduled.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t n = blockIdx.x * kSimtWarps + warp;
    const uint32_t m0 = blockIdx.y * kSimtTokens;
    if (n >= N) return;
    const uint32_t mt = min(kSimtTokens, M - m0);
    const uint8_t* wrow = W + static_cast<size_t>(n) * K;
    const float* srow = scale + static_cast<size_t>(n / 128) * (K / 128);

    float acc[kSimtTokens];
#pragma unroll
    for (uint32_t t = 0; t < kSimtTokens; ++t) acc[t] = 0.f;

    // Lane l covers k in [16 l, 16 l + 16) of every 512-wide chunk: 16 codes, all
    // inside one 128-K scale block. Its 16-term partial is folded into the FP32
    // accumulator with that block's scale.
    for (uint32_t kc = lane * 16; kc < K; kc += 512) {
        const uint4 q = ldg_stream(wrow + kc);
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
        float w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = lut[(words[i >> 2] >> (8 * (i & 3))) & 0xFFu];
        const float s = __ldg(srow + kc / 128);
#pragma unroll
        for (uint32_t t = 0; t < kSimtTokens; ++t) {
            if (t < mt) {
                const __nv_bfloat16* arow = A + static_cast<size_t>(m0 + t) * lda + kc;
                const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(arow));
                const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(arow) + 1);
                const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                float p = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[i]));
                    p = fmaf(f.x, w[2 * i], p);
                    p = fmaf(f.y, w[2 * i + 1], p);
                }
                acc[t] = fmaf(s, p, acc[t]);
            }
        }
    }
    // Fixed butterfly order across lanes: the result does not depend on timing.
#pragma unroll
    for (uint32_t t = 0; t < kSimtTokens; ++t) {
        float v = acc[t];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0 && t < mt) C[static_cast<size_t>(m0 + t) * ldc + n] = __float2bfloat16_rn(v);
    }
}

}  // namespace

int launch_simt(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint32_t flags,
                std::string* err) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(p.grid[0], p.grid[1], 1);
    cfg.blockDim = dim3(p.block[0], 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = (flags & W8A16_FLAG_PDL) ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, w8a16_simt_kernel, static_cast<const __nv_bfloat16*>(g.A),
                                       g.lda, static_cast<const uint8_t*>(g.W), g.scale,
                                       static_cast<__nv_bfloat16*>(g.C), g.ldc, g.M, g.N, g.K);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("SIMT kernel launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
}

}  // namespace w8a16
