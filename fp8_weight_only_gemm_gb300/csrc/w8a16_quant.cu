// Block quantisers for sm_103a. Weights: FP32 or BF16 W -> E4M3 codes + one FP32
// scale per 128x128 block, the format the W8A16 GEMM consumes (page
// "metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs", doc comment of
// `w8a16_gemm_pipelined_m32_strided`: W as FP8 E4M3 [N, K], block_scale FP32
// [N/128, K/128]). Per block: amax = max |w|, scale = amax / 448 (FP32, round to
// nearest), code = E4M3 round-to-nearest-even of w / scale (FP32 quotient,
// saturating at +-448); amax = 0 gives scale 0 and codes 0. NaN inputs do not
// enter amax (fmax ignores them) and encode as the NaN code.
//
// One CTA per block, 8 warps x 16 rows, a lane per 4 consecutive columns: each
// warp instruction reads one 512-byte (FP32) or 256-byte (BF16) row segment and
// writes 128 code bytes. The block's values stay in registers between the
// maximum and the encoding, so W is read once: the kernel is bound by HBM.
//
// Activations (the W8A8 variant's first half; page "metrale_model_layers/layers/
// ops/fp8_act_quant.rs", module doc: per-token 128-element K groups): the same
// rule on 1 x 128 groups, a warp per group. It is queued as a programmatic
// dependent launch: its CTAs may start while the previous kernel of the stream
// runs and wait for that kernel's completion before touching memory; then they
// let the next kernel (a W8A8 GEMM queued with W8A16_FLAG_PDL) start its weight
// prefetch, and that kernel's own dependency wait covers these outputs.
//
// Two-term split (the W8A16 path through the FP8 x FP8 kernel): the same launch
// shape, each group written as hi and lo E4M3 codes with its factor 2^(E-7)
// (w8a16_split.cuh), into the workspace layout codes [2M][K], factors
// [K/128][stride].
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <string>

#include "w8a16_device.cuh"
#include "w8a16_internal.h"
#include "w8a16_split.cuh"

namespace w8a16 {
namespace {

constexpr uint32_t kQRows = 128, kQCols = 128, kQWarps = 8, kQRowsPerWarp = kQRows / kQWarps;

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {   // lo -> byte 0
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <bool BF16>
__global__ void __launch_bounds__(kQWarps * 32)
    quantize_blocks_kernel(const void* __restrict__ W, uint32_t ldw, uint32_t N, uint32_t K,
                           uint8_t* __restrict__ codes, float* __restrict__ scales) {
    __shared__ float warp_max[kQWarps];
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t kb = blockIdx.x, nb = blockIdx.y;
    const uint32_t col = kb * kQCols + 4 * lane;
    const uint32_t row0 = nb * kQRows + warp * kQRowsPerWarp;
    float v[kQRowsPerWarp][4];
    float mx = 0.f;
#pragma unroll
    for (uint32_t r = 0; r < kQRowsPerWarp; ++r) {
        const uint32_t row = row0 + r;
        if (row < N) {
            const size_t off = static_cast<size_t>(row) * ldw + col;
            if constexpr (BF16) {
                const uint2 q = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(W) + off);
                v[r][0] = __uint_as_float(q.x << 16);
                v[r][1] = __uint_as_float(q.x & 0xFFFF0000u);
                v[r][2] = __uint_as_float(q.y << 16);
                v[r][3] = __uint_as_float(q.y & 0xFFFF0000u);
            } else {
                const float4 q = *reinterpret_cast<const float4*>(static_cast<const float*>(W) + off);
                v[r][0] = q.x;
                v[r][1] = q.y;
                v[r][2] = q.z;
                v[r][3] = q.w;
            }
        } else {
            v[r][0] = v[r][1] = v[r][2] = v[r][3] = 0.f;
        }
#pragma unroll
        for (uint32_t e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(v[r][e]));
    }
#pragma unroll
    for (uint32_t o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (lane == 0) warp_max[warp] = mx;
    __syncthreads();
    float amax = warp_max[0];
#pragma unroll
    for (uint32_t w = 1; w < kQWarps; ++w) amax = fmaxf(amax, warp_max[w]);
    const float scale = __fdiv_rn(amax, 448.f);
    if (threadIdx.x == 0) scales[static_cast<size_t>(nb) * (K / kQCols) + kb] = scale;
#pragma unroll
    for (uint32_t r = 0; r < kQRowsPerWarp; ++r) {
        const uint32_t row = row0 + r;
        if (row >= N) break;
        uint32_t word = 0;
        if (scale != 0.f)
            word = e4m3x2(__fdiv_rn(v[r][0], scale), __fdiv_rn(v[r][1], scale)) |
                   (e4m3x2(__fdiv_rn(v[r][2], scale), __fdiv_rn(v[r][3], scale)) << 16);
        *reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(row) * K + col) = word;
    }
}

// Per-token 128-K groups of BF16 activations: a warp per (token, group), a lane
// per 4 values. scales are K-group major: scales[g * scale_stride + m].
__global__ void __launch_bounds__(256)
    quantize_act_kernel(const uint16_t* __restrict__ A, uint32_t lda, uint32_t M, uint32_t K,
                        uint8_t* __restrict__ codes, float* __restrict__ scales, uint32_t scale_stride) {
    grid_dependency_wait();   // A may be the previous kernel's output; codes may be its input
    // only now may the next kernel start: it then overlaps this grid alone, which
    // writes neither its weights nor their scales
    grid_launch_dependents();
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t item = static_cast<uint64_t>(blockIdx.x) * 8u + (threadIdx.x >> 5);
    const uint32_t groups = K / kQCols;
    if (item >= static_cast<uint64_t>(M) * groups) return;
    const uint32_t m = static_cast<uint32_t>(item / groups), g = static_cast<uint32_t>(item % groups);
    const uint32_t col = g * kQCols + 4 * lane;
    const uint2 q = *reinterpret_cast<const uint2*>(A + static_cast<size_t>(m) * lda + col);
    const float v[4] = {__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                        __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u)};
    float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (uint32_t o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    const float scale = __fdiv_rn(mx, 448.f);
    uint32_t word = 0;
    if (scale != 0.f)
        word = e4m3x2(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale)) |
               (e4m3x2(__fdiv_rn(v[2], scale), __fdiv_rn(v[3], scale)) << 16);
    *reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(m) * K + col) = word;
    if (lane == 0) scales[static_cast<size_t>(g) * scale_stride + m] = scale;
}

// A warp per (token, group), lane l holding K 4l..4l+3: the block maximum over
// the finite values (a non-finite value makes the lane's hi codes NaN, so the
// token's outputs are NaN), then the split of the four values.
__global__ void __launch_bounds__(256)
    split_act_kernel(const uint16_t* __restrict__ A, uint32_t lda, uint32_t M, uint32_t K,
                     uint8_t* __restrict__ codes, float* __restrict__ factors, uint32_t factor_stride,
                     uint32_t* __restrict__ counters, uint32_t ncounters) {
    grid_dependency_wait();   // A may be the previous kernel's output; the workspace its input
    grid_launch_dependents();
    // the stream-K tile counters of the GEMM that follows start at zero
    for (uint64_t c = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < ncounters;
         c += static_cast<uint64_t>(gridDim.x) * blockDim.x)
        counters[c] = 0u;
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t item = static_cast<uint64_t>(blockIdx.x) * 8u + (threadIdx.x >> 5);
    const uint32_t groups = K / kQCols;
    if (item >= static_cast<uint64_t>(M) * groups) return;
    const uint32_t m = static_cast<uint32_t>(item / groups), g = static_cast<uint32_t>(item % groups);
    const uint32_t col = g * kQCols + 4 * lane;
    const uint2 q = *reinterpret_cast<const uint2*>(A + static_cast<size_t>(m) * lda + col);
    float x[4] = {__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                  __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u)};
    float mx = 0.f;
    bool bad = false;
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) {
        const float a = fabsf(x[e]);
        if (a <= 3.4028235e38f) mx = fmaxf(mx, a);
        else bad = true;   // NaN or infinity
    }
    mx = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mx)));   // |x| orders as its bits
    const int E = block_exponent(mx);
    float p1, p2;
    split_scales(E, p1, p2);
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) x[e] = (x[e] * p1) * p2;
    uint32_t hw, lw;
    two_terms4(x, hw, lw);
    if (bad) hw = 0x7F7F7F7Fu;
    *reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(m) * K + col) = hw;
    *reinterpret_cast<uint32_t*>(codes + (static_cast<size_t>(M) + m) * K + col) = lw;
    if (lane == 0) factors[static_cast<size_t>(g) * factor_stride + m] = fold_factor(E, mx);
}

}  // namespace

int launch_split_act(const void* A, uint32_t lda, uint32_t M, uint32_t K, void* codes, float* factors,
                     uint32_t factor_stride, uint32_t* counters, uint32_t ncounters, cudaStream_t s,
                     std::string* err) {
    const uint64_t items = static_cast<uint64_t>(M) * (K / kQCols);
    const uint64_t blocks = (items + 7) / 8;
    if (blocks > 0x7FFFFFFFull) {
        *err = "activation split: too many groups";
        return W8A16_ERR_RANGE;
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, split_act_kernel, static_cast<const uint16_t*>(A), lda, M, K,
                                       static_cast<uint8_t*>(codes), factors, factor_stride, counters,
                                       ncounters);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("activation split launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
}

int launch_quantize_act(const void* A, uint32_t lda, uint32_t M, uint32_t K, void* codes, float* scales,
                        uint32_t scale_stride, cudaStream_t s, std::string* err) {
    const uint64_t items = static_cast<uint64_t>(M) * (K / kQCols);
    const uint64_t blocks = (items + 7) / 8;
    if (blocks > 0x7FFFFFFFull) {
        *err = "activation quantiser: too many groups";
        return W8A16_ERR_RANGE;
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_act_kernel, static_cast<const uint16_t*>(A), lda, M, K,
                                       static_cast<uint8_t*>(codes), scales, scale_stride);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("activation quantiser launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
}

int launch_quantize(const void* W, bool bf16, uint32_t ldw, uint32_t N, uint32_t K, void* codes,
                    float* scales, cudaStream_t s, std::string* err) {
    const dim3 grid(K / kQCols, (N + kQRows - 1) / kQRows, 1);
    if (bf16)
        quantize_blocks_kernel<true><<<grid, kQWarps * 32, 0, s>>>(W, ldw, N, K,
                                                                   static_cast<uint8_t*>(codes), scales);
    else
        quantize_blocks_kernel<false><<<grid, kQWarps * 32, 0, s>>>(W, ldw, N, K,
                                                                    static_cast<uint8_t*>(codes), scales);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("quantiser launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
}

}  // namespace w8a16
