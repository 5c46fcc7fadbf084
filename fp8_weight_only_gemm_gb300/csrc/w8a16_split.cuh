// The two-term E4M3 split of BF16 activations, shared by the kernel that splits
// its activation tiles itself (w8a16_tc8.cu) and the split pre-pass
// (w8a16_quant.cu) that feeds the same arithmetic through a workspace.
//
// Per token and 128-K block: E = floor(log2(max |a|)), x = a * 2^(7-E) (exact,
// |x| < 256), hi = e4m3_rne(x), lo = e4m3_rne(32 (x - hi)); then x = hi + lo / 32
// exactly for every a with |a| >= 2^-14 max |a| and within 2^-22 max |a|
// otherwise, and the product of a weight row with the block is recovered in
// FP32 as 2^(E-7) * (P_hi + P_lo / 32).
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace w8a16 {
namespace {

// Two FP32 values to E4M3 (round to nearest even, saturating): lo in byte 0.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// Two E4M3 codes (byte 0 and 1) back to FP32.
__device__ __forceinline__ void e4m3x2_to_f32x2(uint32_t codes, float& lo, float& hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(codes)));
    const __half2 v = *reinterpret_cast<const __half2*>(&h2);
    lo = __low2float(v);
    hi = __high2float(v);
}

// E = floor(log2(mx)) of a block maximum from its bits (mx may be an FP32 subnormal).
__device__ __forceinline__ int block_exponent(float mx) {
    const uint32_t mb = __float_as_uint(mx);
    const int ef = static_cast<int>(mb >> 23);
    return ef != 0 ? ef - 127 : (mb != 0 ? -118 - __clz(mb) : 0);
}
// 2^(7-E) as two exact FP32 powers of two (7 - E spans -120..156).
__device__ __forceinline__ void split_scales(int E, float& p1, float& p2) {
    const int e1 = (7 - E) / 2, e2 = (7 - E) - e1;
    p1 = __int_as_float((127 + e1) << 23);
    p2 = __int_as_float((127 + e2) << 23);
}
// 2^(E-7) as FP32 (subnormal or zero for very small blocks); 0 for an all-zero block.
__device__ __forceinline__ float fold_factor(int E, float mx) {
    const int ie = E - 7;
    if (!(mx > 0.f)) return 0.f;
    return ie >= -126 ? __int_as_float((127 + ie) << 23)
                      : (ie >= -149 ? __int_as_float(1 << (ie + 149)) : 0.f);
}
// hi/lo E4M3 codes of four consecutive scaled values (byte i = value i).
__device__ __forceinline__ void two_terms4(const float* x, uint32_t& hw, uint32_t& lw) {
    const uint32_t h0 = f32x2_to_e4m3x2(x[0], x[1]), h1 = f32x2_to_e4m3x2(x[2], x[3]);
    float hf[4];   // the hi terms' values (exact)
    e4m3x2_to_f32x2(h0, hf[0], hf[1]);
    e4m3x2_to_f32x2(h1, hf[2], hf[3]);
    const uint32_t l0 = f32x2_to_e4m3x2((x[0] - hf[0]) * 32.f, (x[1] - hf[1]) * 32.f);
    const uint32_t l1 = f32x2_to_e4m3x2((x[2] - hf[2]) * 32.f, (x[3] - hf[3]) * 32.f);
    hw = h0 | (h1 << 16);
    lw = l0 | (l1 << 16);
}

}  // namespace
}  // namespace w8a16
