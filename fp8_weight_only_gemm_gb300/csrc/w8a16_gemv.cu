// Decode-sized W8A16 kernel for sm_103a: one or two tokens, every CTA's weight
// share on chip before the grid-dependency wait (tcgen05.mma kind::f8f6f4 + TMA).
//
// Same operation, arithmetic and reduction order as the two-term FP8 kernel
// (page "metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs": one FP32
// fold of the block scale per 128-K step, split-K partials added in step order;
// each BF16 activation enters the tensor core as two E4M3 terms, hi + lo / 32,
// scaled by 2^(E-7) per token and 128-K block). What differs is the schedule,
// made for decode, where a call streams a few MiB of weights and the work after
// the dependency wait sets the rate of back-to-back calls:
//
//   * a cluster of split_k CTAs per 128-row weight tile, each on at most 8 K
//     steps, and at most one CTA per SM for the whole grid (the planner's rule),
//     so the CTAs of the next call fit beside this call's (two per SM: below
//     113 KiB of shared memory and 128 TMEM columns each);
//   * every weight tile-step of the CTA is requested before the dependency wait:
//     five 16 KiB shared-memory slots, and the first steps are copied into TMEM
//     (the MMA reads them there), which frees their slots for the last ones;
//   * after the wait, warp w splits the activations of step w and issues that
//     step's 4 MMAs; the steps write disjoint column pairs of one 16-column
//     accumulator (the B rows of the other steps are zero), so one TMEM read after
//     the last MMA holds every step's product for the fold, which then runs in
//     step order exactly as the two-term kernel's does;
//   * split-K partials go to the rank that owns the row over distributed shared
//     memory and are summed in rank (= K) order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "w8a16_cluster.cuh"
#include "w8a16_device.cuh"
#include "w8a16_internal.h"
#include "w8a16_split.cuh"

namespace w8a16 {

__device__ DeviceStatus g_gemv_status;

namespace {

constexpr uint32_t kWTileBytes = kTcRows * kKStep;   // 16 KiB of E4M3 per tile-step

enum : uint32_t {
    kWaitW = 41, kWaitMoved = 42, kWaitAccZero = 43, kWaitMma = 44, kWaitFact = 45, kWaitRed = 46,
    kWaitOwn = 47
};

// barriers: wfull[slots], moved[resident], acc zeroed, all MMAs, all factors,
// split-K receive, own[8] (each issuing warp's MMAs, waited for before TMEM is freed)
constexpr uint32_t kNumBars = kGvSlots + kGvResident + 4 + kGvMaxSteps;
static_assert(kNumBars * 8 + 8 <= 256, "barrier area");
static_assert(kGvThreads / 32 == kGvMaxSteps, "one warp per step");

__device__ __forceinline__ bool gv_warp_wait(uint32_t bar, uint32_t parity, uint64_t deadline,
                                             volatile int* abort_flag, uint32_t detail) {
    const bool ok = mbar_wait(bar, parity, deadline, abort_flag, &g_gemv_status, detail);
    return __all_sync(0xFFFFFFFFu, ok);
}

// One token's 128-K block split on the whole warp (lane l holds K 4l..4l+3 as four
// BF16 values, lowest K first): the hi codes go to row rh, the lo codes to row rl
// of a 128-byte-row operand with the 128-byte swizzle; returns the fold factor
// 2^(E-7) (0 for an all-zero block). A non-finite value makes the hi codes NaN.
__device__ __forceinline__ float split_block_w32(uint2 av, uint8_t* bs, uint32_t rh, uint32_t rl,
                                                 uint32_t lane) {
    float x[4] = {__uint_as_float(av.x << 16), __uint_as_float(av.x & 0xFFFF0000u),
                  __uint_as_float(av.y << 16), __uint_as_float(av.y & 0xFFFF0000u)};
    float mx = 0.f;
    bool bad = false;
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) {
        const float a = fabsf(x[e]);
        if (a <= 3.4028235e38f) mx = fmaxf(mx, a);
        else bad = true;   // NaN or infinity
    }
    // the block maximum: |x| >= 0 orders as its bit pattern
    mx = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mx)));
    bad = __any_sync(0xFFFFFFFFu, bad);
    const int E = block_exponent(mx);
    float p1, p2;
    split_scales(E, p1, p2);
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) x[e] = (x[e] * p1) * p2;
    uint32_t hw, lw;
    two_terms4(x, hw, lw);
    if (bad) hw = 0x7F7F7F7Fu;   // a non-finite value: NaN codes for the whole block
    // 4 bytes at K 4l: 16-byte chunk l / 4, stored at chunk (l / 4) ^ (row & 7)
    const uint32_t in_chunk = (lane & 3u) << 2;
    *reinterpret_cast<uint32_t*>(bs + rh * 128u + ((((lane >> 2) ^ (rh & 7u)) << 4) + in_chunk)) = hw;
    *reinterpret_cast<uint32_t*>(bs + rl * 128u + ((((lane >> 2) ^ (rl & 7u)) << 4) + in_chunk)) = lw;
    return fold_factor(E, mx);
}

// MT: tokens (1 or 2). Q8: the activations are already E4M3 codes (A [M][lda bytes])
// with one FP32 scale per token and 128-K group (a_scale [K/128][a_scale_stride]), the
// W8A8 variant: each step's codes are copied into the hi rows (the lo rows stay zero)
// and the fold multiplies by s_w * s_a.
template <uint32_t MT, bool Q8>
__global__ void __launch_bounds__(kGvThreads, 2)
    w8a16_gemv_kernel(const __grid_constant__ CUtensorMap tmW, const float* __restrict__ scale,
                      __nv_bfloat16* __restrict__ C, uint32_t ldc, const void* __restrict__ A,
                      uint32_t lda, const float* __restrict__ a_scale, uint32_t a_scale_stride, uint32_t N,
                      uint32_t K, uint32_t split_k, uint64_t timeout_ns) {
    // steps per 16-column accumulator: each step takes MT column pairs (hi, lo)
    constexpr uint32_t kQ = 8u / MT;
    constexpr uint32_t kAcc = kGvMaxSteps / kQ;   // accumulators (16 columns each)
    static_assert(kGvResident * 32u + kAcc * 16u <= kGvTmemCols, "TMEM budget");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sW = smem;                                              // slots x 16 KiB weights
    uint8_t* sB = sW + kGvSlots * kWTileBytes;                       // steps x 2 KiB MMA B operands
    float* sF = reinterpret_cast<float*>(sB + kGvMaxSteps * kGvBStepBytes);   // [step][token] factors
    float* sRed = sF + kGvMaxSteps * kGvMaxTokens;                   // [rank][row][4] partials
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sRed) + kGvRedBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    const uint32_t wfull0 = bar0;                           // kGvSlots: a step landed in a slot
    const uint32_t moved0 = wfull0 + 8u * kGvSlots;         // kGvResident: a step copied to TMEM
    const uint32_t zero_bar = moved0 + 8u * kGvResident;    // the accumulators are zero
    const uint32_t mma_bar = zero_bar + 8u;                 // every step's MMAs are done
    const uint32_t fact_bar = mma_bar + 8u;                 // every step's factors are written
    const uint32_t red_bar = fact_bar + 8u;                 // split-K partials received
    const uint32_t own0 = red_bar + 8u;                     // kGvMaxSteps: one warp's MMAs done

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tile = blockIdx.x / split_k;
    const uint32_t rank = blockIdx.x - tile * split_k;
    const uint32_t ksteps = K / kKStep;
    const uint32_t s_begin = static_cast<uint32_t>(static_cast<uint64_t>(rank) * ksteps / split_k);
    const uint32_t s_end = static_cast<uint32_t>(static_cast<uint64_t>(rank + 1) * ksteps / split_k);
    const uint32_t nsteps = s_end - s_begin;                // 1..kGvMaxSteps (the planner's rule)
    const uint32_t nres = nsteps > kGvSlots ? nsteps - kGvSlots : 0u;   // steps moved to TMEM
    const uint32_t npre = nsteps < kGvSlots ? nsteps : kGvSlots;
    const uint32_t rows_valid = min(kTcRows, N - tile * kTcRows);
    const uint32_t my_row0 = owned_row0(rank, split_k);
    const uint32_t my_rows = owned_row0(rank + 1, split_k) - my_row0;
    uint64_t deadline = globaltimer_ns() + timeout_ns;      // restarted after the dependency wait
    uint32_t loads_issued = 0;                              // thread 0: weight copies queued

    if (warp == 0) {
        for (uint32_t b = lane; b < kNumBars; b += 32) {
            const uint32_t addr = bar0 + 8u * b;
            uint32_t count = 1;
            if (addr >= moved0 && addr <= zero_bar) count = 4;                  // the 4 mover warps
            else if (addr == mma_bar || addr == fact_bar) count = nsteps;       // a warp per step
            mbar_init(addr, count);
        }
        if (lane == 0) *abort_flag = 0;
        fence_barrier_init();
        __syncwarp();
    }
    if (threadIdx.x == 0) {
        if (split_k > 1) mbar_arrive_expect_tx(red_bar, (split_k - 1) * my_rows * 16u);   // the other ranks'
        // every weight tile-step that has a slot, before anything else (under a
        // programmatic launch the caller guarantees the previous grid writes no W)
        const uint64_t pol_w = l2_policy_evict_first();
        for (uint32_t i = 0; i < npre; ++i) {
            mbar_arrive_expect_tx(wfull0 + 8u * i, kWTileBytes);
            tma_load_2d(smem_u32(sW + i * kWTileBytes), &tmW, wfull0 + 8u * i,
                        static_cast<int32_t>((s_begin + i) * kKStep), static_cast<int32_t>(tile * kTcRows),
                        pol_w);
        }
        loads_issued = npre;
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kGvTmemCols);
        tmem_relinquish();
    }
    // The B operands start as zeros: a step fills only its own column pairs' rows.
    for (uint32_t i = threadIdx.x; i < kGvMaxSteps * kGvBStepBytes / 16u; i += kGvThreads)
        reinterpret_cast<uint4*>(sB)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();   // ... as the tensor core will read them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (split_k > 1) cluster_arrive();
    if (threadIdx.x == 0) grid_launch_dependents();
    const uint32_t tbase = *tmem_slot;
    const uint32_t tW = tbase;                              // kGvResident x 32 weight columns
    const uint32_t tAcc = tbase + 32u * kGvResident;        // kAcc x 16 accumulator columns
    const uint32_t quarter = warp & 3u;
    const uint32_t row = quarter * 32u + lane;              // mover / fold row (warps 4..7)
    const uint32_t lane_bits = (quarter * 32u) << 16;
    const bool is_mover = warp >= 4;

    // ------------------------------------------------ before the dependency wait
    float sc = 0.f;   // fold warps: lane l holds the block scale of step l
    if (is_mover) {
        sc = lane < nsteps ? __ldg(scale + static_cast<size_t>(tile) * ksteps + s_begin + lane) : 0.f;
        uint32_t z[32];
#pragma unroll
        for (uint32_t c = 0; c < 32; ++c) z[c] = 0u;
        tmem_st_32x32b_x32(tAcc + lane_bits, z);             // kAcc x 16 = 32 columns
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(zero_bar);
        // steps 0..nres-1: row `row` of the landed tile (128-byte swizzle: chunk c at
        // c ^ (row & 7)) into TMEM lane `row`, 32 columns, K bytes in column order
        for (uint32_t i = 0; i < nres; ++i) {
            if (!gv_warp_wait(wfull0 + 8u * i, 0, deadline, abort_flag, kWaitW)) break;
            const uint8_t* rp = sW + i * kWTileBytes + row * 128u;
            uint32_t w[32];
#pragma unroll
            for (uint32_t c = 0; c < 8; ++c) {
                const uint4 q = *reinterpret_cast<const uint4*>(rp + ((c ^ (row & 7u)) << 4));
                w[4 * c] = q.x;
                w[4 * c + 1] = q.y;
                w[4 * c + 2] = q.z;
                w[4 * c + 3] = q.w;
            }
            fence_proxy_async_smem();   // these reads come before the slot's next TMA write
            tmem_st_32x32b_x32(tW + lane_bits + 32u * i, w);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(moved0 + 8u * i);
        }
    } else if (warp == 0 && lane == 0) {
        // the last steps go to the slots the moved ones freed (step i reuses the
        // slot of step i - kGvSlots < nres)
        const uint64_t pol_w = l2_policy_evict_first();
        for (uint32_t i = npre; i < nsteps; ++i) {
            const uint32_t s = i % kGvSlots;
            if (!mbar_wait(moved0 + 8u * (i - kGvSlots), 0, deadline, abort_flag, &g_gemv_status, kWaitMoved))
                break;
            mbar_arrive_expect_tx(wfull0 + 8u * s, kWTileBytes);
            tma_load_2d(smem_u32(sW + s * kWTileBytes), &tmW, wfull0 + 8u * s,
                        static_cast<int32_t>((s_begin + i) * kKStep), static_cast<int32_t>(tile * kTcRows),
                        pol_w);
            loads_issued = i + 1;
        }
    }
    __syncwarp();

    // ------------------------------------------------- after the dependency wait
    // A may be written by the previous grid in the stream.
    deadline = deadline_after_dependency(timeout_ns);
    bool issued = false;
    if (warp < nsteps) {
        // split step w = warp and issue its MMAs
        const uint32_t w = warp;
        const uint32_t acc_idx = w / kQ;
        const uint32_t pair0 = (w % kQ) * MT;
        uint8_t* bs = sB + w * kGvBStepBytes;
        if constexpr (Q8) {
            // the step's codes into the hi rows (4 bytes a lane, 128-byte swizzle); the
            // factor is the token's group scale (both may be the previous grid's
            // output: read through L2)
            const uint8_t* src = static_cast<const uint8_t*>(A) + static_cast<size_t>(s_begin + w) * kKStep + 4u * lane;
            uint32_t cw[MT];
#pragma unroll
            for (uint32_t t = 0; t < MT; ++t)
                cw[t] = __ldcg(reinterpret_cast<const unsigned int*>(src + static_cast<size_t>(t) * lda));
            const uint32_t in_chunk = (lane & 3u) << 2;
#pragma unroll
            for (uint32_t t = 0; t < MT; ++t) {
                const uint32_t rh = 2u * (pair0 + t);
                *reinterpret_cast<uint32_t*>(bs + rh * 128u + ((((lane >> 2) ^ (rh & 7u)) << 4) + in_chunk)) = cw[t];
                if (lane == 0)
                    sF[w * kGvMaxTokens + t] = __ldcg(a_scale + static_cast<size_t>(s_begin + w) * a_scale_stride + t);
            }
        } else {
            const uint16_t* src = static_cast<const uint16_t*>(A) + static_cast<size_t>(s_begin + w) * kKStep + 4u * lane;
            uint2 av[MT];
#pragma unroll
            for (uint32_t t = 0; t < MT; ++t)
                av[t] = *reinterpret_cast<const uint2*>(src + static_cast<size_t>(t) * lda);
#pragma unroll
            for (uint32_t t = 0; t < MT; ++t) {
                const float f = split_block_w32(av[t], bs, 2u * (pair0 + t), 2u * (pair0 + t) + 1u, lane);
                if (lane == 0) sF[w * kGvMaxTokens + t] = f;
            }
        }
        fence_proxy_async_smem();   // the tensor core reads these terms
        __syncwarp();
        bool ok = true;
        if (lane == 0) {
            mbar_arrive(fact_bar);
            ok = mbar_wait(zero_bar, 0, deadline, abort_flag, &g_gemv_status, kWaitAccZero);
            if (ok)
                ok = w < nres ? mbar_wait(moved0 + 8u * w, 0, deadline, abort_flag, &g_gemv_status, kWaitMoved)
                              : mbar_wait(wfull0 + 8u * (w % kGvSlots), (w / kGvSlots) & 1u, deadline, abort_flag,
                                          &g_gemv_status, kWaitW);
            if (ok) {
                tc_fence_after();
                constexpr uint32_t idesc = idesc_e4m3_f32(kTcRows, 16);
                const uint64_t db = smem_desc_kmajor_sw128(smem_u32(bs));
                const uint32_t d = tAcc + 16u * acc_idx;
                if (w < nres) {
#pragma unroll
                    for (uint32_t kk = 0; kk < kKStep / 32; ++kk)   // 32 K bytes = 8 columns per MMA
                        tc_mma_ts_f8(d, tW + 32u * w + 8u * kk, db + 2u * kk, idesc, 1u);
                } else {
                    const uint64_t dw = smem_desc_kmajor_sw128(smem_u32(sW + (w % kGvSlots) * kWTileBytes));
#pragma unroll
                    for (uint32_t kk = 0; kk < kKStep / 32; ++kk)
                        tc_mma_ss_f8(d, dw + 2u * kk, db + 2u * kk, idesc, 1u);
                }
                tc_commit(mma_bar);
                tc_commit(own0 + 8u * w);
                issued = true;
            }
        }
        __syncwarp();
    }

    if (is_mover) {
        // --------------- fold: acc[t] += scale(s) * 2^(E-7) * (P_hi + P_lo / 32), s in order
        float acc[MT];
#pragma unroll
        for (uint32_t t = 0; t < MT; ++t) acc[t] = 0.f;
        const bool ok = gv_warp_wait(mma_bar, 0, deadline, abort_flag, kWaitMma) &&
                        gv_warp_wait(fact_bar, 0, deadline, abort_flag, kWaitFact);
        if (ok) {
            tc_fence_after();
            float v[kAcc][16];
#pragma unroll
            for (uint32_t a = 0; a < kAcc; ++a) tmem_ld_32x32b_x16(tAcc + lane_bits + 16u * a, v[a]);
            tc_wait_ld();
#pragma unroll
            for (uint32_t s = 0; s < kGvMaxSteps; ++s) {
                const float sw = __shfl_sync(0xFFFFFFFFu, sc, s);
                if (s < nsteps) {
#pragma unroll
                    for (uint32_t t = 0; t < MT; ++t) {
                        const uint32_t col = 2u * ((s % kQ) * MT + t);
                        if constexpr (Q8) {   // acc += (s_w * s_a) * P, as the W8A8 kernel folds
                            acc[t] = fmaf(sw * sF[s * kGvMaxTokens + t], v[s / kQ][col], acc[t]);
                        } else {
                            const float pt = fmaf(v[s / kQ][col + 1], 0.03125f, v[s / kQ][col]) *
                                             sF[s * kGvMaxTokens + t];
                            acc[t] = fmaf(sw, pt, acc[t]);
                        }
                    }
                }
            }
        }
        if (split_k == 1) {
            if (row < rows_valid) {
                const uint32_t n = tile * kTcRows + row;
#pragma unroll
                for (uint32_t t = 0; t < MT; ++t) C[static_cast<size_t>(t) * ldc + n] = __float2bfloat16_rn(acc[t]);
            }
        } else {
            cluster_wait();
            // the last rank r with r * 128 / split_k <= row owns the row
            const uint32_t owner = ((row + 1u) * split_k - 1u) / kTcRows;
            const uint32_t lrow = row - owned_row0(owner, split_k);
            const uint32_t off = (rank * tc_red_rows(split_k) + lrow) * 16u;
            if (owner != rank)   // rows this CTA owns stay in registers
                st_async_v4f32(dsmem_map(smem_u32(sRed) + off, owner), dsmem_map(red_bar, owner), acc[0],
                               MT > 1 ? acc[MT - 1] : 0.f, 0.f, 0.f);
            // the partials are other CTAs' st.async writes: acquire at cluster scope
            const bool got = mbar_wait<true>(red_bar, 0, deadline + timeout_ns, abort_flag, &g_gemv_status,
                                             kWaitRed);
            if (__all_sync(0xFFFFFFFFu, got) && row >= my_row0 && row < my_row0 + my_rows && row < rows_valid) {
                const uint32_t lr = row - my_row0;
                float r[2] = {0.f, 0.f};
                for (uint32_t src = 0; src < split_k; ++src) {   // rank order, this rank's from registers
                    const float4 q = src == rank ? make_float4(acc[0], MT > 1 ? acc[MT - 1] : 0.f, 0.f, 0.f)
                                                 : *reinterpret_cast<const float4*>(
                                                       sRed + (src * tc_red_rows(split_k) + lr) * 4u);
                    r[0] += q.x;
                    r[1] += q.y;
                }
                const uint32_t n = tile * kTcRows + row;
#pragma unroll
                for (uint32_t t = 0; t < MT; ++t) C[static_cast<size_t>(t) * ldc + n] = __float2bfloat16_rn(r[t]);
            }
        }
    }

    // ------------------------------------------------------------ teardown
    // Each warp that issued MMAs waits for them before TMEM is released, and every
    // weight copy lands before the CTA may exit (the last use of each slot; earlier
    // uses were waited for before their slot was reused).
    if (warp < nsteps && lane == 0 && issued) {
        volatile int never = 0;
        mbar_wait(own0 + 8u * warp, 0, globaltimer_ns() + timeout_ns, &never, &g_gemv_status, kWaitOwn);
    }
    if (threadIdx.x == 0) {
        volatile int never = 0;
        const uint64_t dl = globaltimer_ns() + timeout_ns;
        for (uint32_t j = loads_issued > kGvSlots ? loads_issued - kGvSlots : 0u; j < loads_issued; ++j)
            mbar_wait(wfull0 + 8u * (j % kGvSlots), (j / kGvSlots) & 1u, dl, &never, &g_gemv_status, kWaitW);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kGvTmemCols);
    }
}

using GemvKernelFn = void (*)(CUtensorMap, const float*, __nv_bfloat16*, uint32_t, const void*, uint32_t,
                              const float*, uint32_t, uint32_t, uint32_t, uint32_t, uint64_t);
// [Q8][MT - 1]
const GemvKernelFn kGemvKernels[2][2] = {{&w8a16_gemv_kernel<1, false>, &w8a16_gemv_kernel<2, false>},
                                         {&w8a16_gemv_kernel<1, true>, &w8a16_gemv_kernel<2, true>}};

cudaError_t ensure_gemv_attributes(int device) {
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (done[device]) return cudaSuccess;
    for (GemvKernelFn fn : {kGemvKernels[0][0], kGemvKernels[0][1], kGemvKernels[1][0], kGemvKernels[1][1]}) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(gemv_smem_bytes()));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    done[device] = true;
    return cudaSuccess;
}

}  // namespace

namespace {

int launch_gemv_any(const GemmArgs& g, const float* a_scale, uint32_t a_scale_stride, bool q8,
                    const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns, uint32_t flags, std::string* err) {
    if (g.M < 1 || g.M > kGvMaxTokens) {
        *err = "decode kernel: M=" + std::to_string(g.M) + " is outside 1.." + std::to_string(kGvMaxTokens);
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_gemv_attributes(dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("decode kernel attribute setup failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    CUtensorMap mw;
    if (!tc_tensor_map_w(g, dev, &mw, err)) return W8A16_ERR_LAUNCH;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(p.grid[0], 1, 1);
    cfg.blockDim = dim3(kGvThreads, 1, 1);
    cfg.dynamicSmemBytes = gemv_smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.split_k;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = (flags & W8A16_FLAG_PDL) ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kGemvKernels[q8 ? 1 : 0][g.M - 1], mw, g.scale, static_cast<__nv_bfloat16*>(g.C),
                           g.ldc, g.A, g.lda, a_scale, a_scale_stride, g.N, g.K, p.split_k, timeout_ns);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("decode kernel launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
}

}  // namespace

int launch_gemv(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
                uint32_t flags, std::string* err) {
    return launch_gemv_any(g, nullptr, 0u, false, p, s, timeout_ns, flags, err);
}

int launch_gemv_w8a8(const W8A8Args& a, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
                     uint32_t flags, std::string* err) {
    GemmArgs g{};
    g.A = a.A;
    g.lda = a.lda;
    g.W = a.W;
    g.scale = a.scale;
    g.C = a.C;
    g.ldc = a.ldc;
    g.M = a.M;
    g.N = a.N;
    g.K = a.K;
    return launch_gemv_any(g, a.a_scale, a.a_scale_stride, true, p, s, timeout_ns, flags, err);
}

int gemv_cluster_capacity(uint32_t cluster, uint32_t* ctas, std::string* err) {
    if (cluster < 1 || cluster > 16) {
        *err = "decode kernel: cluster size outside 1..16";
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_gemv_attributes(dev);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(cluster * 64, 1, 1);
    cfg.blockDim = dim3(kGvThreads, 1, 1);
    cfg.dynamicSmemBytes = gemv_smem_bytes();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kGemvKernels[0][0]), &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("cudaOccupancyMaxActiveClusters failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_DEVICE;
    }
    *ctas = static_cast<uint32_t>(n) * cluster;
    return W8A16_OK;
}

cudaError_t gemv_status_read(StatusWord* out, bool clear, cudaStream_t s) {
    DeviceStatus st;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&st, g_gemv_status, sizeof st, 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    out->code = st.code;
    out->where = st.where;
    out->detail = st.detail;
    if (clear) {
        const DeviceStatus zero{0, 0, 0};
        e = cudaMemcpyToSymbolAsync(g_gemv_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace w8a16
