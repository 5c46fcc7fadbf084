// FP8-datapath tensor-core W8A16 kernel for sm_103a (tcgen05.mma kind::f8f6f4 + TMA).
//
// Same operation, checks and reduction order as the BF16 tensor-core kernel
// (page "metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs": one
// FP32 fold of the block scale per 128-K step, split-K partials added in step
// order), with the E4M3 weights fed to the tensor core as they arrive:
//
//   * the weight tile TMA lands in shared memory (128 rows x 128 K, 128-byte
//     swizzle) is the MMA's A operand as is: the tensor core decodes E4M3
//     exactly, so there is no conversion work and no TMEM operand traffic, and
//     one K=32 MMA covers twice the weights of a BF16 K=16 MMA;
//   * each BF16 activation row of a 128-K block is written as two E4M3 terms,
//     x = a * 2^(7-E) = hi + lo / 32 with E the exponent of the block's largest
//     |a| (hi = e4m3_rne(x), lo = e4m3_rne(32 (x - hi))): exact for every a with
//     |a| >= 2^-14 max|a|, and within 2^-22 max|a| otherwise. The two terms are
//     the MMA's B rows [0, TN) and [TN, 2 TN), so one MMA of N = 2 TN computes
//     both products;
//   * the fold recombines them in FP32: acc += scale * 2^(E-7) * (P_hi + P_lo / 32).
// A non-finite activation makes its token's outputs NaN (E4M3 has no infinity).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "w8a16_cluster.cuh"
#include "w8a16_device.cuh"
#include "w8a16_internal.h"
#include "w8a16_split.cuh"

namespace w8a16 {

__device__ DeviceStatus g_tc8_status;

namespace {

constexpr uint32_t kWTileBytes = kTcRows * kKStep;   // 16 KiB of E4M3 per stage

enum : uint32_t {
    kWaitW = 11, kWaitX = 12, kWaitXEmpty = 13, kWaitB = 14, kWaitMdone = 15, kWaitPEmpty = 16,
    kWaitDone = 17, kWaitDrain = 18, kWaitRed = 19
};

template <uint32_t TN, uint32_t STAGES>
struct T8Cfg {
    static constexpr uint32_t SA = tc8_act_stages(TN);     // BF16 activation staging ring
    static constexpr uint32_t SB = tc8_b_stages(TN);       // E4M3 two-term activation ring
    static constexpr uint32_t NP = tc8_p_bufs(TN);         // TMEM product buffers (2 TN cols)
    static constexpr uint32_t NS = tc8_split_warps(TN);
    static constexpr uint32_t NF = tc8_fold_warps(TN);
    static constexpr uint32_t kTmemCols = tc8_tmem_cols(TN);
    static constexpr uint32_t kXBytes = TN * kKStep * 2;
    static constexpr uint32_t kBBytes = 2 * TN * kKStep;
    static constexpr uint32_t kSplit0 = 3;                 // first splitter warp
    static constexpr uint32_t kFold0 = kSplit0 + NS;       // first fold warp
    static constexpr uint32_t kTokPerFold = TN * 4 / NF;
    // Step-parallel mode (few tokens): splitter warp w takes steps w, w+NS, ... and
    // issues their MMAs itself. Every ring then has exactly NS slots, so warp w
    // always uses slot w of each and waits only on barriers it alone feeds or that
    // complete once per step of its own.
    static constexpr bool kStepPar = STAGES == NS && SA == NS && SB == NS && NP == NS;

    static constexpr uint32_t ND = STAGES > SB ? (STAGES > NP ? STAGES : NP) : (SB > NP ? SB : NP);
    // barriers: wfull[S], xfull[SA], xempty[SA], bfull[SB], mdone[ND], pempty[NP], done, red
    static constexpr uint32_t kNumBars = STAGES + 2 * SA + SB + ND + NP + 2;
    static_assert(NP * 2 * TN <= kTmemCols, "TMEM budget");
    static_assert(kTokPerFold % 16 == 0, "fold loads whole x16 column groups");
    static_assert(kNumBars * 8 + 16 <= 1024, "barrier area");
};




template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait8(uint32_t bar, uint32_t parity, uint64_t deadline,
                                           volatile int* abort_flag, uint32_t detail) {
    const bool ok = mbar_wait<CLUSTER>(bar, parity, deadline, abort_flag, &g_tc8_status, detail);
    return __all_sync(0xFFFFFFFFu, ok);
}


__device__ __forceinline__ void drain_ring8(uint32_t bar_base, uint32_t depth, uint32_t issued,
                                            uint64_t timeout_ns) {
    const uint64_t dl = globaltimer_ns() + timeout_ns;
    for (uint32_t j = issued > depth ? issued - depth : 0; j < issued; ++j) {
        volatile int never = 0;
        mbar_wait(bar_base + 8u * (j % depth), (j / depth) & 1, dl, &never, &g_tc8_status, kWaitDrain);
    }
}



// The four K=32 MMAs of one 128-K step: D[128 x 2TN] (FP32, TMEM) = W tile x terms.
template <uint32_t TN>
__device__ __forceinline__ void step_mmas(uint32_t d_tmem, uint64_t dw, uint64_t db) {
    constexpr uint32_t idesc = idesc_e4m3_f32(kTcRows, 2 * TN);
#pragma unroll
    for (uint32_t kk = 0; kk < kKStep / 32; ++kk)   // 32 bytes of K per MMA
        tc_mma_ss_f8(d_tmem, dw + 2 * kk, db + 2 * kk, idesc, kk > 0);
}

// Split one token's 128-K block with the whole warp, 4 values per lane (used for
// one or two tokens, where a lane per 4 values keeps all 32 lanes busy). Lane l
// holds K 4l..4l+3 (av: 4 BF16 values, lowest K first).
template <uint32_t TN>
__device__ __forceinline__ void split_token_w32(uint2 av, uint8_t* bs, float* inv, uint32_t t,
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
    // the block maximum: |x| >= 0 orders as its bit pattern, one warp reduction
    mx = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mx)));
    const int E = block_exponent(mx);
    float p1, p2;
    split_scales(E, p1, p2);
#pragma unroll
    for (uint32_t e = 0; e < 4; ++e) x[e] = (x[e] * p1) * p2;
    uint32_t hw, lw;
    two_terms4(x, hw, lw);
    if (bad) hw = 0x7F7F7F7Fu;   // a non-finite value: NaN codes
    // E4M3 rows t (hi) and TN + t (lo): 4 bytes at K 4l, chunk l / 4 (swizzled), byte 4 (l % 4)
    const uint32_t pos = (((lane >> 2) ^ (t & 7)) << 4) + ((lane & 3) << 2);
    *reinterpret_cast<uint32_t*>(bs + t * 128 + pos) = hw;
    *reinterpret_cast<uint32_t*>(bs + (TN + t) * 128 + pos) = lw;
    if (lane == 0) inv[t] = fold_factor(E, mx);
}

// Split P passes of four tokens' blocks (tokens t0 + p*dt .. +3 for p < P), 8 lanes
// per token, 16 values per lane: lane c of a token holds K 8c..8c+7 and
// 64+8c..64+8c+7 (16-byte chunk c of each BF16 box, so the 8 lanes of a token read
// one 128-byte row without conflicts). All loads come first and all stores last,
// so the P passes' dependency chains interleave.
template <uint32_t TN, uint32_t P>
__device__ __forceinline__ void split_tokens_w8(const uint8_t* xs, uint8_t* bs, float* inv,
                                                uint32_t t0, uint32_t dt, uint32_t lane) {
    const uint32_t tt = lane >> 3, c = lane & 7;
    uint32_t w[P][8];
#pragma unroll
    for (uint32_t p = 0; p < P; ++p) {
        const uint32_t t = t0 + p * dt + tt;
        const uint8_t* xr = xs + t * 128 + ((c ^ (t & 7)) << 4);
        const uint4 a0 = *reinterpret_cast<const uint4*>(xr);
        const uint4 a1 = *reinterpret_cast<const uint4*>(xr + TN * 128);
        w[p][0] = a0.x; w[p][1] = a0.y; w[p][2] = a0.z; w[p][3] = a0.w;
        w[p][4] = a1.x; w[p][5] = a1.y; w[p][6] = a1.z; w[p][7] = a1.w;
    }
    float mx[P], x[P][16];
    bool bad[P];
#pragma unroll
    for (uint32_t p = 0; p < P; ++p) {
        mx[p] = 0.f;
        bad[p] = false;
#pragma unroll
        for (uint32_t e = 0; e < 8; ++e) {
            x[p][2 * e] = __uint_as_float(w[p][e] << 16);
            x[p][2 * e + 1] = __uint_as_float(w[p][e] & 0xFFFF0000u);
        }
#pragma unroll
        for (uint32_t e = 0; e < 16; ++e) {
            const float a = fabsf(x[p][e]);
            if (a <= 3.4028235e38f) mx[p] = fmaxf(mx[p], a);
            else bad[p] = true;   // NaN or infinity
        }
    }
#pragma unroll
    for (uint32_t o = 4; o > 0; o >>= 1)
#pragma unroll
        for (uint32_t p = 0; p < P; ++p) mx[p] = fmaxf(mx[p], __shfl_xor_sync(0xFFFFFFFFu, mx[p], o));
    int E[P];
#pragma unroll
    for (uint32_t p = 0; p < P; ++p) {
        E[p] = block_exponent(mx[p]);
        float p1, p2;
        split_scales(E[p], p1, p2);
#pragma unroll
        for (uint32_t e = 0; e < 16; ++e) x[p][e] = (x[p][e] * p1) * p2;
    }
    uint32_t hw[P][4], lw[P][4];
#pragma unroll
    for (uint32_t p = 0; p < P; ++p)
#pragma unroll
        for (uint32_t q = 0; q < 4; ++q) {
            two_terms4(x[p] + 4 * q, hw[p][q], lw[p][q]);
            if (bad[p]) hw[p][q] = 0x7F7F7F7Fu;   // a non-finite value: NaN codes
        }
    // E4M3 rows t (hi) and TN + t (lo), 128 bytes each, 128-byte swizzle: K 8c.. is
    // 8 bytes in chunk c/2, K 64+8c.. in chunk 4 + c/2. Odd tokens store their
    // second half first so that the two tokens of a half-warp write disjoint banks.
    const bool odd = tt & 1;
#pragma unroll
    for (uint32_t p = 0; p < P; ++p) {
        const uint32_t t = t0 + p * dt + tt, sw7 = t & 7;
        const uint32_t posA = (((c >> 1) ^ sw7) << 4) + ((c & 1) << 3);
        const uint32_t posB = ((((c >> 1) + 4) ^ sw7) << 4) + ((c & 1) << 3);
        const uint32_t p_1 = odd ? posB : posA, p_2 = odd ? posA : posB;
        const uint2 h_1 = odd ? make_uint2(hw[p][2], hw[p][3]) : make_uint2(hw[p][0], hw[p][1]);
        const uint2 h_2 = odd ? make_uint2(hw[p][0], hw[p][1]) : make_uint2(hw[p][2], hw[p][3]);
        const uint2 l_1 = odd ? make_uint2(lw[p][2], lw[p][3]) : make_uint2(lw[p][0], lw[p][1]);
        const uint2 l_2 = odd ? make_uint2(lw[p][0], lw[p][1]) : make_uint2(lw[p][2], lw[p][3]);
        uint8_t* rh = bs + t * 128;
        uint8_t* rl = bs + (TN + t) * 128;
        *reinterpret_cast<uint2*>(rh + p_1) = h_1;
        *reinterpret_cast<uint2*>(rh + p_2) = h_2;
        *reinterpret_cast<uint2*>(rl + p_1) = l_1;
        *reinterpret_cast<uint2*>(rl + p_2) = l_2;
        if (c == 0) inv[t] = fold_factor(E[p], mx[p]);
    }
}

template <uint32_t TN, uint32_t STAGES>
__global__ void __launch_bounds__(tc8_threads(TN), TN == 16 ? 2 : 1)
    w8a16_tc8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                     const float* __restrict__ scale, __nv_bfloat16* __restrict__ C, uint32_t ldc,
                     const uint16_t* __restrict__ A, uint32_t lda, uint32_t M, uint32_t N,
                     uint32_t K, uint32_t split_k, uint64_t timeout_ns) {
    using Cfg = T8Cfg<TN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sW = smem;                                   // STAGES x 16 KiB E4M3 weights
    uint8_t* sB = sW + STAGES * kWTileBytes;              // SB x 2TN x 128 E4M3 activation terms
    uint8_t* sX = sB + Cfg::SB * Cfg::kBBytes;            // SA x TN x 128 BF16 activations
    float* sInv = reinterpret_cast<float*>(sX + Cfg::SA * Cfg::kXBytes);   // NP x TN factors
    float* sRed = sInv + Cfg::NP * TN;                    // split-K receive slots
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sRed) +
                                                 tc_red_bytes(TN, split_k));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    // mdone[i % ND] completes when the MMAs of step i have: it frees weight slot
    // i % STAGES and term slot i % SB, and fills product buffer i % NP.
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t wfull0 = bar0;
    const uint32_t xfull0 = wfull0 + 8u * STAGES, xempty0 = xfull0 + 8u * Cfg::SA;
    const uint32_t bfull0 = xempty0 + 8u * Cfg::SA;
    const uint32_t mdone0 = bfull0 + 8u * Cfg::SB;
    const uint32_t pempty0 = mdone0 + 8u * Cfg::ND;
    const uint32_t done_bar = pempty0 + 8u * Cfg::NP;
    const uint32_t red_bar = done_bar + 8u;

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tile = blockIdx.x / split_k;
    const uint32_t rank = blockIdx.x % split_k;
    const uint32_t token0 = blockIdx.y * TN;
    const uint32_t ksteps = K / kKStep;
    const uint32_t s_begin = static_cast<uint32_t>(static_cast<uint64_t>(rank) * ksteps / split_k);
    const uint32_t s_end = static_cast<uint32_t>(static_cast<uint64_t>(rank + 1) * ksteps / split_k);
    const uint32_t nsteps = s_end - s_begin;
    uint64_t deadline = globaltimer_ns() + timeout_ns;   // restarted by each role after the dependency wait
    const uint32_t my_row0 = owned_row0(rank, split_k);
    const uint32_t my_rows = owned_row0(rank + 1, split_k) - my_row0;
    const uint32_t npre = nsteps < STAGES ? nsteps : STAGES;
    const uint32_t rows_valid = min(kTcRows, N - tile * kTcRows);
    const uint32_t toks_valid = min(TN, M - token0);
    // up to 8 tokens: a splitter warp splits whole steps (two passes at most)
    const bool step_par = Cfg::kStepPar && toks_valid <= 8;
    // one or two tokens: the splitters read A straight from global memory (the
    // tensor-memory-access unit is busy with weight tiles, and a 256-byte row
    // waits behind them), so the activation producer has nothing to do
    const bool direct_x = step_par && toks_valid <= 2;

    if (warp == 0) {
        for (uint32_t b = lane; b < Cfg::kNumBars; b += 32) {
            const uint32_t addr = bar0 + 8u * b;
            uint32_t count = 1;
            if (addr >= xempty0 && addr < mdone0) count = step_par ? 1u : Cfg::NS;   // splitters
            else if (addr >= pempty0 && addr < done_bar) count = Cfg::NF;   // fold warps
            else if (addr == done_bar) count = step_par ? Cfg::NS : 1u;      // MMA issuers
            mbar_init(addr, count);
        }
        if (lane == 0) *abort_flag = 0;
        fence_barrier_init();
        __syncwarp();
    }
    if (threadIdx.x == 0) {
        if (split_k > 1)
            mbar_arrive_expect_tx(red_bar, (split_k - 1) * my_rows * red_row_bytes<TN, Cfg::kTokPerFold>(toks_valid));
        // First weight tiles before anything else; weights are requested before
        // waiting on the previous grid (under a programmatic launch the caller
        // guarantees that grid does not write W).
        const uint64_t pol_w = l2_policy_evict_first();
        for (uint32_t i = 0; i < npre; ++i) {
            mbar_arrive_expect_tx(wfull0 + 8u * i, kWTileBytes);
            tma_load_2d(smem_u32(sW + i * kWTileBytes), &tmW, wfull0 + 8u * i,
                        static_cast<int32_t>((s_begin + i) * kKStep),
                        static_cast<int32_t>(tile * kTcRows), pol_w);
        }
        tma_prefetch_desc(&tmA);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (split_k > 1) cluster_arrive();
    if (threadIdx.x == 0) grid_launch_dependents();
    const uint32_t tP = *tmem_slot;                 // NP x 2TN columns: FP32 products
    const uint32_t quarter = warp & 3;
    const uint32_t row = quarter * 32 + lane;
    const uint32_t lane_bits = (quarter * 32) << 16;
    const bool is_split = warp >= Cfg::kSplit0 && warp < Cfg::kFold0;
    const bool is_fold = warp >= Cfg::kFold0;

    if (warp == 0) {
        // ------------------------------------------------ weight producer (TMA)
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            uint32_t issued = npre;
            if (npre < nsteps) deadline = deadline_after_dependency(timeout_ns);   // slots free after MMAs
            for (uint32_t i = npre; i < nsteps; ++i) {
                const uint32_t s = i % STAGES, q = i - STAGES;   // slot s last held step q
                if (!mbar_wait(mdone0 + 8u * (q % Cfg::ND), (q / Cfg::ND) & 1, deadline, abort_flag,
                               &g_tc8_status, kWaitMdone))
                    break;
                mbar_arrive_expect_tx(wfull0 + 8u * s, kWTileBytes);
                tma_load_2d(smem_u32(sW + s * kWTileBytes), &tmW, wfull0 + 8u * s,
                            static_cast<int32_t>((s_begin + i) * kKStep),
                            static_cast<int32_t>(tile * kTcRows), pol_w);
                issued = i + 1;
            }
            drain_ring8(wfull0, STAGES, issued, timeout_ns);
        }
    } else if (warp == 2) {
        // -------------------------------------------- activation producer (TMA)
        if (lane == 0 && !direct_x) {
            const uint64_t pol_a = l2_policy_evict_last();
            // A may be written by the previous grid in the stream
            deadline = deadline_after_dependency(timeout_ns);
            uint32_t issued = 0;
            for (uint32_t i = 0; i < nsteps; ++i) {
                const uint32_t j = i % Cfg::SA;
                if (i >= Cfg::SA && !mbar_wait(xempty0 + 8u * j, ((i / Cfg::SA) - 1) & 1, deadline,
                                               abort_flag, &g_tc8_status, kWaitXEmpty))
                    break;
                mbar_arrive_expect_tx(xfull0 + 8u * j, Cfg::kXBytes);
                const int32_t k = static_cast<int32_t>((s_begin + i) * kKStep);
                const uint32_t dst = smem_u32(sX + j * Cfg::kXBytes);
                tma_load_2d(dst, &tmA, xfull0 + 8u * j, k, static_cast<int32_t>(token0), pol_a);
                tma_load_2d(dst + TN * 128, &tmA, xfull0 + 8u * j, k + 64,
                            static_cast<int32_t>(token0), pol_a);
                issued = i + 1;
            }
            drain_ring8(xfull0, Cfg::SA, issued, timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // (token-parallel mode; in step-parallel mode the splitters issue)
        if (lane == 0) {
            // The fold of step i - NP has freed product buffer i % NP once bfull[i]
            // completes: the splitters of step i wait for that before arriving.
            const uint64_t dw0 = smem_desc_kmajor_sw128(smem_u32(sW));   // + (offset >> 4)
            const uint64_t db0 = smem_desc_kmajor_sw128(smem_u32(sB));
            if (!step_par) deadline = deadline_after_dependency(timeout_ns);   // the terms come after it
            for (uint32_t i = 0; i < (step_par ? 0u : nsteps); ++i) {
                const uint32_t s = i % STAGES, b = i % Cfg::SB, p = i % Cfg::NP;
                if (!mbar_wait(wfull0 + 8u * s, (i / STAGES) & 1, deadline, abort_flag, &g_tc8_status,
                               kWaitW))
                    break;
                if (!mbar_wait(bfull0 + 8u * b, (i / Cfg::SB) & 1, deadline, abort_flag,
                               &g_tc8_status, kWaitB))
                    break;
                tc_fence_after();
                const uint64_t dw = dw0 + ((s * kWTileBytes) >> 4);
                const uint64_t db = db0 + ((b * Cfg::kBBytes) >> 4);
                step_mmas<TN>(tP + p * 2 * TN, dw, db);
                tc_commit(mdone0 + 8u * (i % Cfg::ND));
            }
            if (!step_par) tc_commit(done_bar);
            volatile int never = 0;
            mbar_wait(done_bar, 0, globaltimer_ns() + timeout_ns, &never, &g_tc8_status, kWaitDone);
        }
    } else if (is_split) {
        // ---------------- splitters: BF16 activations -> two E4M3 terms per value
        // Token-parallel mode: warp w takes 4-token passes w, w+NS, ... of every
        // step. Step-parallel mode (up to 8 tokens): warp w takes every pass of
        // steps w, w+NS, ...; with one or two tokens a pass is one token on all
        // 32 lanes.
        const uint32_t sw = warp - Cfg::kSplit0;
        const uint32_t i_first = step_par ? sw : 0u, di = step_par ? Cfg::NS : 1u;
        const uint32_t t_first = step_par ? 0u : 4u * sw, dt = step_par ? 4u : 4u * Cfg::NS;
        const uint64_t dw0 = smem_desc_kmajor_sw128(smem_u32(sW));   // + (offset >> 4)
        const uint64_t db0 = smem_desc_kmajor_sw128(smem_u32(sB));
        // direct_x: lane l's 4 values at K 4l of tokens 0 and 1, one step ahead
        const uint16_t* arow = A + static_cast<size_t>(token0) * lda + 4u * lane;
        auto load_x = [&](uint32_t i, uint2* v) {
            const uint16_t* src = arow + static_cast<size_t>(s_begin + i) * kKStep;
            v[0] = *reinterpret_cast<const uint2*>(src);
            v[1] = toks_valid > 1 ? *reinterpret_cast<const uint2*>(src + lda) : make_uint2(0u, 0u);
        };
        uint2 xnext[2] = {make_uint2(0u, 0u), make_uint2(0u, 0u)};
        // A may be written by the previous grid in the stream
        deadline = deadline_after_dependency(timeout_ns);
        if (direct_x && i_first < nsteps) load_x(i_first, xnext);
        for (uint32_t i = i_first; i < nsteps; i += di) {
            const uint32_t j = i % Cfg::SA, b = i % Cfg::SB, f = i % Cfg::NP;
            uint2 xcur[2] = {xnext[0], xnext[1]};
            if (direct_x) {
                if (i + di < nsteps) load_x(i + di, xnext);
            } else if (!warp_wait8(xfull0 + 8u * j, (i / Cfg::SA) & 1, deadline, abort_flag, kWaitX)) {
                break;
            }
            if (i >= Cfg::SB) {   // term slot b last held step i - SB
                const uint32_t q = i - Cfg::SB;
                if (!warp_wait8(mdone0 + 8u * (q % Cfg::ND), (q / Cfg::ND) & 1, deadline, abort_flag,
                                kWaitMdone))
                    break;
            }
            if (i >= Cfg::NP && !warp_wait8(pempty0 + 8u * f, ((i / Cfg::NP) - 1) & 1, deadline,
                                            abort_flag, kWaitPEmpty))
                break;   // factor slot f and product buffer f are read by the fold of step i - NP
            const uint8_t* xs = sX + j * Cfg::kXBytes;
            uint8_t* bs = sB + b * Cfg::kBBytes;
            float* inv = sInv + f * TN;
            if (direct_x) {
                for (uint32_t t = 0; t < toks_valid; ++t) split_token_w32<TN>(xcur[t], bs, inv, t, lane);
            } else {
                // rows past the last token are TMA zero fill: splitting them is harmless
                uint32_t t0 = t_first;
                if constexpr (TN >= 32) {   // two passes at once where registers allow
                    for (; t0 + dt < toks_valid; t0 += 2 * dt)
                        split_tokens_w8<TN, 2>(xs, bs, inv, t0, dt, lane);
                }
                for (; t0 < toks_valid; t0 += dt) split_tokens_w8<TN, 1>(xs, bs, inv, t0, dt, lane);
            }
            fence_proxy_async_smem();   // the tensor core reads these terms
            __syncwarp();
            if (step_par) {
                // This warp issues step i's MMAs: slot b = i % NS also holds step i's
                // weights, and step i - NS's MMAs (this warp's, awaited above) freed it.
                bool ok = true;
                if (lane == 0) {
                    if (!direct_x) mbar_arrive(xempty0 + 8u * j);
                    ok = mbar_wait(wfull0 + 8u * b, (i / STAGES) & 1, deadline, abort_flag,
                                   &g_tc8_status, kWaitW);
                    if (ok) {
                        tc_fence_after();
                        step_mmas<TN>(tP + f * 2 * TN, dw0 + ((b * kWTileBytes) >> 4),
                                      db0 + ((b * Cfg::kBBytes) >> 4));
                        tc_commit(mdone0 + 8u * (i % Cfg::ND));
                    }
                }
                if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) break;
            } else if (lane == 0) {
                mbar_arrive(bfull0 + 8u * b);
                mbar_arrive(xempty0 + 8u * j);
            }
        }
        if (step_par && lane == 0) tc_commit(done_bar);   // after this warp's last MMAs
    } else if (is_fold) {
        // --------- fold: acc += scale * 2^(E-7) * (P_hi + P_lo / 32) per token
        const uint32_t fh = (warp - Cfg::kFold0) >> 2;
        float acc[Cfg::kTokPerFold];
#pragma unroll
        for (uint32_t t = 0; t < Cfg::kTokPerFold; ++t) acc[t] = 0.f;
        const float* srow = scale + static_cast<size_t>(tile) * ksteps + s_begin;
        // The block scales of this CTA's steps, 32 per register (lane l holds step
        // 32c + l of chunk c), read at once instead of one load per step: under a
        // programmatic launch the caller guarantees they are not being written.
        float sc_cur = lane < nsteps ? __ldg(srow + lane) : 0.f;
        float sc_next = lane + 32u < nsteps ? __ldg(srow + 32u + lane) : 0.f;
        deadline = deadline_after_dependency(timeout_ns);   // the products come after it
        for (uint32_t i = 0; i < nsteps; ++i) {
            if (i != 0 && (i & 31u) == 0) {
                sc_cur = sc_next;
                sc_next = i + 32u + lane < nsteps ? __ldg(srow + i + 32u + lane) : 0.f;
            }
            const uint32_t p = i % Cfg::NP;
            if (!warp_wait8(mdone0 + 8u * (i % Cfg::ND), (i / Cfg::ND) & 1, deadline, abort_flag,
                            kWaitMdone))
                break;
            tc_fence_after();
            const float sc = __shfl_sync(0xFFFFFFFFu, sc_cur, i & 31u);
            const uint32_t pcol = tP + lane_bits + p * 2 * TN + fh * Cfg::kTokPerFold;
            const float* inv = sInv + p * TN + fh * Cfg::kTokPerFold;
#pragma unroll
            for (uint32_t c = 0; c < Cfg::kTokPerFold; c += 16) {
                float vh[16], vl[16];
                tmem_ld_32x32b_x16(pcol + c, vh);
                tmem_ld_32x32b_x16(pcol + TN + c, vl);
                tc_wait_ld();
                // two tokens per packed FP32 instruction, each with the arithmetic of
                // acc = fmaf(sc, fmaf(lo, 1/32, hi) * f, acc)
                const uint64_t sc2 = pack_f32x2(sc, sc), k32 = pack_f32x2(0.03125f, 0.03125f);
#pragma unroll
                for (uint32_t t = 0; t < 16; t += 2) {
                    const float2 f = *reinterpret_cast<const float2*>(inv + c + t);
                    const uint64_t pt = fma_f32x2(pack_f32x2(vl[t], vl[t + 1]), k32, pack_f32x2(vh[t], vh[t + 1]));
                    const float2 a = unpack_f32x2(fma_f32x2(sc2, mul_f32x2(pt, pack_f32x2(f.x, f.y)),
                                                            pack_f32x2(acc[c + t], acc[c + t + 1])));
                    acc[c + t] = a.x;
                    acc[c + t + 1] = a.y;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty0 + 8u * p);
        }
        if (split_k == 1) {
            if (row < rows_valid) {
                const uint32_t n = tile * kTcRows + row;
#pragma unroll
                for (uint32_t t = 0; t < Cfg::kTokPerFold; ++t) {
                    const uint32_t m = fh * Cfg::kTokPerFold + t;
                    if (m < toks_valid)
                        C[static_cast<size_t>(token0 + m) * ldc + n] = __float2bfloat16_rn(acc[t]);
                }
            }
        } else {
            cluster_wait();
            // the last rank r with r * 128 / split_k <= row (no division by split_k)
            const uint32_t owner = ((row + 1) * split_k - 1) / kTcRows;
            const uint32_t lrow = row - owned_row0(owner, split_k);
            // receive layout [slot][row][token]: this thread's tokens are contiguous
            // and go as 16-byte groups; the owner reads them back the same way
            const uint32_t off =
                ((tc_red_slot(rank, owner) * tc_red_rows(split_k) + lrow) * tc_red_stride(TN) +
                 fh * Cfg::kTokPerFold) * 4u;
            const uint32_t dst = dsmem_map(smem_u32(sRed) + off, owner);
            const uint32_t dbar = dsmem_map(red_bar, owner);
            const uint32_t ngroups = push_bytes(toks_valid, fh * Cfg::kTokPerFold, Cfg::kTokPerFold) / 16u;
            if (owner != rank) {   // rows this CTA owns stay in registers
#pragma unroll
                for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g)   // groups past M are not sent
                    if (g < ngroups)
                        st_async_v4f32(dst + 16u * g, dbar, acc[4 * g], acc[4 * g + 1], acc[4 * g + 2],
                                       acc[4 * g + 3]);
            }
            // This CTA's own rows: the thread holding row `row` of the tile (and
            // tokens fh*kTokPerFold..) adds the ranks' partials in rank order, its
            // own rank's from its registers.
            // the partials are other CTAs' st.async writes: acquire at cluster scope
            const bool got = warp_wait8<true>(red_bar, 0, deadline + timeout_ns, abort_flag, kWaitRed);
            if (got && row >= my_row0 && row < my_row0 + my_rows && row < rows_valid) {
                const uint32_t lr = row - my_row0;
                const uint32_t rank_stride = tc_red_rows(split_k) * tc_red_stride(TN);   // floats
                const float* src_row = sRed + lr * tc_red_stride(TN);
#pragma unroll
                for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g) {
                    const uint32_t t = fh * Cfg::kTokPerFold + 4u * g;
                    if (t >= toks_valid) break;
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                    for (uint32_t src = 0; src < split_k; ++src) {   // rank order
                        const float4 q =
                            src == rank ? make_float4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3])
                                        : *reinterpret_cast<const float4*>(
                                              src_row + tc_red_slot(src, rank) * rank_stride + t);
                        v.x += q.x;
                        v.y += q.y;
                        v.z += q.z;
                        v.w += q.w;
                    }
                    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (uint32_t u = 0; u < 4; ++u)
                        if (t + u < toks_valid)
                            C[static_cast<size_t>(token0 + t + u) * ldc + tile * kTcRows + row] =
                                __float2bfloat16_rn(vv[u]);
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tP, Cfg::kTmemCols);
    }

}

using Tc8KernelFn = void (*)(CUtensorMap, CUtensorMap, const float*, __nv_bfloat16*, uint32_t,
                             const uint16_t*, uint32_t, uint32_t, uint32_t, uint32_t, uint32_t,
                             uint64_t);
struct Tc8Instance {
    uint32_t tn, stages;
    Tc8KernelFn fn;
};
#define W8A16_TC8_INST(TN_, ST_) {TN_, ST_, &w8a16_tc8_kernel<TN_, ST_>}
const Tc8Instance kTc8Instances[] = {
    W8A16_TC8_INST(16, 4), W8A16_TC8_INST(16, 6), W8A16_TC8_INST(16, 8),
    W8A16_TC8_INST(32, 4), W8A16_TC8_INST(32, 6), W8A16_TC8_INST(32, 8),
    W8A16_TC8_INST(64, 4), W8A16_TC8_INST(64, 6),
};
#undef W8A16_TC8_INST
constexpr int kNumTc8 = sizeof(kTc8Instances) / sizeof(kTc8Instances[0]);

int find_tc8(uint32_t tn, uint32_t stages) {
    for (int i = 0; i < kNumTc8; ++i)
        if (kTc8Instances[i].tn == tn && kTc8Instances[i].stages == stages) return i;
    return -1;
}

cudaError_t ensure_attributes8(int inst, int device) {
    static std::mutex mu;
    static bool done[64][kNumTc8] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (done[device][inst]) return cudaSuccess;
    const Tc8Instance& k = kTc8Instances[inst];
    uint32_t most = 0;
    for (uint32_t sp = 1; sp <= 16; ++sp) {
        const uint32_t b = tc8_smem_bytes(k.tn, k.stages, sp);
        if (b <= kMaxDynSmem && b > most) most = b;
    }
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(k.fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(most));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(k.fn),
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) done[device][inst] = true;
    return e;
}

}  // namespace

bool tc8_supported_stages(uint32_t tn, uint32_t stages) { return find_tc8(tn, stages) >= 0; }

int launch_tc8(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
               uint32_t flags, std::string* err) {
    const int inst = find_tc8(p.token_tile, p.stages);
    if (inst < 0) {
        *err = "no TC8 kernel instance for token_tile=" + std::to_string(p.token_tile) +
               " stages=" + std::to_string(p.stages);
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_attributes8(inst, dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("TC8 kernel attribute setup failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    CUtensorMap mw, ma;
    if (!tc_tensor_map_w(g, dev, &mw, err) || !tc_tensor_map_a(g, p.token_tile, dev, &ma, err))
        return W8A16_ERR_LAUNCH;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(p.grid[0], p.grid[1], 1);
    cfg.blockDim = dim3(tc8_threads(p.token_tile), 1, 1);
    cfg.dynamicSmemBytes = tc8_smem_bytes(p.token_tile, p.stages, p.split_k);
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
    e = cudaLaunchKernelEx(&cfg, kTc8Instances[inst].fn, mw, ma, g.scale,
                           static_cast<__nv_bfloat16*>(g.C), g.ldc,
                           static_cast<const uint16_t*>(g.A), g.lda, g.M, g.N, g.K, p.split_k,
                           timeout_ns);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("TC8 kernel launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
}

int tc8_cluster_capacity(uint32_t tn, uint32_t stages, uint32_t cluster, uint32_t* ctas,
                         std::string* err) {
    const int inst = find_tc8(tn, stages);
    if (inst < 0 || cluster < 1 || cluster > 16) {
        *err = "no TC8 kernel instance, or cluster size outside 1..16";
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_attributes8(inst, dev);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(cluster * 64, 1, 1);
    cfg.blockDim = dim3(tc8_threads(tn), 1, 1);
    cfg.dynamicSmemBytes = tc8_smem_bytes(tn, stages, cluster);
    if (cfg.dynamicSmemBytes > kMaxDynSmem) {
        *ctas = 0;
        return W8A16_OK;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kTc8Instances[inst].fn),
                                           &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("cudaOccupancyMaxActiveClusters failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_DEVICE;
    }
    *ctas = static_cast<uint32_t>(n) * cluster;
    return W8A16_OK;
}

cudaError_t tc8_status_read(StatusWord* out, bool clear, cudaStream_t s) {
    DeviceStatus st;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&st, g_tc8_status, sizeof st, 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    out->code = st.code;
    out->where = st.where;
    out->detail = st.detail;
    if (clear) {
        const DeviceStatus zero{0, 0, 0};
        e = cudaMemcpyToSymbolAsync(g_tc8_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace w8a16
