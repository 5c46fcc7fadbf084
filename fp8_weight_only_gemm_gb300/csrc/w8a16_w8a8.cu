// W8A8 tensor-core kernel for sm_103a: E4M3 activations (per-token 128-K group
// scales) times E4M3 weights (128x128 block scales), tcgen05.mma kind::f8f6f4.
//
// The adjacent precision variant of the W8A16 GEMM: the activations come already
// quantised (page "metrale_model_layers/layers/ops/fp8_act_quant.rs", module
// doc: per-token quantisation in 128-element K groups), so each 128-K step is one
// FP8 x FP8 product P = A_q W_q^T folded as acc += s_w * s_a[token] * P, with
// the same tiles, rings, split-K and reduction order as the two-term kernel
// (w8a16_tc8.cu) but no activation split: the activation codes are the MMA's
// B operand as TMA lands them (N = TN, one MMA per 32 K).
//
// The same kernel computes the W8A16 product from the two-term split of the BF16
// activations (TERMS = 2; the split is the one w8a16_split.cuh describes, written
// to a workspace by a pre-pass): the hi and lo codes of a token tile are the MMA's
// B rows [0, TN) and [TN, 2 TN), one MMA of N = 2 TN computes both products, and
// the fold takes acc += s_w * 2^(E-7) * (P_hi + P_lo / 32), as the kernel that
// splits its own tiles does (w8a16_tc8.cu).
//
// Warp roles: 0 weight producer (TMA), 1 TMEM owner + MMA issuer for even steps,
// 2 activation producer (TMA: the step's codes), 3 MMA issuer for odd steps, then
// NF fold warps. Two issuers each wait only on their own steps' slots (every ring
// has an even number of slots), so one thread's waits overlap the other's MMAs.
// Both rings hold only MMA operands and are freed by MMA completion. The per-token
// factors come from global memory: each fold warp loads its tokens' factors one
// step ahead (lane l, token l) and stages them in its own shared buffer with
// ordinary stores, so no generic access meets TMA-written memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "w8a16_cluster.cuh"
#include "w8a16_device.cuh"
#include "w8a16_internal.h"

namespace w8a16 {

__device__ DeviceStatus g_w8a8_status;

namespace {

constexpr uint32_t kWTileBytes = kTcRows * kKStep;   // 16 KiB of E4M3 weights per stage

enum : uint32_t {
    kWaitW = 21, kWaitX = 22, kWaitXSlot = 23, kWaitMdone = 24, kWaitPEmpty = 25, kWaitDone = 26,
    kWaitDrain = 27, kWaitRed = 28, kWaitFlush = 29
};

template <uint32_t TN, uint32_t STAGES, uint32_t TERMS>
struct A8Cfg {
    static constexpr uint32_t SA = w8a8_act_stages(TN, TERMS);   // activation ring (codes + factors)
    static constexpr uint32_t NP = w8a8_p_bufs(TN, TERMS);       // TMEM product buffers
    static constexpr uint32_t NB = TERMS * TN;                   // MMA N: B rows per step
    static constexpr uint32_t NF = w8a8_fold_warps(TN, TERMS);
    static constexpr uint32_t kTmemCols = w8a8_tmem_cols(TN, TERMS);
    static constexpr uint32_t kCodeBytes = NB * kKStep;    // one step's E4M3 activation tile(s)
    static constexpr uint32_t kFold0 = 4;                  // first fold warp
    static constexpr uint32_t kTokPerFold = TN * 4 / NF;
    static constexpr uint32_t ND = STAGES > SA ? (STAGES > NP ? STAGES : NP) : (SA > NP ? SA : NP);
    // barriers: wfull[S], xfull[SA], mdone[ND], pempty[NP], done, red, fsync[2] (stream-K)
    static constexpr uint32_t kNumBars = STAGES + SA + ND + NP + 4;
    static constexpr uint32_t kFactorRegs = (kTokPerFold + 31) / 32;   // per lane
    static_assert(STAGES % 2 == 0 && SA % 2 == 0 && NP % 2 == 0, "rings of even depth");
    static_assert(NP * NB <= kTmemCols, "TMEM budget");
    static_assert(TERMS == 1 || TERMS == 2, "one or two activation terms");
    static_assert(kTokPerFold % 16 == 0, "fold loads are whole x16 column groups");
    static_assert(kNumBars * 8 + 16 <= 1024, "barrier area");
};

template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait_a8(uint32_t bar, uint32_t parity, uint64_t deadline,
                                             volatile int* abort_flag, uint32_t detail) {
    const bool ok = mbar_wait<CLUSTER>(bar, parity, deadline, abort_flag, &g_w8a8_status, detail);
    return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ void drain_ring_a8(uint32_t bar_base, uint32_t depth, uint32_t issued,
                                              uint64_t timeout_ns) {
    const uint64_t dl = globaltimer_ns() + timeout_ns;
    for (uint32_t j = issued > depth ? issued - depth : 0; j < issued; ++j) {
        volatile int never = 0;
        mbar_wait(bar_base + 8u * (j % depth), (j / depth) & 1, dl, &never, &g_w8a8_status, kWaitDrain);
    }
}

// acc[t] += g[t] * P[t] for CW tokens, g = s_w * f (the step's block scale times the
// token's factor, staged per step), two tokens per packed FP32 instruction. With two
// terms P = hi + lo / 32 (fmaf(lo, 1/32, hi), exact); f is then a power of two, so
// fmaf(g, P, acc) rounds as fmaf(s_w, P * f, acc) does wherever s_w * f stays a
// normal FP32 number.
template <uint32_t TERMS, uint32_t CW>
__device__ __forceinline__ void fold_cols(float* acc, const float* v, const float* vl, const float* g) {
#pragma unroll
    for (uint32_t t = 0; t < CW; t += 2) {
        const float2 gg = *reinterpret_cast<const float2*>(g + t);
        const uint64_t p = TERMS == 2 ? fma_f32x2(pack_f32x2(vl[t], vl[t + 1]), pack_f32x2(0.03125f, 0.03125f),
                                                  pack_f32x2(v[t], v[t + 1]))
                                      : pack_f32x2(v[t], v[t + 1]);
        const float2 a = unpack_f32x2(fma_f32x2(pack_f32x2(gg.x, gg.y), p, pack_f32x2(acc[t], acc[t + 1])));
        acc[t] = a.x;
        acc[t + 1] = a.y;
    }
}

// SK: the persistent stream-K instance (two terms, up to 32 tokens); its fold code is
// compiled only there, so the cluster split-K instances keep their register budget.
template <uint32_t TN, uint32_t STAGES, uint32_t TERMS, bool SK = false>
__global__ void __launch_bounds__(w8a8_threads(TN, TERMS), w8a8_max_ctas_by_regs(TN))
    w8a16_w8a8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const float* __restrict__ a_scale, uint32_t a_stride, const float* __restrict__ scale,
                      __nv_bfloat16* __restrict__ C, uint32_t ldc, uint32_t M, uint32_t N, uint32_t K,
                      uint32_t split_k, uint32_t tile0, uint32_t tok_major, const StreamK sk,
                      uint64_t timeout_ns) {
    using Cfg = A8Cfg<TN, STAGES, TERMS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sW = smem;                                        // STAGES x 16 KiB weights
    uint8_t* sX = sW + STAGES * kWTileBytes;                   // SA x NB x 128 activation codes
    float* sF = reinterpret_cast<float*>(sX + Cfg::SA * Cfg::kCodeBytes);   // fold warps' factors
    // split-K receive slots: after the rings, or (alias) in the rings' memory, then
    // written by peers only once every rank of the cluster is past its last K step
    const bool alias = w8a8_red_alias(TN, STAGES, split_k, TERMS);
    const uint32_t ring = w8a8_ring_bytes(TN, STAGES, TERMS), red = tc_red_bytes(TN, split_k);
    float* sRed = reinterpret_cast<float*>(alias ? smem : smem + ring);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (alias ? (ring > red ? ring : red) : ring + red));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* sk_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);   // stream-K: last of a tile

    // mdone[i % ND] completes when step i's MMAs have: it frees weight slot
    // i % STAGES and activation slot i % SA and fills product buffer i % NP.
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t wfull0 = bar0;
    const uint32_t xfull0 = wfull0 + 8u * STAGES;
    const uint32_t mdone0 = xfull0 + 8u * Cfg::SA;
    const uint32_t pempty0 = mdone0 + 8u * Cfg::ND;
    const uint32_t done_bar = pempty0 + 8u * Cfg::NP;
    const uint32_t red_bar = done_bar + 8u;
    const uint32_t fsync0 = red_bar + 8u, fsync1 = fsync0 + 8u;   // stream-K: fold warps meet

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tok_major (no split): the token tiles of one weight tile are consecutive CTAs, so
    // beyond the token tile the later ones find the tile's weights in L2
    const uint32_t bx = tok_major ? blockIdx.y : blockIdx.x, by = tok_major ? blockIdx.x : blockIdx.y;
    const uint32_t cta_tile = bx / split_k;
    const uint32_t rank = bx - cta_tile * split_k;
    const uint32_t tile = tile0 + cta_tile;                    // 128-row weight tile
    const uint32_t token0 = by * TN;
    const uint32_t ksteps = K / kKStep;                        // < 2^24: products fit 32 bits
    const uint32_t s_begin = rank * ksteps / split_k;
    const uint32_t s_end = (rank + 1) * ksteps / split_k;
    // The CTA's steps as units (128-row tile, 128-K step) in tile-major order: the
    // range [u_first, u_first + nsteps) is one tile's [s_begin, s_end) under the
    // cluster split-K schedule, and the CTA's share of all units under stream-K.
    static_assert(!SK || (TERMS == 2 && TN <= 32), "stream-K instances: two terms, up to 32 tokens");
    constexpr bool sk_mode = SK;
    const uint32_t u_first = sk_mode ? static_cast<uint32_t>(static_cast<uint64_t>(blockIdx.x) * sk.units / gridDim.x)
                                     : tile * ksteps + s_begin;
    const uint32_t nsteps =
        sk_mode ? static_cast<uint32_t>(static_cast<uint64_t>(blockIdx.x + 1) * sk.units / gridDim.x) - u_first
                : s_end - s_begin;
    uint64_t deadline = globaltimer_ns() + timeout_ns;   // restarted by each role after the dependency wait
    const uint32_t my_row0 = owned_row0(rank, split_k);
    const uint32_t my_rows = owned_row0(rank + 1, split_k) - my_row0;
    const uint32_t npre = nsteps < STAGES ? nsteps : STAGES;
    const uint32_t rows_valid = min(kTcRows, N - tile * kTcRows);
    const uint32_t toks_valid = min(TN, M - token0);

    if (warp == 0) {
        for (uint32_t b = lane; b < Cfg::kNumBars; b += 32) {
            const uint32_t addr = bar0 + 8u * b;
            uint32_t count = 1;
            if ((addr >= pempty0 && addr < done_bar) || addr == fsync0) count = Cfg::NF;   // fold warps
            else if (addr == done_bar) count = 2;                           // MMA issuers
            mbar_init(addr, count);
        }
        if (lane == 0) *abort_flag = 0;
        fence_barrier_init();
        __syncwarp();
    }
    if (threadIdx.x == 0) {
        if (split_k > 1)
            mbar_arrive_expect_tx(red_bar,
                                  (split_k - 1) * my_rows * red_row_bytes<TN, Cfg::kTokPerFold>(toks_valid));
        // weights before the dependency wait (a programmatic launch's caller
        // guarantees the previous grid writes neither W nor its scales)
        const uint64_t pol_w = l2_policy_evict_first();
        for (uint32_t i = 0; i < npre; ++i) {
            mbar_arrive_expect_tx(wfull0 + 8u * i, kWTileBytes);
            const uint32_t u = u_first + i;
            tma_load_2d(smem_u32(sW + i * kWTileBytes), &tmW, wfull0 + 8u * i,
                        static_cast<int32_t>((SK ? u % ksteps : s_begin + i) * kKStep),
                        static_cast<int32_t>((SK ? u / ksteps : tile) * kTcRows),
                        pol_w);
        }
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Without aliasing, peers may push as soon as this CTA's receive barrier is
    // initialised: a relaxed arrive (fence.mbarrier_init released the
    // initialisation to the cluster), which does not wait for in-flight loads.
    if (split_k > 1 && !alias) cluster_arrive();
    if (threadIdx.x == 0) grid_launch_dependents();
    const uint32_t tP = *tmem_slot;                            // NP x TN columns: FP32 products
    const uint32_t quarter = warp & 3;
    const uint32_t row = quarter * 32 + lane;
    const uint32_t lane_bits = (quarter * 32) << 16;
    const bool is_fold = warp >= Cfg::kFold0 && warp < Cfg::kFold0 + Cfg::NF;

    if (warp == 0) {
        // ------------------------------------------------ weight producer (TMA)
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            uint32_t issued = npre;
            if (npre < nsteps) deadline = deadline_after_dependency(timeout_ns);   // slots free after MMAs
            for (uint32_t i = npre; i < nsteps; ++i) {
                const uint32_t s = i % STAGES, q = i - STAGES;   // slot s last held step q
                if (!mbar_wait(mdone0 + 8u * (q % Cfg::ND), (q / Cfg::ND) & 1, deadline, abort_flag,
                               &g_w8a8_status, kWaitMdone))
                    break;
                mbar_arrive_expect_tx(wfull0 + 8u * s, kWTileBytes);
                const uint32_t u = u_first + i;
                tma_load_2d(smem_u32(sW + s * kWTileBytes), &tmW, wfull0 + 8u * s,
                            static_cast<int32_t>((SK ? u % ksteps : s_begin + i) * kKStep),
                            static_cast<int32_t>((SK ? u / ksteps : tile) * kTcRows), pol_w);
                issued = i + 1;
            }
            drain_ring_a8(wfull0, STAGES, issued, timeout_ns);
        }
        __syncwarp();
        if (split_k > 1 && alias) cluster_arrive_release();
    } else if (warp == 2) {
        // ------------------------------------ activation producer (TMA): codes
        if (lane == 0) {
            const uint64_t pol_a = l2_policy_evict_last();
            // the activations may be the previous grid's output
            deadline = deadline_after_dependency(timeout_ns);
            uint32_t issued = 0;
            for (uint32_t i = 0; i < nsteps; ++i) {
                const uint32_t j = i % Cfg::SA;
                const uint32_t q = i - Cfg::SA;   // slot j last held step q
                if (i >= Cfg::SA && !mbar_wait(mdone0 + 8u * (q % Cfg::ND), (q / Cfg::ND) & 1, deadline,
                                               abort_flag, &g_w8a8_status, kWaitXSlot))
                    break;
                mbar_arrive_expect_tx(xfull0 + 8u * j, Cfg::kCodeBytes);
                const int32_t kx = static_cast<int32_t>((SK ? (u_first + i) % ksteps : s_begin + i) * kKStep);
                tma_load_2d(smem_u32(sX + j * Cfg::kCodeBytes), &tmX, xfull0 + 8u * j, kx,
                            static_cast<int32_t>(token0), pol_a);
                if (TERMS == 2)   // lo terms: rows M + token0.. of the [2M][K] codes
                    tma_load_2d(smem_u32(sX + j * Cfg::kCodeBytes + TN * kKStep), &tmX, xfull0 + 8u * j, kx,
                                static_cast<int32_t>(M + token0), pol_a);
                issued = i + 1;
            }
            drain_ring_a8(xfull0, Cfg::SA, issued, timeout_ns);
        }
        __syncwarp();
        if (split_k > 1 && alias) cluster_arrive_release();
    } else if (warp == 1 || warp == 3) {
        // ----------------------------------- MMA issuers: even steps, odd steps
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kTcRows, Cfg::NB);
            const uint64_t dw0 = smem_desc_kmajor_sw128(smem_u32(sW));   // + (offset >> 4)
            const uint64_t dx0 = smem_desc_kmajor_sw128(smem_u32(sX));
            deadline = deadline_after_dependency(timeout_ns);   // the activations come after it
            for (uint32_t i = (warp == 1 ? 0u : 1u); i < nsteps; i += 2) {
                const uint32_t s = i % STAGES, j = i % Cfg::SA, p = i % Cfg::NP;
                if (!mbar_wait(wfull0 + 8u * s, (i / STAGES) & 1, deadline, abort_flag, &g_w8a8_status,
                               kWaitW))
                    break;
                if (!mbar_wait(xfull0 + 8u * j, (i / Cfg::SA) & 1, deadline, abort_flag, &g_w8a8_status,
                               kWaitX))
                    break;
                if (i >= Cfg::NP && !mbar_wait(pempty0 + 8u * p, ((i / Cfg::NP) - 1) & 1, deadline,
                                               abort_flag, &g_w8a8_status, kWaitPEmpty))
                    break;
                tc_fence_after();
                const uint64_t dw = dw0 + ((s * kWTileBytes) >> 4);
                const uint64_t dx = dx0 + ((j * Cfg::kCodeBytes) >> 4);
#pragma unroll
                for (uint32_t kk = 0; kk < kKStep / 32; ++kk)   // 32 bytes of K per MMA
                    tc_mma_ss_f8(tP + p * Cfg::NB, dw + 2 * kk, dx + 2 * kk, idesc, kk > 0);
                tc_commit(mdone0 + 8u * (i % Cfg::ND));
            }
            tc_commit(done_bar);   // this thread's MMAs, before TMEM is released
            volatile int never = 0;
            mbar_wait(done_bar, 0, globaltimer_ns() + timeout_ns, &never, &g_w8a8_status, kWaitDone);
        }
        __syncwarp();
        if (split_k > 1 && alias) cluster_arrive_release();
    } else if (is_fold) {
        // ------------------------- fold: acc += s_w * s_a[token] * P per token
        const uint32_t fh = (warp - Cfg::kFold0) >> 2;
        float acc[Cfg::kTokPerFold];
#pragma unroll
        for (uint32_t t = 0; t < Cfg::kTokPerFold; ++t) acc[t] = 0.f;
        const float* srow = scale + u_first;   // block_scale [tiles][ksteps] is unit-major
        // this CTA's weight block scales, 32 per register (lane l: step 32c + l)
        float sc_cur = lane < nsteps ? __ldg(srow + lane) : 0.f;
        float sc_next = lane + 32u < nsteps ? __ldg(srow + 32u + lane) : 0.f;
        // this warp's per-token factors of a step: lane l holds token r*32 + l of the
        // warp's tokens, loaded kAhead steps ahead into a queue of registers (a step
        // can be shorter than an L2 round trip), after the dependency wait (the
        // factors may be the previous grid's output; L2 only, never a stale L1)
        float* fbuf = sF + (warp - Cfg::kFold0) * Cfg::kTokPerFold;
        const uint32_t tokf = token0 + fh * Cfg::kTokPerFold;
        const auto load_factors = [&](uint32_t step, float (&f)[Cfg::kFactorRegs]) {
            // the step's 128-K group: s_begin + step, or under stream-K the unit's
            const uint32_t kg = SK ? (u_first + step) % ksteps : s_begin + step;
#pragma unroll
            for (uint32_t r = 0; r < Cfg::kFactorRegs; ++r) {
                const uint32_t t = r * 32u + lane;
                f[r] = (t < Cfg::kTokPerFold && tokf + t < M)
                           ? __ldcg(a_scale + static_cast<size_t>(kg) * a_stride + tokf + t)
                           : 0.f;
            }
        };
        constexpr uint32_t kAhead = 4;
        deadline = deadline_after_dependency(timeout_ns);
        float fq[kAhead][Cfg::kFactorRegs];
#pragma unroll
        for (uint32_t d = 0; d < kAhead; ++d) {
            if (d < nsteps) {
                load_factors(d, fq[d]);
            } else {
#pragma unroll
                for (uint32_t r = 0; r < Cfg::kFactorRegs; ++r) fq[d][r] = 0.f;
            }
        }
        // Stream-K: the fold's current tile and step, and whether its segment started at
        // the tile's first step. When a segment ends (the tile's last step, or the CTA's),
        // a whole tile goes straight to C and part of one to its slot of the partials.
        uint32_t seg_tile = u_first / ksteps, seg_k = u_first % ksteps;
        bool seg_from0 = seg_k == 0, loop_done = false;
        const uint32_t m0 = fh * Cfg::kTokPerFold;   // this thread's first token of the tile
        const auto sk_store = [&](uint32_t t, bool whole) {
            if (whole) {
                const uint32_t rows_v = min(kTcRows, N - t * kTcRows);
                if (row < rows_v) {
                    __nv_bfloat16* crow = C + static_cast<size_t>(t) * kTcRows + row;
#pragma unroll
                    for (uint32_t tt = 0; tt < Cfg::kTokPerFold; ++tt)
                        if (m0 + tt < toks_valid)
                            crow[static_cast<size_t>(token0 + m0 + tt) * ldc] = __float2bfloat16_rn(acc[tt]);
                }
            } else {
                const uint32_t cf = stream_cta_of(static_cast<uint64_t>(t) * ksteps, sk.units, gridDim.x);
                float4* mine = reinterpret_cast<float4*>(
                    sk.parts + ((static_cast<size_t>(t) * sk.maxseg + (blockIdx.x - cf)) * kTcRows + row) * TN + m0);
#pragma unroll
                for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g)
                    mine[g] = make_float4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]);
            }
        };
        for (uint32_t i = 0; i < nsteps; ++i) {
            if (i != 0 && (i & 31u) == 0) {
                sc_cur = sc_next;
                sc_next = i + 32u + lane < nsteps ? __ldg(srow + i + 32u + lane) : 0.f;
            }
            const uint32_t p = i % Cfg::NP;
            const float sw = __shfl_sync(0xFFFFFFFFu, sc_cur, i & 31u);
            __syncwarp();   // the previous step's reads of fbuf are done
            // staged as g = s_w * f: one FMA per product in the fold
#pragma unroll
            for (uint32_t r = 0; r < Cfg::kFactorRegs; ++r)
                if (r * 32u + lane < Cfg::kTokPerFold) fbuf[r * 32u + lane] = fq[0][r] * sw;
            __syncwarp();   // ... and this step's factors are visible to the whole warp
#pragma unroll
            for (uint32_t d = 0; d + 1 < kAhead; ++d)
#pragma unroll
                for (uint32_t r = 0; r < Cfg::kFactorRegs; ++r) fq[d][r] = fq[d + 1][r];
            if (i + kAhead < nsteps) load_factors(i + kAhead, fq[kAhead - 1]);
            if (!warp_wait_a8(mdone0 + 8u * (i % Cfg::ND), (i / Cfg::ND) & 1, deadline, abort_flag,
                              kWaitMdone))
                break;
            tc_fence_after();
            const uint32_t pcol = tP + lane_bits + p * Cfg::NB + fh * Cfg::kTokPerFold;
#pragma unroll
            for (uint32_t c = 0; c < Cfg::kTokPerFold; c += 16) {
                float v[16], vl[16];
                tmem_ld_32x32b_x16(pcol + c, v);
                if (TERMS == 2) tmem_ld_32x32b_x16(pcol + TN + c, vl);
                tc_wait_ld();
                fold_cols<TERMS, 16>(acc + c, v, vl, fbuf + c);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty0 + 8u * p);
            if (sk_mode) {
                if (seg_k == ksteps - 1 || i == nsteps - 1) {
                    sk_store(seg_tile, seg_from0 && seg_k == ksteps - 1);
#pragma unroll
                    for (uint32_t t = 0; t < Cfg::kTokPerFold; ++t) acc[t] = 0.f;
                    seg_from0 = true;
                }
                if (++seg_k == ksteps) {
                    seg_k = 0;
                    ++seg_tile;
                }
            }
            loop_done = i == nsteps - 1;
        }
        if (sk_mode) {
            // Only a CTA's first and last tiles can be partial; their segments are in
            // the partials. The fold warps meet once on two mbarriers (bounded waits, so
            // a failed role elsewhere cannot leave them waiting): every warp's partials
            // are written before the leader's fence and counts, and the counts' verdict
            // comes back through sk_flag. The CTA that brings a tile's count of
            // segments to its total adds them in segment (= K) order and writes C.
            const uint32_t u_last = u_first + nsteps - 1;
            const uint32_t tf = u_first / ksteps, tl = u_last / ksteps;
            const bool part_f = u_first % ksteps != 0 || (tf == tl && u_last % ksteps != ksteps - 1);
            const bool part_l = tl != tf && u_last % ksteps != ksteps - 1;
            if (part_f || part_l) {
                __syncwarp();
                if (lane == 0) mbar_arrive(fsync0);
                bool ok = warp_wait_a8(fsync0, 0, deadline, abort_flag, kWaitFlush) && loop_done;
                if (warp == Cfg::kFold0 && lane == 0) {
                    int bits = 0;
                    if (ok && *abort_flag == 0) {
                        __threadfence();   // the CTA's partials, ordered by the meeting, before the counts
                        const uint32_t cf = part_f ? atomicAdd(sk.counters + tf, 1u) : 0u;
                        const uint32_t cl = part_l ? atomicAdd(sk.counters + tl, 1u) : 0u;
                        if (part_f && cf == stream_segments(tf, ksteps, sk.units, gridDim.x) - 1) bits |= 1;
                        if (part_l && cl == stream_segments(tl, ksteps, sk.units, gridDim.x) - 1) bits |= 2;
                        __threadfence();
                    }
                    *sk_flag = bits;
                    mbar_arrive(fsync1);
                }
                ok = warp_wait_a8(fsync1, 0, deadline, abort_flag, kWaitFlush) && ok;
                const int bits = ok ? *sk_flag : 0;
                // Each thread copies its slice of every segment into the (then idle)
                // weight ring with 16-byte asynchronous copies (one round trip), reads
                // back only its own copies and adds them in order.
                constexpr uint32_t kRingSegs = STAGES * kWTileBytes / (kTcRows * TN * 4u);
                float* mine = reinterpret_cast<float*>(sW) + static_cast<size_t>(row) * TN + m0;
                for (uint32_t j = 0; j < 2; ++j) {
                    if (!(bits & (1 << j))) continue;
                    const uint32_t t = j == 0 ? tf : tl;
                    const uint32_t nseg = stream_segments(t, ksteps, sk.units, gridDim.x);
                    const float* base = sk.parts + (static_cast<size_t>(t) * sk.maxseg * kTcRows + row) * TN + m0;
#pragma unroll
                    for (uint32_t tt = 0; tt < Cfg::kTokPerFold; ++tt) acc[tt] = 0.f;
                    for (uint32_t s0 = 0; s0 < nseg; s0 += kRingSegs) {
                        const uint32_t s1 = min(nseg, s0 + kRingSegs);
                        for (uint32_t sg = s0; sg < s1; ++sg) {
                            const float* src = base + static_cast<size_t>(sg) * kTcRows * TN;
                            float* dst = mine + static_cast<size_t>(sg - s0) * kTcRows * TN;
#pragma unroll
                            for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g)
                                cp_async_16(smem_u32(dst + 4 * g), src + 4 * g);
                        }
                        cp_async_commit();
                        cp_async_wait_group<0>();
                        for (uint32_t sg = s0; sg < s1; ++sg) {   // segment (= K) order
                            const float4* q4 =
                                reinterpret_cast<const float4*>(mine + static_cast<size_t>(sg - s0) * kTcRows * TN);
#pragma unroll
                            for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g) {
                                const float4 q = q4[g];
                                acc[4 * g] += q.x;
                                acc[4 * g + 1] += q.y;
                                acc[4 * g + 2] += q.z;
                                acc[4 * g + 3] += q.w;
                            }
                        }
                    }
                    sk_store(t, true);
                    if (warp == Cfg::kFold0 && lane == 0) sk.counters[t] = 0u;   // ready for the next call
                }
            }
        } else if (split_k == 1) {
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
            if (alias) cluster_arrive_release();
            cluster_wait();   // (alias) every rank's loads and MMAs are done: the rings may be overwritten
            // the last rank r with r * 128 / split_k <= row (no division by split_k)
            const uint32_t owner = ((row + 1) * split_k - 1) / kTcRows;
            const uint32_t lrow = row - owned_row0(owner, split_k);
            // receive layout [slot][row][token]: this thread's tokens are contiguous
            // and go as 16-byte groups; the owner reads them back the same way. Rows
            // this CTA owns stay in registers (its own slot of the layout is unused).
            const uint32_t off =
                ((tc_red_slot(rank, owner) * tc_red_rows(split_k) + lrow) * tc_red_stride(TN) +
                 fh * Cfg::kTokPerFold) * 4u;
            const uint32_t dst = dsmem_map(smem_u32(sRed) + off, owner);
            const uint32_t dbar = dsmem_map(red_bar, owner);
            const uint32_t ngroups = push_bytes(toks_valid, fh * Cfg::kTokPerFold, Cfg::kTokPerFold) / 16u;
            if (owner != rank) {
#pragma unroll
                for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g)   // groups past M are not sent
                    if (g < ngroups)
                        st_async_v4f32(dst + 16u * g, dbar, acc[4 * g], acc[4 * g + 1], acc[4 * g + 2],
                                       acc[4 * g + 3]);
            }
            // This CTA's own rows: the thread holding row `row` (and tokens
            // fh*kTokPerFold..) adds the ranks' partials in rank order, its own
            // rank's from its registers.
            // the partials are other CTAs' st.async writes: acquire at cluster scope
            const bool got = warp_wait_a8<true>(red_bar, 0, deadline + timeout_ns, abort_flag, kWaitRed);
            if (got && row >= my_row0 && row < my_row0 + my_rows && row < rows_valid) {
                const uint32_t lr = row - my_row0;
                const uint32_t rank_stride = tc_red_rows(split_k) * tc_red_stride(TN);   // floats
                const float* src_row = sRed + lr * tc_red_stride(TN);
                // Two ranks (the common split): the other rank's partials of every group
                // loaded first, then straight-line sums in rank order. Not in the 640-thread
                // instance, whose 96 registers a thread cannot hold them beside the fold's.
                constexpr bool kFlat2 = w8a8_threads(TN, TERMS) <= 384u;
                if (kFlat2 && split_k == 2) {
                    float4 q[Cfg::kTokPerFold / 4];
#pragma unroll
                    for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g)   // slot 0: the other rank
                        q[g] = *reinterpret_cast<const float4*>(src_row + fh * Cfg::kTokPerFold + 4u * g);
#pragma unroll
                    for (uint32_t g = 0; g < Cfg::kTokPerFold / 4; ++g) {
                        const uint32_t t = fh * Cfg::kTokPerFold + 4u * g;
                        const float mine[4] = {acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]};
                        const float other[4] = {q[g].x, q[g].y, q[g].z, q[g].w};
#pragma unroll
                        for (uint32_t u = 0; u < 4; ++u) {
                            float v = 0.f;   // as the general loop: 0 + rank 0's + rank 1's
                            v += rank == 0 ? mine[u] : other[u];
                            v += rank == 0 ? other[u] : mine[u];
                            if (t + u < toks_valid)
                                C[static_cast<size_t>(token0 + t + u) * ldc + tile * kTcRows + row] =
                                    __float2bfloat16_rn(v);
                        }
                    }
                } else {
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
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tP, Cfg::kTmemCols);
    }
}

using A8KernelFn = void (*)(CUtensorMap, CUtensorMap, const float*, uint32_t, const float*, __nv_bfloat16*,
                            uint32_t, uint32_t, uint32_t, uint32_t, uint32_t, uint32_t, uint32_t, StreamK,
                            uint64_t);
struct A8Instance {
    uint32_t tn, stages, terms;
    bool stream_k;
    A8KernelFn fn;
};
#define W8A16_A8_INST(TN_, ST_, T_) {TN_, ST_, T_, false, &w8a16_w8a8_kernel<TN_, ST_, T_>}
#define W8A16_A8_SK(TN_, ST_) {TN_, ST_, 2, true, &w8a16_w8a8_kernel<TN_, ST_, 2, true>}
const A8Instance kA8Instances[] = {
    W8A16_A8_INST(16, 4, 1), W8A16_A8_INST(16, 6, 1), W8A16_A8_INST(32, 4, 1), W8A16_A8_INST(32, 6, 1),
    W8A16_A8_INST(64, 4, 1), W8A16_A8_INST(64, 6, 1), W8A16_A8_INST(128, 4, 1),
    W8A16_A8_INST(16, 4, 2), W8A16_A8_INST(32, 4, 2), W8A16_A8_INST(32, 6, 2), W8A16_A8_INST(64, 4, 2),
    W8A16_A8_INST(64, 6, 2), W8A16_A8_INST(128, 4, 2),
    W8A16_A8_SK(16, 4), W8A16_A8_SK(32, 4),
};
#undef W8A16_A8_INST
#undef W8A16_A8_SK
constexpr int kNumA8 = sizeof(kA8Instances) / sizeof(kA8Instances[0]);

int find_a8(uint32_t tn, uint32_t stages, uint32_t terms, bool stream_k = false) {
    for (int i = 0; i < kNumA8; ++i)
        if (kA8Instances[i].tn == tn && kA8Instances[i].stages == stages && kA8Instances[i].terms == terms &&
            kA8Instances[i].stream_k == stream_k)
            return i;
    return -1;
}

cudaError_t ensure_attributes_a8(int inst, int device) {
    static std::mutex mu;
    static bool done[64][kNumA8] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (done[device][inst]) return cudaSuccess;
    const A8Instance& k = kA8Instances[inst];
    uint32_t most = 0;
    for (uint32_t sp = 1; sp <= 16; ++sp) {
        const uint32_t b = w8a8_smem_bytes(k.tn, k.stages, sp, k.terms);
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

bool w8a8_supported_stages(uint32_t tn, uint32_t stages, uint32_t terms) {
    return find_a8(tn, stages, terms) >= 0;
}

int launch_w8a8(const W8A8Args& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
                uint32_t flags, std::string* err) {
    const int inst = find_a8(p.token_tile, p.stages, g.terms, g.sk.units != 0);
    if (inst < 0) {
        *err = "no FP8 x FP8 kernel instance for token_tile=" + std::to_string(p.token_tile) +
               " stages=" + std::to_string(p.stages) + " terms=" + std::to_string(g.terms) +
               (g.sk.units ? " (stream-K)" : "");
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_attributes_a8(inst, dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("W8A8 kernel attribute setup failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    GemmArgs wg{};
    wg.W = g.W;
    wg.N = g.N;
    wg.K = g.K;
    CUtensorMap mw, mx;
    if (!tc_tensor_map_w(wg, dev, &mw, err) ||
        !tensor_map_act_codes(g.A, g.M * g.terms, g.K, g.lda, p.token_tile, dev, &mx, err))
        return W8A16_ERR_LAUNCH;
    const uint32_t row_tiles = (g.N + kTcRows - 1) / kTcRows;
    if (g.sk.units != 0) {
        // Stream-K: grid[0] persistent CTAs share the units in contiguous ranges, one
        // token tile, no clusters.
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3(p.grid[0], 1, 1);
        cfg.blockDim = dim3(w8a8_threads(p.token_tile, g.terms), 1, 1);
        cfg.dynamicSmemBytes = w8a8_smem_bytes(p.token_tile, p.stages, 1, g.terms);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = (flags & W8A16_FLAG_PDL) ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kA8Instances[inst].fn, mw, mx, g.a_scale, g.a_scale_stride, g.scale,
                               static_cast<__nv_bfloat16*>(g.C), g.ldc, g.M, g.N, g.K, 1u, 0u, 0u, g.sk, timeout_ns);
        if (e != cudaSuccess) {
            cudaGetLastError();
            *err = std::string("W8A8 kernel launch failed: ") + cudaGetErrorString(e);
            return W8A16_ERR_LAUNCH;
        }
        return W8A16_OK;
    }
    // One launch, or (a split-K tail) two: whole tiles [0, T - tail) at the plan's
    // split, then tiles [T - tail, T) over clusters of tail_split CTAs, queued as a
    // programmatic dependent launch of the first (which writes neither W nor its scales).
    const uint32_t tail = p.tail_split > 1 ? p.tail_tiles : 0u;
    for (uint32_t part = 0; part < (tail ? 2u : 1u); ++part) {
        const uint32_t split = part == 0 ? p.split_k : p.tail_split;
        const uint32_t tile0 = part == 0 ? 0u : row_tiles - tail;
        const uint32_t ctas = part == 0 ? p.grid[0] : tail * p.tail_split;
        if (ctas == 0) continue;
        const uint32_t tok_major = (split == 1 && p.grid[1] > 1 && ctas <= 65535u) ? 1u : 0u;
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = tok_major ? dim3(p.grid[1], ctas, 1) : dim3(ctas, p.grid[1], 1);
        cfg.blockDim = dim3(w8a8_threads(p.token_tile, g.terms), 1, 1);
        cfg.dynamicSmemBytes = w8a8_smem_bytes(p.token_tile, p.stages, split, g.terms);
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = split;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = (part == 1 || (flags & W8A16_FLAG_PDL)) ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kA8Instances[inst].fn, mw, mx, g.a_scale, g.a_scale_stride, g.scale,
                               static_cast<__nv_bfloat16*>(g.C), g.ldc, g.M, g.N, g.K, split, tile0,
                               tok_major, StreamK{}, timeout_ns);
        if (e != cudaSuccess) {
            cudaGetLastError();
            *err = std::string("W8A8 kernel launch failed: ") + cudaGetErrorString(e);
            return W8A16_ERR_LAUNCH;
        }
    }
    return W8A16_OK;
}

int w8a8_cluster_capacity(uint32_t tn, uint32_t stages, uint32_t terms, uint32_t cluster, uint32_t* ctas,
                          std::string* err) {
    const int inst = find_a8(tn, stages, terms);
    if (inst < 0 || cluster < 1 || cluster > 16) {
        *err = "no W8A8 kernel instance, or cluster size outside 1..16";
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_attributes_a8(inst, dev);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(cluster * 64, 1, 1);
    cfg.blockDim = dim3(w8a8_threads(tn, terms), 1, 1);
    cfg.dynamicSmemBytes = w8a8_smem_bytes(tn, stages, cluster, terms);
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
        e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kA8Instances[inst].fn), &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("cudaOccupancyMaxActiveClusters failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_DEVICE;
    }
    *ctas = static_cast<uint32_t>(n) * cluster;
    return W8A16_OK;
}

cudaError_t w8a8_status_read(StatusWord* out, bool clear, cudaStream_t s) {
    DeviceStatus st;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&st, g_w8a8_status, sizeof st, 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    out->code = st.code;
    out->where = st.where;
    out->detail = st.detail;
    if (clear) {
        const DeviceStatus zero{0, 0, 0};
        e = cudaMemcpyToSymbolAsync(g_w8a8_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace w8a16
