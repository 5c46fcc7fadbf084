// Tensor-core W8A16 kernel for sm_103a (tcgen05 + TMA), and its launcher.
//
// Operation and checks: page "metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs"
// (doc comment of `w8a16_gemm_pipelined_m32_strided`). The page's GB10 design
// (32x32 output tile, cp.async staging, an E4M3 table in shared memory, an 8-warp
// skinny body) is prior art; what is kept is its arithmetic: 128-K steps equal to
// the scale block, each step's product folded into an FP32 accumulator with that
// block's scale (doc comments of `W8A16_M32_K_BLOCK` and the module doc's "fold
// points"), and split-K partials added in a fixed step order (doc comment of
// `W8A16_M16_MAX_ROWS`).
//
// Mapping to Blackwell:
//   * swap-AB: 128 weight rows are the MMA's M, the tokens (rows of A, padded to
//     the token tile TN = 16..128) are its N, so a decode call wastes no MMA rows
//     on padding and the whole token range of one tile streams W exactly once;
//   * warp 0 (one thread) streams 128x128 E4M3 weight tiles with TMA (128-byte
//     swizzle) into a ring of STAGES shared-memory slots; the first slots are
//     requested before the CTA barrier, and before waiting on the previous grid
//     (programmatic dependent launch: the caller guarantees W is not written);
//   * warp 2 (one thread) waits on the previous grid, then streams the TNx128
//     BF16 activation tile of each K step into its own ring;
//   * NC converter warps (16 for TN <= 32, else 8) take 32 weight rows x a K
//     slice of a step each, convert E4M3 to BF16 in registers (exact) and write
//     them with tcgen05.st into one of NA TMEM operand buffers;
//   * warp 1 (one thread) allocates TMEM and issues 8 tcgen05.mma (K = 16 each)
//     per step with A in TMEM and the activations in shared memory, into one of
//     NP TMEM product buffers P, committing each step to an mbarrier;
//   * NF fold warps read P back (tcgen05.ld) and fold acc += scale * P in FP32
//     registers, one scale per (tile, step), then store or push the partials;
//   * split-K: a cluster of split_k CTAs shares one weight tile, each CTA on a
//     contiguous range of K steps; every CTA owns a slice of the tile's rows and
//     receives the other ranks' partials of that slice in shared memory
//     (st.async over distributed shared memory), summing them in rank (= K)
//     order. No global scratch, no atomics: deterministic.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

#include "w8a16_cluster.cuh"
#include "w8a16_device.cuh"
#include "w8a16_internal.h"

namespace w8a16 {

__device__ DeviceStatus g_tc_status;

namespace {

constexpr uint32_t kWTileBytes = kTcRows * kKStep;   // 16 KiB of E4M3 per stage
constexpr uint32_t kABufCols = kKStep / 2;            // TMEM columns of one BF16 W tile

// Wait-detail codes (which barrier a timed-out wait was on).
enum : uint32_t {
    kWaitFull = 1, kWaitEmpty = 2, kWaitAFull = 3, kWaitAEmpty = 4, kWaitPFull = 5,
    kWaitPEmpty = 6, kWaitMmaDone = 7, kWaitDrain = 8, kWaitRed = 9
};

template <uint32_t TN, uint32_t STAGES>
struct TcCfg {
    static constexpr uint32_t SA = tc_act_stages(TN);          // activation ring depth
    static constexpr uint32_t kActBytes = TN * kKStep * 2;     // BF16, two 64-K boxes
    static constexpr uint32_t kTmemCols = tc_tmem_cols(TN);
    static constexpr uint32_t NC = tc_conv_warps(TN);
    static constexpr uint32_t kKPerConv = kKStep * 4 / NC;     // K of a step per converter warp
    static constexpr uint32_t NA = tc_a_bufs(TN);
    static constexpr uint32_t ND = SA > NA ? SA : NA;          // MMA-completion barriers (>= 4)
    static constexpr uint32_t NF = tc_fold_warps(TN);
    static constexpr uint32_t NP = tc_p_bufs(TN);
    static constexpr uint32_t kConv0 = 3;                       // first converter warp
    static constexpr uint32_t kFold0 = kConv0 + NC;             // first fold warp
    static constexpr uint32_t kTokPerFold = TN * 4 / NF;        // tokens per fold thread
    // barriers: wfull/wempty[S], xfull[SA], tfull[NA], mdone[ND], pempty[NP], done, red
    static constexpr uint32_t kNumBars = 2 * STAGES + SA + NA + ND + NP + 2;
    static_assert(NA >= 2 && NA * 64 + NP * TN <= kTmemCols, "TMEM budget");
    static_assert(ND >= SA && ND >= NA && ND >= NP, "a completion barrier is never lapped");
    static_assert(kKPerConv == 32 || kKPerConv == 64, "converter K slice");
    static_assert(kTokPerFold % 8 == 0, "fold loads are whole x8 column groups");
    static_assert(kNumBars * 8 + 16 <= 1024, "barrier area");
    // Two MMA issuers take alternate steps; each waits only on steps of its own
    // parity, so a slot index it waits on must recur on its own steps.
    static_assert(SA % 2 == 0 && NA % 2 == 0 && NP % 2 == 0, "rings of even depth");
    static constexpr uint32_t kIssuer2 = kFold0 + NF;        // warp of the second MMA issuer
};






template <uint32_t NREG>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[NREG]) {
    if constexpr (NREG == 32) {
        tmem_st_32x32b_x32(taddr, r);
    } else {
        static_assert(NREG == 16, "16 or 32 columns per converter store");
        tmem_st_32x32b_x16(taddr, r);
    }
}

// Warp-uniform bounded wait: every lane polls; the warp proceeds only if all did.
template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t deadline,
                                          volatile int* abort_flag, uint32_t detail) {
    const bool ok = mbar_wait<CLUSTER>(bar, parity, deadline, abort_flag, &g_tc_status, detail);
    return __all_sync(0xFFFFFFFFu, ok);
}


// Wait until the last `depth` copies a producer issued into a ring have landed.
__device__ __forceinline__ void drain_ring(uint32_t bar_base, uint32_t depth, uint32_t issued,
                                           uint64_t timeout_ns) {
    const uint64_t dl = globaltimer_ns() + timeout_ns;
    for (uint32_t j = issued > depth ? issued - depth : 0; j < issued; ++j) {
        volatile int never = 0;
        mbar_wait(bar_base + 8u * (j % depth), (j / depth) & 1, dl, &never, &g_tc_status,
                  kWaitDrain);
    }
}

template <uint32_t TN, uint32_t STAGES>
__global__ void __launch_bounds__(tc_threads(TN), 1)
    w8a16_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                    const float* __restrict__ scale, __nv_bfloat16* __restrict__ C, uint32_t ldc,
                    uint32_t M, uint32_t N, uint32_t K, uint32_t split_k, uint32_t tile0,
                    uint32_t tok_major, uint64_t timeout_ns) {
    using Cfg = TcCfg<TN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sW = smem;                                    // STAGES x 16 KiB of E4M3 codes
    uint8_t* sX = smem + STAGES * kWTileBytes;             // SA x TN x 128 BF16 activations
    float* sRed = reinterpret_cast<float*>(sX + Cfg::SA * Cfg::kActBytes);   // split-K slots
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sRed) +
                                                 tc_red_bytes(TN, split_k));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    // mdone[i % ND] completes when the MMAs of step i have: it frees activation
    // slot i % SA, TMEM operand buffer i % NA, and fills product buffer i % NP.
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t wfull0 = bar0, wempty0 = wfull0 + 8u * STAGES;
    const uint32_t xfull0 = wempty0 + 8u * STAGES;
    const uint32_t tfull0 = xfull0 + 8u * Cfg::SA;
    const uint32_t mdone0 = tfull0 + 8u * Cfg::NA;
    const uint32_t pempty0 = mdone0 + 8u * Cfg::ND;
    const uint32_t done_bar = pempty0 + 8u * Cfg::NP;
    const uint32_t red_bar = done_bar + 8u;

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tok_major (no split): the token tiles of one weight tile are consecutive CTAs, so
    // beyond 128 tokens the later ones find the tile's weights in L2
    const uint32_t bx = tok_major ? blockIdx.y : blockIdx.x, by = tok_major ? blockIdx.x : blockIdx.y;
    const uint32_t tile = tile0 + bx / split_k;   // cluster = split_k consecutive CTAs
    const uint32_t rank = bx % split_k;           // == rank in the cluster
    const uint32_t token0 = by * TN;
    const uint32_t ksteps = K / kKStep;
    const uint32_t s_begin = static_cast<uint32_t>(static_cast<uint64_t>(rank) * ksteps / split_k);
    const uint32_t s_end = static_cast<uint32_t>(static_cast<uint64_t>(rank + 1) * ksteps / split_k);
    const uint32_t nsteps = s_end - s_begin;
    uint64_t deadline = globaltimer_ns() + timeout_ns;   // restarted by each role after the dependency wait
    const uint32_t my_row0 = owned_row0(rank, split_k);
    const uint32_t my_rows = owned_row0(rank + 1, split_k) - my_row0;
    const uint32_t npre = nsteps < STAGES ? nsteps : STAGES;
    const uint32_t toks_valid = min(TN, M - token0);

    if (warp == 0) {
        // barrier b is initialised by lane b % 32 (arrival counts by kind)
        for (uint32_t b = lane; b < Cfg::kNumBars; b += 32) {
            const uint32_t addr = bar0 + 8u * b;
            uint32_t count = 1;
            if (addr >= wempty0 && addr < xfull0) count = Cfg::NC;        // converters
            else if (addr >= tfull0 && addr < mdone0) count = Cfg::NC;    // converters
            else if (addr >= pempty0 && addr < done_bar) count = Cfg::NF; // fold warps
            else if (addr == done_bar) count = 2;                           // MMA issuers
            mbar_init(addr, count);
        }
        if (lane == 0) *abort_flag = 0;
        fence_barrier_init();
        __syncwarp();
    }
    if (threadIdx.x == 0) {
        if (split_k > 1)   // every other rank pushes its partials of my rows here
            mbar_arrive_expect_tx(red_bar,
                                  (split_k - 1) * my_rows * red_row_bytes<TN, Cfg::kTokPerFold>(toks_valid));
        // The first ring's weight tiles go out before anything else (TMEM
        // allocation, the CTA barrier), so their HBM latency overlaps the set-up.
        // Weights are requested before waiting on the previous grid in the
        // stream: under a programmatic launch the caller guarantees that grid
        // does not write W.
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
    // Peers may push into this CTA's receive buffer once the cluster barrier
    // completes; arrive now, wait only before the first push.
    if (split_k > 1) cluster_arrive();
    // Dependents may be scheduled from here on: this CTA holds its TMEM already.
    if (threadIdx.x == 0) grid_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tA = tmem_base;                         // NA x 64 columns: BF16 weight tiles
    const uint32_t tP = tmem_base + Cfg::NA * kABufCols;   // NP x TN columns: FP32 products
    const uint32_t quarter = warp & 3;                     // TMEM lanes this warp may access
    const uint32_t row = quarter * 32 + lane;              // weight row within the tile
    const uint32_t lane_bits = (quarter * 32) << 16;
    const bool is_conv = warp >= Cfg::kConv0 && warp < Cfg::kFold0;
    const bool is_fold = warp >= Cfg::kFold0 && warp < Cfg::kFold0 + Cfg::NF;
    const uint32_t rows_valid = min(kTcRows, N - tile * kTcRows);

    if (warp == 0) {
        // ------------------------------------------- weight producer (TMA)
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();   // W is streamed once
            uint32_t issued = npre;                            // issued at set-up
            for (uint32_t i = npre; i < nsteps; ++i) {
                const uint32_t s = i % STAGES;
                // Converters release the slots of the first NA + 1 steps before any
                // MMA has run; later slots free only after the dependency wait.
                if (i == STAGES + Cfg::NA + 1) deadline = deadline_after_dependency(timeout_ns);
                if (!mbar_wait(wempty0 + 8u * s, ((i / STAGES) - 1) & 1, deadline, abort_flag,
                               &g_tc_status, kWaitEmpty))
                    break;
                mbar_arrive_expect_tx(wfull0 + 8u * s, kWTileBytes);
                tma_load_2d(smem_u32(sW + s * kWTileBytes), &tmW, wfull0 + 8u * s,
                            static_cast<int32_t>((s_begin + i) * kKStep),
                            static_cast<int32_t>(tile * kTcRows), pol_w);
                issued = i + 1;
            }
            // every issued copy lands before the CTA may exit
            drain_ring(wfull0, STAGES, issued, timeout_ns);
        }
    } else if (warp == 2) {
        // --------------------------------------- activation producer (TMA)
        if (lane == 0) {
            const uint64_t pol_a = l2_policy_evict_last();    // A is re-read by every tile
            // A may be written by the previous grid in the stream: wait for it
            // (returns at once unless launched as a programmatic dependent).
            deadline = deadline_after_dependency(timeout_ns);
            uint32_t issued = 0;
            for (uint32_t i = 0; i < nsteps; ++i) {
                const uint32_t j = i % Cfg::SA;
                if (i >= Cfg::SA) {   // slot j last held step i - SA: wait for its MMAs
                    const uint32_t q = i - Cfg::SA;
                    if (!mbar_wait(mdone0 + 8u * (q % Cfg::ND), (q / Cfg::ND) & 1, deadline,
                                   abort_flag, &g_tc_status, kWaitEmpty))
                        break;
                }
                mbar_arrive_expect_tx(xfull0 + 8u * j, Cfg::kActBytes);
                const int32_t k = static_cast<int32_t>((s_begin + i) * kKStep);
                const uint32_t dst = smem_u32(sX + j * Cfg::kActBytes);
                tma_load_2d(dst, &tmA, xfull0 + 8u * j, k, static_cast<int32_t>(token0), pol_a);
                tma_load_2d(dst + TN * 128, &tmA, xfull0 + 8u * j, k + 64,
                            static_cast<int32_t>(token0), pol_a);
                issued = i + 1;
            }
            drain_ring(xfull0, Cfg::SA, issued, timeout_ns);
        }
    } else if (warp == 1 || warp == Cfg::kIssuer2) {
        // --------------------------------------------------------- MMA issuers
        // Two threads, even and odd steps: one thread's waits and fence overlap
        // the other's MMAs, so the tensor pipe rather than one issuing thread
        // sets the pace. Each commits its own steps (a commit covers the
        // issuing thread's MMAs only).
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTcRows, TN);
            deadline = deadline_after_dependency(timeout_ns);   // the activations come after it
            for (uint32_t i = (warp == 1 ? 0u : 1u); i < nsteps; i += 2) {
                const uint32_t a = i % Cfg::NA, p = i % Cfg::NP, j = i % Cfg::SA;
                if (!mbar_wait(tfull0 + 8u * a, (i / Cfg::NA) & 1, deadline, abort_flag,
                               &g_tc_status, kWaitAFull))
                    break;
                if (!mbar_wait(xfull0 + 8u * j, (i / Cfg::SA) & 1, deadline, abort_flag,
                               &g_tc_status, kWaitFull))
                    break;
                if (i >= Cfg::NP && !mbar_wait(pempty0 + 8u * p, ((i / Cfg::NP) - 1) & 1, deadline,
                                               abort_flag, &g_tc_status, kWaitPEmpty))
                    break;
                tc_fence_after();
                const uint32_t act = smem_u32(sX + j * Cfg::kActBytes);
#pragma unroll
                for (uint32_t kk = 0; kk < kKStep / 16; ++kk) {
                    const uint64_t bdesc =
                        smem_desc_kmajor_sw128(act + (kk >> 2) * (TN * 128) + (kk & 3) * 32);
                    tc_mma_a_tmem(tP + p * TN, tA + a * kABufCols + kk * 8, bdesc, idesc, kk > 0);
                }
                tc_commit(mdone0 + 8u * (i % Cfg::ND));
            }
            // All MMAs this thread issued must finish before TMEM is released.
            tc_commit(done_bar);
            volatile int never = 0;
            mbar_wait(done_bar, 0, globaltimer_ns() + timeout_ns, &never, &g_tc_status,
                      kWaitMmaDone);
        }
    } else if (is_conv) {
        // -------------------------------------- converters: E4M3 -> BF16 in TMEM
        // The NC/4 converter warps of one TMEM lane quarter split each step's K
        // into slices of kKPerConv codes (32 or 64) per row.
        const uint32_t slice = (warp - Cfg::kConv0) >> 2;
        constexpr uint32_t kChunks = Cfg::kKPerConv / 16;           // 16-byte chunks per row
        const uint32_t swz = row & 7;
        for (uint32_t i = 0; i < nsteps; ++i) {
            const uint32_t a = i % Cfg::NA, s = i % STAGES;
            if (!warp_wait(wfull0 + 8u * s, (i / STAGES) & 1, deadline, abort_flag, kWaitFull)) break;
            // Row `row`'s codes of this slice sit in 16-byte chunks slice*kChunks.., chunk
            // c at position c ^ (row & 7) (TMA's 128-byte swizzle).
            const uint8_t* rp = sW + s * kWTileBytes + row * 128;
            uint4 q[kChunks];
#pragma unroll
            for (uint32_t c = 0; c < kChunks; ++c)
                q[c] = *reinterpret_cast<const uint4*>(rp + (((slice * kChunks + c) ^ swz) << 4));
            // the codes are in registers; TMA refills the slot next, so order these
            // generic reads before that async-proxy write
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(wempty0 + 8u * s);
            uint32_t w[kChunks * 8];
#pragma unroll
            for (uint32_t c = 0; c < kChunks; ++c) {
                uint32_t o[8];
                e4m3x16_to_bf16x16(q[c], o);
#pragma unroll
                for (uint32_t t = 0; t < 8; ++t) w[8 * c + t] = o[t];
            }
            if (i >= Cfg::NA) {   // buffer a last held step i - NA: wait for its MMAs
                if (i == Cfg::NA) deadline = deadline_after_dependency(timeout_ns);
                const uint32_t q2 = i - Cfg::NA;
                if (!warp_wait(mdone0 + 8u * (q2 % Cfg::ND), (q2 / Cfg::ND) & 1, deadline, abort_flag,
                               kWaitAEmpty))
                    break;
            }
            tc_fence_after();
            tmem_st_cols<kChunks * 8>(tA + lane_bits + a * kABufCols + slice * (kChunks * 8), w);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tfull0 + 8u * a);
        }
    } else if (is_fold) {
        // ------------------------------- fold: acc += scale(step) * P(step)
        const uint32_t fh = (warp - Cfg::kFold0) >> 2;   // token group of this fold warp
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
            if (!warp_wait(mdone0 + 8u * (i % Cfg::ND), (i / Cfg::ND) & 1, deadline, abort_flag,
                           kWaitPFull))
                break;
            tc_fence_after();
            const float sc = __shfl_sync(0xFFFFFFFFu, sc_cur, i & 31u);
            const uint32_t pcol = tP + lane_bits + p * TN + fh * Cfg::kTokPerFold;
            // up to 32 columns per wait (16 when the accumulators are wide, to
            // bound register use)
            constexpr uint32_t kChunk = Cfg::kTokPerFold > 32 ? 16u : 32u;
#pragma unroll
            for (uint32_t c = 0; c < Cfg::kTokPerFold; c += kChunk) {
                float v0[16], v1[16];
                tmem_ld_32x32b_x16(pcol + c, v0);
                if (kChunk == 32 && c + 16 < Cfg::kTokPerFold) tmem_ld_32x32b_x16(pcol + c + 16, v1);
                tc_wait_ld();
#pragma unroll
                for (uint32_t t = 0; t < 16; ++t) acc[c + t] = fmaf(sc, v0[t], acc[c + t]);
                if (kChunk == 32 && c + 16 < Cfg::kTokPerFold) {
#pragma unroll
                    for (uint32_t t = 0; t < 16; ++t) acc[c + 16 + t] = fmaf(sc, v1[t], acc[c + 16 + t]);
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
            // Split-K: push this row's partial to the rank owning the row (slot =
            // this CTA's rank). No CTA reads another's shared memory, so none has
            // to wait for the others before it exits.
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
            const bool got = warp_wait<true>(red_bar, 0, deadline + timeout_ns, abort_flag, kWaitRed);
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
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }

}

// One CTA, one thread: waits on an mbarrier nothing arrives on, so the bounded
// wait must run out, record W8A16_STATUS_WAIT_TIMEOUT and return. It lets a
// programmatic dependent start at once, so a call queued after it with
// W8A16_FLAG_PDL runs its set-up while this wait is still going.
__global__ void w8a16_wait_selftest_kernel(uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    grid_launch_dependents();
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    const uint64_t deadline = globaltimer_ns() + timeout_ns;
    mbar_wait(smem_u32(&bar), 0, deadline, &abort_flag, &g_tc_status, 0xFFu);
}

// ------------------------------------------------------ host: TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct MapKey {
    uint64_t ptr, rows, cols, stride;
    uint32_t box_rows, kind;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && rows == o.rows && cols == o.cols && stride == o.stride &&
               box_rows == o.box_rows && kind == o.kind;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
        h ^= (k.rows + 0x632BE59BD9B4E019ull + (h << 6) + (h >> 2));
        h ^= (k.cols + 0x85EBCA77C2B2AE63ull + (h << 6) + (h >> 2));
        h ^= (k.stride + (static_cast<uint64_t>(k.box_rows) << 32 | k.kind) + (h << 6) + (h >> 2));
        return static_cast<size_t>(h);
    }
};

// Descriptors depend only on (pointer, shape, pitch, box, device); a small cache
// keeps their encoding off the per-call path. Bounded: cleared when full.
bool get_map(const MapKey& key, int device, CUtensorMap* out, std::string* err) {
    static std::mutex mu;
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache[64];
    std::lock_guard<std::mutex> lock(mu);
    auto& c = cache[device & 63];
    auto it = c.find(key);
    if (it != c.end()) {
        *out = it->second;
        return true;
    }
    auto enc = encode_fn();
    if (!enc) {
        *err = "cuTensorMapEncodeTiled is not available from the CUDA driver";
        return false;
    }
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    // kinds: 0 E4M3 weights and 2 E4M3 activation codes (128-byte rows of a box),
    // 1 BF16 activations (64-value rows); all with the 128-byte swizzle
    const bool u8 = key.kind == 0 || key.kind == 2;
    const cuuint64_t dims[2] = {key.cols, key.rows};
    const cuuint64_t strides[1] = {key.stride};
    const cuuint32_t box[2] = {u8 ? 128u : 64u, key.box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     reinterpret_cast<void*>(key.ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed (CUresult " + std::to_string(static_cast<int>(r)) + ")";
        return false;
    }
    if (c.size() >= 256) c.clear();
    c.emplace(key, m);
    *out = m;
    return true;
}

using TcKernelFn = void (*)(CUtensorMap, CUtensorMap, const float*, __nv_bfloat16*, uint32_t,
                           uint32_t, uint32_t, uint32_t, uint32_t, uint32_t, uint32_t, uint64_t);

struct TcInstance {
    uint32_t tn, stages;
    TcKernelFn fn;
};

#define W8A16_TC_INST(TN_, ST_) {TN_, ST_, &w8a16_tc_kernel<TN_, ST_>}
const TcInstance kTcInstances[] = {
    W8A16_TC_INST(16, 4),  W8A16_TC_INST(16, 6),  W8A16_TC_INST(16, 8), W8A16_TC_INST(16, 10),
    W8A16_TC_INST(32, 3),  W8A16_TC_INST(32, 4),  W8A16_TC_INST(32, 6), W8A16_TC_INST(32, 8),
    W8A16_TC_INST(64, 4),  W8A16_TC_INST(64, 6),  W8A16_TC_INST(64, 8),
    W8A16_TC_INST(128, 4), W8A16_TC_INST(128, 6),
};
#undef W8A16_TC_INST
constexpr int kNumTcInstances = sizeof(kTcInstances) / sizeof(kTcInstances[0]);

int find_instance(uint32_t tn, uint32_t stages) {
    for (int i = 0; i < kNumTcInstances; ++i)
        if (kTcInstances[i].tn == tn && kTcInstances[i].stages == stages) return i;
    return -1;
}

// Function attributes (dynamic shared memory above 48 KiB, cluster sizes above
// 8) are per device: set once per (device, instance).
cudaError_t ensure_attributes(int inst, int device) {
    static std::mutex mu;
    static bool done[64][kNumTcInstances] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (done[device][inst]) return cudaSuccess;
    const TcInstance& k = kTcInstances[inst];
    // the largest request any split of this instance makes (capped at the limit)
    uint32_t most = 0;
    for (uint32_t sp = 1; sp <= 16; ++sp) {
        const uint32_t b = tc_smem_bytes(k.tn, k.stages, sp);
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

bool tc_supported_token_tile(uint32_t tn) {
    return tn == 16 || tn == 32 || tn == 64 || tn == 128;
}

bool tc_supported_stages(uint32_t tn, uint32_t stages) { return find_instance(tn, stages) >= 0; }

int launch_tc(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
              uint32_t flags, std::string* err) {
    const int inst = find_instance(p.token_tile, p.stages);
    if (inst < 0) {
        *err = "no TC kernel instance for token_tile=" + std::to_string(p.token_tile) +
               " stages=" + std::to_string(p.stages);
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_attributes(inst, dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("TC kernel attribute setup failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    CUtensorMap mw, ma;
    if (!get_map({reinterpret_cast<uint64_t>(g.W), g.N, g.K, g.K, kTcRows, 0}, dev, &mw, err) ||
        !get_map({reinterpret_cast<uint64_t>(g.A), g.M, g.K, static_cast<uint64_t>(g.lda) * 2,
                  p.token_tile, 1},
                 dev, &ma, err))
        return W8A16_ERR_LAUNCH;

    // One launch, or (a split-K tail) two: whole tiles [0, T - tail) at the plan's
    // split, then tiles [T - tail, T) over clusters of tail_split CTAs, queued as a
    // programmatic dependent launch of the first (which writes neither W nor its scales).
    const uint32_t row_tiles = (g.N + kTcRows - 1) / kTcRows;
    const uint32_t tail = p.tail_split > 1 ? p.tail_tiles : 0u;
    for (uint32_t part = 0; part < (tail ? 2u : 1u); ++part) {
        const uint32_t split = part == 0 ? p.split_k : p.tail_split;
        const uint32_t ctas = part == 0 ? p.grid[0] : tail * p.tail_split;
        if (ctas == 0) continue;
        const uint32_t tok_major = (split == 1 && p.grid[1] > 1 && ctas <= 65535u) ? 1u : 0u;
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = tok_major ? dim3(p.grid[1], ctas, 1) : dim3(ctas, p.grid[1], 1);
        cfg.blockDim = dim3(tc_threads(p.token_tile), 1, 1);
        cfg.dynamicSmemBytes = tc_smem_bytes(p.token_tile, p.stages, split);
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
        e = cudaLaunchKernelEx(&cfg, kTcInstances[inst].fn, mw, ma, g.scale,
                               static_cast<__nv_bfloat16*>(g.C), g.ldc, g.M, g.N, g.K, split,
                               part == 0 ? 0u : row_tiles - tail, tok_major, timeout_ns);
        if (e != cudaSuccess) {
            cudaGetLastError();
            *err = std::string("TC kernel launch failed: ") + cudaGetErrorString(e);
            return W8A16_ERR_LAUNCH;
        }
    }
    return W8A16_OK;
}

bool tc_tensor_map_w(const GemmArgs& g, int device, CUtensorMap* out, std::string* err) {
    return get_map({reinterpret_cast<uint64_t>(g.W), g.N, g.K, g.K, kTcRows, 0}, device, out, err);
}

bool tensor_map_act_codes(const void* codes, uint32_t M, uint32_t K, uint32_t row_stride,
                          uint32_t token_tile, int device, CUtensorMap* out, std::string* err) {
    return get_map({reinterpret_cast<uint64_t>(codes), M, K, row_stride, token_tile, 2}, device, out,
                   err);
}

bool tc_tensor_map_a(const GemmArgs& g, uint32_t token_tile, int device, CUtensorMap* out,
                     std::string* err) {
    return get_map({reinterpret_cast<uint64_t>(g.A), g.M, g.K, static_cast<uint64_t>(g.lda) * 2,
                    token_tile, 1},
                   device, out, err);
}

int tc_cluster_capacity(uint32_t tn, uint32_t stages, uint32_t cluster, uint32_t* ctas,
                        std::string* err) {
    const int inst = find_instance(tn, stages);
    if (inst < 0 || cluster < 1 || cluster > 16) {
        *err = "no TC kernel instance, or cluster size outside 1..16";
        return W8A16_ERR_PLAN;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = ensure_attributes(inst, dev);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(cluster * 64, 1, 1);
    cfg.blockDim = dim3(tc_threads(tn), 1, 1);
    cfg.dynamicSmemBytes = tc_smem_bytes(tn, stages, cluster);
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
        e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kTcInstances[inst].fn),
                                           &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("cudaOccupancyMaxActiveClusters failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_DEVICE;
    }
    *ctas = static_cast<uint32_t>(n) * cluster;
    return W8A16_OK;
}

int launch_wait_selftest(uint64_t timeout_ns, cudaStream_t s, std::string* err) {
    w8a16_wait_selftest_kernel<<<1, 32, 0, s>>>(timeout_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("self-test launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
}

cudaError_t tc_status_read(StatusWord* out, bool clear, cudaStream_t s) {
    DeviceStatus st;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&st, g_tc_status, sizeof st, 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    out->code = st.code;
    out->where = st.where;
    out->detail = st.detail;
    if (clear) {
        const DeviceStatus zero{0, 0, 0};
        e = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace w8a16
