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
//   * warp 0 (one thread) streams 128x128 E4M3 weight tiles and the TNx128 BF16
//     activation tile of each K step with TMA (128-byte swizzle) into a ring of
//     STAGES shared-memory slots;
//   * 8 converter warps each take 32 weight rows x 64 K of a step, convert E4M3
//     to BF16 in registers (exact) and write them with tcgen05.st into one of two
//     TMEM operand buffers;
//   * warp 1 (one thread) issues 8 tcgen05.mma (K = 16 each) per step with A in
//     TMEM and the activations in shared memory, into one of two TMEM product
//     buffers P, and commits to mbarriers;
//   * the converter warps read P back (tcgen05.ld) and fold acc += scale * P in
//     FP32 registers, one scale per (tile, step);
//   * split-K: a cluster of split_k CTAs shares one weight tile, each CTA on a
//     contiguous range of K steps; partials meet in shared memory and each CTA
//     sums a slice of the outputs over the cluster's CTAs in rank (= K) order via
//     distributed shared memory. No global scratch, no atomics: deterministic.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

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
    kWaitPEmpty = 6, kWaitMmaDone = 7, kWaitDrain = 8
};

template <uint32_t TN, uint32_t STAGES>
struct TcCfg {
    static constexpr uint32_t kActBytes = TN * kKStep * 2;   // BF16, two 64-K boxes
    static constexpr uint32_t kStageBytes = kWTileBytes + kActBytes;
    static constexpr uint32_t kTmemCols = tc_tmem_cols(TN);
    static constexpr uint32_t kHalf = TN / 2;                 // tokens per converter warp
    static constexpr uint32_t kNumBars = 2 * STAGES + 9;
};

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Warp-uniform bounded wait: every lane polls; the warp proceeds only if all did.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t deadline,
                                          volatile int* abort_flag, uint32_t detail) {
    const bool ok = mbar_wait(bar, parity, deadline, abort_flag, &g_tc_status, detail);
    return __all_sync(0xFFFFFFFFu, ok);
}

template <uint32_t N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
    if constexpr (N == 8) {
        tmem_ld_32x32b_x8(taddr, v);
    } else {
        static_assert(N % 16 == 0, "token half must be 8 or a multiple of 16");
#pragma unroll
        for (uint32_t c = 0; c < N / 16; ++c) {
            float t[16];
            tmem_ld_32x32b_x16(taddr + 16 * c, t);
#pragma unroll
            for (uint32_t i = 0; i < 16; ++i) v[16 * c + i] = t[i];
        }
    }
}

template <uint32_t TN, uint32_t STAGES>
__global__ void __launch_bounds__(kTcThreads, TN <= 64 ? 2 : 1)
    w8a16_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                    const float* __restrict__ scale, __nv_bfloat16* __restrict__ C, uint32_t ldc,
                    uint32_t M, uint32_t N, uint32_t K, uint32_t split_k, uint64_t timeout_ns) {
    using Cfg = TcCfg<TN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sW = smem;                                   // STAGES x 16 KiB
    uint8_t* sA = smem + STAGES * kWTileBytes;            // STAGES x kActBytes
    uint64_t* bars = reinterpret_cast<uint64_t*>(sA + STAGES * Cfg::kActBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
    auto afull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + b); };
    auto aempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    auto pfull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 4 + b); };
    auto pempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 6 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 8);

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tile = blockIdx.x / split_k;     // cluster = split_k consecutive CTAs
    const uint32_t rank = blockIdx.x % split_k;     // == rank in the cluster
    const uint32_t token0 = blockIdx.y * TN;
    const uint32_t ksteps = K / kKStep;
    const uint32_t s_begin = static_cast<uint32_t>(static_cast<uint64_t>(rank) * ksteps / split_k);
    const uint32_t s_end = static_cast<uint32_t>(static_cast<uint64_t>(rank + 1) * ksteps / split_k);
    const uint32_t nsteps = s_end - s_begin;
    const uint64_t deadline = globaltimer_ns() + timeout_ns;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kTcConvWarps + 1);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(afull_bar(b), kTcConvWarps);
            mbar_init(aempty_bar(b), 1);
            mbar_init(pfull_bar(b), 1);
            mbar_init(pempty_bar(b), kTcConvWarps);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmA);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Dependents may be scheduled from here on: this CTA holds its TMEM already.
    if (threadIdx.x == 0) grid_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tA = tmem_base;                    // 2 x 64 columns: BF16 weight tiles
    const uint32_t tP = tmem_base + 2 * kABufCols;    // 2 x TN columns: FP32 step products

    float acc[Cfg::kHalf];
#pragma unroll
    for (uint32_t t = 0; t < Cfg::kHalf; ++t) acc[t] = 0.f;
    const uint32_t cw = warp - 2;                     // converter index 0..7
    const uint32_t quarter = warp & 3;                // TMEM lanes this warp may access
    const uint32_t khalf = cw >> 2;                   // which 64 K of a step / which token half
    const uint32_t row = quarter * 32 + lane;         // weight row within the tile
    const uint32_t lane_bits = (quarter * 32) << 16;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();   // W is streamed once
            const uint64_t pol_a = l2_policy_evict_last();    // A is re-read by every tile
            // The first ring's weight tiles are requested before waiting on the
            // previous grid in the stream (under a programmatic launch the caller
            // guarantees that grid does not write W); A is only read after the
            // wait. Without a programmatic launch the wait returns at once.
            const uint32_t npre = nsteps < STAGES ? nsteps : STAGES;
            for (uint32_t i = 0; i < npre; ++i) {
                mbar_arrive_expect_tx(full_bar(i), Cfg::kStageBytes);
                tma_load_2d(smem_u32(sW + i * kWTileBytes), &tmW, full_bar(i),
                            static_cast<int32_t>((s_begin + i) * kKStep),
                            static_cast<int32_t>(tile * kTcRows), pol_w);
            }
            grid_dependency_wait();
            for (uint32_t i = 0; i < npre; ++i) {
                const int32_t k = static_cast<int32_t>((s_begin + i) * kKStep);
                const uint32_t a_dst = smem_u32(sA + i * Cfg::kActBytes);
                tma_load_2d(a_dst, &tmA, full_bar(i), k, static_cast<int32_t>(token0), pol_a);
                tma_load_2d(a_dst + TN * 128, &tmA, full_bar(i), k + 64,
                            static_cast<int32_t>(token0), pol_a);
            }
            uint32_t issued = npre;
            for (uint32_t i = npre; i < nsteps; ++i) {
                const uint32_t s = i % STAGES, round = i / STAGES;
                if (!mbar_wait(empty_bar(s), (round - 1) & 1, deadline, abort_flag, &g_tc_status,
                               kWaitEmpty))
                    break;
                mbar_arrive_expect_tx(full_bar(s), Cfg::kStageBytes);
                const int32_t k = static_cast<int32_t>((s_begin + i) * kKStep);
                tma_load_2d(smem_u32(sW + s * kWTileBytes), &tmW, full_bar(s), k,
                            static_cast<int32_t>(tile * kTcRows), pol_w);
                const uint32_t a_dst = smem_u32(sA + s * Cfg::kActBytes);
                tma_load_2d(a_dst, &tmA, full_bar(s), k, static_cast<int32_t>(token0), pol_a);
                tma_load_2d(a_dst + TN * 128, &tmA, full_bar(s), k + 64,
                            static_cast<int32_t>(token0), pol_a);
                issued = i + 1;
            }
            // Every issued copy must land before the CTA may exit or reuse its
            // shared memory (on the normal path they already have).
            const uint64_t drain_deadline = globaltimer_ns() + timeout_ns;
            for (uint32_t j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j) {
                volatile int never = 0;
                mbar_wait(full_bar(j % STAGES), (j / STAGES) & 1, drain_deadline, &never,
                          &g_tc_status, kWaitDrain);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTcRows, TN);
            for (uint32_t i = 0; i < nsteps; ++i) {
                const uint32_t b = i & 1, use = i >> 1, s = i % STAGES;
                if (!mbar_wait(afull_bar(b), use & 1, deadline, abort_flag, &g_tc_status, kWaitAFull))
                    break;
                if (!mbar_wait(full_bar(s), (i / STAGES) & 1, deadline, abort_flag, &g_tc_status,
                               kWaitFull))
                    break;
                if (use > 0 && !mbar_wait(pempty_bar(b), (use - 1) & 1, deadline, abort_flag,
                                          &g_tc_status, kWaitPEmpty))
                    break;
                tc_fence_after();
                const uint32_t act = smem_u32(sA + s * Cfg::kActBytes);
#pragma unroll
                for (uint32_t j = 0; j < kKStep / 16; ++j) {
                    const uint64_t bdesc =
                        smem_desc_kmajor_sw128(act + (j >> 2) * (TN * 128) + (j & 3) * 32);
                    tc_mma_a_tmem(tP + b * TN, tA + b * kABufCols + j * 8, bdesc, idesc, j > 0);
                }
                tc_commit(pfull_bar(b));
                tc_commit(aempty_bar(b));
                tc_commit(empty_bar(s));
            }
            // All MMAs this thread issued must finish before TMEM is released.
            tc_commit(done_bar);
            volatile int never = 0;
            mbar_wait(done_bar, 0, globaltimer_ns() + timeout_ns, &never, &g_tc_status,
                      kWaitMmaDone);
        }
    } else {
        // ------------------------------------------- converters and scale fold
        const float* srow = scale + static_cast<size_t>(tile) * ksteps + s_begin;
        auto fold = [&](uint32_t j) -> bool {
            const uint32_t b = j & 1;
            if (!warp_wait(pfull_bar(b), (j >> 1) & 1, deadline, abort_flag, kWaitPFull))
                return false;
            tc_fence_after();
            float p[Cfg::kHalf];
            tmem_ld_cols<Cfg::kHalf>(tP + lane_bits + b * TN + khalf * Cfg::kHalf, p);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty_bar(b));
            const float sc = __ldg(srow + j);
#pragma unroll
            for (uint32_t t = 0; t < Cfg::kHalf; ++t) acc[t] = fmaf(sc, p[t], acc[t]);
            return true;
        };

        bool ok = true;
        const uint32_t swz = row & 7;
        for (uint32_t i = 0; i < nsteps && ok; ++i) {
            const uint32_t b = i & 1, use = i >> 1, s = i % STAGES;
            if (!warp_wait(full_bar(s), (i / STAGES) & 1, deadline, abort_flag, kWaitFull)) {
                ok = false;
                break;
            }
            // This thread's 64 codes: row `row`, K [64 khalf, 64 khalf + 64) of the
            // step, stored as 16-byte chunks 4 khalf + c at chunk (4 khalf + c) ^ (row & 7)
            // (TMA's 128-byte swizzle).
            const uint8_t* rp = sW + s * kWTileBytes + row * 128;
            uint4 q[4];
#pragma unroll
            for (uint32_t c = 0; c < 4; ++c)
                q[c] = *reinterpret_cast<const uint4*>(rp + (((4 * khalf + c) ^ swz) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));

            uint32_t w[32];
#pragma unroll
            for (uint32_t c = 0; c < 4; ++c) {
                uint32_t o[8];
                e4m3x16_to_bf16x16(q[c], o);
#pragma unroll
                for (uint32_t t = 0; t < 8; ++t) w[8 * c + t] = o[t];
            }
            if (use > 0 &&
                !warp_wait(aempty_bar(b), (use - 1) & 1, deadline, abort_flag, kWaitAEmpty)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st_32x32b_x32(tA + lane_bits + b * kABufCols + khalf * 32, w);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull_bar(b));
            if (i > 0 && !fold(i - 1)) ok = false;
        }
        if (ok && nsteps > 0) ok = fold(nsteps - 1);
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }

    const uint32_t rows_valid = min(kTcRows, N - tile * kTcRows);
    const uint32_t toks_valid = min(TN, M - token0);
    if (split_k == 1) {
        if (warp >= 2 && row < rows_valid) {
            const uint32_t n = tile * kTcRows + row;
#pragma unroll
            for (uint32_t t = 0; t < Cfg::kHalf; ++t) {
                const uint32_t m = khalf * Cfg::kHalf + t;
                if (m < toks_valid)
                    C[static_cast<size_t>(token0 + m) * ldc + n] = __float2bfloat16_rn(acc[t]);
            }
        }
        return;
    }

    // Split-K: partials to shared memory as red[token][row] (over the drained
    // ring), then every CTA of the cluster sums its slice of the outputs over
    // ranks 0..split_k-1 in order.
    float* red = reinterpret_cast<float*>(smem);
    if (warp >= 2) {
#pragma unroll
        for (uint32_t t = 0; t < Cfg::kHalf; ++t) red[(khalf * Cfg::kHalf + t) * kTcRows + row] = acc[t];
    }
    cluster_sync_all();
    {
        const uint32_t total = toks_valid * kTcRows;
        const uint32_t beg = static_cast<uint32_t>(static_cast<uint64_t>(rank) * total / split_k);
        const uint32_t end = static_cast<uint32_t>(static_cast<uint64_t>(rank + 1) * total / split_k);
        const uint32_t red_local = smem_u32(red);
        for (uint32_t idx = beg + threadIdx.x; idx < end; idx += kTcThreads) {
            const uint32_t tok = idx / kTcRows, r = idx % kTcRows;
            if (r >= rows_valid) continue;
            float v = 0.f;
            for (uint32_t src = 0; src < split_k; ++src)
                v += dsmem_ld_f32(dsmem_map(red_local + 4u * idx, src));
            C[static_cast<size_t>(token0 + tok) * ldc + tile * kTcRows + r] = __float2bfloat16_rn(v);
        }
    }
    cluster_sync_all();   // no CTA leaves while others still read its shared memory
}

// One CTA, one thread: waits on an mbarrier nothing arrives on, so the bounded
// wait must run out, record W8A16_STATUS_WAIT_TIMEOUT and return.
__global__ void w8a16_wait_selftest_kernel(uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
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
    const bool is_w = key.kind == 0;
    const cuuint64_t dims[2] = {key.cols, key.rows};
    const cuuint64_t strides[1] = {key.stride};
    const cuuint32_t box[2] = {is_w ? 128u : 64u, key.box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&m, is_w ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     reinterpret_cast<void*>(key.ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
                           uint32_t, uint32_t, uint32_t, uint32_t, uint64_t);

struct TcInstance {
    uint32_t tn, stages;
    TcKernelFn fn;
};

#define W8A16_TC_INST(TN_, ST_) {TN_, ST_, &w8a16_tc_kernel<TN_, ST_>}
const TcInstance kTcInstances[] = {
    W8A16_TC_INST(16, 4), W8A16_TC_INST(16, 6), W8A16_TC_INST(16, 8),
    W8A16_TC_INST(32, 4), W8A16_TC_INST(32, 6), W8A16_TC_INST(32, 8),
    W8A16_TC_INST(64, 3), W8A16_TC_INST(64, 4), W8A16_TC_INST(64, 6),
    W8A16_TC_INST(128, 4),
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
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(k.fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(tc_smem_bytes(k.tn, k.stages)));
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

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(p.grid[0], p.grid[1], 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = tc_smem_bytes(p.token_tile, p.stages);
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
    e = cudaLaunchKernelEx(&cfg, kTcInstances[inst].fn, mw, ma, g.scale,
                           static_cast<__nv_bfloat16*>(g.C), g.ldc, g.M, g.N, g.K, p.split_k,
                           timeout_ns);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *err = std::string("TC kernel launch failed: ") + cudaGetErrorString(e);
        return W8A16_ERR_LAUNCH;
    }
    return W8A16_OK;
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
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = tc_smem_bytes(tn, stages);
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
