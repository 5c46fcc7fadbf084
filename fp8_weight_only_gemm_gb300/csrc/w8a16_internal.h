// Definitions shared by the host dispatcher and the kernel translation units.
#pragma once

#include <cstdint>
#include <string>

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "w8a16.h"

namespace w8a16 {

struct GemmArgs {
    const void* A;
    uint32_t lda;
    const void* W;
    const float* scale;
    void* C;
    uint32_t ldc;
    uint32_t M, N, K;
};

// Persistent stream-K schedule of the FP8 x FP8 kernel (units = 0: the cluster
// split-K schedule instead). The grid's CTAs split the units (128-row weight
// tile, 128-K step), in tile-major order, into contiguous equal ranges; a tile
// whose steps fall to several CTAs is summed through `parts` (FP32 partials
// [tile][segment][128 rows][token tile]) by whichever of them finishes last,
// in segment (= K) order; `counters` [tiles] count finished segments and are
// zero when the kernel starts (the split pre-pass clears them; the last CTA of a
// tile resets its counter).
struct StreamK {
    float* parts;
    uint32_t* counters;
    uint32_t units;
    uint32_t maxseg;
};
// The CTA (of P) whose contiguous range [c U / P, (c + 1) U / P) holds unit u.
__host__ __device__ constexpr uint32_t stream_cta_of(uint64_t u, uint64_t units, uint64_t ctas) {
    return static_cast<uint32_t>(((u + 1) * ctas - 1) / units);
}
// How many CTAs' ranges cover tile t's units [t ksteps, (t + 1) ksteps).
__host__ __device__ constexpr uint32_t stream_segments(uint32_t t, uint32_t ksteps, uint64_t units, uint64_t ctas) {
    return stream_cta_of(static_cast<uint64_t>(t) * ksteps + ksteps - 1, units, ctas) -
           stream_cta_of(static_cast<uint64_t>(t) * ksteps, units, ctas) + 1;
}


// Operands of the FP8 x FP8 kernel: E4M3 activation codes with FP32 factors per
// token and 128-K group [K/128][a_scale_stride], the weights and C as in GemmArgs.
// terms = 1 (W8A8): codes [M][lda bytes], factors the group scales. terms = 2 (the
// W8A16 two-term split): codes [2M][lda bytes], hi terms in rows [0, M), lo terms
// (x32) in rows [M, 2M); factors 2^(E-7).
struct W8A8Args {
    const void* A;
    uint32_t lda;
    const float* a_scale;
    uint32_t a_scale_stride;
    const void* W;
    const float* scale;
    void* C;
    uint32_t ldc;
    uint32_t M, N, K;
    uint32_t terms;
    StreamK sk;   // zero-initialised: the cluster split-K schedule
};

struct StatusWord {
    uint32_t code, where, detail;
};


// Tiling constants of the tensor-core variant.
constexpr uint32_t kTcRows = 128;      // weight rows per tile (tcgen05 MMA M)
constexpr uint32_t kKStep = 128;       // K per pipeline stage == one scale block
constexpr uint32_t kTcMaxTokenTile = 128;
constexpr uint32_t kMaxDynSmem = 232448;   // per-CTA dynamic shared memory limit (227 KiB)

// Warp roles per CTA: a weight-tile TMA producer, the MMA issuer, an
// activation-tile TMA producer, 8 converter warps (E4M3 -> BF16 into TMEM) and
// fold warps (step products -> FP32 accumulators).
constexpr uint32_t tc_conv_warps(uint32_t tn) { return tn <= 32 ? 16u : 8u; }
constexpr uint32_t tc_fold_warps(uint32_t tn) { return tn <= 32 ? 4u : 8u; }
// + one warp whose lane 0 is the second MMA issuer (odd steps)
constexpr uint32_t tc_threads(uint32_t tn) {
    return 128u + 32u * (tc_conv_warps(tn) + tc_fold_warps(tn));
}
// Activation ring depth per token tile (its slots are held until the MMA that
// reads them completes; the weight ring's are released as soon as converted).
constexpr uint32_t tc_act_stages(uint32_t tn) {
    return tn == 16 ? 8u : tn == 32 ? 4u : 2u;   // even: two MMA issuers alternate steps
}
// TMEM: NA operand buffers of 64 columns (one BF16 128x128 weight tile) and NP
// product buffers of TN FP32 columns.
constexpr uint32_t tc_tmem_cols(uint32_t) { return 512u; }   // one CTA per SM
constexpr uint32_t tc_p_bufs(uint32_t tn) { return tn == 16 ? 4u : 2u; }
constexpr uint32_t tc_a_bufs(uint32_t tn) {   // even: two MMA issuers alternate steps
    return (tc_tmem_cols(tn) - tc_p_bufs(tn) * tn) / 64u >= 4u ? 4u : 2u;   // 4 for every TN
}
// Split-K receive buffer of one CTA: a slot per other cluster rank (a CTA's own
// partials of the rows it owns stay in registers) holding those rows (at most
// ceil(128/split)) x TN FP32 partials.
constexpr uint32_t tc_red_rows(uint32_t split) { return (kTcRows + split - 1) / split; }
// Receive layout [slot][row][token]: a row's TN partials are contiguous (16-byte
// pushes), rows padded by 4 floats so that consecutive rows start in different banks.
constexpr uint32_t tc_red_stride(uint32_t tn) { return tn + 4u; }
constexpr uint32_t tc_red_bytes(uint32_t tn, uint32_t split) {
    return split <= 1 ? 0u : (split - 1) * tc_red_rows(split) * tc_red_stride(tn) * 4u;
}
// The slot of rank src's partials in the receive buffer of rank owner (src != owner;
// 0 for src == owner, which has no slot, so that the index stays in range).
constexpr uint32_t tc_red_slot(uint32_t src, uint32_t owner) {
    return src < owner ? src : (src > owner ? src - 1u : 0u);
}
// A CTA that allocates all 512 TMEM columns must be alone on its SM (a second
// one would block in tcgen05.alloc): its dynamic shared memory is padded so that
// two can never fit in the SM's 228 KiB.
constexpr uint32_t kAloneSmem = 116u * 1024u;
constexpr uint32_t alone_if_full_tmem(uint32_t bytes, uint32_t tmem_cols) {
    return tmem_cols >= 512u && bytes < kAloneSmem ? kAloneSmem : bytes;
}
// Dynamic shared memory: 1 KiB alignment slack, the weight ring (`stages`
// 16 KiB slots), the activation ring, the receive buffer, barriers and flags.
constexpr uint32_t tc_smem_bytes(uint32_t tn, uint32_t stages, uint32_t split) {
    return alone_if_full_tmem(1024u + stages * kTcRows * kKStep + tc_act_stages(tn) * tn * kKStep * 2u +
                                  tc_red_bytes(tn, split) + 1024u,
                              tc_tmem_cols(tn));
}

// FP8-datapath variant (TC8): E4M3 weights straight from the TMA ring into
// kind::f8f6f4 MMAs, activations as two E4M3 terms (2 TN MMA columns).
constexpr uint32_t tc8_act_stages(uint32_t tn) { return tn <= 32 ? 4u : 2u; }
constexpr uint32_t tc8_b_stages(uint32_t tn) { return tn <= 32 ? 4u : 2u; }
constexpr uint32_t tc8_p_bufs(uint32_t) { return 4u; }
constexpr uint32_t tc8_split_warps(uint32_t tn) { return tn <= 32 ? 4u : 8u; }
constexpr uint32_t tc8_fold_warps(uint32_t tn) { return tn <= 32 ? 4u : 8u; }
constexpr uint32_t tc8_threads(uint32_t tn) {
    return 96u + 32u * (tc8_split_warps(tn) + tc8_fold_warps(tn));
}
constexpr uint32_t tc8_tmem_cols(uint32_t tn) {
    return tc8_p_bufs(tn) * 2u * tn <= 128u ? 128u : tc8_p_bufs(tn) * 2u * tn <= 256u ? 256u : 512u;
}
constexpr uint32_t tc8_smem_bytes(uint32_t tn, uint32_t stages, uint32_t split) {
    return alone_if_full_tmem(1024u + stages * kTcRows * kKStep + tc8_b_stages(tn) * 2u * tn * kKStep +
                                  tc8_act_stages(tn) * tn * kKStep * 2u + tc8_p_bufs(tn) * tn * 4u +
                                  tc_red_bytes(tn, split) + 1024u,
                              tc8_tmem_cols(tn));
}

// FP8 x FP8 kernel (W8A8, terms = 1; W8A16 from a two-term split, terms = 2): an
// activation ring of SA slots (terms x TN x 128 codes), NP product buffers of
// terms x TN columns, 4 fold warps (8 from a 64-token tile), two MMA issuers and
// the two producers in the first four warps; each fold warp stages its tokens'
// FP32 factors of a step in a private buffer. The 128-token two-term tile has
// room in TMEM for 2 product buffers of 256 columns.
// Activation-code stages: 4, and 2 for the 32-token two-term tile (4 measured no
// faster there; 2 keeps its split-K receive buffer beside the rings at two CTAs per
// SM with room to spare: no aliasing, so the partials go out as soon as a CTA's
// fold is done).
constexpr uint32_t w8a8_act_stages(uint32_t tn, uint32_t terms = 1) { return terms == 2 && tn == 32 ? 2u : 4u; }
constexpr uint32_t w8a8_p_bufs(uint32_t tn, uint32_t terms = 1) { return terms == 2 && tn >= 128 ? 2u : 4u; }
// (16 for the 128-token two-term tile, whose fold reads two 128-column halves)
constexpr uint32_t w8a8_fold_warps(uint32_t tn, uint32_t terms = 1) {
    return tn <= 32 ? 4u : (terms == 2 && tn >= 128 ? 16u : 8u);
}
constexpr uint32_t w8a8_threads(uint32_t tn, uint32_t terms = 1) { return 128u + 32u * w8a8_fold_warps(tn, terms); }
constexpr uint32_t pow2_at_least(uint32_t x, uint32_t p = 32u) { return p >= x ? p : pow2_at_least(x, 2u * p); }
constexpr uint32_t w8a8_tmem_cols(uint32_t tn, uint32_t terms = 1) {
    return pow2_at_least(w8a8_p_bufs(tn, terms) * terms * tn);
}
// Registers: the 64- and 128-token instances (384 or 640 threads) run one CTA per
// SM; the smaller ones are built for two.
constexpr uint32_t w8a8_max_ctas_by_regs(uint32_t tn) { return tn >= 64 ? 1u : 2u; }
// The fold warps' factor buffers: kTokPerFold FP32 per warp, 4 x TN in all.
constexpr uint32_t w8a8_factor_bytes(uint32_t tn) { return 16u * tn; }
constexpr uint32_t w8a8_ring_bytes(uint32_t tn, uint32_t stages, uint32_t terms = 1) {
    return stages * kTcRows * kKStep + w8a8_act_stages(tn, terms) * terms * tn * kKStep + w8a8_factor_bytes(tn);
}
// The split-K receive buffer normally follows the rings. Where that would not fit,
// or would cost CTAs per SM, it reuses the rings' memory instead ("alias"): then
// partials are pushed only after every rank of the cluster is past its K steps (a
// cluster barrier at the end of the loops rather than at set-up).
constexpr uint32_t w8a8_min3(uint32_t a, uint32_t b, uint32_t c) { return a < b ? (a < c ? a : c) : (b < c ? b : c); }
constexpr uint32_t w8a8_ctas_for(uint32_t bytes, uint32_t tn, uint32_t terms) {
    return w8a8_min3(233472u / (alone_if_full_tmem(bytes, w8a8_tmem_cols(tn, terms)) + 1024u),
                     512u / w8a8_tmem_cols(tn, terms), w8a8_max_ctas_by_regs(tn));
}
constexpr bool w8a8_red_alias(uint32_t tn, uint32_t stages, uint32_t split, uint32_t terms = 1) {
    return split > 1 &&
           (2048u + w8a8_ring_bytes(tn, stages, terms) + tc_red_bytes(tn, split) > kMaxDynSmem ||
            w8a8_ctas_for(2048u + w8a8_ring_bytes(tn, stages, terms) + tc_red_bytes(tn, split), tn, terms) <
                w8a8_ctas_for(2048u + (w8a8_ring_bytes(tn, stages, terms) > tc_red_bytes(tn, split)
                                           ? w8a8_ring_bytes(tn, stages, terms)
                                           : tc_red_bytes(tn, split)),
                              tn, terms));
}
constexpr uint32_t w8a8_smem_bytes(uint32_t tn, uint32_t stages, uint32_t split, uint32_t terms = 1) {
    return alone_if_full_tmem(
        2048u + (!w8a8_red_alias(tn, stages, split, terms)
                     ? w8a8_ring_bytes(tn, stages, terms) + tc_red_bytes(tn, split)
                     : (w8a8_ring_bytes(tn, stages, terms) > tc_red_bytes(tn, split) ? w8a8_ring_bytes(tn, stages, terms)
                                                                                     : tc_red_bytes(tn, split))),
        w8a8_tmem_cols(tn, terms));
}
// Decode kernel (W8A16_VARIANT_GEMV): one or two tokens; a cluster of split_k CTAs
// per 128-row weight tile, each on at most kGvMaxSteps 128-K steps, all of which
// are on chip before the grid-dependency wait: kGvSlots shared-memory slots, and
// the first kGvResident steps moved to TMEM to free theirs. Per CTA: 256 threads,
// < 113 KiB of shared memory and 128 TMEM columns (two CTAs per SM, so a call's
// CTAs fit beside the previous call's).
constexpr uint32_t kGvSlots = 5;
constexpr uint32_t kGvMaxSteps = 8;
constexpr uint32_t kGvResident = kGvMaxSteps - kGvSlots;
constexpr uint32_t kGvThreads = 256;
constexpr uint32_t kGvTmemCols = 128;          // kGvResident x 32 weight columns + 2 x 16 accumulators
constexpr uint32_t kGvMaxTokens = 2;
constexpr uint32_t kGvBStepBytes = 16u * kKStep;   // MMA B operand of one step: 16 rows x 128 K
constexpr uint32_t kGvRedBytes = 2304;         // >= split x ceil(128 / split) x 16 B for split <= 16
constexpr uint32_t gemv_smem_bytes() {
    return 1024u + kGvSlots * kTcRows * kKStep + kGvMaxSteps * kGvBStepBytes + kGvMaxSteps * kGvMaxTokens * 4u +
           kGvRedBytes + 256u;
}
static_assert(2u * (gemv_smem_bytes() + 1024u) <= 233472u, "two decode CTAs per SM");

// Stream-K workspace after the split's codes and factors: tile counters (256-byte
// aligned) and the partials [tiles][maxseg][128][token tile] FP32.
constexpr uint64_t align256(uint64_t x) { return (x + 255u) / 256u * 256u; }

// Workspace of the two-term split: codes [2M][K] (hi rows, then lo rows) and
// factors [K/128][round_up(M, 4)] FP32.
constexpr uint64_t split_ws_scale_stride(uint32_t M) { return (static_cast<uint64_t>(M) + 3u) / 4u * 4u; }
constexpr uint64_t split_ws_bytes(uint32_t M, uint32_t K) {
    return 2ull * M * K + 4ull * (K / kKStep) * split_ws_scale_stride(M);
}

// Kernel launchers (implemented in the kernel translation units). They assume
// the arguments and plan were validated; they return a W8A16_* code and, on
// failure, a message in *err.
int launch_simt(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint32_t flags,
                std::string* err);
int launch_tc(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
              uint32_t flags, std::string* err);
// CTAs of the TC instance (tn, stages) that can be co-resident on the current
// device when launched in clusters of `cluster` CTAs.
int tc_cluster_capacity(uint32_t tn, uint32_t stages, uint32_t cluster, uint32_t* ctas,
                        std::string* err);
// E4M3 activation codes [M][row_stride bytes] of the FP8 x FP8 kernel.
bool tensor_map_act_codes(const void* codes, uint32_t M, uint32_t K, uint32_t row_stride,
                          uint32_t token_tile, int device, CUtensorMap* out, std::string* err);
int launch_quantize(const void* W, bool bf16, uint32_t ldw, uint32_t N, uint32_t K, void* codes,
                    float* scales, cudaStream_t s, std::string* err);
int launch_w8a8(const W8A8Args& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
                uint32_t flags, std::string* err);
bool w8a8_supported_stages(uint32_t tn, uint32_t stages, uint32_t terms = 1);
int w8a8_cluster_capacity(uint32_t tn, uint32_t stages, uint32_t terms, uint32_t cluster, uint32_t* ctas,
                          std::string* err);
// The two-term split of BF16 activations into the workspace layout above.
int launch_split_act(const void* A, uint32_t lda, uint32_t M, uint32_t K, void* codes, float* factors,
                     uint32_t factor_stride, uint32_t* counters, uint32_t ncounters, cudaStream_t s,
                     std::string* err);
cudaError_t w8a8_status_read(StatusWord* out, bool clear, cudaStream_t s);
int launch_quantize_act(const void* A, uint32_t lda, uint32_t M, uint32_t K, void* codes, float* scales,
                        uint32_t scale_stride, cudaStream_t s, std::string* err);
int launch_tc8(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
               uint32_t flags, std::string* err);
int tc8_cluster_capacity(uint32_t tn, uint32_t stages, uint32_t cluster, uint32_t* ctas,
                         std::string* err);
bool tc8_supported_stages(uint32_t tn, uint32_t stages);
int launch_wait_selftest(uint64_t timeout_ns, cudaStream_t s, std::string* err);
int launch_gemv(const GemmArgs& g, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
                uint32_t flags, std::string* err);
// The decode kernel on E4M3 activations with per-token group scales (the W8A8 variant).
int launch_gemv_w8a8(const W8A8Args& a, const w8a16_plan_t& p, cudaStream_t s, uint64_t timeout_ns,
                     uint32_t flags, std::string* err);
int gemv_cluster_capacity(uint32_t cluster, uint32_t* ctas, std::string* err);
cudaError_t gemv_status_read(StatusWord* out, bool clear, cudaStream_t s);

// TMA descriptors of W ([N][K] E4M3, 128x128 boxes) and A ([M][K] BF16 at the
// caller's pitch, 64 x token_tile boxes), 128-byte swizzle; cached per device.
bool tc_tensor_map_w(const GemmArgs& g, int device, CUtensorMap* out, std::string* err);
bool tc_tensor_map_a(const GemmArgs& g, uint32_t token_tile, int device, CUtensorMap* out,
                     std::string* err);

// Device status of the translation units whose kernels wait.
cudaError_t tc_status_read(StatusWord* out, bool clear, cudaStream_t s);
cudaError_t tc8_status_read(StatusWord* out, bool clear, cudaStream_t s);

bool tc_supported_token_tile(uint32_t tn);
bool tc_supported_stages(uint32_t tn, uint32_t stages);

}  // namespace w8a16
