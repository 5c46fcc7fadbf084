// C ABI of libw8a16.so: argument checks, planning, dispatch, errors, status.
//
// The checks are those of the page "metrale_model_layers/layers/ops/
// w8a16_gemm_pipelined_m32.rs" (the `ensure!` clauses of
// `w8a16_gemm_pipelined_m32_strided`: m >= 1; K a positive multiple of 128; row
// pitches covering K and N; a_row_stride a multiple of 8), in that order, each
// with its own code and a message naming the values, followed by this library's
// own (N >= 1, pointers, alignment, index ranges). All of them run before any
// device work.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "w8a16_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

int ok() {
    g_last_error.clear();
    return W8A16_OK;
}

std::string u(uint64_t v) { return std::to_string(v); }

// Bounded-wait limit for the kernels: W8A16_WAIT_TIMEOUT_MS, read once.
struct TimeoutSetting {
    uint64_t ns = 2000ull * 1000 * 1000;
    bool valid = true;
    std::string raw;
};

const TimeoutSetting& timeout_setting() {
    static TimeoutSetting t;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* v = std::getenv("W8A16_WAIT_TIMEOUT_MS");
        if (v && *v) {
            char* end = nullptr;
            const unsigned long long ms = std::strtoull(v, &end, 10);
            if (end && *end == '\0' && ms >= 1 && ms <= 600000ull) {
                t.ns = ms * 1000ull * 1000ull;
            } else {
                t.valid = false;
                t.raw = v;
            }
        }
    });
    return t;
}

struct DeviceInfo {
    bool checked = false;
    bool ok = false;
    int sm_count = 0;
    int major = 0, minor = 0;
};

int current_device_info(DeviceInfo* out, std::string* err) {
    static std::mutex mu;
    static DeviceInfo infos[64];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        *err = std::string("no usable CUDA device: ") + cudaGetErrorString(e);
        return W8A16_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = infos[dev];
    if (!d.checked) {
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaGetLastError();
        d.ok = (d.major == 10 && d.minor == 3);
        d.checked = true;
    }
    *out = d;
    if (!d.ok) {
        *err = "device " + std::to_string(dev) + " is sm_" + std::to_string(d.major) +
               std::to_string(d.minor) + "; this library is built for sm_103a (GB300) only";
        return W8A16_ERR_DEVICE;
    }
    return W8A16_OK;
}

uint32_t ceil_div(uint32_t a, uint32_t b) { return (a + b - 1) / b; }

uint32_t token_tile_for(uint32_t M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    return 128;
}

// Tensor-core variants: TC (BF16 datapath) and TC8 (FP8 datapath, token tiles
// up to 64). Per-variant sizes come from the shared constants.
bool is_tc_variant(int32_t v) {
    return v == W8A16_VARIANT_TC || v == W8A16_VARIANT_TC8 || v == W8A16_VARIANT_W8A8 ||
           v == W8A16_VARIANT_PRESPLIT || v == W8A16_VARIANT_STREAM;
}
bool is_stream(int32_t v) { return v == W8A16_VARIANT_STREAM; }
bool is_fp8_act_variant(int32_t v) {
    return v == W8A16_VARIANT_W8A8 || v == W8A16_VARIANT_PRESPLIT || v == W8A16_VARIANT_STREAM;
}
bool is_gemv(int32_t v) { return v == W8A16_VARIANT_GEMV; }
uint32_t v_terms(int32_t v) { return v == W8A16_VARIANT_PRESPLIT || v == W8A16_VARIANT_STREAM ? 2u : 1u; }
uint32_t max_token_tile(int32_t v) { return v == W8A16_VARIANT_TC8 ? 64u : 128u; }
uint32_t v_threads(int32_t v, uint32_t tn) {
    return is_gemv(v)                ? w8a16::kGvThreads
           : v == W8A16_VARIANT_TC8   ? w8a16::tc8_threads(tn)
           : is_fp8_act_variant(v) ? w8a16::w8a8_threads(tn, v_terms(v))
                                   : w8a16::tc_threads(tn);
}
uint32_t v_smem(int32_t v, uint32_t tn, uint32_t st, uint32_t split) {
    return is_gemv(v)                ? w8a16::gemv_smem_bytes()
           : v == W8A16_VARIANT_TC8   ? w8a16::tc8_smem_bytes(tn, st, split)
           : is_fp8_act_variant(v) ? w8a16::w8a8_smem_bytes(tn, st, split, v_terms(v))
                                   : w8a16::tc_smem_bytes(tn, st, split);
}
uint32_t v_tmem(int32_t v, uint32_t tn) {
    return is_gemv(v)                ? w8a16::kGvTmemCols
           : v == W8A16_VARIANT_TC8   ? w8a16::tc8_tmem_cols(tn)
           : is_fp8_act_variant(v) ? w8a16::w8a8_tmem_cols(tn, v_terms(v))
                                   : w8a16::tc_tmem_cols(tn);
}
bool v_supported(int32_t v, uint32_t tn, uint32_t st) {
    return is_gemv(v)                ? (tn == w8a16::kGvMaxTokens && st == w8a16::kGvSlots)
           : v == W8A16_VARIANT_TC8   ? w8a16::tc8_supported_stages(tn, st)
           : is_fp8_act_variant(v) ? w8a16::w8a8_supported_stages(tn, st, v_terms(v))
                                   : w8a16::tc_supported_stages(tn, st);
}
uint32_t default_stages(int32_t v, uint32_t tn) {
    if (is_fp8_act_variant(v)) return 4;
    if (v == W8A16_VARIANT_TC8) return tn == 16 ? 4 : tn == 32 ? 6 : 4;   // 16: two CTAs per SM
    return tn == 16 ? 8 : tn == 32 ? 4 : tn == 64 ? 6 : 4;
}
// The variant the planner uses for a token count: the two-term FP8 kernel while
// its activation split is cheap (a 16-token tile), the BF16 kernel beyond.
int32_t auto_variant(uint32_t M) { return M <= 16 ? W8A16_VARIANT_TC8 : W8A16_VARIANT_TC; }

// CTAs of one tensor-core plan that fit on an SM: shared memory (228 KiB per
// SM, 1 KiB reserved per CTA), TMEM (512 columns), threads (2048), and the
// kernels' launch bounds (registers sized for one CTA per SM).
uint32_t tc_ctas_per_sm(int32_t v, uint32_t tn, uint32_t stages, uint32_t split) {
    const uint32_t smem = v_smem(v, tn, stages, split);
    const uint32_t by_smem = 233472u / (smem + 1024u);
    const uint32_t by_tmem = 512u / v_tmem(v, tn);
    const uint32_t by_threads = 2048u / v_threads(v, tn);
    uint32_t c = by_smem < by_tmem ? by_smem : by_tmem;
    c = c < by_threads ? c : by_threads;
    if (is_fp8_act_variant(v) && c > w8a16::w8a8_max_ctas_by_regs(tn)) c = w8a16::w8a8_max_ctas_by_regs(tn);
    return c < 1u ? 1u : c;
}

// Fill a tensor-core plan for a given variant, token tile, stage count and split.
void fill_tc(int32_t v, uint32_t M, uint32_t N, uint32_t tn, uint32_t stages, uint32_t split,
             w8a16_plan_t* p) {
    std::memset(p, 0, sizeof *p);
    p->variant = v;
    p->token_tile = tn;
    p->split_k = split;
    p->stages = stages;
    p->ctas_per_sm = tc_ctas_per_sm(v, tn, stages, split);
    p->grid[0] = ceil_div(N, w8a16::kTcRows) * split;
    p->grid[1] = ceil_div(M, tn);
    p->grid[2] = 1;
    p->block[0] = v_threads(v, tn);
    p->block[1] = p->block[2] = 1;
    p->cluster[0] = split;
    p->cluster[1] = p->cluster[2] = 1;
    p->smem_bytes = v_smem(v, tn, stages, split);
    p->tmem_cols = v_tmem(v, tn);
}

void fill_simt(uint32_t M, uint32_t N, w8a16_plan_t* p) {
    std::memset(p, 0, sizeof *p);
    p->variant = W8A16_VARIANT_SIMT;
    p->token_tile = 8;
    p->split_k = 1;
    p->stages = 0;
    p->ctas_per_sm = 8;
    p->grid[0] = ceil_div(N, 8);
    p->grid[1] = ceil_div(M, 8);
    p->grid[2] = 1;
    p->block[0] = 256;
    p->block[1] = p->block[2] = 1;
    p->cluster[0] = p->cluster[1] = p->cluster[2] = 1;
}

// Persistent stream-K plans of the pre-split path (W8A16_VARIANT_STREAM): 3..32
// tokens in one token tile of 16 or 32, 4 weight stages, two CTAs per SM.
constexpr uint32_t kStreamMinTokens = 3, kStreamMaxTokens = 32, kStreamStages = 4;

struct StreamLayout {
    uint64_t counters_off, parts_off, total;
    uint32_t maxseg;
};
// The largest number of CTAs any tile's steps fall to, with P CTAs over the units.
uint32_t stream_maxseg(uint32_t tiles, uint32_t ksteps, uint32_t P) {
    const uint64_t U = static_cast<uint64_t>(tiles) * ksteps;
    uint32_t most = 1;
    for (uint32_t t = 0; t < tiles; ++t) {
        const uint64_t u = static_cast<uint64_t>(t) * ksteps;
        const uint32_t n = w8a16::stream_cta_of(u + ksteps - 1, U, P) - w8a16::stream_cta_of(u, U, P) + 1;
        most = n > most ? n : most;
    }
    return most;
}
// Workspace: the split's codes and factors, the tile counters, the partials.
StreamLayout stream_layout(uint32_t M, uint32_t N, uint32_t K, uint32_t tn, uint32_t P) {
    StreamLayout L;
    const uint32_t tiles = ceil_div(N, w8a16::kTcRows);
    L.maxseg = stream_maxseg(tiles, K / w8a16::kKStep, P);
    L.counters_off = w8a16::align256(w8a16::split_ws_bytes(M, K));
    L.parts_off = w8a16::align256(L.counters_off + 4ull * tiles);
    L.total = L.parts_off + static_cast<uint64_t>(tiles) * L.maxseg * w8a16::kTcRows * tn * 4ull;
    return L;
}
bool stream_applies(uint32_t M, uint32_t N, uint32_t K) {
    return M >= kStreamMinTokens && M <= kStreamMaxTokens &&
           static_cast<uint64_t>(ceil_div(N, w8a16::kTcRows)) * (K / w8a16::kKStep) < (1ull << 31);
}

// Decode kernel plan: a cluster of `split` CTAs per 128-row weight tile, one token
// tile of up to kGvMaxTokens tokens.
void fill_gemv(uint32_t N, uint32_t split, w8a16_plan_t* p) {
    std::memset(p, 0, sizeof *p);
    p->variant = W8A16_VARIANT_GEMV;
    p->token_tile = w8a16::kGvMaxTokens;
    p->split_k = split;
    p->stages = w8a16::kGvSlots;
    p->ctas_per_sm = tc_ctas_per_sm(W8A16_VARIANT_GEMV, w8a16::kGvMaxTokens, w8a16::kGvSlots, split);
    p->grid[0] = ceil_div(N, w8a16::kTcRows) * split;
    p->grid[1] = p->grid[2] = 1;
    p->block[0] = w8a16::kGvThreads;
    p->block[1] = p->block[2] = 1;
    p->cluster[0] = split;
    p->cluster[1] = p->cluster[2] = 1;
    p->smem_bytes = w8a16::gemv_smem_bytes();
    p->tmem_cols = w8a16::kGvTmemCols;
}

// Stream-K plan: `ctas` persistent CTAs (0: two per SM), one token tile.
void fill_stream(uint32_t M, uint32_t N, uint32_t K, uint32_t sm_count, uint32_t ctas, w8a16_plan_t* p) {
    const uint32_t tn = M <= 16 ? 16u : 32u;
    const uint64_t units = static_cast<uint64_t>(ceil_div(N, w8a16::kTcRows)) * (K / w8a16::kKStep);
    fill_tc(W8A16_VARIANT_STREAM, M, N, tn, kStreamStages, 1, p);
    const uint64_t slots = static_cast<uint64_t>(sm_count ? sm_count : 152u) * p->ctas_per_sm;
    const uint64_t P = ctas ? ctas : (units < slots ? units : slots);
    p->grid[0] = static_cast<uint32_t>(P);
    p->grid[1] = 1;
}

// Whether a decode-kernel split can run (N, K): each CTA on at most kGvMaxSteps K
// steps, and no more CTAs than SMs, so the next call's CTAs fit beside them.
bool gemv_split_ok(uint32_t N, uint32_t K, uint32_t split, uint32_t sm_count) {
    const uint32_t ksteps = K / w8a16::kKStep;
    const uint32_t sms = sm_count ? sm_count : 152u;
    return split >= 1 && split <= 16 && split <= ksteps && ceil_div(ksteps, split) <= w8a16::kGvMaxSteps &&
           static_cast<uint64_t>(ceil_div(N, w8a16::kTcRows)) * split <= sms;
}

// The decode kernel's split for (M, N, K), or 0 where it does not apply: the
// largest split whose clusters stay portable (<= 8 CTAs), that fits the rule above
// and that leaves every CTA at least two K steps where K has them (more CTAs stream
// the weights from more SMs and leave each fewer steps after the dependency wait,
// but a CTA of a single step pays a cluster reduction for almost no streaming: on
// GB300 N = K = 256 takes 2.00 us a call at split 1 against 2.26 at split 2, and
// N = K = 1024 2.41 us at split 4 against 2.50 at split 8); cap[s] (NULL: assume it
// runs) = 0 rules cluster size s out.
uint32_t gemv_split(uint32_t M, uint32_t N, uint32_t K, uint32_t sm_count, const uint32_t* cap) {
    if (M < 1 || M > w8a16::kGvMaxTokens) return 0;
    const uint32_t ksteps = K / w8a16::kKStep;
    uint32_t single_step = 0;   // the largest admissible split of one step a CTA, if nothing else fits
    for (uint32_t s = 8; s >= 1; --s) {
        if (!gemv_split_ok(N, K, s, sm_count) || (cap && cap[s] == 0)) continue;
        if (ksteps / s >= 2 || ksteps < 2) return s;   // every CTA at least two steps
        if (single_step == 0) single_step = s;
    }
    return single_step;
}

// Choose the split-K factor by a load model: a CTA's time is its share of K
// steps plus a fixed start-up and drain (5 steps' worth); CTAs beyond the
// co-resident slots for that cluster size stretch the launch in proportion (a
// partial second wave costs only its share, since launches overlap); each rank
// of a split adds a little reduction work. cap[s] = co-resident CTAs in clusters
// of s (0 = cannot run).
uint32_t choose_split(uint32_t row_tiles, uint32_t token_tiles, uint32_t ksteps,
                      const uint32_t* cap) {
    const uint32_t max_split = ksteps < 16u ? ksteps : 16u;
    double best = 1e300;
    uint32_t best_s = 1;
    for (uint32_t s = 1; s <= max_split; ++s) {
        const uint32_t slots = cap[s];
        if (slots == 0) continue;
        const double ctas = static_cast<double>(row_tiles) * token_tiles * s;
        const double load = ctas > slots ? ctas / slots : 1.0;
        const double steps = static_cast<double>((ksteps + s - 1) / s);
        const double cost = load * (steps + 5.0) + 0.25 * s;
        if (cost < best - 1e-9) {
            best = cost;
            best_s = s;
        }
    }
    return best_s;
}

int check_sizes(uint32_t a_row_stride, uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K) {
    if (M < 1) return fail(W8A16_ERR_M_ZERO, "w8a16_gemm: m=0 has no rows to compute");
    if (K < w8a16::kKStep || K % w8a16::kKStep != 0)
        return fail(W8A16_ERR_K_BLOCK, "w8a16_gemm: K=" + u(K) +
                                           " must be a positive multiple of 128 (one FP8 scale "
                                           "block per K-step)");
    if (a_row_stride < K || c_row_stride < N)
        return fail(W8A16_ERR_PITCH, "w8a16_gemm: row pitches (a=" + u(a_row_stride) +
                                         ", c=" + u(c_row_stride) + ") must cover the used extents (k=" +
                                         u(K) + ", n=" + u(N) + ")");
    if (a_row_stride % 8 != 0)
        return fail(W8A16_ERR_A_PITCH_ALIGN, "w8a16_gemm: a_row_stride=" + u(a_row_stride) +
                                                 " must keep rows 16B-aligned (multiple of 8)");
    if (N < 1) return fail(W8A16_ERR_N_ZERO, "w8a16_gemm: n=0 has no columns to compute");
    if (M > 0x7FFFFFFFu || N > 0x7FFFFFFFu || K > 0x7FFFFFFFu)
        return fail(W8A16_ERR_RANGE, "w8a16_gemm: M, N and K must each be below 2^31 (M=" + u(M) +
                                         ", N=" + u(N) + ", K=" + u(K) + ")");
    if (ceil_div(M, 16) > 65535u * 8u)
        return fail(W8A16_ERR_RANGE, "w8a16_gemm: M=" + u(M) + " needs more token tiles than grid.y allows");
    return W8A16_OK;
}

int check_ptrs(const void* A, const void* W, const float* S, const void* C) {
    if (!A || !W || !S || !C)
        return fail(W8A16_ERR_NULL, std::string("w8a16_gemm: NULL ") +
                                        (!A ? "A" : !W ? "W" : !S ? "block_scale" : "C") + " pointer");
    const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(A) % 16 || addr(W) % 16 || addr(S) % 4 || addr(C) % 2)
        return fail(W8A16_ERR_ALIGN,
                    "w8a16_gemm: alignment (A and W need 16 bytes, block_scale 4, C 2); got A%16=" +
                        u(addr(A) % 16) + " W%16=" + u(addr(W) % 16) + " scale%4=" + u(addr(S) % 4) +
                        " C%2=" + u(addr(C) % 2));
    return W8A16_OK;
}

int validate_plan(uint32_t M, uint32_t N, uint32_t K, const w8a16_plan_t& p) {
    const uint32_t ksteps = K / w8a16::kKStep;
    if (p.variant == W8A16_VARIANT_SIMT) {
        if (p.grid[0] != ceil_div(N, 8) || p.grid[1] != ceil_div(M, 8) || p.block[0] != 256)
            return fail(W8A16_ERR_PLAN, "SIMT plan does not match the shape");
        return W8A16_OK;
    }
    if (is_gemv(p.variant)) {
        if (M > w8a16::kGvMaxTokens)
            return fail(W8A16_ERR_PLAN, "decode plan: M=" + u(M) + " is above " + u(w8a16::kGvMaxTokens));
        if (p.split_k < 1 || p.split_k > 16 || p.split_k > ksteps ||
            ceil_div(ksteps, p.split_k) > w8a16::kGvMaxSteps)
            return fail(W8A16_ERR_PLAN, "decode plan: split_k=" + u(p.split_k) + " must be in 1..min(16, K/128) "
                                        "with at most " + u(w8a16::kGvMaxSteps) + " K steps per CTA");
        w8a16_plan_t ref;
        fill_gemv(N, p.split_k, &ref);
        if (p.grid[0] != ref.grid[0] || p.grid[1] != 1 || p.cluster[0] != p.split_k ||
            p.token_tile != ref.token_tile || p.stages != ref.stages || p.tail_tiles || p.tail_split)
            return fail(W8A16_ERR_PLAN, "decode plan does not match the shape");
        return W8A16_OK;
    }
    if (is_stream(p.variant)) {
        const uint64_t units = static_cast<uint64_t>(ceil_div(N, w8a16::kTcRows)) * ksteps;
        if (!stream_applies(M, N, K) || (p.token_tile != 16 && p.token_tile != 32) || M > p.token_tile ||
            p.stages != kStreamStages || p.split_k != 1 || p.grid[1] != 1 || p.grid[0] < 1 ||
            p.grid[0] > units || p.cluster[0] != 1 || p.tail_tiles || p.tail_split)
            return fail(W8A16_ERR_PLAN, "stream-K plan: needs " + u(kStreamMinTokens) + " <= M <= " +
                                            u(kStreamMaxTokens) + " tokens in one token tile, 1..units CTAs, "
                                            "split 1, no tail");
        return W8A16_OK;
    }
    if (!is_tc_variant(p.variant))
        return fail(W8A16_ERR_PLAN, "unknown variant " + std::to_string(p.variant));
    if (!v_supported(p.variant, p.token_tile, p.stages))
        return fail(W8A16_ERR_PLAN, "TC plan: token_tile=" + u(p.token_tile) + " stages=" +
                                        u(p.stages) + " has no kernel instance for variant " +
                                        std::to_string(p.variant));
    if (p.split_k < 1 || p.split_k > 16 || p.split_k > ksteps)
        return fail(W8A16_ERR_PLAN, "TC plan: split_k=" + u(p.split_k) +
                                        " must be in 1..min(16, K/128=" + u(ksteps) + ")");
    w8a16_plan_t ref;
    fill_tc(p.variant, M, N, p.token_tile, p.stages, p.split_k, &ref);
    if (p.tail_tiles != 0 || p.tail_split != 0) {
        const uint32_t row_tiles = ceil_div(N, w8a16::kTcRows);
        if (!(is_fp8_act_variant(p.variant) || p.variant == W8A16_VARIANT_TC) || ref.grid[1] != 1)
            return fail(W8A16_ERR_PLAN, "a split-K tail needs the BF16 or FP8 x FP8 kernel and one token tile");
        if (p.tail_tiles < 1 || p.tail_tiles >= row_tiles || p.tail_split < 2 || p.tail_split > 16 ||
            p.tail_split > ksteps)
            return fail(W8A16_ERR_PLAN, "split-K tail: tail_tiles=" + u(p.tail_tiles) + " must be in 1.." +
                                            u(row_tiles - 1) + " and tail_split=" + u(p.tail_split) +
                                            " in 2..min(16, K/128)");
        if (v_smem(p.variant, p.token_tile, p.stages, p.tail_split) > w8a16::kMaxDynSmem)
            return fail(W8A16_ERR_PLAN, "split-K tail: tail_split=" + u(p.tail_split) +
                                            " does not fit in shared memory");
        ref.grid[0] = (row_tiles - p.tail_tiles) * p.split_k;
    }
    if (p.grid[0] != ref.grid[0] || p.grid[1] != ref.grid[1] || p.cluster[0] != ref.cluster[0])
        return fail(W8A16_ERR_PLAN, "TC plan grid does not match the shape");
    if (ref.grid[1] > 65535u) return fail(W8A16_ERR_RANGE, "TC plan: too many token tiles");
    if (ref.smem_bytes > w8a16::kMaxDynSmem)
        return fail(W8A16_ERR_PLAN, "TC plan: token_tile=" + u(p.token_tile) + " stages=" +
                                        u(p.stages) + " split_k=" + u(p.split_k) + " needs " +
                                        u(ref.smem_bytes) + " bytes of shared memory");
    return W8A16_OK;
}

// Co-resident CTAs per cluster size on `sm_count` SMs: whole clusters of CTAs
// that fit per SM at that split (the split-K receive buffer grows shared memory).
void model_capacity(int32_t v, uint32_t tn, uint32_t stages, uint32_t sm_count, uint32_t* cap) {
    cap[0] = 0;
    for (uint32_t c = 1; c <= 16; ++c)
        cap[c] = ((sm_count ? sm_count : 152u) * tc_ctas_per_sm(v, tn, stages, c) / c) * c;
}

uint32_t token_tile_for(int32_t v, uint32_t M) {
    const uint32_t tn = token_tile_for(M);
    return tn > max_token_tile(v) ? max_token_tile(v) : tn;
}

// W8A8 plan: split and stage count from a stream model. A launch costs a fixed
// start-up and drain per wave of co-resident CTAs (a partial wave costs as much as
// a full one), plus the longer of two floors: the weight bytes at the bandwidth
// its in-flight loads can sustain (bytes in flight / latency, capped at HBM
// bandwidth; a CTA has at most `stages` weight tiles, and no more than its K
// steps, in flight) and the CTAs' K steps at a per-step cost growing with the
// token tile (MMAs and fold); plus a little reduction work per split rank. As for
// the BF16 kernel, wide tiles (64 and 128 tokens) that already cover half the SMs
// are not split. live[i] (NULL: model only) is the device's cluster table for
// kA8Stages[i]; a zero entry rules that cluster size out.
constexpr uint32_t kA8Stages[2] = {4, 6};
// Stage counts the model may pick, from sweeps on GB300: six-stage rings did not
// pay where two CTAs share an SM (decode, skinny, 32-token tiles), nor for
// 128-token tiles.
bool a8_stage_allowed(int32_t, uint32_t, uint32_t st) { return st == 4u; }

void choose_w8a8(int32_t v, uint32_t tn, uint32_t row_tiles, uint32_t token_tiles, uint32_t ksteps,
                 uint32_t sm_count, const uint32_t* const live[2], uint32_t* split_out,
                 uint32_t* stages_out) {
    constexpr double kWaveSeconds = 6.0e-6, kLatency = 2.5e-6, kHbm = 6.8e12, kPerRank = 5.0e-8;
    const double step_seconds = 4.5e-7 * tn / 128.0 * (v == W8A16_VARIANT_PRESPLIT ? 1.3 : 1.0);
    const double wbytes = static_cast<double>(row_tiles) * token_tiles * w8a16::kTcRows * w8a16::kKStep * ksteps;
    const uint32_t sms = sm_count ? sm_count : 152u;
    const uint32_t max_split = (tn >= 64 && 2u * row_tiles * token_tiles >= sms) ? 1u : (ksteps < 16u ? ksteps : 16u);
    double best = 1e300;
    *split_out = 1;
    *stages_out = kA8Stages[0];
    for (uint32_t i = 0; i < 2; ++i) {
        const uint32_t st = kA8Stages[i];
        if (!v_supported(v, tn, st) || !a8_stage_allowed(v, tn, st)) continue;
        uint32_t cap[17];
        model_capacity(v, tn, st, sm_count, cap);
        for (uint32_t sp = 1; sp <= max_split; ++sp) {
            if (v_smem(v, tn, st, sp) > w8a16::kMaxDynSmem || cap[sp] == 0) continue;
            if (live && live[i] && live[i][sp] == 0) continue;
            const double ctas = static_cast<double>(row_tiles) * token_tiles * sp;
            const double waves = std::ceil(ctas / cap[sp]);
            const uint32_t per_cta = ceil_div(ksteps, sp) < st ? ceil_div(ksteps, sp) : st;
            const double inflight = (ctas < cap[sp] ? ctas : cap[sp]) * per_cta * w8a16::kTcRows * w8a16::kKStep;
            const double bw = inflight / kLatency < kHbm ? inflight / kLatency : kHbm;
            const double compute = waves * ceil_div(ksteps, sp) * step_seconds;
            const double t = waves * kWaveSeconds + (wbytes / bw > compute ? wbytes / bw : compute) + kPerRank * sp;
            if (t < best * (1.0 - 1e-9)) {
                best = t;
                *split_out = sp;
                *stages_out = st;
            }
        }
    }
}

// Split-K tail for the FP8 x FP8 kernel: a plan of whole tiles (split 1, one token
// tile) that needs a second, partial wave runs its last tiles in a second launch
// instead, split over the largest cluster size whose CTAs all fit in one wave, so
// that tail costs a fraction of a tile's time instead of a whole one. live (NULL:
// model only) rules out cluster sizes the device cannot run.
void add_tail(w8a16_plan_t* p, uint32_t M, uint32_t N, uint32_t K, uint32_t sm_count, const uint32_t* live) {
    const uint32_t row_tiles = ceil_div(N, w8a16::kTcRows), ksteps = K / w8a16::kKStep;
    if (!(is_fp8_act_variant(p->variant) || p->variant == W8A16_VARIANT_TC) || p->split_k != 1 ||
        ceil_div(M, p->token_tile) != 1)
        return;
    uint32_t cap[17];
    model_capacity(p->variant, p->token_tile, p->stages, sm_count, cap);
    if (row_tiles <= cap[1] || row_tiles > 2u * cap[1]) return;
    const uint32_t tail = row_tiles - cap[1];
    uint32_t best = 0;
    for (uint32_t k = 2; k <= (ksteps < 16u ? ksteps : 16u); ++k) {
        if (v_smem(p->variant, p->token_tile, p->stages, k) > w8a16::kMaxDynSmem) continue;
        if (live && live[k] == 0) continue;
        if (tail * k <= cap[k]) best = k;
    }
    if (best < 2) return;
    p->tail_tiles = tail;
    p->tail_split = best;
    p->grid[0] = cap[1];
}

// Pure planner: variant by M (or as given), token tile by M, stage count by
// token tile, split from the wave model over `cap` (NULL: every cluster size
// fills every SM slot). The W8A8 variant has its own model (choose_w8a8).
int plan_core(int32_t v, uint32_t M, uint32_t N, uint32_t K, uint32_t sm_count,
              const uint32_t* cap, w8a16_plan_t* out) {
    if (v == W8A16_VARIANT_AUTO || is_gemv(v)) {
        const uint32_t gs = gemv_split(M, N, K, sm_count, nullptr);
        if (gs) {
            fill_gemv(N, gs, out);
            return W8A16_OK;
        }
        if (is_gemv(v)) return W8A16_ERR_PLAN;
    }
    if (v == W8A16_VARIANT_AUTO) v = auto_variant(M);
    if (is_fp8_act_variant(v)) {
        const uint32_t tn = token_tile_for(v, M);
        uint32_t sp = 1, st = kA8Stages[0];
        choose_w8a8(v, tn, ceil_div(N, w8a16::kTcRows), ceil_div(M, tn), K / w8a16::kKStep, sm_count, nullptr,
                    &sp, &st);
        fill_tc(v, M, N, tn, st, sp, out);
        add_tail(out, M, N, K, sm_count, nullptr);
        return W8A16_OK;
    }
    const uint32_t tn = token_tile_for(v, M);
    const uint32_t stages = default_stages(v, tn);
    const uint32_t row_tiles = ceil_div(N, w8a16::kTcRows);
    const uint32_t token_tiles = ceil_div(M, tn);
    const uint32_t ksteps = K / w8a16::kKStep;
    uint32_t model[17];
    if (!cap) {
        model_capacity(v, tn, stages, sm_count, model);
        cap = model;
    }
    uint32_t usable[17];
    for (uint32_t c = 0; c <= 16; ++c)   // splits whose shared memory does not fit are out
        usable[c] = (c >= 1 && v_smem(v, tn, stages, c) <= w8a16::kMaxDynSmem) ? cap[c] : 0u;
    // The BF16 kernel runs one CTA per SM and is bound by its MMA pipe: once the
    // tiles cover half the SMs, splitting K only adds waves and reductions.
    const uint32_t sms = sm_count ? sm_count : 152u;
    const uint32_t split = (v == W8A16_VARIANT_TC && 2u * row_tiles * token_tiles >= sms)
                               ? 1u
                               : choose_split(row_tiles, token_tiles, ksteps, usable);
    fill_tc(v, M, N, tn, stages, split, out);
    add_tail(out, M, N, K, sm_count, cap);
    return W8A16_OK;
}

// Live capacity table of the current device for (variant, tn, stages), cached.
int live_capacity(int32_t v, uint32_t tn, uint32_t stages, uint32_t* cap, std::string* err) {
    static std::mutex mu;
    struct Entry { int dev; int32_t v; uint32_t tn, stages; uint32_t cap[17]; };
    static Entry cache[128];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].dev == dev && cache[i].v == v && cache[i].tn == tn &&
                cache[i].stages == stages) {
                std::memcpy(cap, cache[i].cap, sizeof(uint32_t) * 17);
                return W8A16_OK;
            }
    }
    Entry e{dev, v, tn, stages, {0}};
    for (uint32_t c = 1; c <= 16; ++c) {
        int rc = is_gemv(v)                ? w8a16::gemv_cluster_capacity(c, &e.cap[c], err)
                 : v == W8A16_VARIANT_TC8    ? w8a16::tc8_cluster_capacity(tn, stages, c, &e.cap[c], err)
                 : is_fp8_act_variant(v)   ? w8a16::w8a8_cluster_capacity(tn, stages, v_terms(v), c, &e.cap[c], err)
                                           : w8a16::tc_cluster_capacity(tn, stages, c, &e.cap[c], err);
        if (rc) return rc;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (used < 128) cache[used++] = e;
    std::memcpy(cap, e.cap, sizeof(uint32_t) * 17);
    return W8A16_OK;
}

// The live table decides which cluster sizes can run at all; the slot counts are
// the model's (SMs x CTAs per SM), because the cluster occupancy query reports one
// CTA per SM even where two co-reside (launches of two-per-SM plans do run all
// their CTAs at once).
int plan_live(int32_t v, uint32_t M, uint32_t N, uint32_t K, const DeviceInfo& info, w8a16_plan_t* out,
              std::string* err) {
    if (v == W8A16_VARIANT_AUTO && gemv_split(M, N, K, static_cast<uint32_t>(info.sm_count), nullptr)) {
        uint32_t cap[17];
        const int rc = live_capacity(W8A16_VARIANT_GEMV, w8a16::kGvMaxTokens, w8a16::kGvSlots, cap, err);
        if (rc) return rc;
        const uint32_t gs = gemv_split(M, N, K, static_cast<uint32_t>(info.sm_count), cap);
        if (gs) {
            fill_gemv(N, gs, out);
            return W8A16_OK;
        }
    }
    if (v == W8A16_VARIANT_AUTO) v = auto_variant(M);
    const uint32_t tn = token_tile_for(v, M);
    if (is_fp8_act_variant(v)) {
        uint32_t tables[2][17] = {};
        const uint32_t* live[2] = {nullptr, nullptr};
        for (uint32_t i = 0; i < 2; ++i) {
            if (!v_supported(v, tn, kA8Stages[i])) continue;
            const int rc = live_capacity(v, tn, kA8Stages[i], tables[i], err);
            if (rc) return rc;
            live[i] = tables[i];
        }
        uint32_t sp = 1, st = kA8Stages[0];
        choose_w8a8(v, tn, ceil_div(N, w8a16::kTcRows), ceil_div(M, tn), K / w8a16::kKStep,
                    static_cast<uint32_t>(info.sm_count), live, &sp, &st);
        fill_tc(v, M, N, tn, st, sp, out);
        add_tail(out, M, N, K, static_cast<uint32_t>(info.sm_count), live[st == kA8Stages[0] ? 0 : 1]);
        return W8A16_OK;
    }
    const uint32_t stages = default_stages(v, tn);
    uint32_t cap[17];
    int rc = live_capacity(v, tn, stages, cap, err);
    if (rc) return rc;
    uint32_t model[17];
    model_capacity(v, tn, stages, static_cast<uint32_t>(info.sm_count), model);
    for (uint32_t c = 1; c <= 16; ++c) cap[c] = cap[c] == 0 ? 0u : model[c];
    return plan_core(v, M, N, K, static_cast<uint32_t>(info.sm_count), cap, out);
}

int run(const w8a16::GemmArgs& g, const w8a16_plan_t* forced, uint32_t flags,
        cudaStream_t stream) {
    if (flags & ~static_cast<uint32_t>(W8A16_FLAG_PDL))
        return fail(W8A16_ERR_ARG, "w8a16_gemm: unknown flag bits " + u(flags));
    int rc = check_sizes(g.lda, g.ldc, g.M, g.N, g.K);
    if (rc) return rc;
    rc = check_ptrs(g.A, g.W, g.scale, g.C);
    if (rc) return rc;
    const TimeoutSetting& ts = timeout_setting();
    if (!ts.valid)
        return fail(W8A16_ERR_ARG, "W8A16_WAIT_TIMEOUT_MS='" + ts.raw +
                                       "' is not an integer number of milliseconds in 1..600000");
    if (forced) {
        if (forced->variant == W8A16_VARIANT_W8A8)
            return fail(W8A16_ERR_PLAN, "w8a16_gemm: a W8A8 plan needs FP8 activations "
                                        "(w8a16_gemm_w8a8_with_plan)");
        if (forced->variant == W8A16_VARIANT_PRESPLIT)
            return fail(W8A16_ERR_PLAN, "w8a16_gemm: a pre-split plan needs a workspace (w8a16_gemm_ws)");
        rc = validate_plan(g.M, g.N, g.K, *forced);
        if (rc) return rc;
    }
    DeviceInfo info;
    std::string err;
    rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    w8a16_plan_t plan;
    if (forced) {
        plan = *forced;
    } else {
        rc = plan_live(W8A16_VARIANT_AUTO, g.M, g.N, g.K, info, &plan, &err);
        if (rc) return fail(rc, err);
    }
    if (plan.variant == W8A16_VARIANT_SIMT)
        rc = w8a16::launch_simt(g, plan, stream, flags, &err);
    else if (is_gemv(plan.variant))
        rc = w8a16::launch_gemv(g, plan, stream, ts.ns, flags, &err);
    else if (plan.variant == W8A16_VARIANT_TC8)
        rc = w8a16::launch_tc8(g, plan, stream, ts.ns, flags, &err);
    else
        rc = w8a16::launch_tc(g, plan, stream, ts.ns, flags, &err);
    if (rc) return fail(rc, err);
    return ok();
}

// W8A8: the same size rules as w8a16_gemm, plus the activation code pitch (a
// multiple of 16 bytes: TMA row stride) and the scale pitch (>= M, a multiple of 4).
// The stream-K operands in a workspace laid out by stream_layout.
w8a16::StreamK stream_args(uint32_t M, uint32_t N, uint32_t K, const w8a16_plan_t& plan, uint8_t* ws) {
    const StreamLayout L = stream_layout(M, N, K, plan.token_tile, plan.grid[0]);
    w8a16::StreamK sk{};
    sk.parts = reinterpret_cast<float*>(ws + L.parts_off);
    sk.counters = reinterpret_cast<uint32_t*>(ws + L.counters_off);
    sk.units = ceil_div(N, w8a16::kTcRows) * (K / w8a16::kKStep);
    sk.maxseg = L.maxseg;
    return sk;
}

// The W8A16 product through the two-term split: the split pre-pass into the
// workspace, then the FP8 x FP8 kernel on it. Both are queued as programmatic
// dependent launches; the kernel's weight prefetch overlaps only the split,
// which writes neither the weights nor their scales. A stream-K plan also gets the
// tile counters (cleared by the split) and the partials from the workspace.
int run_presplit(const w8a16::GemmArgs& g, const w8a16_plan_t& plan, void* ws, uint64_t ts_ns,
                 cudaStream_t stream) {
    std::string err;
    const uint32_t fstride = static_cast<uint32_t>(w8a16::split_ws_scale_stride(g.M));
    uint8_t* codes = static_cast<uint8_t*>(ws);
    float* factors = reinterpret_cast<float*>(codes + 2ull * g.M * g.K);
    const w8a16::StreamK sk = is_stream(plan.variant) ? stream_args(g.M, g.N, g.K, plan, codes) : w8a16::StreamK{};
    int rc = w8a16::launch_split_act(g.A, g.lda, g.M, g.K, codes, factors, fstride, sk.counters,
                                     sk.counters ? ceil_div(g.N, w8a16::kTcRows) : 0u, stream, &err);
    if (rc) return fail(rc, err);
    const w8a16::W8A8Args a{codes, g.K, factors, fstride, g.W, g.scale, g.C, g.ldc, g.M, g.N, g.K, 2u, sk};
    rc = w8a16::launch_w8a8(a, plan, stream, ts_ns, W8A16_FLAG_PDL, &err);
    if (rc) return fail(rc, err);
    return ok();
}

// Workspace bytes of the stream-K plan for (M, N, K) on `sm_count` SMs (0 where it
// does not apply).
uint64_t stream_ws_bytes(uint32_t M, uint32_t N, uint32_t K, uint32_t sm_count) {
    if (!stream_applies(M, N, K)) return 0;
    w8a16_plan_t p;
    fill_stream(M, N, K, sm_count, 0, &p);
    return stream_layout(M, N, K, p.token_tile, p.grid[0]).total;
}

// The plan w8a16_gemm_ws takes without a forced plan, given `have` bytes of
// workspace: the pre-split path on the cluster split-K schedule for M > 16 (its
// terms fit), else w8a16_gemm's own plan (*presplit = false). The persistent
// stream-K plan is never chosen here: on GB300 it measured slower than both (its
// fix-up of tiles split between CTAs costs several loaded memory round trips at
// the end of every CTA), so it runs only when forced.
int plan_ws_choice(uint32_t M, uint32_t N, uint32_t K, uint64_t have, const DeviceInfo& info,
                   w8a16_plan_t* plan, bool* presplit, std::string* err) {
    *presplit = true;
    if (M > 16 && have >= w8a16::split_ws_bytes(M, K))
        return plan_live(W8A16_VARIANT_PRESPLIT, M, N, K, info, plan, err);
    *presplit = false;
    return plan_live(W8A16_VARIANT_AUTO, M, N, K, info, plan, err);
}

int run_ws(const w8a16::GemmArgs& g, const w8a16_plan_t* forced, void* ws, uint64_t ws_bytes,
           uint32_t flags, cudaStream_t stream) {
    if (flags & ~static_cast<uint32_t>(W8A16_FLAG_PDL))
        return fail(W8A16_ERR_ARG, "w8a16_gemm_ws: unknown flag bits " + u(flags));
    int rc = check_sizes(g.lda, g.ldc, g.M, g.N, g.K);
    if (rc) return rc;
    rc = check_ptrs(g.A, g.W, g.scale, g.C);
    if (rc) return rc;
    if (ws && reinterpret_cast<uintptr_t>(ws) % 16 != 0)
        return fail(W8A16_ERR_ALIGN, "w8a16_gemm_ws: the workspace must be 16-byte aligned");
    const uint64_t need = w8a16::split_ws_bytes(g.M, g.K);
    const uint64_t have = ws ? ws_bytes : 0;
    const bool pre = forced && (forced->variant == W8A16_VARIANT_PRESPLIT || is_stream(forced->variant));
    if (forced && !pre) return run(g, forced, flags, stream);
    if (pre) {
        rc = validate_plan(g.M, g.N, g.K, *forced);
        if (rc) return rc;
        const uint64_t want = is_stream(forced->variant)
                                  ? stream_layout(g.M, g.N, g.K, forced->token_tile, forced->grid[0]).total
                                  : need;
        if (have < want)
            return fail(W8A16_ERR_ARG, "w8a16_gemm_ws: this plan needs a workspace of " + std::to_string(want) +
                                           " bytes (have " + std::to_string(have) + ")");
    }
    const TimeoutSetting& ts = timeout_setting();
    if (!ts.valid)
        return fail(W8A16_ERR_ARG, "W8A16_WAIT_TIMEOUT_MS='" + ts.raw +
                                       "' is not an integer number of milliseconds in 1..600000");
    DeviceInfo info;
    std::string err;
    rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    w8a16_plan_t plan;
    if (forced) {
        plan = *forced;
    } else {
        bool presplit = false;
        rc = plan_ws_choice(g.M, g.N, g.K, have, info, &plan, &presplit, &err);
        if (rc) return fail(rc, err);
        if (!presplit) return run(g, nullptr, flags, stream);
    }
    return run_presplit(g, plan, ws, ts.ns, stream);
}

// Scratch of the allocation-free entry point: a fixed device array in this
// module, so a call allocates nothing. Its device address is looked up on every
// call (cudaGetSymbolAddress allocates nothing), so it stays right after a device
// reset or under another context, where the module is loaded anew. Calls that
// overlap in time (other streams, other host threads) share it and race.
constexpr uint64_t kNoAllocScratchBytes = 32ull << 20;
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

int noalloc_scratch(void** out, std::string* err) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        *err = std::string("scratch buffer address: ") + cudaGetErrorString(e);
        return W8A16_ERR_DEVICE;
    }
    *out = addr;
    return W8A16_OK;
}

int run_w8a8(const w8a16::W8A8Args& g, const w8a16_plan_t* forced, uint32_t flags,
             cudaStream_t stream) {
    if (flags & ~static_cast<uint32_t>(W8A16_FLAG_PDL))
        return fail(W8A16_ERR_ARG, "w8a16_gemm_w8a8: unknown flag bits " + u(flags));
    if (g.M < 1) return fail(W8A16_ERR_M_ZERO, "w8a16_gemm_w8a8: m=0 has no rows to compute");
    if (g.K < w8a16::kKStep || g.K % w8a16::kKStep != 0)
        return fail(W8A16_ERR_K_BLOCK, "w8a16_gemm_w8a8: K=" + u(g.K) + " must be a positive multiple of 128");
    if (g.lda < g.K || g.ldc < g.N || g.a_scale_stride < g.M)
        return fail(W8A16_ERR_PITCH, "w8a16_gemm_w8a8: pitches (a=" + u(g.lda) + ", c=" + u(g.ldc) +
                                         ", a_scale=" + u(g.a_scale_stride) + ") must cover k=" + u(g.K) +
                                         ", n=" + u(g.N) + ", m=" + u(g.M));
    if (g.lda % 16 != 0 || g.a_scale_stride % 4 != 0)
        return fail(W8A16_ERR_A_PITCH_ALIGN, "w8a16_gemm_w8a8: a_row_stride=" + u(g.lda) +
                                                 " must be a multiple of 16 bytes and a_scale_stride=" +
                                                 u(g.a_scale_stride) + " a multiple of 4");
    if (g.N < 1) return fail(W8A16_ERR_N_ZERO, "w8a16_gemm_w8a8: n=0 has no columns to compute");
    if (g.M > 0x7FFFFFFFu || g.N > 0x7FFFFFFFu || g.K > 0x7FFFFFFFu || ceil_div(g.M, 16) > 65535u * 8u)
        return fail(W8A16_ERR_RANGE, "w8a16_gemm_w8a8: M, N or K out of range");
    if (!g.A || !g.a_scale || !g.W || !g.scale || !g.C)
        return fail(W8A16_ERR_NULL, "w8a16_gemm_w8a8: NULL operand pointer");
    const auto addr = [](const void* q) { return reinterpret_cast<uintptr_t>(q); };
    if (addr(g.A) % 16 || addr(g.a_scale) % 16 || addr(g.W) % 16 || addr(g.scale) % 4 || addr(g.C) % 2)
        return fail(W8A16_ERR_ALIGN, "w8a16_gemm_w8a8: alignment (A, a_scale and W need 16 bytes, "
                                     "block_scale 4, C 2)");
    const TimeoutSetting& ts = timeout_setting();
    if (!ts.valid)
        return fail(W8A16_ERR_ARG, "W8A16_WAIT_TIMEOUT_MS='" + ts.raw +
                                       "' is not an integer number of milliseconds in 1..600000");
    if (forced) {
        if (forced->variant != W8A16_VARIANT_W8A8 && !is_gemv(forced->variant))
            return fail(W8A16_ERR_PLAN, "w8a16_gemm_w8a8: the plan is neither a W8A8 nor a decode plan");
        const int rc = validate_plan(g.M, g.N, g.K, *forced);
        if (rc) return rc;
    }
    DeviceInfo info;
    std::string err;
    int rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    w8a16_plan_t plan;
    if (forced) {
        plan = *forced;
    } else {
        // one or two tokens: the decode kernel where its rule admits the shape (the
        // same plan as for W8A16), else the W8A8 kernel
        rc = plan_live(W8A16_VARIANT_AUTO, g.M, g.N, g.K, info, &plan, &err);
        if (rc || !is_gemv(plan.variant)) {
            rc = plan_live(W8A16_VARIANT_W8A8, g.M, g.N, g.K, info, &plan, &err);
            if (rc) return fail(rc, err);
        }
    }
    rc = is_gemv(plan.variant) ? w8a16::launch_gemv_w8a8(g, plan, stream, ts.ns, flags, &err)
                               : w8a16::launch_w8a8(g, plan, stream, ts.ns, flags, &err);
    if (rc) return fail(rc, err);
    return ok();
}

}  // namespace

extern "C" {

int w8a16_check_args(const void* A, uint32_t a_row_stride, const void* W, const float* block_scale,
                     const void* C, uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K) {
    int rc = check_sizes(a_row_stride, c_row_stride, M, N, K);
    if (rc) return rc;
    const auto misaligned = [](const void* p, uintptr_t a) {
        return p != nullptr && reinterpret_cast<uintptr_t>(p) % a != 0;
    };
    if (misaligned(A, 16) || misaligned(W, 16) || misaligned(block_scale, 4) || misaligned(C, 2))
        return fail(W8A16_ERR_ALIGN,
                    "w8a16_gemm: alignment (A and W need 16 bytes, block_scale 4, C 2)");
    return ok();
}

int w8a16_quantize_weights(const void* W, uint32_t w_dtype, uint32_t w_row_stride, uint32_t N,
                           uint32_t K, void* codes, float* block_scale, w8a16_stream_t stream) {
    if (N < 1) return fail(W8A16_ERR_N_ZERO, "w8a16_quantize_weights: n=0 has no rows to quantise");
    if (K < w8a16::kKStep || K % w8a16::kKStep != 0)
        return fail(W8A16_ERR_K_BLOCK, "w8a16_quantize_weights: K=" + u(K) +
                                           " must be a positive multiple of 128 (one scale per 128x128 block)");
    if (w_row_stride < K)
        return fail(W8A16_ERR_PITCH, "w8a16_quantize_weights: w_row_stride=" + u(w_row_stride) +
                                         " must cover K=" + u(K));
    if (w_row_stride % 4 != 0)
        return fail(W8A16_ERR_A_PITCH_ALIGN, "w8a16_quantize_weights: w_row_stride=" + u(w_row_stride) +
                                                 " must be a multiple of 4 (vector loads of 4 values)");
    if (w_dtype != W8A16_WEIGHTS_F32 && w_dtype != W8A16_WEIGHTS_BF16)
        return fail(W8A16_ERR_ARG, "w8a16_quantize_weights: unknown weight type " + u(w_dtype));
    if (N > 0x7FFFFFFFu || K > 0x7FFFFFFFu || (N + 127u) / 128u > 65535u)
        return fail(W8A16_ERR_RANGE, "w8a16_quantize_weights: N=" + u(N) + " K=" + u(K) + " out of range");
    if (!W || !codes || !block_scale)
        return fail(W8A16_ERR_NULL, std::string("w8a16_quantize_weights: NULL ") +
                                        (!W ? "W" : !codes ? "codes" : "block_scale") + " pointer");
    const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
    if (addr(W) % 16 || addr(codes) % 4 || addr(block_scale) % 4)
        return fail(W8A16_ERR_ALIGN,
                    "w8a16_quantize_weights: alignment (W needs 16 bytes, codes and block_scale 4)");
    DeviceInfo info;
    std::string err;
    int rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    rc = w8a16::launch_quantize(W, w_dtype == W8A16_WEIGHTS_BF16, w_row_stride, N, K, codes, block_scale,
                                static_cast<cudaStream_t>(stream), &err);
    if (rc) return fail(rc, err);
    return ok();
}

int w8a16_gemm_w8a8(const void* A, uint32_t a_row_stride, const float* a_scale, uint32_t a_scale_stride,
                    const void* W, const float* block_scale, void* C, uint32_t c_row_stride, uint32_t M,
                    uint32_t N, uint32_t K, uint32_t flags, w8a16_stream_t stream) {
    const w8a16::W8A8Args g{A, a_row_stride, a_scale, a_scale_stride, W, block_scale, C, c_row_stride, M, N, K, 1u};
    return run_w8a8(g, nullptr, flags, static_cast<cudaStream_t>(stream));
}

int w8a16_gemm_w8a8_with_plan(const void* A, uint32_t a_row_stride, const float* a_scale,
                              uint32_t a_scale_stride, const void* W, const float* block_scale, void* C,
                              uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K,
                              const w8a16_plan_t* plan, uint32_t flags, w8a16_stream_t stream) {
    if (!plan) return fail(W8A16_ERR_NULL, "w8a16_gemm_w8a8_with_plan: NULL plan");
    const w8a16::W8A8Args g{A, a_row_stride, a_scale, a_scale_stride, W, block_scale, C, c_row_stride, M, N, K, 1u};
    return run_w8a8(g, plan, flags, static_cast<cudaStream_t>(stream));
}

uint64_t w8a16_workspace_bytes(uint32_t M, uint32_t K) {
    if (M == 0 || K == 0 || K % w8a16::kKStep != 0) return 0;
    return w8a16::split_ws_bytes(M, K);
}

uint64_t w8a16_workspace_bytes_for(uint32_t M, uint32_t N, uint32_t K) {
    if (M == 0 || N == 0 || K == 0 || K % w8a16::kKStep != 0) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        sms = 152;
    }
    const uint64_t pre = M > 16 ? w8a16::split_ws_bytes(M, K) : 0;
    const uint64_t sk = stream_ws_bytes(M, N, K, static_cast<uint32_t>(sms));
    return sk > pre ? sk : pre;
}

int w8a16_gemm_noalloc(const void* A, uint32_t a_row_stride, const void* W, const float* block_scale,
                       void* C, uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K, uint32_t flags,
                       w8a16_stream_t stream) {
    int rc = check_sizes(a_row_stride, c_row_stride, M, N, K);
    if (rc) return rc;
    const uint64_t need = w8a16::split_ws_bytes(M, K);
    if (M > 16 && need > kNoAllocScratchBytes)
        return fail(W8A16_ERR_RANGE, "w8a16_gemm_noalloc: M=" + u(M) + ", K=" + u(K) + " need " +
                                         std::to_string(need) + " bytes of scratch, above the fixed " +
                                         std::to_string(kNoAllocScratchBytes));
    rc = check_ptrs(A, W, block_scale, C);
    if (rc) return rc;
    void* scratch = nullptr;
    if (M > 16) {
        std::string err;
        rc = noalloc_scratch(&scratch, &err);
        if (rc) return fail(rc, err);
    }
    const w8a16::GemmArgs g{A, a_row_stride, W, block_scale, C, c_row_stride, M, N, K};
    return run_ws(g, nullptr, scratch, scratch ? kNoAllocScratchBytes : 0, flags,
                  static_cast<cudaStream_t>(stream));
}

uint64_t w8a16_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int w8a16_split_activations(const void* A, uint32_t a_row_stride, uint32_t M, uint32_t K, void* workspace,
                            uint64_t workspace_bytes, w8a16_stream_t stream) {
    int rc = check_sizes(a_row_stride, 1, M, 1, K);
    if (rc) return rc;
    if (!A || !workspace)
        return fail(W8A16_ERR_NULL, std::string("w8a16_split_activations: NULL ") + (!A ? "A" : "workspace") +
                                        " pointer");
    if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(workspace) % 16)
        return fail(W8A16_ERR_ALIGN, "w8a16_split_activations: A and the workspace need 16-byte alignment");
    const uint64_t need = w8a16::split_ws_bytes(M, K);
    if (workspace_bytes < need)
        return fail(W8A16_ERR_ARG, "w8a16_split_activations: the workspace needs " + std::to_string(need) +
                                       " bytes (have " + std::to_string(workspace_bytes) + ")");
    DeviceInfo info;
    std::string err;
    rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    const uint32_t fstride = static_cast<uint32_t>(w8a16::split_ws_scale_stride(M));
    uint8_t* codes = static_cast<uint8_t*>(workspace);
    float* factors = reinterpret_cast<float*>(codes + 2ull * M * K);
    rc = w8a16::launch_split_act(A, a_row_stride, M, K, codes, factors, fstride, nullptr, 0u,
                                 static_cast<cudaStream_t>(stream), &err);
    if (rc) return fail(rc, err);
    return ok();
}

int w8a16_gemm_split_terms(const void* workspace, uint64_t workspace_bytes, const void* W,
                           const float* block_scale, void* C, uint32_t c_row_stride, uint32_t M, uint32_t N,
                           uint32_t K, uint32_t flags, w8a16_stream_t stream) {
    if (flags & ~static_cast<uint32_t>(W8A16_FLAG_PDL))
        return fail(W8A16_ERR_ARG, "w8a16_gemm_split_terms: unknown flag bits " + u(flags));
    int rc = check_sizes(K, c_row_stride, M, N, K);
    if (rc) return rc;
    rc = check_ptrs(workspace, W, block_scale, C);
    if (rc) return rc;
    const uint64_t need = w8a16::split_ws_bytes(M, K);
    if (workspace_bytes < need)
        return fail(W8A16_ERR_ARG, "w8a16_gemm_split_terms: the workspace holds " +
                                       std::to_string(workspace_bytes) + " bytes, the split of (M, K) needs " +
                                       std::to_string(need));
    const TimeoutSetting& ts = timeout_setting();
    if (!ts.valid)
        return fail(W8A16_ERR_ARG, "W8A16_WAIT_TIMEOUT_MS='" + ts.raw +
                                       "' is not an integer number of milliseconds in 1..600000");
    DeviceInfo info;
    std::string err;
    rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    w8a16_plan_t plan;
    rc = plan_live(W8A16_VARIANT_PRESPLIT, M, N, K, info, &plan, &err);
    if (rc) return fail(rc, err);
    const uint32_t fstride = static_cast<uint32_t>(w8a16::split_ws_scale_stride(M));
    const uint8_t* codes = static_cast<const uint8_t*>(workspace);
    const float* factors = reinterpret_cast<const float*>(codes + 2ull * M * K);
    const w8a16::W8A8Args a{codes, K, factors, fstride, W, block_scale, C, c_row_stride, M, N, K, 2u};
    rc = w8a16::launch_w8a8(a, plan, static_cast<cudaStream_t>(stream), ts.ns, flags, &err);
    if (rc) return fail(rc, err);
    return ok();
}

int w8a16_gemm_ws(const void* A, uint32_t a_row_stride, const void* W, const float* block_scale, void* C,
                  uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K, const w8a16_plan_t* plan,
                  void* workspace, uint64_t workspace_bytes, uint32_t flags, w8a16_stream_t stream) {
    const w8a16::GemmArgs g{A, a_row_stride, W, block_scale, C, c_row_stride, M, N, K};
    return run_ws(g, plan, workspace, workspace_bytes, flags, static_cast<cudaStream_t>(stream));
}

int w8a16_quantize_activations(const void* A, uint32_t a_row_stride, uint32_t M, uint32_t K, void* codes,
                               float* scales, uint32_t scale_stride, w8a16_stream_t stream) {
    if (M < 1) return fail(W8A16_ERR_M_ZERO, "w8a16_quantize_activations: m=0 has no rows");
    if (K < w8a16::kKStep || K % w8a16::kKStep != 0)
        return fail(W8A16_ERR_K_BLOCK, "w8a16_quantize_activations: K=" + u(K) +
                                           " must be a positive multiple of 128 (one scale per 128-K group)");
    if (a_row_stride < K || scale_stride < M)
        return fail(W8A16_ERR_PITCH, "w8a16_quantize_activations: a_row_stride=" + u(a_row_stride) +
                                         " must cover K=" + u(K) + " and scale_stride=" + u(scale_stride) +
                                         " must cover M=" + u(M));
    if (a_row_stride % 8 != 0 || scale_stride % 4 != 0)
        return fail(W8A16_ERR_A_PITCH_ALIGN, "w8a16_quantize_activations: a_row_stride=" + u(a_row_stride) +
                                                 " must be a multiple of 8 and scale_stride=" +
                                                 u(scale_stride) + " a multiple of 4");
    if (M > 0x7FFFFFFFu || K > 0x7FFFFFFFu)
        return fail(W8A16_ERR_RANGE, "w8a16_quantize_activations: M or K out of range");
    if (!A || !codes || !scales)
        return fail(W8A16_ERR_NULL, std::string("w8a16_quantize_activations: NULL ") +
                                        (!A ? "A" : !codes ? "codes" : "scales") + " pointer");
    const auto addr = [](const void* q) { return reinterpret_cast<uintptr_t>(q); };
    if (addr(A) % 16 || addr(codes) % 16 || addr(scales) % 16)
        return fail(W8A16_ERR_ALIGN, "w8a16_quantize_activations: A, codes and scales need 16-byte alignment");
    DeviceInfo info;
    std::string err;
    int rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    rc = w8a16::launch_quantize_act(A, a_row_stride, M, K, codes, scales, scale_stride,
                                    static_cast<cudaStream_t>(stream), &err);
    if (rc) return fail(rc, err);
    return ok();
}

int w8a16_plan_for(uint32_t M, uint32_t N, uint32_t K, uint32_t sm_count,
                   const uint32_t* cluster_ctas, w8a16_plan_t* out) {
    if (!out) return fail(W8A16_ERR_NULL, "w8a16_plan_for: NULL plan pointer");
    int rc = check_sizes(K, N, M, N, K);
    if (rc) return rc;
    plan_core(W8A16_VARIANT_AUTO, M, N, K, sm_count, cluster_ctas, out);
    return ok();
}

int w8a16_plan_current(uint32_t M, uint32_t N, uint32_t K, w8a16_plan_t* out) {
    if (!out) return fail(W8A16_ERR_NULL, "w8a16_plan_current: NULL plan pointer");
    int rc = check_sizes(K, N, M, N, K);
    if (rc) return rc;
    DeviceInfo info;
    std::string err;
    rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    rc = plan_live(W8A16_VARIANT_AUTO, M, N, K, info, out, &err);
    if (rc) return fail(rc, err);
    return ok();
}

int w8a16_plan_ws(uint32_t M, uint32_t N, uint32_t K, uint64_t workspace_bytes, w8a16_plan_t* out) {
    if (!out) return fail(W8A16_ERR_NULL, "w8a16_plan_ws: NULL plan pointer");
    int rc = check_sizes(K, N, M, N, K);
    if (rc) return rc;
    DeviceInfo info;
    std::string err;
    rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    bool presplit = false;
    rc = plan_ws_choice(M, N, K, workspace_bytes, info, out, &presplit, &err);
    if (rc) return fail(rc, err);
    return ok();
}

int w8a16_cluster_capacity(int32_t variant, uint32_t token_tile, uint32_t stages,
                           uint32_t out[17]) {
    if (!out) return fail(W8A16_ERR_NULL, "w8a16_cluster_capacity: NULL output");
    if (!(is_tc_variant(variant) || is_gemv(variant)) || !v_supported(variant, token_tile, stages))
        return fail(W8A16_ERR_PLAN, "w8a16_cluster_capacity: no kernel instance for variant " +
                                        std::to_string(variant) + " token_tile=" + u(token_tile) +
                                        " stages=" + u(stages));
    DeviceInfo info;
    std::string err;
    int rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    rc = live_capacity(variant, token_tile, stages, out, &err);
    if (rc) return fail(rc, err);
    return ok();
}

int w8a16_plan_variant(uint32_t M, uint32_t N, uint32_t K, int32_t variant, uint32_t split_k,
                       uint32_t stages, uint32_t sm_count, w8a16_plan_t* out) {
    if (!out) return fail(W8A16_ERR_NULL, "w8a16_plan_variant: NULL plan pointer");
    int rc = check_sizes(K, N, M, N, K);
    if (rc) return rc;
    w8a16_plan_t p;
    if (variant == W8A16_VARIANT_AUTO) {
        plan_core(W8A16_VARIANT_AUTO, M, N, K, sm_count, nullptr, &p);
    } else if (variant == W8A16_VARIANT_SIMT) {
        fill_simt(M, N, &p);
    } else if (is_stream(variant)) {
        if (!stream_applies(M, N, K) || (stages && stages != kStreamStages) || (split_k && split_k != 1))
            return fail(W8A16_ERR_PLAN, "w8a16_plan_variant: the stream-K plan takes " + u(kStreamMinTokens) +
                                            " <= M <= " + u(kStreamMaxTokens) + ", split 1 and " +
                                            u(kStreamStages) + " stages");
        fill_stream(M, N, K, sm_count, 0, &p);
    } else if (is_gemv(variant)) {
        const uint32_t sp = split_k ? split_k : gemv_split(M, N, K, sm_count, nullptr);
        if (sp == 0 || M > w8a16::kGvMaxTokens || (stages && stages != w8a16::kGvSlots))
            return fail(W8A16_ERR_PLAN, "w8a16_plan_variant: the decode kernel takes M <= " +
                                            u(w8a16::kGvMaxTokens) + " and at most " + u(w8a16::kGvMaxSteps) +
                                            " K steps per CTA on at most one CTA per SM");
        fill_gemv(N, sp, &p);
    } else if (is_tc_variant(variant)) {
        w8a16_plan_t a;
        plan_core(variant, M, N, K, sm_count, nullptr, &a);
        const uint32_t st = stages ? stages : a.stages;
        const uint32_t sp = split_k ? split_k : a.split_k;
        fill_tc(variant, M, N, a.token_tile, st, sp, &p);
        if (!split_k) add_tail(&p, M, N, K, sm_count, nullptr);   // an explicit split has none
    } else {
        return fail(W8A16_ERR_PLAN, "w8a16_plan_variant: unknown variant " + std::to_string(variant));
    }
    rc = validate_plan(M, N, K, p);
    if (rc) return rc;
    *out = p;
    return ok();
}

int w8a16_gemm(const void* A, uint32_t a_row_stride, const void* W, const float* block_scale,
               void* C, uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K,
               w8a16_stream_t stream) {
    return run({A, a_row_stride, W, block_scale, C, c_row_stride, M, N, K}, nullptr, 0,
               reinterpret_cast<cudaStream_t>(stream));
}

int w8a16_gemm_ex(const void* A, uint32_t a_row_stride, const void* W, const float* block_scale,
                  void* C, uint32_t c_row_stride, uint32_t M, uint32_t N, uint32_t K,
                  uint32_t flags, w8a16_stream_t stream) {
    return run({A, a_row_stride, W, block_scale, C, c_row_stride, M, N, K}, nullptr, flags,
               reinterpret_cast<cudaStream_t>(stream));
}

int w8a16_gemm_contiguous(const void* A, const void* W, const float* block_scale, void* C,
                          uint32_t M, uint32_t N, uint32_t K, w8a16_stream_t stream) {
    return w8a16_gemm(A, K, W, block_scale, C, N, M, N, K, stream);
}

int w8a16_gemm_with_plan(const void* A, uint32_t a_row_stride, const void* W,
                         const float* block_scale, void* C, uint32_t c_row_stride, uint32_t M,
                         uint32_t N, uint32_t K, const w8a16_plan_t* plan, uint32_t flags,
                         w8a16_stream_t stream) {
    if (!plan) return fail(W8A16_ERR_NULL, "w8a16_gemm_with_plan: NULL plan pointer");
    return run({A, a_row_stride, W, block_scale, C, c_row_stride, M, N, K}, plan, flags,
               reinterpret_cast<cudaStream_t>(stream));
}

int w8a16_gemm_host(const void* A_host, uint32_t a_row_stride, const void* W_host,
                    const float* scale_host, void* C_host, uint32_t c_row_stride, uint32_t M,
                    uint32_t N, uint32_t K, void* dA, void* dW, float* dScale, void* dC,
                    int copy_weights, w8a16_stream_t stream) {
    int rc = check_sizes(a_row_stride, c_row_stride, M, N, K);
    if (rc) return rc;
    if (!A_host || !C_host || (copy_weights && (!W_host || !scale_host)))
        return fail(W8A16_ERR_NULL, "w8a16_gemm_host: NULL host pointer");
    rc = check_ptrs(dA, dW, dScale, dC);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t scale_bytes = static_cast<size_t>(ceil_div(N, 128)) * (K / 128) * sizeof(float);
    cudaError_t e = cudaMemcpy2DAsync(dA, static_cast<size_t>(a_row_stride) * 2, A_host,
                                      static_cast<size_t>(a_row_stride) * 2, static_cast<size_t>(K) * 2,
                                      M, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && copy_weights)
        e = cudaMemcpyAsync(dW, W_host, static_cast<size_t>(N) * K, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && copy_weights)
        e = cudaMemcpyAsync(dScale, scale_host, scale_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(W8A16_ERR_COPY, std::string("w8a16_gemm_host: upload failed: ") + cudaGetErrorString(e));
    }
    rc = w8a16_gemm(dA, a_row_stride, dW, dScale, dC, c_row_stride, M, N, K, stream);
    if (rc) return rc;
    e = cudaMemcpy2DAsync(C_host, static_cast<size_t>(c_row_stride) * 2, dC,
                          static_cast<size_t>(c_row_stride) * 2, static_cast<size_t>(N) * 2, M,
                          cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(W8A16_ERR_COPY, std::string("w8a16_gemm_host: download failed: ") + cudaGetErrorString(e));
    }
    return ok();
}

const char* w8a16_last_error(void) { return g_last_error.c_str(); }

const char* w8a16_strerror(int code) {
    switch (code) {
        case W8A16_OK: return "success";
        case W8A16_ERR_M_ZERO: return "M is 0: no rows to compute";
        case W8A16_ERR_K_BLOCK: return "K is not a positive multiple of 128";
        case W8A16_ERR_PITCH: return "a row pitch is shorter than K (A) or N (C)";
        case W8A16_ERR_A_PITCH_ALIGN: return "a_row_stride is not a multiple of 8";
        case W8A16_ERR_N_ZERO: return "N is 0: no columns to compute";
        case W8A16_ERR_NULL: return "a required pointer is NULL";
        case W8A16_ERR_ALIGN: return "a pointer is not aligned (A, W: 16 B; block_scale: 4 B; C: 2 B)";
        case W8A16_ERR_RANGE: return "a size is beyond what the kernels address";
        case W8A16_ERR_DEVICE: return "no usable sm_103 CUDA device";
        case W8A16_ERR_LAUNCH: return "the CUDA launch failed";
        case W8A16_ERR_PLAN: return "the requested plan cannot run this shape";
        case W8A16_ERR_COPY: return "a host/device copy could not be queued";
        case W8A16_ERR_ARG: return "invalid argument";
        default: return "unknown error code";
    }
}

int w8a16_device_status(w8a16_stream_t stream, int clear, uint32_t* status, uint32_t* where,
                        uint32_t* detail) {
    w8a16::StatusWord w{0, 0, 0}, w8{0, 0, 0}, wa{0, 0, 0}, wg{0, 0, 0};
    cudaError_t e = w8a16::tc_status_read(&w, clear != 0, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess)
        e = w8a16::tc8_status_read(&w8, clear != 0, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess)
        e = w8a16::w8a8_status_read(&wa, clear != 0, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess)
        e = w8a16::gemv_status_read(&wg, clear != 0, reinterpret_cast<cudaStream_t>(stream));
    if (w.code == 0) w = w8;
    if (w.code == 0) w = wa;
    if (w.code == 0) w = wg;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(W8A16_ERR_DEVICE, std::string("w8a16_device_status: ") + cudaGetErrorString(e));
    }
    if (status) *status = w.code;
    if (where) *where = w.where;
    if (detail) *detail = w.detail;
    return ok();
}

int w8a16_selftest_wait_timeout(uint32_t timeout_us, w8a16_stream_t stream) {
    DeviceInfo info;
    std::string err;
    int rc = current_device_info(&info, &err);
    if (rc) return fail(rc, err);
    if (timeout_us < 1 || timeout_us > 10u * 1000u * 1000u)
        return fail(W8A16_ERR_ARG, "w8a16_selftest_wait_timeout: timeout_us must be in 1..10^7");
    rc = w8a16::launch_wait_selftest(static_cast<uint64_t>(timeout_us) * 1000ull,
                                     reinterpret_cast<cudaStream_t>(stream), &err);
    if (rc) return fail(rc, err);
    return ok();
}

const char* w8a16_version(void) { return "w8a16 0.1.0 (sm_103a)"; }

}  // extern "C"
