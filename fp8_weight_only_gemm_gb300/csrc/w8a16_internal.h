// Definitions shared by the host dispatcher and the kernel translation units.
#pragma once

#include <cstdint>
#include <string>

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

struct StatusWord {
    uint32_t code, where, detail;
};

// Tiling constants of the tensor-core variant.
constexpr uint32_t kTcRows = 128;      // weight rows per tile (tcgen05 MMA M)
constexpr uint32_t kKStep = 128;       // K per pipeline stage == one scale block
constexpr uint32_t kTcConvWarps = 8;   // converter / fold warps
constexpr uint32_t kTcThreads = 64 + 32 * kTcConvWarps;
constexpr uint32_t kTcMaxTokenTile = 128;

// Shared-memory bytes the TC kernel needs for a token tile and stage count.
constexpr uint32_t tc_smem_bytes(uint32_t tn, uint32_t stages) {
    return 1024 /* alignment slack */ + stages * (kTcRows * kKStep + tn * kKStep * 2) +
           /* barriers, tmem slot, flags */ 256;
}
constexpr uint32_t tc_tmem_cols(uint32_t tn) {
    return (2 * (kKStep / 2) + 2 * tn) <= 256 ? 256u : 512u;
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
int launch_wait_selftest(uint64_t timeout_ns, cudaStream_t s, std::string* err);

// Device status of the TC translation unit (the only one with waits).
cudaError_t tc_status_read(StatusWord* out, bool clear, cudaStream_t s);

bool tc_supported_token_tile(uint32_t tn);
bool tc_supported_stages(uint32_t tn, uint32_t stages);

}  // namespace w8a16
