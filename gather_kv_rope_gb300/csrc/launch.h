// Internal interface between the host ABI (api.cu) and the kernel launchers.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace gkr {

// Validated arguments of one insert launch (all device pointers).
struct InsertParams {
    const void* kv;            // bf16 [num_tokens, 512]
    int64_t num_tokens;
    uint8_t* cache;
    int64_t page_stride;
    int32_t block_size;
    int32_t num_slots;         // num_pages * block_size (< 2^31, checked on the host)
    const int64_t* slots;
    const int64_t* positions;
    const float* csc;          // fp32 [max_pos, 64]
    int64_t max_pos;
    int32_t* err;              // nullable
};

// Validated arguments of one gather launch.
struct GatherParams {
    const uint8_t* cache;
    int64_t page_stride;
    int32_t block_size;
    int32_t num_slots;
    const int32_t* indices;
    int64_t num_indices;
    void* out;                 // bf16 [num_indices, 512]
    int32_t* err;              // nullable
};

// Launch-shape helpers (api.cu).  `resident_warps` returns how many warps of `func`
// (launched with `threads` threads and `smem` dynamic shared bytes per block) fit
// on the current device at once: SM count x resident blocks per SM x warps per
// block.  Results are cached per device and kernel; the first call for a kernel
// on a device also raises its dynamic shared-memory limit when it needs more than
// the default 48 KiB.
cudaError_t resident_warps(const void* func, int threads, size_t smem, int64_t* warps);
// Whether launches carry the programmatic-dependent-launch attribute.
bool pdl_enabled();

// Launch `kernel` with the PDL attribute when enabled.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), int64_t blocks, int threads, size_t smem,
                          cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Split `n` items over at most one wave of warps: returns the items per warp
// (chunk) and the number of blocks of `warps_per_block` warps.
inline void one_wave_split(int64_t n, int64_t wave_warps, int warps_per_block, int64_t* chunk,
                           int64_t* blocks) {
    if (wave_warps < 1) wave_warps = 1;
    *chunk = (n + wave_warps - 1) / wave_warps;
    const int64_t warps = (n + *chunk - 1) / *chunk;
    *blocks = (warps + warps_per_block - 1) / warps_per_block;
}

cudaError_t launch_insert_v41(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_insert_v4(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream);
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream);

}  // namespace gkr
