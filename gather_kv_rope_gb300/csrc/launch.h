// Internal interface between the host ABI (api.cu) and the kernel launchers.
#pragma once

#include <cstdint>
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

cudaError_t launch_insert_v41(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_insert_v4(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream);
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream);

}  // namespace gkr
