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
    int64_t max_pos;           // < 2^31 (checked on the host)
    int64_t ratio;             // compress ratio >= 1 (1 for the plain insert)
    const float* fp8_scale;    // fp8 rows (record 512): the cache's scale; else unused
    int32_t* err;              // nullable
    int32_t early_metadata;    // 1: slots / positions may be read before the PDL wait
    int32_t pdl;               // 1: launch with the programmatic-dependent-launch attribute
    int64_t staged_min;        // token counts from which the insert stages rows in shared
    int64_t stream_min;        //   memory / streams them (launch policy of this call)
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
    const float* fp8_scale;    // fp8 rows (record 512): the cache's scale; else unused
    int32_t* err;              // nullable
    int32_t early_metadata;    // 1: indices may be read before the PDL wait
    int32_t pdl;               // 1: launch with the programmatic-dependent-launch attribute
};

// Query side of the fused attention write (gkr_qnorm_rope_kv_insert).
struct QSideParams {
    const void* q_in;          // bf16 [num_tokens, num_heads, 512]
    void* q_out;               // bf16 [num_tokens, num_heads_padded, 512], or e4m3 codes
    const float* q_scale;      // nullptr: bf16 q_out; else the e4m3 q_out's fp32 scale
    int32_t num_heads;
    int32_t num_heads_padded;  // >= num_heads, > 0 (0 is the plain KV insert)
    float eps;
    int32_t apply_norm;        // 1: divide each head by sqrt(mean(x^2) + eps)
};

// Validated arguments of one fused gather + logits launch (gkr_sparse_logits).
struct LogitsParams {
    const void* q;             // bf16 [num_queries, num_heads, 512]
    int32_t num_heads;         // 1 .. logits_max_heads()
    const uint8_t* cache;
    int64_t page_stride;
    int32_t block_size;
    int32_t num_slots;
    const int32_t* indices;    // [num_queries, topk]
    int64_t num_queries;
    int64_t topk;              // a multiple of 4
    int64_t chunks;            // ceil(topk / logits_chunk_keys())
    float sm_scale;
    const float* fp8_scale;    // fp8 rows (record 512): the cache's scale; else unused
    float* out;                // fp32 [num_queries, num_heads, topk]
    int32_t* err;              // nullable
    int32_t pdl;
};

// Row geometry of the four cache formats ("record" = bytes a token occupies):
//   528  V4.1 MXFP8 record: 512 B e4m3 data row + 16 B scale row;
//   584  V4 record: 576 B data row (448 e4m3 + 64 bf16) + 8 B scale row;
//   512  fp8 e4m3 row, one fp32 scale for the whole cache, no scale row;
//   1024 bf16 row, no scale row.
// A page holds block_size data rows, then block_size scale rows.
template <int kRecord>
struct Fmt {
    static constexpr uint32_t D =
        kRecord == 528 ? 512u : kRecord == 584 ? 576u : static_cast<uint32_t>(kRecord);
    static constexpr uint32_t S = kRecord == 528 ? 16u : kRecord == 584 ? 8u : 0u;
    // bytes of a row that lane L owns at 8L-dim granularity: 8 e4m3 or 16 bf16 bytes
    static constexpr int kLaneBytes = kRecord == 1024 ? 16 : 8;
    static constexpr bool kPacked = kRecord == 528 || kRecord == 584;
};

// Launch-shape helpers (api.cu).  `resident_warps` returns how many warps of `func`
// (launched with `threads` threads and `smem` dynamic shared bytes per block) fit
// on the current device at once: SM count x resident blocks per SM x warps per
// block.  Results are cached per device and kernel; the first call for a kernel
// on a device also raises its dynamic shared-memory limit when it needs more than
// the default 48 KiB.
cudaError_t resident_warps(const void* func, int threads, size_t smem, int64_t* warps);

// Launch `kernel`, with the programmatic-dependent-launch attribute when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), int64_t blocks, int threads, size_t smem,
                          cudaStream_t stream, int32_t pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl != 0 ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// How the items (tokens or indices) of a launch are dealt to its warps.  Warp w owns
// items base(w) + j * step for j in [0, count(w)):
//   chunked  (step 1):      base = w * chunk, a contiguous run of `chunk` items;
//   cyclic   (step = warps): base = w, so the warps active at one moment touch one
//                            contiguous window of items.
// Either way the grid is at most one resident wave of warps.
struct WorkMap {
    int64_t n;        // items in the launch
    int64_t chunk;    // chunked: items per warp
    int64_t warps;    // warps launched
    int32_t cyclic;   // 1 = cyclic, 0 = chunked
};

// max_chunk caps the items per warp (chunked maps only): larger launches then become
// several waves of short-lived warps, which the block scheduler balances at the end.
inline WorkMap make_work_map(int64_t n, int64_t wave_warps, bool cyclic, int64_t granule = 1,
                             int64_t max_chunk = 0) {
    WorkMap m;
    m.n = n;
    m.cyclic = cyclic ? 1 : 0;
    if (wave_warps < 1) wave_warps = 1;
    m.chunk = (n + wave_warps - 1) / wave_warps;
    if (!cyclic && max_chunk > 0 && m.chunk > max_chunk) m.chunk = max_chunk;
    m.chunk = (m.chunk + granule - 1) / granule * granule;   // whole warp iterations
    m.warps = cyclic ? (n < wave_warps ? n : wave_warps) : (n + m.chunk - 1) / m.chunk;
    return m;
}

// The items of warp `gw` under a work map: item j is base + j * step, j < n.
struct WarpItems {
    int64_t base, step;
    int n;
    __host__ __device__ int64_t at(int j) const { return base + j * step; }
};

__host__ __device__ inline WarpItems warp_items(const WorkMap& m, int64_t gw) {
    WarpItems w;
    if (gw >= m.warps) {         // spare warps of the last block
        w.base = 0;
        w.step = 1;
        w.n = 0;
        return w;
    }
    if (m.cyclic) {
        w.base = gw;
        w.step = m.warps;
        w.n = gw < m.n ? static_cast<int>((m.n - 1 - gw) / m.warps + 1) : 0;
    } else {
        w.base = gw * m.chunk;
        w.step = 1;
        const int64_t r = m.n - w.base;
        w.n = r <= 0 ? 0 : static_cast<int>(r < m.chunk ? r : m.chunk);
    }
    return w;
}

cudaError_t launch_insert_v41(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_insert_v4(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_insert_fp8(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_insert_bf16(const InsertParams& p, cudaStream_t stream);
// Compressed-KV insert: only group-boundary tokens are written; NaN -> 0 if sanitize.
cudaError_t launch_rope_quant_insert_v41(const InsertParams& p, bool sanitize,
                                         cudaStream_t stream);
cudaError_t launch_rope_quant_insert_v4(const InsertParams& p, bool sanitize,
                                        cudaStream_t stream);
// Query heads normed and rotated, padded heads zeroed, and the KV rows inserted (any of
// the four cache formats), in one launch.
cudaError_t launch_qnorm_rope_kv_insert(int32_t record, const InsertParams& p,
                                        const QSideParams& qp, cudaStream_t stream);
// Sparse decode logits from the cache records, gathered and dequantised on chip.
cudaError_t launch_sparse_logits(int32_t record, const LogitsParams& p, cudaStream_t stream);
int32_t logits_chunk_keys(int32_t record);   // keys per work item
int32_t logits_max_heads();    // heads per query at most
cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream);
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream);
cudaError_t launch_gather_fp8(const GatherParams& p, cudaStream_t stream);
cudaError_t launch_gather_bf16(const GatherParams& p, cudaStream_t stream);

}  // namespace gkr
