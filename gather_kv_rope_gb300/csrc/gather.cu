// Dequantise-and-gather of paged KV records back to bf16 [N, 512] (also from the two
// plain caches: bf16 rows are copied, fp8 e4m3 rows multiplied by the cache's scale).
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "实现拆解" item 4: the gather reads a record by its width and
// dequantises e4m3 * 2^(scale - 127) per group -- 512 dims in 32-dim groups for
// V4.1, 448 dims in 64-dim groups plus a copied bf16 tail for V4; FlashMLA overview
// page, DSA section: an index of -1 is an invalid entry, which emits zeros).
//
// Launch shape: one warp per record, lane L owning output dims [8L, 8L+8) and
// [256+8L, 256+8L+8), U records per warp, all their loads issued before the first is
// converted.  Every load and store instruction covers one contiguous 256- or 512-byte
// span.  A random-record gather is latency-bound, so the kernel favours many resident
// warps (few registers) over deep per-warp pipelines.
#include "decode.cuh"
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

#ifndef GKR_GATHER_PER_WARP
#define GKR_GATHER_PER_WARP 2
#endif
constexpr int kPerWarp = GKR_GATHER_PER_WARP;   // records per warp


// Dequantise one loaded record (zeros for an invalid one) and write its output row.
template <int kRecord>
__device__ __forceinline__ void convert_store(const Loaded<kRecord>& r, uint8_t* orow, int lane,
                                              float scale) {
    uint4 oa, ob;
    convert<kRecord>(r, lane, scale, oa, ob);
    st_stream16(orow, oa);
    st_stream16(orow + 512, ob);
}

// One warp per U consecutive indices; lanes 0..U-1 decode them in parallel and the
// offsets are broadcast with shuffles, so each record costs two shuffles, four loads,
// the dequantisation and two stores.  Short-lived warps (U records each) keep many
// warps resident and let the block scheduler balance the end of a large gather.
template <int kRecord, int U, bool kEarly>
__global__ void __launch_bounds__(kThreads, kRecord == 584 ? 6 : 8)
    gather_kernel(const GatherParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * U;
    // lane u < U decodes index i0 + u; with early metadata (gkr_set_early_metadata, the
    // kEarly instantiation) the index is read before waiting for the previous kernel,
    // every other access after
    int32_t idx = -1;
    if constexpr (kEarly) {
        if (lane < U && i0 + lane < p.num_indices) idx = __ldg(p.indices + i0 + lane);
    }
    pdl_wait_previous();
    pdl_release_next();
    if (i0 >= p.num_indices) return;  // warp-uniform

    // fp8 rows: the cache's scale, read once per warp; not a positive finite number ->
    // every row of the warp is written as zeros and the error bit is set
    float scale = 1.0f;
    bool scale_bad = false;
    if constexpr (kRecord == 512) {
        scale = __ldg(p.fp8_scale);
        scale_bad = !scale_ok(scale);
        if (scale_bad && lane == 0) report(p.err, kErrScale);
    }

    // data-row offset (-1 = emit zeros), scale-row offset
    int64_t off = -1, soff = 0;
    bool bad = false;
    if (lane < U && i0 + lane < p.num_indices && !scale_bad) {
        using R = Fmt<kRecord>;
        if constexpr (!kEarly) idx = __ldg(p.indices + i0 + lane);
        if (idx >= 0 && idx < p.num_slots) {
            const uint32_t s = static_cast<uint32_t>(idx);
            const uint32_t bs = static_cast<uint32_t>(p.block_size);
            uint32_t page, row;
            page_row(s, bs, page, row);
            const int64_t base = static_cast<int64_t>(page) * p.page_stride;
            off = base + row * R::D;
            soff = base + bs * R::D + row * R::S;
        } else {
            bad = idx != -1;
        }
    }
    LaneBases lb;
    lb.a = p.cache + Fmt<kRecord>::kLaneBytes * lane;
    lb.tail = p.cache + 448 + 16 * (lane >= 24 ? lane - 24 : 0);
    lb.s = p.cache + (kRecord == 528 ? (lane >> 2) : (lane >> 3));
    Loaded<kRecord> r[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        load_record<kRecord>(__shfl_sync(kFull, off, u), __shfl_sync(kFull, soff, u), lb, lane, r[u]);
    // the error bit while the record loads are in flight
    if (__ballot_sync(kFull, bad) != 0u && lane == 0) report(p.err, 4);
    uint8_t* orow = static_cast<uint8_t*>(p.out) + i0 * 1024 + 16 * lane;
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (i0 + u < p.num_indices) convert_store<kRecord>(r[u], orow + u * 1024, lane, scale);
}

template <int kRecord, int U>
cudaError_t launch(const GatherParams& p, cudaStream_t stream) {
    if (p.num_indices <= 0) return cudaSuccess;
    const int64_t per_block = static_cast<int64_t>(kWarpsPerBlock) * U;
    const int64_t blocks = (p.num_indices + per_block - 1) / per_block;
    return p.early_metadata != 0
               ? launch_kernel(gather_kernel<kRecord, U, true>, blocks, kThreads, 0, stream, p.pdl, p)
               : launch_kernel(gather_kernel<kRecord, U, false>, blocks, kThreads, 0, stream, p.pdl, p);
}

}  // namespace

cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream) {
    return launch<528, kPerWarp>(p, stream);
}
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream) {
    return launch<584, kPerWarp>(p, stream);
}
cudaError_t launch_gather_fp8(const GatherParams& p, cudaStream_t stream) {
    return launch<512, kPerWarp>(p, stream);
}
cudaError_t launch_gather_bf16(const GatherParams& p, cudaStream_t stream) {
    return launch<1024, kPerWarp>(p, stream);
}

}  // namespace gkr
