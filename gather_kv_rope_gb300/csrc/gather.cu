// Dequantise-and-gather of paged KV records back to bf16 [N, 512].
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "实现拆解" item 4: the gather reads a record by its width and
// dequantises e4m3 * 2^(scale - 127) per group -- 512 dims in 32-dim groups for
// V4.1, 448 dims in 64-dim groups plus a copied bf16 tail for V4; FlashMLA overview
// page, DSA section: an index of -1 is an invalid entry, which emits zeros).
//
// Launch shape: exactly one wave of warps; each warp walks a contiguous chunk of
// indices, loading 32 indices with one coalesced load and keeping S records in
// flight in a per-warp shared-memory ring filled by cp.async (the 512 / 576 data
// bytes as one 16-byte piece per lane, the scale row by one lane).  Output rows are
// written with streaming stores (each 1 KiB row is written once).
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

constexpr int kGatherDepth = 4;  // records in flight per warp

template <int kRecord>
struct Rec {
    static constexpr uint32_t D = kRecord == 528 ? 512u : 576u;   // data row bytes
    static constexpr uint32_t S = kRecord == 528 ? 16u : 8u;      // scale row bytes
    static constexpr int kSlot = kRecord == 528 ? 528 : 592;      // ring slot (16 B multiple)
};

__device__ __forceinline__ int32_t load_index_group(const GatherParams& p, int64_t i_begin, int n,
                                                    int g, int lane) {
    const int i = 32 * g + lane;
    return i < n ? __ldg(p.indices + i_begin + i) : -1;
}

// Stage the record of slot idx into ring slot k % S, then close one commit group.
template <int kRecord, int S>
__device__ __forceinline__ void stage(const GatherParams& p, uint8_t* ring, int k, int32_t idx,
                                      int lane) {
    using R = Rec<kRecord>;
    if (idx >= 0 && idx < p.num_slots) {
        const uint32_t s = static_cast<uint32_t>(idx);
        const uint32_t bs = static_cast<uint32_t>(p.block_size);
        const uint32_t page = s / bs, row = s - page * bs;
        const uint8_t* base = p.cache + static_cast<int64_t>(page) * p.page_stride;
        const uint8_t* data = base + row * R::D;
        const uint8_t* srow = base + bs * R::D + row * R::S;
        uint8_t* dst = ring + (k % S) * R::kSlot;
        cp_async16(dst + 16 * lane, data + 16 * lane);
        if (kRecord == 528) {
            if (lane == 0) cp_async16(dst + 512, srow);
        } else {
            if (lane < 4) cp_async16(dst + 512 + 16 * lane, data + 512 + 16 * lane);
            if (lane == 4) cp_async8(dst + 576, srow);
        }
    }
    cp_async_commit();
}

template <int kRecord, int S>
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherParams p, int64_t chunk) {
    using R = Rec<kRecord>;
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_wait_previous();
    pdl_release_next();
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t i_begin = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib) * chunk;
    if (i_begin >= p.num_indices) return;  // warp-uniform
    const int n = static_cast<int>(chunk < p.num_indices - i_begin ? chunk : p.num_indices - i_begin);
    uint8_t* ring = smem + wib * (S * R::kSlot);

    int32_t cur = load_index_group(p, i_begin, n, 0, lane);
    int32_t nxt = load_index_group(p, i_begin, n, 1, lane);
#pragma unroll
    for (int k = 0; k < S - 1; ++k) {
        const int32_t idx = __shfl_sync(kFull, cur, k);
        if (k < n) stage<kRecord, S>(p, ring, k, idx, lane);
        else cp_async_commit();
    }
    for (int j = 0; j < n; ++j) {
        const int k = j + S - 1;
        __syncwarp();                        // every lane is done reading ring slot k % S
        if (k < n) {
            const int32_t idx = __shfl_sync(kFull, ((k >> 5) == (j >> 5)) ? cur : nxt, k & 31);
            stage<kRecord, S>(p, ring, k, idx, lane);
        } else {
            cp_async_commit();
        }
        cp_async_wait<S - 1>();              // this lane's pieces of record j have landed
        __syncwarp();                        // ... and every other lane's

        const int32_t idx = __shfl_sync(kFull, cur, j & 31);
        uint4 oa = make_uint4(0u, 0u, 0u, 0u), ob = oa;
        if (idx >= 0 && idx < p.num_slots) {
            const uint8_t* src = ring + (j % S) * R::kSlot;
            const uint2 ca = lds8(src + 8 * lane);
            if (kRecord == 528) {
                const uint4 sc = lds16(src + 512);
                oa = dequant8(ca, byte_of(sc, lane >> 2));
                ob = dequant8(lds8(src + 256 + 8 * lane), byte_of(sc, 8 + (lane >> 2)));
            } else {
                const uint2 sc = lds8(src + 576);
                oa = dequant8(ca, byte_of(sc, lane >> 3));
                ob = (lane < 24) ? dequant8(lds8(src + 256 + 8 * lane), byte_of(sc, 4 + (lane >> 3)))
                                 : lds16(src + 448 + 16 * (lane - 24));
            }
        } else if (idx != -1 && lane == 0) {
            report(p.err, 4);
        }
        uint8_t* orow = static_cast<uint8_t*>(p.out) + (i_begin + j) * 1024;
        st_stream16(orow + 16 * lane, oa);
        st_stream16(orow + 512 + 16 * lane, ob);
        if ((j & 31) == 31) {
            cur = nxt;
            nxt = load_index_group(p, i_begin, n, (j >> 5) + 2, lane);
        }
    }
    cp_async_wait<0>();
}

template <int kRecord, int S>
cudaError_t launch(const GatherParams& p, cudaStream_t stream) {
    if (p.num_indices <= 0) return cudaSuccess;
    auto kernel = gather_kernel<kRecord, S>;
    const size_t smem = static_cast<size_t>(kWarpsPerBlock) * S * Rec<kRecord>::kSlot;
    int64_t wave = 0;
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(kernel), kThreads, smem, &wave);
    if (e != cudaSuccess) return e;
    int64_t chunk = 0, blocks = 0;
    one_wave_split(p.num_indices, wave, kWarpsPerBlock, &chunk, &blocks);
    return launch_kernel(kernel, blocks, kThreads, smem, stream, p, chunk);
}

}  // namespace

cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream) {
    return launch<528, kGatherDepth>(p, stream);
}
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream) {
    return launch<584, kGatherDepth>(p, stream);
}

}  // namespace gkr
