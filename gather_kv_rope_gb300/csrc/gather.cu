// Dequantise-and-gather of paged KV records back to bf16 [N, 512].
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "实现拆解" item 4: the gather reads a record by its width and
// dequantises e4m3 * 2^(scale - 127) per group -- 512 dims in 32-dim groups for
// V4.1, 448 dims in 64-dim groups plus a copied bf16 tail for V4; FlashMLA overview
// page, DSA section: an index of -1 is an invalid entry, which emits zeros).
//
// Launch shape: one warp per index, U indices per warp with all record loads
// issued before any is consumed, 8 warps per block.  Output rows are written with
// streaming stores (each 1 KiB row is written once and not re-read here).
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

__device__ __forceinline__ bool index_ok(const GatherParams& p, int32_t idx, bool in, int lane) {
    if (idx >= 0 && idx < p.num_slots) return true;
    if (in && idx != -1 && lane == 0) report(p.err, 4);
    return false;
}

struct RecordLoads {
    uint2 a;      // e4m3 codes of chunk A
    uint4 b;      // e4m3 codes of chunk B (.x/.y), or the V4 bf16 tail (all four words)
    uint4 sc;     // scale row (V4.1: 16 bytes; V4: 8 bytes in .x/.y)
};

template <int kRecord>
__device__ __forceinline__ void load_record(const GatherParams& p, int32_t idx, int lane,
                                            RecordLoads& L) {
    constexpr uint32_t D = kRecord == 528 ? 512u : 576u;
    constexpr uint32_t S = kRecord == 528 ? 16u : 8u;
    const uint32_t s = static_cast<uint32_t>(idx);
    const uint32_t bs = static_cast<uint32_t>(p.block_size);
    const uint32_t page = s / bs, row = s - page * bs;
    const uint8_t* base = p.cache + static_cast<int64_t>(page) * p.page_stride;
    const uint8_t* data = base + row * D;
    L.a = ld_ro8(data + 8 * lane);
    if (kRecord == 528) {
        const uint2 t = ld_ro8(data + 256 + 8 * lane);
        L.b = make_uint4(t.x, t.y, 0u, 0u);
        L.sc = ld_ro16(base + bs * D + row * S);
    } else {
        if (lane < 24) {
            const uint2 t = ld_ro8(data + 256 + 8 * lane);
            L.b = make_uint4(t.x, t.y, 0u, 0u);
        } else {
            L.b = ld_ro16(data + 448 + 16 * (lane - 24));
        }
        const uint2 t = ld_ro8(base + bs * D + row * S);
        L.sc = make_uint4(t.x, t.y, 0u, 0u);
    }
}

template <int kRecord, int U>
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * U;
    if (i0 >= p.num_indices) return;

    int32_t idx[U];
    bool in[U], ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        in[u] = i0 + u < p.num_indices;
        idx[u] = in[u] ? __ldg(p.indices + i0 + u) : -1;
    }
    RecordLoads L[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        ok[u] = index_ok(p, idx[u], in[u], lane);
        if (ok[u]) load_record<kRecord>(p, idx[u], lane, L[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!in[u]) continue;
        uint4 oa = make_uint4(0u, 0u, 0u, 0u), ob = oa;
        if (ok[u]) {
            if (kRecord == 528) {
                oa = dequant8(L[u].a, byte_of(L[u].sc, lane >> 2));
                ob = dequant8(make_uint2(L[u].b.x, L[u].b.y), byte_of(L[u].sc, 8 + (lane >> 2)));
            } else {
                const uint2 sc = make_uint2(L[u].sc.x, L[u].sc.y);
                oa = dequant8(L[u].a, byte_of(sc, lane >> 3));
                ob = (lane < 24) ? dequant8(make_uint2(L[u].b.x, L[u].b.y), byte_of(sc, 4 + (lane >> 3)))
                                 : L[u].b;
            }
        }
        uint8_t* orow = static_cast<uint8_t*>(p.out) + (i0 + u) * 1024;
        st_stream16(orow + 16 * lane, oa);
        st_stream16(orow + 512 + 16 * lane, ob);
    }
}

template <int kRecord, int U>
cudaError_t launch(const GatherParams& p, cudaStream_t stream) {
    if (p.num_indices <= 0) return cudaSuccess;
    const int64_t per_block = static_cast<int64_t>(kWarpsPerBlock) * U;
    const int64_t blocks = (p.num_indices + per_block - 1) / per_block;
    gather_kernel<kRecord, U><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

constexpr int kGatherIndicesPerWarp = 2;

cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream) {
    return launch<528, kGatherIndicesPerWarp>(p, stream);
}
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream) {
    return launch<584, kGatherIndicesPerWarp>(p, stream);
}

}  // namespace gkr
