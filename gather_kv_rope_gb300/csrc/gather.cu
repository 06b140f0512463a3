// Dequantise-and-gather of paged KV records back to bf16 [N, 512].
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "实现拆解" item 4: the gather reads a record by its width and
// dequantises e4m3 * 2^(scale - 127) per group -- 512 dims in 32-dim groups for
// V4.1, 448 dims in 64-dim groups plus a copied bf16 tail for V4; FlashMLA overview
// page, DSA section: an index of -1 is an invalid entry, which emits zeros).
//
// Launch shape: at most one wave of warps, each walking its own list of indices
// (see WorkMap); one warp per record, lane L owning output dims [8L, 8L+8) and
// [256+8L, 256+8L+8).  Per group of 32 indices, lane i decodes index i once
// (validity, the record's byte offset, the distance to its scale row), so a record
// costs three shuffles, four coalesced loads (two 8-byte code pieces, two scale
// bytes), the dequantisation and two 16-byte streaming stores.  Records are loaded
// straight into registers in batches of P, the next batch's loads issued before the
// current batch is converted, so 2P records per warp are in flight.
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

#ifndef GKR_GATHER_BATCH
#define GKR_GATHER_BATCH 2
#endif
#ifndef GKR_GATHER_CYCLIC
#define GKR_GATHER_CYCLIC 0
#endif
constexpr int kBatch = GKR_GATHER_BATCH;   // records per batch (a power of two <= 16)

template <int kRecord>
struct Rec {
    static constexpr uint32_t D = kRecord == 528 ? 512u : 576u;   // data row bytes
    static constexpr uint32_t S = kRecord == 528 ? 16u : 8u;      // scale row bytes
};

// Read-only loads that do not allocate in L1 (each record is read once).
__device__ __forceinline__ uint2 ldg_na8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg_na16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u8(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Lane-parallel decode of one group of 32 indices: for this lane's index, the
// record's byte offset in the cache (-1 when the index is -1 or out of range) and the
// distance from the data row to the scale row.  Out-of-range indices set GKR_ERR_INDEX.
template <int kRecord>
__device__ __forceinline__ void decode_group(const GatherParams& p, const WarpItems& w, int g,
                                             int lane, int64_t& off, int32_t& delta) {
    using R = Rec<kRecord>;
    const int i = 32 * g + lane;
    off = -1;
    delta = 0;
    bool bad = false;
    if (i < w.n) {
        const int32_t idx = __ldg(p.indices + w.at(i));
        if (idx >= 0 && idx < p.num_slots) {
            const uint32_t s = static_cast<uint32_t>(idx);
            const uint32_t bs = static_cast<uint32_t>(p.block_size);
            const uint32_t page = s / bs, row = s - page * bs;
            off = static_cast<int64_t>(page) * p.page_stride + row * R::D;
            delta = static_cast<int32_t>(bs * R::D + row * R::S - row * R::D);
        } else {
            bad = idx != -1;
        }
    }
    if (__ballot_sync(kFull, bad) != 0u && lane == 0) report(p.err, 4);
}

struct Loaded {
    uint2 a;        // codes of chunk A
    uint4 b;        // codes of chunk B (.x, .y) or, for the V4 tail lanes, 8 bf16
    uint32_t sa, sb;
    bool valid;
};

template <int kRecord>
__device__ __forceinline__ void load_record(const GatherParams& p, int64_t off, int32_t delta,
                                            int lane, Loaded& r) {
    r.valid = off >= 0;
    if (!r.valid) return;
    const uint8_t* data = p.cache + off;
    const uint8_t* srow = data + delta;
    r.a = ldg_na8(data + 8 * lane);
    if (kRecord == 528) {
        const uint2 t = ldg_na8(data + 256 + 8 * lane);
        r.b = make_uint4(t.x, t.y, 0u, 0u);
        r.sa = ldg_u8(srow + (lane >> 2));
        r.sb = ldg_u8(srow + 8 + (lane >> 2));
    } else {
        if (lane < 24) {
            const uint2 t = ldg_na8(data + 256 + 8 * lane);
            r.b = make_uint4(t.x, t.y, 0u, 0u);
            r.sb = ldg_u8(srow + 4 + (lane >> 3));
        } else {
            r.b = ldg_na16(data + 448 + 16 * (lane - 24));
            r.sb = 0u;
        }
        r.sa = ldg_u8(srow + (lane >> 3));
    }
}

template <int kRecord>
__device__ __forceinline__ void convert_store(const Loaded& r, uint8_t* orow, int lane) {
    uint4 oa = make_uint4(0u, 0u, 0u, 0u), ob = oa;
    if (r.valid) {
        oa = dequant8(r.a, r.sa);
        if (kRecord == 528 || lane < 24) ob = dequant8(make_uint2(r.b.x, r.b.y), r.sb);
        else ob = r.b;
    }
    st_stream16(orow + 16 * lane, oa);
    st_stream16(orow + 512 + 16 * lane, ob);
}

template <int kRecord, int P>
__device__ __forceinline__ void load_batch(const GatherParams& p, int j, int n, bool same,
                                           int64_t cur_off, int32_t cur_delta, int64_t nxt_off,
                                           int32_t nxt_delta, int lane, Loaded* r) {
#pragma unroll
    for (int u = 0; u < P; ++u) {
        const int64_t off = __shfl_sync(kFull, same ? cur_off : nxt_off, (j + u) & 31);
        const int32_t delta = __shfl_sync(kFull, same ? cur_delta : nxt_delta, (j + u) & 31);
        load_record<kRecord>(p, j + u < n ? off : -1, delta, lane, r[u]);
    }
}

template <int kRecord, int P>
__global__ void __launch_bounds__(kThreads, kRecord == 584 ? 3 : GKR_MIN_BLOCKS) gather_kernel(const GatherParams p,
                                                                          const WorkMap m) {
    static_assert((P & (P - 1)) == 0 && P >= 1 && P <= 16, "batch: power of two <= 16");
    pdl_wait_previous();
    pdl_release_next();
    const int lane = threadIdx.x & 31;
    const WarpItems w = warp_items(m, static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock +
                                          (threadIdx.x >> 5));
    if (w.n <= 0) return;  // warp-uniform
    const int n = w.n;
    uint8_t* out = static_cast<uint8_t*>(p.out);

    // cur describes the group (32 items) holding the batch being converted, nxt the next
    int64_t cur_off, nxt_off;
    int32_t cur_delta, nxt_delta;
    decode_group<kRecord>(p, w, 0, lane, cur_off, cur_delta);
    decode_group<kRecord>(p, w, 1, lane, nxt_off, nxt_delta);

    // Batches of P items [j, j + P), aligned so a batch never straddles two groups.
    Loaded A[P], B[P];
    load_batch<kRecord, P>(p, 0, n, true, cur_off, cur_delta, nxt_off, nxt_delta, lane, A);
    for (int j0 = 0; j0 < n; j0 += 2 * P) {
        const int j1 = j0 + P, j2 = j0 + 2 * P;
        load_batch<kRecord, P>(p, j1, n, (j1 >> 5) == (j0 >> 5), cur_off, cur_delta, nxt_off,
                               nxt_delta, lane, B);
#pragma unroll
        for (int u = 0; u < P; ++u)
            if (j0 + u < n) convert_store<kRecord>(A[u], out + w.at(j0 + u) * 1024, lane);
        if ((j1 & 31) == 0) {                // batch j1 opens a new group
            cur_off = nxt_off;
            cur_delta = nxt_delta;
            decode_group<kRecord>(p, w, (j1 >> 5) + 1, lane, nxt_off, nxt_delta);
        }
        load_batch<kRecord, P>(p, j2, n, (j2 >> 5) == (j1 >> 5), cur_off, cur_delta, nxt_off,
                               nxt_delta, lane, A);
#pragma unroll
        for (int u = 0; u < P; ++u)
            if (j1 + u < n) convert_store<kRecord>(B[u], out + w.at(j1 + u) * 1024, lane);
        if ((j2 & 31) == 0) {                // batch j2 opens a new group
            cur_off = nxt_off;
            cur_delta = nxt_delta;
            decode_group<kRecord>(p, w, (j2 >> 5) + 1, lane, nxt_off, nxt_delta);
        }
    }
}

template <int kRecord, int P>
cudaError_t launch(const GatherParams& p, cudaStream_t stream) {
    if (p.num_indices <= 0) return cudaSuccess;
    auto kernel = gather_kernel<kRecord, P>;
    int64_t wave = 0;
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(kernel), kThreads, 0, &wave);
    if (e != cudaSuccess) return e;
    const WorkMap m = make_work_map(p.num_indices, wave, GKR_GATHER_CYCLIC != 0);
    const int64_t blocks = (m.warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_kernel(kernel, blocks, kThreads, 0, stream, p, m);
}

}  // namespace

cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream) {
    return launch<528, kBatch>(p, stream);
}
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream) {
    return launch<584, kBatch>(p, stream);
}

}  // namespace gkr
