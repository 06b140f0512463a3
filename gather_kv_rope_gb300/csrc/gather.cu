// Dequantise-and-gather of paged KV records back to bf16 [N, 512].
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "实现拆解" item 4: the gather reads a record by its width and
// dequantises e4m3 * 2^(scale - 127) per group -- 512 dims in 32-dim groups for
// V4.1, 448 dims in 64-dim groups plus a copied bf16 tail for V4; FlashMLA overview
// page, DSA section: an index of -1 is an invalid entry, which emits zeros).
//
// Launch shape: at most one wave of warps, each walking its own list of indices
// (see WorkMap), two indices per iteration -- one per half-warp, lane q of a half
// owning output dims [32q, 32q + 32).  Per group of 32 indices, lane i decodes index
// i once (validity, the record's byte offset, the distance to its scale row), so the
// per-index cost is two shuffles, the copies and the dequantisation.  A per-warp ring
// in shared memory, filled by cp.async, keeps S iterations (2S records) in flight;
// each lane's slice of a staged record is padded by 16 bytes so the 16-byte shared
// loads of 8 consecutive lanes fall in distinct bank groups.  Output rows are
// written with streaming stores (each 1 KiB row is written once).
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

#ifndef GKR_GATHER_DEPTH
#define GKR_GATHER_DEPTH 4
#endif
#ifndef GKR_GATHER_CYCLIC
#define GKR_GATHER_CYCLIC 0
#endif
constexpr int kGatherDepth = GKR_GATHER_DEPTH;  // iterations in flight per warp

template <int kRecord>
struct Rec {
    static constexpr uint32_t D = kRecord == 528 ? 512u : 576u;    // data row bytes
    static constexpr uint32_t S = kRecord == 528 ? 16u : 8u;       // scale row bytes
    static constexpr int kLane = kRecord == 528 ? 48 : 80;         // staged bytes per lane (+16 pad)
    static constexpr int kScale = 16 * kLane;                      // scale row offset in the item
    static constexpr int kItem = kScale + 16;                      // staged bytes per record
};

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

// Stage this half-warp's record (byte offset `off`, -1 = none) into ring slot
// `it % S`, half `h`; then close one commit group (every lane, every iteration).
template <int kRecord, int S>
__device__ __forceinline__ void stage(const GatherParams& p, uint8_t* ring, int it, int h, int q,
                                      int64_t off, int32_t delta) {
    using R = Rec<kRecord>;
    if (off >= 0) {
        const uint8_t* data = p.cache + off;
        uint8_t* dst = ring + (it & (S - 1)) * (2 * R::kItem) + h * R::kItem + q * R::kLane;
        if (kRecord == 528 || q < 14) {
            cp_async16(dst, data + 32 * q);
            cp_async16(dst + 16, data + 32 * q + 16);
        } else {                                   // V4 bf16 tail: dims 448..511
            const uint8_t* t = data + 448 + 64 * (q - 14);
            cp_async16(dst, t);
            cp_async16(dst + 16, t + 16);
            cp_async16(dst + 32, t + 32);
            cp_async16(dst + 48, t + 48);
        }
        if (q == 0) {
            uint8_t* sdst = ring + (it & (S - 1)) * (2 * R::kItem) + h * R::kItem + R::kScale;
            if (kRecord == 528) cp_async16(sdst, data + delta);
            else cp_async8(sdst, data + delta);
        }
    }
    cp_async_commit();
}

template <int kRecord, int S>
__global__ void __launch_bounds__(kThreads, GKR_MIN_BLOCKS) gather_kernel(const GatherParams p, const WorkMap m) {
    static_assert((S & (S - 1)) == 0 && S >= 2 && S <= 16, "ring depth: power of two <= 16");
    using R = Rec<kRecord>;
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_wait_previous();
    pdl_release_next();
    const int lane = threadIdx.x & 31;
    const int h = lane >> 4, q = lane & 15;
    const int wib = threadIdx.x >> 5;
    const WarpItems w = warp_items(m, static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib);
    if (w.n <= 0) return;  // warp-uniform
    const int n = w.n;
    const int iters = (n + 1) >> 1;
    uint8_t* ring = smem + wib * (S * 2 * R::kItem);

    int64_t cur_off, nxt_off;
    int32_t cur_delta, nxt_delta;
    decode_group<kRecord>(p, w, 0, lane, cur_off, cur_delta);
    decode_group<kRecord>(p, w, 1, lane, nxt_off, nxt_delta);
#pragma unroll
    for (int k = 0; k < S - 1; ++k) {        // prologue: iterations 0 .. S-2 (group 0)
        const int64_t off = __shfl_sync(kFull, cur_off, 2 * k + h);
        const int32_t delta = __shfl_sync(kFull, cur_delta, 2 * k + h);
        stage<kRecord, S>(p, ring, k, h, q, k < iters ? off : -1, delta);
    }
    uint8_t* out = static_cast<uint8_t*>(p.out);
    for (int it = 0; it < iters; ++it) {
        const int k = it + S - 1;
        __syncwarp();                         // every lane is done reading ring slot k % S
        {
            const bool same = (k >> 4) == (it >> 4);
            const int src = (2 * k + h) & 31;
            const int64_t off = __shfl_sync(kFull, same ? cur_off : nxt_off, src);
            const int32_t delta = __shfl_sync(kFull, same ? cur_delta : nxt_delta, src);
            stage<kRecord, S>(p, ring, k, h, q, k < iters ? off : -1, delta);
        }
        cp_async_wait<S - 1>();               // this lane's copies of iteration `it` landed
        __syncwarp();                         // ... and every other lane's

        const int i = 2 * it + h;             // this half's item
        const int64_t off = __shfl_sync(kFull, cur_off, (2 * it + h) & 31);
        const uint8_t* slot = ring + (it & (S - 1)) * (2 * R::kItem) + h * R::kItem;
        uint32_t o[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) o[t] = 0u;
        if (off >= 0) {
            const uint8_t* src = slot + q * R::kLane;
            if (kRecord == 528 || q < 14) {
                const uint4 a = lds16(src), b = lds16(src + 16);
                const uint32_t c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                dequant32(c, slot[R::kScale + (kRecord == 528 ? q : (q >> 1))], o);
            } else {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint4 v = lds16(src + 16 * t);
                    o[4 * t] = v.x; o[4 * t + 1] = v.y; o[4 * t + 2] = v.z; o[4 * t + 3] = v.w;
                }
            }
        }
        if (i < n) {
            uint8_t* orow = out + w.at(i) * 1024 + 64 * q;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                st_stream16(orow + 16 * t, make_uint4(o[4 * t], o[4 * t + 1], o[4 * t + 2], o[4 * t + 3]));
        }
        if ((it & 15) == 15) {
            cur_off = nxt_off;
            cur_delta = nxt_delta;
            decode_group<kRecord>(p, w, (it >> 4) + 2, lane, nxt_off, nxt_delta);
        }
    }
    cp_async_wait<0>();
}

template <int kRecord, int S>
cudaError_t launch(const GatherParams& p, cudaStream_t stream) {
    if (p.num_indices <= 0) return cudaSuccess;
    auto kernel = gather_kernel<kRecord, S>;
    const size_t smem = static_cast<size_t>(kWarpsPerBlock) * S * 2 * Rec<kRecord>::kItem;
    int64_t wave = 0;
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(kernel), kThreads, smem, &wave);
    if (e != cudaSuccess) return e;
    const WorkMap m = make_work_map(p.num_indices, wave, GKR_GATHER_CYCLIC != 0, 2);
    const int64_t blocks = (m.warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_kernel(kernel, blocks, kThreads, smem, stream, p, m);
}

}  // namespace

cudaError_t launch_gather_v41(const GatherParams& p, cudaStream_t stream) {
    return launch<528, kGatherDepth>(p, stream);
}
cudaError_t launch_gather_v4(const GatherParams& p, cudaStream_t stream) {
    return launch<584, kGatherDepth>(p, stream);
}

}  // namespace gkr
