// RoPE + MXFP8 quantise + paged KV insert (V4.1 528 B and legacy V4 584 B records).
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "关键源码片段", the insert kernel of fused_compress_quant_cache.py,
// and section "功能与动机" for the legacy record): per token, skip on slot < 0;
// rotate adjacent pairs of dims 448..511 with the position's cos/sin row; pick one
// UE8M0 scale per block (32 dims for V4.1 after rotation, 64 NoPE dims for V4);
// store e4m3 codes in the page's data region and the scale bytes in its scale region.
//
// Launch shape: one warp per token, U tokens per warp with all their loads issued
// before any is consumed (memory-level parallelism), 8 warps per block.  The grid
// depends only on the token count, so large inserts keep every warp busy (the pages'
// reduced-grid kernel idled 7 of 8 warps above ~16k tokens; PR #56441, review notes).
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

// Per-token validity, identical in every lane (warp-uniform), with error reporting.
__device__ __forceinline__ bool token_ok(const InsertParams& p, int64_t slot, int64_t pos,
                                         int lane) {
    if (slot < 0) return false;
    if (slot >= p.num_slots) {
        if (lane == 0) report(p.err, 1);
        return false;
    }
    if (pos < 0 || pos >= p.max_pos) {
        if (lane == 0) report(p.err, 2);
        return false;
    }
    return true;
}

struct TokenLoads {
    uint4 a, b;       // bf16 chunks A and B
    float4 c, s;      // cos / sin of the 4 pairs in chunk B (lanes 24..31 only)
};

__device__ __forceinline__ void load_token(const InsertParams& p, int64_t t, int64_t pos,
                                           int lane, TokenLoads& L) {
    const uint8_t* row = static_cast<const uint8_t*>(p.kv) + t * 1024;
    L.a = ld_stream16(row + 16 * lane);
    L.b = ld_stream16(row + 512 + 16 * lane);
    if (lane >= 24) {
        const float* cs = p.csc + pos * 64 + 4 * (lane - 24);
        L.c = ld_ro_f4(cs);
        L.s = ld_ro_f4(cs + 32);
    }
}

// V4.1: 16 blocks of 32 dims.  Chunk A of lane L is in block L/4, chunk B in 8 + L/4.
__device__ __forceinline__ void encode_store_v41(const InsertParams& p, const TokenLoads& L,
                                                 int64_t slot, int lane) {
    float a[8], b[8];
    unpack_bf16x8(L.a, a);
    unpack_bf16x8(L.b, b);
    if (lane >= 24) rope4(b, L.c, L.s);  // dims 448..511 = pairs 4(L-24) .. 4(L-24)+3

    uint32_t sc = ue8m0_byte(amax8(a)) | (ue8m0_byte(amax8(b)) << 16);
    sc = __vmaxu2(sc, __shfl_xor_sync(kFull, sc, 1));
    sc = __vmaxu2(sc, __shfl_xor_sync(kFull, sc, 2));
    const uint32_t ba = sc & 0xFFFFu, bb = sc >> 16;

    const uint2 qa = quantise8(a, ba);
    const uint2 qb = quantise8(b, bb);

    const uint32_t s = static_cast<uint32_t>(slot);
    const uint32_t bs = static_cast<uint32_t>(p.block_size);
    const uint32_t page = s / bs, row = s - page * bs;
    uint8_t* base = p.cache + static_cast<int64_t>(page) * p.page_stride;
    uint8_t* data = base + row * 512u;
    st8(data + 8 * lane, qa);
    st8(data + 256 + 8 * lane, qb);
    if ((lane & 3) == 0) {
        uint8_t* srow = base + bs * 512u + row * 16u;
        srow[lane >> 2] = static_cast<uint8_t>(ba);
        srow[8 + (lane >> 2)] = static_cast<uint8_t>(bb);
    }
}

// V4: 7 blocks of 64 NoPE dims (chunk A of lane L in block L/8; chunk B of lanes 0..23
// in block 4 + L/8), rotated dims 448..511 (chunk B of lanes 24..31) stored as bf16.
__device__ __forceinline__ void encode_store_v4(const InsertParams& p, const TokenLoads& L,
                                                int64_t slot, int lane) {
    float a[8], b[8];
    unpack_bf16x8(L.a, a);
    unpack_bf16x8(L.b, b);
    const bool rope_lane = lane >= 24;
    if (rope_lane) rope4(b, L.c, L.s);

    uint32_t sc = ue8m0_byte(amax8(a)) | (rope_lane ? 0u : (ue8m0_byte(amax8(b)) << 16));
    sc = __vmaxu2(sc, __shfl_xor_sync(kFull, sc, 1));
    sc = __vmaxu2(sc, __shfl_xor_sync(kFull, sc, 2));
    sc = __vmaxu2(sc, __shfl_xor_sync(kFull, sc, 4));
    const uint32_t ba = sc & 0xFFFFu, bb = sc >> 16;

    const uint32_t s = static_cast<uint32_t>(slot);
    const uint32_t bs = static_cast<uint32_t>(p.block_size);
    const uint32_t page = s / bs, row = s - page * bs;
    uint8_t* base = p.cache + static_cast<int64_t>(page) * p.page_stride;
    uint8_t* data = base + row * 576u;

    st8(data + 8 * lane, quantise8(a, ba));
    if (!rope_lane) {
        st8(data + 256 + 8 * lane, quantise8(b, bb));
    } else {
        uint4 h;
        h.x = pack_bf16x2_rn(b[0], b[1]);
        h.y = pack_bf16x2_rn(b[2], b[3]);
        h.z = pack_bf16x2_rn(b[4], b[5]);
        h.w = pack_bf16x2_rn(b[6], b[7]);
        st16(data + 448 + 16 * (lane - 24), h);
    }
    if ((lane & 7) == 0) {
        uint8_t* srow = base + bs * 576u + row * 8u;
        srow[lane >> 3] = static_cast<uint8_t>(ba);          // blocks 0..3
        if (!rope_lane) srow[4 + (lane >> 3)] = static_cast<uint8_t>(bb);  // blocks 4..6
        else srow[7] = 0;                                    // pad byte
    }
}

template <int kRecord, int U>
__global__ void __launch_bounds__(kThreads) insert_kernel(const InsertParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t t0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * U;
    if (t0 >= p.num_tokens) return;

    int64_t slot[U], pos[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t t = t0 + u;
        const bool in = t < p.num_tokens;
        slot[u] = in ? __ldg(p.slots + t) : -1;
        pos[u] = in ? __ldg(p.positions + t) : 0;
    }
    bool ok[U];
    TokenLoads L[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        ok[u] = token_ok(p, slot[u], pos[u], lane);
        if (ok[u]) load_token(p, t0 + u, pos[u], lane, L[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!ok[u]) continue;  // warp-uniform
        if (kRecord == 528) encode_store_v41(p, L[u], slot[u], lane);
        else encode_store_v4(p, L[u], slot[u], lane);
    }
}

template <int kRecord, int U>
cudaError_t launch(const InsertParams& p, cudaStream_t stream) {
    if (p.num_tokens <= 0) return cudaSuccess;
    const int64_t per_block = static_cast<int64_t>(kWarpsPerBlock) * U;
    const int64_t blocks = (p.num_tokens + per_block - 1) / per_block;
    insert_kernel<kRecord, U><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

constexpr int kInsertTokensPerWarp = 2;

cudaError_t launch_insert_v41(const InsertParams& p, cudaStream_t stream) {
    return launch<528, kInsertTokensPerWarp>(p, stream);
}
cudaError_t launch_insert_v4(const InsertParams& p, cudaStream_t stream) {
    return launch<584, kInsertTokensPerWarp>(p, stream);
}

}  // namespace gkr
