// RoPE + MXFP8 quantise + paged KV insert (V4.1 528 B and legacy V4 584 B records).
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "关键源码片段", the insert kernel of fused_compress_quant_cache.py,
// and section "功能与动机" for the legacy record): per token, skip on slot < 0;
// rotate adjacent pairs of dims 448..511 with the position's cos/sin row; pick one
// UE8M0 scale per block (32 dims for V4.1 after rotation, 64 NoPE dims for V4);
// store e4m3 codes in the page's data region and the scale bytes in its scale region.
//
// Launch shape (GB300): one warp per token row at a time, and exactly one wave of
// warps -- the grid is sized from the occupancy so every warp is resident, and each
// warp walks a contiguous chunk of ceil(T / resident warps) tokens.  A warp loads the
// slots and positions of 32 tokens with one coalesced load, then keeps S tokens in
// flight through a per-warp shared-memory ring filled by cp.async (each lane copies
// exactly the 16-byte pieces of the kv row and cos/sin row it later consumes).  The
// grid depends only on T and the device, so large inserts keep every SM streaming
// (the pages' reduced-grid kernel idled 7 of 8 warps above ~16k tokens; page
// "PR #56441 [Perf][DSpark] KV-only context insertion across V4.1 cache formats",
// review notes).
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

constexpr int kInsertSlotBytes = 1024 + 256;  // one kv row + one cos/sin row
constexpr int kInsertDepth = 4;               // tokens in flight per warp

// Slot/position checks, identical in every lane (warp-uniform).
__device__ __forceinline__ bool token_in_range(const InsertParams& p, int64_t slot, int64_t pos) {
    return slot >= 0 && slot < p.num_slots && pos >= 0 && pos < p.max_pos;
}
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
        srow[lane >> 3] = static_cast<uint8_t>(ba);                        // blocks 0..3
        if (!rope_lane) srow[4 + (lane >> 3)] = static_cast<uint8_t>(bb);  // blocks 4..6
        else srow[7] = 0;                                                  // pad byte
    }
}

// Slots and positions of tokens 32g .. 32g+31 of this warp's chunk, one per lane.
__device__ __forceinline__ void load_group(const InsertParams& p, int64_t t_begin, int n, int g,
                                           int lane, int64_t& slot, int64_t& pos) {
    const int i = 32 * g + lane;
    slot = -1;
    pos = 0;
    if (i < n) {
        slot = __ldg(p.slots + t_begin + i);
        pos = __ldg(p.positions + t_begin + i);
    }
}

// Stage token k of the chunk into ring slot k % S (nothing for skipped or invalid
// tokens), then close one commit group.
template <int S>
__device__ __forceinline__ void stage(const InsertParams& p, uint8_t* ring, int64_t t_begin,
                                      int k, int64_t slot, int64_t pos, int lane,
                                      uint64_t policy) {
    if (token_in_range(p, slot, pos)) {
        uint8_t* dst = ring + (k % S) * kInsertSlotBytes;
        const uint8_t* row = static_cast<const uint8_t*>(p.kv) + (t_begin + k) * 1024;
        cp_async16_stream(dst + 16 * lane, row + 16 * lane, policy);
        cp_async16_stream(dst + 512 + 16 * lane, row + 512 + 16 * lane, policy);
        if (lane >= 24) {
            const float* cs = p.csc + pos * 64 + 4 * (lane - 24);
            cp_async16(dst + 1024 + 16 * (lane - 24), cs);
            cp_async16(dst + 1024 + 128 + 16 * (lane - 24), cs + 32);
        }
    }
    cp_async_commit();
}

template <int kRecord, int S>
__global__ void __launch_bounds__(kThreads) insert_kernel(const InsertParams p, int64_t chunk) {
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_wait_previous();
    pdl_release_next();
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t t_begin = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib) * chunk;
    if (t_begin >= p.num_tokens) return;  // warp-uniform
    const int n = static_cast<int>(chunk < p.num_tokens - t_begin ? chunk : p.num_tokens - t_begin);
    uint8_t* ring = smem + wib * (S * kInsertSlotBytes);
    const uint64_t policy = l2_evict_first_policy();

    // lane i of cur holds token 32*g + i of the group being processed; nxt the next group
    int64_t cur_s, cur_p, nxt_s, nxt_p;
    load_group(p, t_begin, n, 0, lane, cur_s, cur_p);
    load_group(p, t_begin, n, 1, lane, nxt_s, nxt_p);

#pragma unroll
    for (int k = 0; k < S - 1; ++k) {  // prologue: tokens 0 .. S-2 (all in group 0)
        const int64_t s = __shfl_sync(kFull, cur_s, k);
        const int64_t q = __shfl_sync(kFull, cur_p, k);
        if (k < n) stage<S>(p, ring, t_begin, k, s, q, lane, policy);
        else cp_async_commit();
    }
    for (int j = 0; j < n; ++j) {
        const int k = j + S - 1;             // token staged this iteration
        if (k < n) {
            const bool same = (k >> 5) == (j >> 5);
            const int64_t s = __shfl_sync(kFull, same ? cur_s : nxt_s, k & 31);
            const int64_t q = __shfl_sync(kFull, same ? cur_p : nxt_p, k & 31);
            stage<S>(p, ring, t_begin, k, s, q, lane, policy);
        } else {
            cp_async_commit();
        }
        cp_async_wait<S - 1>();              // this lane's copies of token j have landed

        const int64_t slot = __shfl_sync(kFull, cur_s, j & 31);
        const int64_t pos = __shfl_sync(kFull, cur_p, j & 31);
        if (token_ok(p, slot, pos, lane)) {
            const uint8_t* src = ring + (j % S) * kInsertSlotBytes;
            TokenLoads L;
            L.a = lds16(src + 16 * lane);
            L.b = lds16(src + 512 + 16 * lane);
            if (lane >= 24) {
                const uint4 c = lds16(src + 1024 + 16 * (lane - 24));
                const uint4 s = lds16(src + 1024 + 128 + 16 * (lane - 24));
                L.c = make_float4(__uint_as_float(c.x), __uint_as_float(c.y),
                                  __uint_as_float(c.z), __uint_as_float(c.w));
                L.s = make_float4(__uint_as_float(s.x), __uint_as_float(s.y),
                                  __uint_as_float(s.z), __uint_as_float(s.w));
            }
            if (kRecord == 528) encode_store_v41(p, L, slot, lane);
            else encode_store_v4(p, L, slot, lane);
        }
        if ((j & 31) == 31) {                // move to the next group of 32 tokens
            cur_s = nxt_s;
            cur_p = nxt_p;
            load_group(p, t_begin, n, (j >> 5) + 2, lane, nxt_s, nxt_p);
        }
    }
    cp_async_wait<0>();
}

template <int kRecord, int S>
cudaError_t launch(const InsertParams& p, cudaStream_t stream) {
    if (p.num_tokens <= 0) return cudaSuccess;
    auto kernel = insert_kernel<kRecord, S>;
    const size_t smem = static_cast<size_t>(kWarpsPerBlock) * S * kInsertSlotBytes;
    int64_t wave = 0;
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(kernel), kThreads, smem, &wave);
    if (e != cudaSuccess) return e;
    int64_t chunk = 0, blocks = 0;
    one_wave_split(p.num_tokens, wave, kWarpsPerBlock, &chunk, &blocks);
    return launch_kernel(kernel, blocks, kThreads, smem, stream, p, chunk);
}

}  // namespace

cudaError_t launch_insert_v41(const InsertParams& p, cudaStream_t stream) {
    return launch<528, kInsertDepth>(p, stream);
}
cudaError_t launch_insert_v4(const InsertParams& p, cudaStream_t stream) {
    return launch<584, kInsertDepth>(p, stream);
}

}  // namespace gkr
