// RoPE + MXFP8 quantise + paged KV insert (V4.1 528 B and legacy V4 584 B records).
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "关键源码片段", the insert kernel of fused_compress_quant_cache.py,
// and section "功能与动机" for the legacy record): per token, skip on slot < 0;
// rotate adjacent pairs of dims 448..511 with the position's cos/sin row; pick one
// UE8M0 scale per block (32 dims for V4.1 after rotation, 64 NoPE dims for V4);
// store e4m3 codes in the page's data region and the scale bytes in its scale region.
//
// Launch shape (GB300): at most one wave of warps (sized from the occupancy), each
// walking its own list of tokens (see WorkMap), two tokens per iteration -- one per
// half-warp, lane q of a half owning dims [32q, 32q + 32), i.e. one V4.1 scale block
// (half a V4 block).  Per group of 32 tokens, lane i decodes token i's slot and
// position once.  A per-warp shared-memory ring filled by cp.async keeps S iterations
// in flight; each lane copies the 64 bytes of its block (padded by 16 bytes so the
// 16-byte shared loads of 8 consecutive lanes hit distinct bank groups) and 16 bytes
// of the cos/sin row.  The 32 rotated pairs are computed by all 16 lanes (two pairs
// each) and handed to the two lanes owning dims 448..511 through a small per-warp
// scratch area.  The grid depends only on T and the device, so large inserts keep
// every SM streaming (the pages' reduced-grid kernel idled 7 of 8 warps above ~16k
// tokens; page "PR #56441 [Perf][DSpark] KV-only context insertion across V4.1 cache
// formats", review notes).
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

#ifndef GKR_INSERT_DEPTH
#define GKR_INSERT_DEPTH 2
#endif
#ifndef GKR_INSERT_CYCLIC
#define GKR_INSERT_CYCLIC 0
#endif
constexpr int kInsertDepth = GKR_INSERT_DEPTH;  // iterations (token pairs) in flight per warp

constexpr int kKvLane = 80;                     // a lane's 64-byte block of the kv row + 16 pad
constexpr int kCscOff = 16 * kKvLane;           // cos/sin row offset in a staged token
constexpr int kTokBytes = kCscOff + 256;        // staged bytes per token
constexpr int kRotSeg = 144;                    // 32 rotated fp32 (128 B) + 16 pad
constexpr int kRotBytes = 4 * kRotSeg;          // per warp: 2 tokens x 2 rope lanes

// Lane-parallel decode of one group of 32 tokens: for this lane's token, the byte
// offset of its data row in the cache (-1 when the token is skipped or invalid), the
// distance from the data row to the scale row, and its position.  Invalid slots and
// positions set GKR_ERR_SLOT / GKR_ERR_POS (one atomic per group at most).
template <int kRecord>
__device__ __forceinline__ void decode_group(const InsertParams& p, const WarpItems& w, int g,
                                             int lane, int64_t& off, int32_t& delta, int32_t& pos) {
    constexpr uint32_t D = kRecord == 528 ? 512u : 576u;
    constexpr uint32_t S = kRecord == 528 ? 16u : 8u;
    const int i = 32 * g + lane;
    off = -1;
    delta = 0;
    pos = 0;
    int32_t err = 0;
    if (i < w.n) {
        const int64_t slot = __ldg(p.slots + w.at(i));
        const int64_t q = __ldg(p.positions + w.at(i));
        if (slot >= p.num_slots) {
            err = 1;
        } else if (slot >= 0) {
            if (q < 0 || q >= p.max_pos) {
                err = 2;
            } else {
                const uint32_t s = static_cast<uint32_t>(slot);
                const uint32_t bs = static_cast<uint32_t>(p.block_size);
                const uint32_t page = s / bs, row = s - page * bs;
                off = static_cast<int64_t>(page) * p.page_stride + row * D;
                delta = static_cast<int32_t>(bs * D + row * S - row * D);
                pos = static_cast<int32_t>(q);
            }
        }
    }
    err = static_cast<int32_t>(__reduce_or_sync(kFull, static_cast<uint32_t>(err)));
    if (err != 0 && lane == 0) report(p.err, err);
}

// Stage this half-warp's token (item i, valid when off >= 0) into ring slot it % S:
// lane q copies dims [32q, 32q + 32) of the kv row and bytes [16q, 16q + 16) of the
// cos/sin row.  Then close one commit group (every lane, every iteration).
template <int S>
__device__ __forceinline__ void stage(const InsertParams& p, uint8_t* ring, const WarpItems& w,
                                      int it, int h, int q, bool valid, int32_t pos) {
    if (valid) {
        uint8_t* dst = ring + (it & (S - 1)) * (2 * kTokBytes) + h * kTokBytes;
        const uint8_t* row = static_cast<const uint8_t*>(p.kv) + w.at(2 * it + h) * 1024 + 64 * q;
        uint8_t* d = dst + q * kKvLane;
        cp_async16(d, row);
        cp_async16(d + 16, row + 16);
        cp_async16(d + 32, row + 32);
        cp_async16(d + 48, row + 48);
        cp_async16(dst + kCscOff + 16 * q,
                   reinterpret_cast<const uint8_t*>(p.csc) + static_cast<int64_t>(pos) * 256 + 16 * q);
    }
    cp_async_commit();
}

template <int kRecord, int S>
__global__ void __launch_bounds__(kThreads, GKR_MIN_BLOCKS) insert_kernel(const InsertParams p, const WorkMap m) {
    static_assert((S & (S - 1)) == 0 && S >= 2 && S <= 16, "ring depth: power of two <= 16");
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_wait_previous();
    pdl_release_next();
    const int lane = threadIdx.x & 31;
    const int h = lane >> 4, q = lane & 15;
    const int wib = threadIdx.x >> 5;
    const WarpItems w = warp_items(m, static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib);
    if (w.n <= 0) return;  // warp-uniform
    const int iters = (w.n + 1) >> 1;
    uint8_t* ring = smem + wib * (S * 2 * kTokBytes + kRotBytes);
    uint8_t* rot = ring + S * 2 * kTokBytes;
    const bool rope_lane = q >= 14;             // owns dims 448..479 (q = 14) or 480..511

    // lane i of cur describes token 32*g + i of the group being processed; nxt the next
    int64_t cur_off, nxt_off;
    int32_t cur_delta, nxt_delta, cur_pos, nxt_pos;
    decode_group<kRecord>(p, w, 0, lane, cur_off, cur_delta, cur_pos);
    decode_group<kRecord>(p, w, 1, lane, nxt_off, nxt_delta, nxt_pos);

#pragma unroll
    for (int k = 0; k < S - 1; ++k) {           // prologue: iterations 0 .. S-2 (group 0)
        const bool valid = __shfl_sync(kFull, cur_off, 2 * k + h) >= 0 && k < iters;
        const int32_t pos = __shfl_sync(kFull, cur_pos, 2 * k + h);
        stage<S>(p, ring, w, k, h, q, valid, pos);
    }
    for (int it = 0; it < iters; ++it) {
        const int k = it + S - 1;
        __syncwarp();                            // every lane is done reading ring slot k % S
        {
            const bool same = (k >> 4) == (it >> 4);
            const int src = (2 * k + h) & 31;
            const bool valid = __shfl_sync(kFull, same ? cur_off : nxt_off, src) >= 0 && k < iters;
            const int32_t pos = __shfl_sync(kFull, same ? cur_pos : nxt_pos, src);
            stage<S>(p, ring, w, k, h, q, valid, pos);
        }
        cp_async_wait<S - 1>();                  // this lane's copies of iteration `it` landed
        __syncwarp();                            // ... and every other lane's

        const int src = (2 * it + h) & 31;
        const int64_t off = __shfl_sync(kFull, cur_off, src);
        const int32_t delta = __shfl_sync(kFull, cur_delta, src);
        const bool valid = off >= 0;             // uniform per half-warp
        const uint8_t* tok = ring + (it & (S - 1)) * (2 * kTokBytes) + h * kTokBytes;

        // RoPE, two pairs per lane: pairs 2q, 2q+1 = dims 448 + 4q .. 448 + 4q + 3, which
        // sit in the staged block of lane 14 + q/8 at byte 8 * (q % 8).
        if (valid) {
            const uint2 e = lds8(tok + (14 + (q >> 3)) * kKvLane + 8 * (q & 7));
            const uint2 cb = lds8(tok + kCscOff + 8 * q);
            const uint2 sb = lds8(tok + kCscOff + 128 + 8 * q);
            float f[4] = {__uint_as_float(e.x << 16), __uint_as_float(e.x & 0xFFFF0000u),
                          __uint_as_float(e.y << 16), __uint_as_float(e.y & 0xFFFF0000u)};
            rope2(f, make_float2(__uint_as_float(cb.x), __uint_as_float(cb.y)),
                  make_float2(__uint_as_float(sb.x), __uint_as_float(sb.y)));
            *reinterpret_cast<float4*>(rot + (2 * h + (q >> 3)) * kRotSeg + 16 * (q & 7)) =
                make_float4(f[0], f[1], f[2], f[3]);
        }
        __syncwarp();

        float v[32];
        if (valid) {
            if (!rope_lane) {
                const uint8_t* b = tok + q * kKvLane;
#pragma unroll
                for (int t = 0; t < 4; ++t) unpack_bf16x8(lds16(b + 16 * t), v + 8 * t);
            } else {
                const uint8_t* r = rot + (2 * h + (q - 14)) * kRotSeg;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const float4 x = *reinterpret_cast<const float4*>(r + 16 * t);
                    v[4 * t] = x.x; v[4 * t + 1] = x.y; v[4 * t + 2] = x.z; v[4 * t + 3] = x.w;
                }
            }
        } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = 0.0f;
        }
        float amax = amax32(v);
        if (kRecord == 584) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));  // 64-dim blocks
        const uint32_t byte = ue8m0_byte(amax);

        if (valid) {
            uint8_t* data = p.cache + off;
            uint8_t* srow = data + delta;
            if (kRecord == 528 || !rope_lane) {
                uint4 lo, hi;
                quantise32(v, byte, lo, hi);
                st16(data + 32 * q, lo);
                st16(data + 32 * q + 16, hi);
            } else {                             // V4: rotated dims stored as bf16
                uint8_t* t = data + 448 + 64 * (q - 14);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st16(t + 16 * c, make_uint4(pack_bf16x2_rn(v[8 * c], v[8 * c + 1]),
                                                pack_bf16x2_rn(v[8 * c + 2], v[8 * c + 3]),
                                                pack_bf16x2_rn(v[8 * c + 4], v[8 * c + 5]),
                                                pack_bf16x2_rn(v[8 * c + 6], v[8 * c + 7])));
            }
            if (kRecord == 528) {
                srow[q] = static_cast<uint8_t>(byte);
            } else if (q < 14) {
                if ((q & 1) == 0) srow[q >> 1] = static_cast<uint8_t>(byte);   // blocks 0..6
            } else if (q == 14) {
                srow[7] = 0;                                                  // pad byte
            }
        }
        if ((it & 15) == 15) {                   // move to the next group of 32 tokens
            cur_off = nxt_off;
            cur_delta = nxt_delta;
            cur_pos = nxt_pos;
            decode_group<kRecord>(p, w, (it >> 4) + 2, lane, nxt_off, nxt_delta, nxt_pos);
        }
    }
    cp_async_wait<0>();
}

template <int kRecord, int S>
cudaError_t launch(const InsertParams& p, cudaStream_t stream) {
    if (p.num_tokens <= 0) return cudaSuccess;
    auto kernel = insert_kernel<kRecord, S>;
    const size_t smem = static_cast<size_t>(kWarpsPerBlock) * (S * 2 * kTokBytes + kRotBytes);
    int64_t wave = 0;
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(kernel), kThreads, smem, &wave);
    if (e != cudaSuccess) return e;
    const WorkMap m = make_work_map(p.num_tokens, wave, GKR_INSERT_CYCLIC != 0, 2);
    const int64_t blocks = (m.warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_kernel(kernel, blocks, kThreads, smem, stream, p, m);
}

}  // namespace

cudaError_t launch_insert_v41(const InsertParams& p, cudaStream_t stream) {
    return launch<528, kInsertDepth>(p, stream);
}
cudaError_t launch_insert_v4(const InsertParams& p, cudaStream_t stream) {
    return launch<584, kInsertDepth>(p, stream);
}

}  // namespace gkr
