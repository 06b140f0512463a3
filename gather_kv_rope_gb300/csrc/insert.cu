// RoPE + MXFP8 quantise + paged KV insert (V4.1 528 B and legacy V4 584 B records),
// and the same rotation into the two plain KV-only caches (bf16 rows; fp8 e4m3 rows
// with one fp32 scale: page "PR #56441 [Perf][DSpark] KV-only context insertion
// across V4.1 cache formats", section "实现拆解" item 1).
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "关键源码片段", the insert kernel of fused_compress_quant_cache.py,
// and section "功能与动机" for the legacy record): per token, skip on slot < 0;
// rotate adjacent pairs of dims 448..511 with the position's cos/sin row; pick one
// UE8M0 scale per block (32 dims for V4.1 after rotation, 64 NoPE dims for V4);
// store e4m3 codes in the page's data region and the scale bytes in its scale region.
//
// Launch shape (GB300): at most one wave of warps (sized from the occupancy), each
// walking its own list of tokens (see WorkMap); one warp per token, lane L owning dims
// [8L, 8L+8) and [256+8L, 256+8L+8).  Per group of 32 tokens, lane i decodes token i's
// slot and position once (data-row offset, scale-row distance, checked position), so
// a token costs a few shuffles plus its own work.  A per-warp shared-memory ring filled
// by cp.async keeps S tokens in flight; every copy instruction moves one contiguous
// 512-byte piece of the kv row (or the 128-byte cos/sin halves), and every store one
// contiguous 256-byte piece of the record.  The grid depends only on T and the
// device, so large inserts keep every SM streaming (the pages' reduced-grid kernel
// idled 7 of 8 warps above ~16k tokens; page "PR #56441 [Perf][DSpark] KV-only context
// insertion across V4.1 cache formats", review notes).
#include "device.cuh"
#include "encode.cuh"
#include "launch.h"

namespace gkr {

namespace {

#ifndef GKR_INSERT_DEPTH
#define GKR_INSERT_DEPTH 4
#endif
#ifndef GKR_INSERT_MAX_CHUNK
#define GKR_INSERT_MAX_CHUNK 16  // tokens per streaming warp at most (0 = one wave)
#endif

constexpr int kInsertDepth = GKR_INSERT_DEPTH;  // tokens in flight per warp
constexpr int kSlotBytes = 1024 + 256;          // staged kv row + cos/sin row


// Slot and position of token t.  With early metadata (gkr_set_early_metadata) the kernels
// below read them before waiting for the previous kernel in the stream; all other reads
// and every write come after the wait.
__device__ __forceinline__ void load_slot_position(const InsertParams& p, int64_t t,
                                                   int64_t& slot, int64_t& q) {
    slot = __ldg(p.slots + t);
    q = __ldg(p.positions + t);
}

// Lane-parallel decode of one group of 32 tokens: for this lane's token, the byte
// offsets in the cache of its data row (-1 when the token is skipped or invalid) and
// of its scale row, and its position.  Invalid slots and positions set GKR_ERR_SLOT /
// GKR_ERR_POS (one atomic per group at most).
template <int kRecord>
__device__ __forceinline__ void decode_group(const InsertParams& p, const WarpItems& w, int g,
                                             int lane, int64_t& off, int64_t& soff, int32_t& pos,
                                             const int64_t* pre = nullptr) {
    constexpr uint32_t D = Fmt<kRecord>::D;
    constexpr uint32_t S = Fmt<kRecord>::S;
    const int i = 32 * g + lane;
    off = -1;
    soff = 0;
    pos = 0;
    int32_t err = 0;
    if (i < w.n) {
        const int64_t slot = pre != nullptr ? pre[0] : __ldg(p.slots + w.at(i));
        const int64_t q = pre != nullptr ? pre[1] : __ldg(p.positions + w.at(i));
        if (slot >= p.num_slots) {
            err = 1;
        } else if (slot >= 0) {
            if (q < 0 || q >= p.max_pos) {
                err = 2;
            } else {
                const uint32_t s = static_cast<uint32_t>(slot);
                const uint32_t bs = static_cast<uint32_t>(p.block_size);
                // a plain division here: one decode per 32 tokens is off the streaming
                // kernel's critical path, and page_row's branch measured slower in its
                // fp8 instantiation
                const uint32_t page = s / bs, row = s - page * bs;
                const int64_t base = static_cast<int64_t>(page) * p.page_stride;
                off = base + row * D;
                soff = base + bs * D + row * S;
                pos = static_cast<int32_t>(q);
            }
        }
    }
    err = static_cast<int32_t>(__reduce_or_sync(kFull, static_cast<uint32_t>(err)));
    if (err != 0 && lane == 0) report(p.err, err);
}

// Stage token k (kv row + cos/sin row) into ring slot k % S, then close one group.
// `kv_lane` = this warp's first kv row + 16L, `kv_step` = bytes between its rows,
// `ring_lane` = ring + 16L, `csc_lane` = cos/sin table + 4(L-24) floats.
template <int S>
__device__ __forceinline__ void stage(const uint8_t* kv_lane, int32_t kv_step, uint8_t* ring_lane,
                                      const float* csc_lane, int k, bool valid, int32_t pos,
                                      int lane) {
    if (valid) {
        uint8_t* dst = ring_lane + (k & (S - 1)) * kSlotBytes;
        const uint8_t* row = kv_lane + static_cast<int64_t>(k) * kv_step;
        cp_async16(dst, row);
        cp_async16(dst + 512, row + 512);
        if (lane >= 24) {  // cos / sin of pairs 4(L-24) .. +3 -> ring + 1024 + 16(L-24)
            const float* cs = csc_lane + static_cast<int64_t>(pos) * 64;
            cp_async16(dst + 1024 - 16 * 24, cs);
            cp_async16(dst + 1024 + 128 - 16 * 24, cs + 32);
        }
    }
    cp_async_commit();
}

template <int kRecord, int S>
__global__ void __launch_bounds__(kThreads, GKR_MIN_BLOCKS) insert_kernel(const InsertParams p,
                                                                          const WorkMap m) {
    static_assert((S & (S - 1)) == 0 && S >= 2 && S <= 16, "ring depth: power of two <= 16");
    extern __shared__ __align__(16) uint8_t smem[];
    using Rows = ScaleRows<kRecord>;
    __shared__ __align__(16) uint8_t srows[kWarpsPerBlock][Rows::kBytes];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const WarpItems w = warp_items(m, static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib);
    if (w.n <= 0) return;  // warp-uniform
    int64_t pre[2] = {-1, 0};  // slot and position of this lane's token in the first group
    if (p.early_metadata != 0 && lane < w.n) load_slot_position(p, w.at(lane), pre[0], pre[1]);
    pdl_wait_previous();
    pdl_release_next();
    if (p.early_metadata == 0 && lane < w.n) load_slot_position(p, w.at(lane), pre[0], pre[1]);
    Scale scale;
    if (!load_scale<kRecord>(p, lane, scale)) return;  // warp-uniform
    const int n = w.n;
    uint8_t* const ring_lane = smem + wib * (S * kSlotBytes) + 16 * lane;
    const uint8_t* const kv_lane = static_cast<const uint8_t*>(p.kv) + w.base * 1024 + 16 * lane;
    const int32_t kv_step = static_cast<int32_t>(w.step * 1024);
    const float* const csc_lane = p.csc + 4 * (lane >= 24 ? lane - 24 : 0);
    uint8_t* const cache_a = p.cache + Fmt<kRecord>::kLaneBytes * lane;            // lane's row part
    constexpr int B = Rows::kRows > 0 ? Rows::kRows : 1;   // tokens per scale-row batch

    // lane i of cur describes token 32*g + i of the group being processed; nxt the next
    int64_t cur_off, nxt_off, cur_soff, nxt_soff;
    int32_t cur_pos, nxt_pos;
    decode_group<kRecord>(p, w, 0, lane, cur_off, cur_soff, cur_pos, pre);
    decode_group<kRecord>(p, w, 1, lane, nxt_off, nxt_soff, nxt_pos);

#pragma unroll
    for (int k = 0; k < S - 1; ++k) {          // prologue: tokens 0 .. S-2 (group 0)
        const bool valid = __shfl_sync(kFull, cur_off, k) >= 0;
        const int32_t pos = __shfl_sync(kFull, cur_pos, k);
        stage<S>(kv_lane, kv_step, ring_lane, csc_lane, k, valid && k < n, pos, lane);
    }
    for (int j = 0; j < n; ++j) {
        const int k = j + S - 1;                // token staged this iteration
        {
            const bool same = (k >> 5) == (j >> 5);
            const bool valid = __shfl_sync(kFull, same ? cur_off : nxt_off, k & 31) >= 0;
            const int32_t pos = __shfl_sync(kFull, same ? cur_pos : nxt_pos, k & 31);
            stage<S>(kv_lane, kv_step, ring_lane, csc_lane, k, valid && k < n, pos, lane);
        }
        cp_async_wait<S - 1>();                 // this lane's copies of token j have landed

        const int64_t off = __shfl_sync(kFull, cur_off, j & 31);
        if (off >= 0) {                         // warp-uniform
            const int64_t soff = __shfl_sync(kFull, cur_soff, j & 31);
            const uint8_t* src = ring_lane + (j & (S - 1)) * kSlotBytes;
            TokenLoads L;
            L.a = lds16(src);
            L.b = lds16(src + 512);
            if (lane >= 24) {
                L.c = *reinterpret_cast<const float4*>(src + 1024 - 16 * 24);
                L.s = *reinterpret_cast<const float4*>(src + 1024 + 128 - 16 * 24);
            }
            encode_store<kRecord>(L, cache_a + off, Rows::row(srows[wib], j % B, lane), lane,
                                  scale);
        }
        if constexpr (Rows::kRows > 0) {
            if (j % B == B - 1 || j == n - 1) {  // store the batch's scale rows (B | 32)
                const int src = ((j - j % B) & 31) + lane;
                const int64_t so = __shfl_sync(kFull, cur_soff, src & 31);
                const bool mine = __shfl_sync(kFull, cur_off, src & 31) >= 0;
                Rows::store(srows[wib], p.cache, so, mine, j % B + 1, lane);
            }
        }
        if ((j & 31) == 31) {                   // move to the next group of 32 tokens
            cur_off = nxt_off;
            cur_soff = nxt_soff;
            cur_pos = nxt_pos;
            decode_group<kRecord>(p, w, (j >> 5) + 2, lane, nxt_off, nxt_soff, nxt_pos);
        }
    }
    cp_async_wait<0>();
}

// Short-lived warps for small and medium inserts: one warp per U consecutive tokens,
// lanes 0..U-1 decode them in parallel, all loads (kv rows and cos/sin rows) go
// straight to registers before the first token is encoded.  Below a few hundred
// thousand tokens an insert is latency-bound, and many small resident warps beat a
// deep per-warp pipeline.
#ifndef GKR_SHORT_MIN_BLOCKS
#define GKR_SHORT_MIN_BLOCKS 5   // 48 registers: 5 blocks per SM (6.14 vs 6.32 us at 4, 16k tokens)
#endif
template <int kRecord, int U>
__global__ void __launch_bounds__(kThreads, GKR_SHORT_MIN_BLOCKS)
    insert_short_kernel(const InsertParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t t0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * U;
    if (t0 >= p.num_tokens) return;  // warp-uniform
    const bool mine = lane < U && t0 + lane < p.num_tokens;  // lane u decodes token t0 + u
    int64_t slot = -1, q = 0;
    if (p.early_metadata != 0 && mine) load_slot_position(p, t0 + lane, slot, q);
    pdl_wait_previous();
    pdl_release_next();
    if (p.early_metadata == 0 && mine) load_slot_position(p, t0 + lane, slot, q);
    Scale scale;
    if (!load_scale<kRecord>(p, lane, scale)) return;  // warp-uniform
    constexpr uint32_t D = Fmt<kRecord>::D;
    constexpr uint32_t S = Fmt<kRecord>::S;

    int64_t off = -1, soff = 0;
    int32_t pos = 0;
    uint32_t err = 0;
    if (mine) {
        if (slot >= p.num_slots) {
            err = 1;
        } else if (slot >= 0) {
            if (q < 0 || q >= p.max_pos) {
                err = 2;
            } else {
                const uint32_t s = static_cast<uint32_t>(slot);
                const uint32_t bs = static_cast<uint32_t>(p.block_size);
                uint32_t page, row;
                page_row(s, bs, page, row);
                const int64_t base = static_cast<int64_t>(page) * p.page_stride;
                off = base + row * D;
                soff = base + bs * D + row * S;
                pos = static_cast<int32_t>(q);
            }
        }
    }
    const uint8_t* kv_lane = static_cast<const uint8_t*>(p.kv) + t0 * 1024 + 16 * lane;
    const float* csc_lane = p.csc + 4 * (lane >= 24 ? lane - 24 : 0);
    TokenLoads L[U];
    bool valid[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        valid[u] = __shfl_sync(kFull, off, u) >= 0;
        const int32_t q = __shfl_sync(kFull, pos, u);
        if (valid[u]) {
            L[u].a = ld_stream16(kv_lane + u * 1024);
            L[u].b = ld_stream16(kv_lane + u * 1024 + 512);
            if (lane >= 24) {
                const float* cs = csc_lane + static_cast<int64_t>(q) * 64;
                L[u].c = ld_ro_f4(cs);
                L[u].s = ld_ro_f4(cs + 32);
            }
        }
    }
    // the error bits while the row loads are in flight
    err = __reduce_or_sync(kFull, err);
    if (err != 0u && lane == 0) report(p.err, static_cast<int32_t>(err));
    uint8_t* const cache_a = p.cache + Fmt<kRecord>::kLaneBytes * lane;
    uint8_t* const cache_s = p.cache + ScaleRows<kRecord>::lane_byte(lane);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t o = __shfl_sync(kFull, off, u);
        const int64_t so = __shfl_sync(kFull, soff, u);
        // scalar products: at 48 registers the two-wide form spills here
        if (valid[u]) encode_store<kRecord, false, false>(L[u], cache_a + o, cache_s + so, lane, scale);
    }
}

// ---------------------------------------------------------------- compressed-KV insert
//
// Operation (same page and kernel text as above): a token is written only when
// (position + 1) % R == 0 -- the last token of a group of R positions -- rotated with
// the cos/sin row of the group's first position, position // R * R = position + 1 - R;
// with NaN sanitising every NaN of the rotated row becomes +0.  Checks, in order:
// slot < 0 skips; a slot past the cache sets GKR_ERR_SLOT; a negative position sets
// GKR_ERR_POS; a position that ends no group skips; a group row past the table sets
// GKR_ERR_POS.

// Decode one token from its slot and position: data-row / scale-row offsets (off = -1
// when nothing is written) and the cos/sin row; returns the error bits.
template <int kRecord>
__device__ __forceinline__ uint32_t decode_compressed(const InsertParams& p, int64_t slot,
                                                      int64_t q, int64_t& off, int64_t& soff,
                                                      int32_t& row) {
    static_assert(Fmt<kRecord>::kPacked, "the compressed insert writes the packed records");
    constexpr uint32_t D = Fmt<kRecord>::D;
    constexpr uint32_t S = Fmt<kRecord>::S;
    if (slot < 0) return 0u;
    if (slot >= p.num_slots) return 1u;
    if (q < 0) return 2u;
    const uint64_t q1 = static_cast<uint64_t>(q) + 1u;
    const uint64_t R = static_cast<uint64_t>(p.ratio);
    // a power-of-two ratio (the usual case) takes a mask instead of a division
    const uint64_t rem = (R & (R - 1u)) == 0u ? (q1 & (R - 1u))
                         : (q1 | R) >> 32 == 0u
                             ? static_cast<uint64_t>(static_cast<uint32_t>(q1) %
                                                     static_cast<uint32_t>(R))
                             : q1 % R;
    if (rem != 0u) return 0u;                        // not the last token of its group
    const uint64_t g = q1 - R;                       // group's first position
    if (g >= static_cast<uint64_t>(p.max_pos)) return 2u;
    const uint32_t s = static_cast<uint32_t>(slot);
    const uint32_t bs = static_cast<uint32_t>(p.block_size);
    uint32_t page, r;
    page_row(s, bs, page, r);
    const int64_t base = static_cast<int64_t>(page) * p.page_stride;
    off = base + r * D;
    soff = base + bs * D + r * S;
    row = static_cast<int32_t>(g);
    return 0u;
}


#ifndef GKR_STAGE_MIN_BLOCKS
#define GKR_STAGE_MIN_BLOCKS 6
#endif


// Short-lived warps with shared-memory staging, for medium inserts: one warp per U
// consecutive tokens, lanes 0..U-1 decode them, then every lane copies its own 16-byte
// pieces of the U kv rows (and, on lanes 24..31, of the cos/sin rows) into the warp's
// staging area with cp.async and waits once.  No payload register is live while the
// loads are in flight, so 6 blocks fit on an SM (4 with register loads) and U (1..3,
// chosen per launch) keeps the grid to about one wave per U.  Measured on GB300: ahead
// of both other kernels from ~24k to ~131k tokens, behind the register-load kernel at
// 16k.
template <int kRecord, int U>
__global__ void __launch_bounds__(kThreads, GKR_STAGE_MIN_BLOCKS)
    insert_staged_kernel(const InsertParams p) {
    static_assert(U >= 1 && U <= 3, "one cp.async group per token, at most 3 in flight");
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t t0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib) * U;
    if (t0 >= p.num_tokens) return;  // warp-uniform
    const bool mine = lane < U && t0 + lane < p.num_tokens;  // lane u decodes token t0 + u
    int64_t slot = -1, q = 0;
    if (p.early_metadata != 0 && mine) load_slot_position(p, t0 + lane, slot, q);
    pdl_wait_previous();
    pdl_release_next();
    if (p.early_metadata == 0 && mine) load_slot_position(p, t0 + lane, slot, q);
    Scale scale;
    if (!load_scale<kRecord>(p, lane, scale)) return;  // warp-uniform
    constexpr uint32_t D = Fmt<kRecord>::D;
    constexpr uint32_t S = Fmt<kRecord>::S;
    const uint8_t* const kv_lane = static_cast<const uint8_t*>(p.kv) + t0 * 1024 + 16 * lane;
    uint8_t* const ring_lane = smem + wib * (U * kSlotBytes) + 16 * lane;

    int64_t off = -1, soff = 0;
    int32_t pos = 0;
    uint32_t err = 0;
    if (mine) {
        if (slot >= p.num_slots) {
            err = 1;
        } else if (slot >= 0) {
            if (q < 0 || q >= p.max_pos) {
                err = 2;
            } else {
                const uint32_t s = static_cast<uint32_t>(slot);
                const uint32_t bs = static_cast<uint32_t>(p.block_size);
                uint32_t page, row;
                page_row(s, bs, page, row);
                const int64_t base = static_cast<int64_t>(page) * p.page_stride;
                off = base + row * D;
                soff = base + bs * D + row * S;
                pos = static_cast<int32_t>(q);
            }
        }
    }
    const float* const csc_lane = p.csc + 4 * (lane >= 24 ? lane - 24 : 0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool valid = __shfl_sync(kFull, off, u) >= 0;
        const int32_t q = __shfl_sync(kFull, pos, u);
        if (valid) {
            uint8_t* dst = ring_lane + u * kSlotBytes;
            cp_async16(dst, kv_lane + u * 1024);
            cp_async16(dst + 512, kv_lane + u * 1024 + 512);
            if (lane >= 24) {  // cos / sin of pairs 4(L-24) .. +3 -> slot + 1024 + 16(L-24)
                const float* cs = csc_lane + static_cast<int64_t>(q) * 64;
                cp_async16(dst + 1024 - 16 * 24, cs);
                cp_async16(dst + 1024 + 128 - 16 * 24, cs + 32);
            }
        }
        cp_async_commit();   // one group per token (empty for a skipped one)
    }
    // the error bits while the copies are in flight
    err = __reduce_or_sync(kFull, err);
    if (err != 0u && lane == 0) report(p.err, static_cast<int32_t>(err));

    uint8_t* const cache_a = p.cache + Fmt<kRecord>::kLaneBytes * lane;
    uint8_t* const cache_s = p.cache + ScaleRows<kRecord>::lane_byte(lane);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t o = __shfl_sync(kFull, off, u);
        const int64_t so = __shfl_sync(kFull, soff, u);
        // token u's copies have landed (this lane's; each lane reads only its own), the
        // later tokens' may still be on their way while this one is encoded
        if (U - 1 - u == 0) cp_async_wait<0>();
        else if (U - 1 - u == 1) cp_async_wait<1>();
        else cp_async_wait<2>();
        if (o >= 0) {  // warp-uniform
            const uint8_t* src = ring_lane + u * kSlotBytes;
            TokenLoads L;
            L.a = lds16(src);
            L.b = lds16(src + 512);
            if (lane >= 24) {
                L.c = *reinterpret_cast<const float4*>(src + 1024 - 16 * 24);
                L.s = *reinterpret_cast<const float4*>(src + 1024 + 128 - 16 * 24);
            }
            encode_store<kRecord>(L, cache_a + o, cache_s + so, lane, scale);
        }
    }
}

template <int kRecord, int U>
cudaError_t launch_staged(const InsertParams& p, cudaStream_t stream) {
    const int64_t per_block = static_cast<int64_t>(kWarpsPerBlock) * U;
    const int64_t blocks = (p.num_tokens + per_block - 1) / per_block;
    const size_t smem = static_cast<size_t>(kWarpsPerBlock) * U * kSlotBytes;
    int64_t wave = 0;  // also raises the kernel's dynamic shared-memory limit above 48 KiB
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(insert_staged_kernel<kRecord, U>),
                                   kThreads, smem, &wave);
    if (e != cudaSuccess) return e;
    return launch_kernel(insert_staged_kernel<kRecord, U>, blocks, kThreads, smem, stream, p.pdl, p);
}

template <int kRecord>
cudaError_t launch(const InsertParams& p, cudaStream_t stream) {
    if (p.num_tokens <= 0) return cudaSuccess;
    if (p.num_tokens < p.staged_min && p.num_tokens < p.stream_min) {
        constexpr int U = 2;
        const int64_t per_block = static_cast<int64_t>(kWarpsPerBlock) * U;
        const int64_t blocks = (p.num_tokens + per_block - 1) / per_block;
        return launch_kernel(insert_short_kernel<kRecord, U>, blocks, kThreads, 0, stream, p.pdl, p);
    }
    if (p.num_tokens < p.stream_min) {
        // tokens per warp: the fewest (1..3) that fit the launch in one wave of warps
        int64_t wave = 0;
        cudaError_t e = resident_warps(reinterpret_cast<const void*>(insert_staged_kernel<kRecord, 3>),
                                       kThreads, static_cast<size_t>(kWarpsPerBlock) * 3 * kSlotBytes,
                                       &wave);
        if (e != cudaSuccess) return e;
        if (p.num_tokens <= wave) return launch_staged<kRecord, 1>(p, stream);
        if (p.num_tokens <= 2 * wave) return launch_staged<kRecord, 2>(p, stream);
        return launch_staged<kRecord, 3>(p, stream);
    }
    constexpr int S = kInsertDepth;
    auto kernel = insert_kernel<kRecord, S>;
    const size_t smem = static_cast<size_t>(kWarpsPerBlock) * S * kSlotBytes;
    int64_t wave = 0;
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(kernel), kThreads, smem, &wave);
    if (e != cudaSuccess) return e;
    const WorkMap m = make_work_map(p.num_tokens, wave, false, 1, GKR_INSERT_MAX_CHUNK);
    const int64_t blocks = (m.warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_kernel(kernel, blocks, kThreads, smem, stream, p.pdl, p, m);
}

#ifndef GKR_SPARSE_MIN_BLOCKS
#define GKR_SPARSE_MIN_BLOCKS 4   // up to 64 registers: the 48-register build spills
#endif
#ifndef GKR_SPARSE_BATCH
#define GKR_SPARSE_BATCH 3
#endif
constexpr int kSparseBatch = GKR_SPARSE_BATCH;  // tokens staged at once by the compressed insert
static_assert(kSparseBatch >= 1 && kSparseBatch <= 3,
              "one cp.async group per staged token, at most 3 in flight");

// The compressed insert: the grid is at most one wave, and each warp takes chunks of
// `chunk` (<= 32) consecutive tokens, striding by the grid's token count.  In a chunk,
// lane i decodes token t0 + i and a ballot collects the tokens to write; they are taken
// up to three at a time, their kv and cos/sin rows copied into the warp's shared-memory
// staging area with cp.async (each lane its own 16-byte pieces) and encoded after one
// wait.  The slot and position loads of the warp's next chunk are issued before this
// chunk's copies, so their latency hides behind its writes.  With chunk about 3R a chunk
// is usually one batch, while tokens that end no group cost only their 16 bytes of slot
// and position.  Measured on GB300 at 262144 tokens, ratio 4, against one chunk per
// warp: 21.5 against 23.1 us back to back, 29.4-29.8 against 30.1-30.4 us after an
// L2-flushing kernel, 26.2-26.6 against 26.9 us launched alone; at ratio 128, 4.4 against
// 4.9 us back to back.  48 registers (5 blocks per SM) spill and measured slower, as did
// chunks of 8R.
template <int kRecord, bool kSanitize>
__global__ void __launch_bounds__(kThreads, GKR_SPARSE_MIN_BLOCKS)
    insert_sparse_staged_kernel(const InsertParams p, const int32_t chunk) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock * chunk;
    int64_t t0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + wib) * chunk;
    if (t0 >= p.num_tokens) return;  // warp-uniform
    const bool mine = lane < chunk && t0 + lane < p.num_tokens;  // lane i decodes t0 + i
    int64_t slot = -1, q = 0;
    if (p.early_metadata != 0 && mine) load_slot_position(p, t0 + lane, slot, q);
    pdl_wait_previous();
    pdl_release_next();
    if (p.early_metadata == 0 && mine) load_slot_position(p, t0 + lane, slot, q);

    const float* const csc_lane = p.csc + 4 * (lane >= 24 ? lane - 24 : 0);
    uint8_t* const ring_lane = smem + wib * (kSparseBatch * kSlotBytes) + 16 * lane;
    uint8_t* const cache_a = p.cache + 8 * lane;
    uint8_t* const cache_s = p.cache + ScaleRows<kRecord>::lane_byte(lane);
    while (true) {
        int64_t off = -1, soff = 0;
        int32_t row = 0;
        uint32_t err = decode_compressed<kRecord>(p, slot, q, off, soff, row);
        err = __reduce_or_sync(kFull, err);
        if (err != 0u && lane == 0) report(p.err, static_cast<int32_t>(err));
        uint32_t todo = __ballot_sync(kFull, off >= 0);
        const uint8_t* const kv_lane = static_cast<const uint8_t*>(p.kv) + t0 * 1024 + 16 * lane;
        // the next chunk's slot / position loads fly while this chunk is written
        const int64_t t1 = t0 + stride;
        slot = -1;
        q = 0;
        if (lane < chunk && t1 + lane < p.num_tokens) {
            slot = __ldg(p.slots + t1 + lane);
            q = __ldg(p.positions + t1 + lane);
        }
        while (todo != 0u) {                             // warp-uniform
            int u[kSparseBatch];
#pragma unroll
            for (int v = 0; v < kSparseBatch; ++v) {
                u[v] = todo != 0u ? __ffs(todo) - 1 : -1;
                todo &= todo - 1u;
            }
#pragma unroll
            for (int v = 0; v < kSparseBatch; ++v) {
                if (u[v] >= 0) {                         // warp-uniform
                    const int32_t r = __shfl_sync(kFull, row, u[v]);
                    uint8_t* dst = ring_lane + v * kSlotBytes;
                    cp_async16(dst, kv_lane + u[v] * 1024);
                    cp_async16(dst + 512, kv_lane + u[v] * 1024 + 512);
                    if (lane >= 24) {
                        const float* cs = csc_lane + static_cast<int64_t>(r) * 64;
                        cp_async16(dst + 1024 - 16 * 24, cs);
                        cp_async16(dst + 1024 + 128 - 16 * 24, cs + 32);
                    }
                }
                cp_async_commit();   // one group per batch place (empty when unused)
            }
#pragma unroll
            for (int v = 0; v < kSparseBatch; ++v) {
                // place v's copies have landed (this lane's; each lane reads only its own)
                if (kSparseBatch - 1 - v == 0) cp_async_wait<0>();
                else if (kSparseBatch - 1 - v == 1) cp_async_wait<1>();
                else cp_async_wait<2>();
                if (u[v] >= 0) {                         // warp-uniform
                    const int64_t o = __shfl_sync(kFull, off, u[v]);
                    const int64_t so = __shfl_sync(kFull, soff, u[v]);
                    const uint8_t* src = ring_lane + v * kSlotBytes;
                    TokenLoads L;
                    L.a = lds16(src);
                    L.b = lds16(src + 512);
                    if (lane >= 24) {
                        L.c = *reinterpret_cast<const float4*>(src + 1024 - 16 * 24);
                        L.s = *reinterpret_cast<const float4*>(src + 1024 + 128 - 16 * 24);
                    }
                    encode_store<kRecord, kSanitize>(L, cache_a + o, cache_s + so, lane,
                                                     Scale{1.0f, 1.0f, false});
                }
            }
        }
        if (t1 >= p.num_tokens) break;  // warp-uniform
        __syncwarp();  // reconverge before the next chunk's shuffles
        t0 = t1;
    }
}

template <int kRecord>
cudaError_t launch_compressed(const InsertParams& p, bool sanitize, cudaStream_t stream) {
    if (p.num_tokens <= 0) return cudaSuccess;
    if (p.ratio == 1 && !sanitize) return launch<kRecord>(p, stream);
    const int32_t chunk = static_cast<int32_t>(
        p.ratio * kSparseBatch >= 32 ? 32 : kSparseBatch * p.ratio);
    const int64_t per_block = static_cast<int64_t>(kWarpsPerBlock) * chunk;
    const int64_t blocks = (p.num_tokens + per_block - 1) / per_block;
    const size_t smem = static_cast<size_t>(kWarpsPerBlock) * kSparseBatch * kSlotBytes;
    auto kernel = sanitize ? insert_sparse_staged_kernel<kRecord, true>
                           : insert_sparse_staged_kernel<kRecord, false>;
    int64_t wave = 0;  // also raises the kernel's dynamic shared-memory limit above 48 KiB
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(kernel), kThreads, smem, &wave);
    if (e != cudaSuccess) return e;
    const int64_t resident = wave / kWarpsPerBlock;          // the grid is at most one wave
    return launch_kernel(kernel, blocks < resident ? blocks : resident, kThreads, smem, stream, p.pdl, p,
                         chunk);
}

}  // namespace

cudaError_t launch_insert_v41(const InsertParams& p, cudaStream_t stream) {
    return launch<528>(p, stream);
}
cudaError_t launch_insert_v4(const InsertParams& p, cudaStream_t stream) {
    return launch<584>(p, stream);
}
cudaError_t launch_insert_fp8(const InsertParams& p, cudaStream_t stream) {
    return launch<512>(p, stream);
}
cudaError_t launch_insert_bf16(const InsertParams& p, cudaStream_t stream) {
    return launch<1024>(p, stream);
}
cudaError_t launch_rope_quant_insert_v41(const InsertParams& p, bool sanitize,
                                         cudaStream_t stream) {
    return launch_compressed<528>(p, sanitize, stream);
}
cudaError_t launch_rope_quant_insert_v4(const InsertParams& p, bool sanitize,
                                        cudaStream_t stream) {
    return launch_compressed<584>(p, sanitize, stream);
}

}  // namespace gkr
