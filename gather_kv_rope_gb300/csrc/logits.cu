// The dequant-gather fused into its consumer: sparse decode logits.
//
// Operation (FlashMLA overview page, DSA section: each decode query attends to the top-k
// cache entries listed by its index row, -1 marking an invalid entry, and FP8 entries
// are dequantised to bf16 before the matrix product; page "PR #56893 [DSv4.1] Store the
// whole KV in MXFP8 (FlashMLA V4.1 record)", section "实现拆解" item 4, for the dequant):
//   out[q, h, k] = sm_scale * sum_d Q[q, h, d] * K[q, k, d]
// where K[q, k, :] is exactly the bf16 row kv_gather returns for index indices[q, k];
// an invalid index (-1) gives -inf, and so does an index outside the cache (which also
// sets GKR_ERR_INDEX).  The gathered rows never leave the SM: the bf16 intermediate that
// kv_gather writes (1 KB per index) and a separate product kernel reads back is gone.
//
// Launch shape (sm_103a, 5th-generation tensor cores): a persistent kernel, one CTA of 21
// warps per SM, each CTA taking a contiguous run of work items (query, chunk of 128 keys)
// in query-major order.
//   * A, the query's heads (up to 128, zero-padded; M = 128 x K = 512, bf16), lives in
//     tensor memory next to the two accumulators, so shared memory is left to the records.
//     The 4 epilogue warps write it (tcgen05.st) at launch and when the run reaches a new
//     query, once the products that read the old one are done, and signal each half of K
//     as soon as it is written, so that the new query's first low-half products start
//     while the high half is loaded; one thread prefetches the run's query tiles into L2
//     at launch.
//   * 16 producer warps, 4 keys of each 64-key group each: a ring of raw records per warp
//     in shared memory, filled with cp.async two groups ahead (the loads in flight cost no
//     registers); each group is dequantised twice, its low 256 dims and then its high 256,
//     into B stages of 64 keys x 256 dims (K-major, 128-byte swizzle, a ring of 3).
//   * one warp, once all producers have filled a stage, issues its 16 tcgen05.mma
//     (kind::f16, N = 64, K = 16 each, A from tensor memory) into the group's 64 columns of
//     one of two 128-column accumulators and commits them to the stage's mbarrier (the
//     stage may then be refilled); after an item's last stage it commits the accumulator.
//   * the 4 epilogue warps, one per quarter of the tensor-memory lanes (heads), drain
//     each item's accumulator while the next item is multiplied into the other one, 32
//     columns (entries) at a time: each lane writes its head's 32 logits (entries that are
//     not records: -inf) into the warp's swizzled tile and one lane hands the tile to a
//     TMA tensor store.
// Every wait on an mbarrier sleeps in try_wait (a suspend hint, so waiting warps take no
// issue slots) and is bounded (20 ms of %globaltimer): past it the CTA sets
// GKR_ERR_TIMEOUT, stops waiting, still frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

constexpr int kM = 128;                  // heads per tile (MMA rows)
constexpr int kN = 64;                   // keys per group (MMA columns)
constexpr int kHalfK = 256;              // dims per B stage: a group's keys, half of K
constexpr int kStages = 3;               // B ring depth (half-groups)
constexpr int kChunk = 128;              // keys per work item
constexpr int kGroups = kChunk / kN;     // groups per item
constexpr int kTiles = 2 * kGroups;      // B stages per item (low, high half per group)
constexpr int kProducerWarps = 16;       // warps 0..15: gather + dequantise
constexpr int kEpilogueWarps = 4;        // warps 16..19: A in, accumulators out (warp w
                                         // owns tensor-memory lanes 32 (w % 4) .. +31)
constexpr int kFirstEpilogue = kProducerWarps;
constexpr int kMmaWarp = kProducerWarps + kEpilogueWarps;   // warp 20: tcgen05.mma issue;
                                                            // allocates and frees TMEM too
constexpr int kKeysPerWarp = kN / kProducerWarps;           // keys of a group per producer
constexpr int kLogitThreads = (kMmaWarp + 1) * 32;          // 21 warps: up to 80 registers
constexpr int kRowBytes = 128;           // one swizzle row: 64 bf16 of K
constexpr int kBBytes = kN * kHalfK * 2; // 32 KB per stage
constexpr uint32_t kTmemCols = 512;      // accumulators at columns 0 and 128, A at 256
constexpr uint32_t kACol = 2 * kChunk;   // A: 512 bf16 a row, two to a column
constexpr int kTileCols = 32;            // entries per drain step
constexpr int kTileWarpBytes = 32 * kTileCols * 4;   // an epilogue warp's 32 x 32 fp32 tile
constexpr int kTileBytes = kEpilogueWarps * kTileWarpBytes;
constexpr int kWindow = 32 / kKeysPerWarp;  // groups whose indices one register holds
constexpr int kSmemLimit = 227 * 1024;   // shared memory a CTA may use
constexpr int32_t kErrIndex = 4;
constexpr int32_t kErrTimeout = 16;
constexpr uint64_t kWaitNs = 20000000;    // a wait gives up after 20 ms (a normal one takes us)

// A producer warp's ring of raw records: kSlots groups of kKeysPerWarp records, each as
// the cache holds it (data row, then scale row) at a 16-byte aligned stride; as many
// groups as the shared memory left by the B stages and the drain tiles holds.
template <int kRecord>
struct Raw {
    static constexpr int stride = kRecord == 584 ? 592 : kRecord;   // 576 data + 8 scale
    static constexpr int fixed = 1024 + kStages * kBBytes + 1024 + kTileBytes + 256;
    static constexpr int slots =
        (kSmemLimit - fixed) / (kProducerWarps * kKeysPerWarp * stride);
    static constexpr int bytes = kProducerWarps * slots * kKeysPerWarp * stride;
    // the drain tiles follow the rings, 1024-byte aligned (the TMA's 128-byte swizzle)
    static constexpr int tile_off = (kStages * kBBytes + bytes + 1023) / 1024 * 1024;
    static constexpr int smem = 1024 + tile_off + kTileBytes;   // + the barriers
};

static_assert(kN % kProducerWarps == 0 && kN % 16 == 0 && kN <= 256 && kEpilogueWarps == 4 &&
                  kFirstEpilogue % 4 == 0,
              "whole keys per producer; N of an M = 128 product is a multiple of 16; one "
              "epilogue warp per quarter of the tensor-memory lanes, in order");
static_assert(kChunk % kN == 0 && kChunk % kTileCols == 0 && 2 * kChunk + 256 <= kTmemCols,
              "whole groups and drain steps per item; two accumulators and A fit");
static_assert(Raw<528>::slots >= 3 && Raw<584>::slots >= 3 && Raw<512>::slots >= 3 &&
                  Raw<1024>::slots >= 1 && Raw<528>::slots * kKeysPerWarp <= 32 &&
                  Raw<512>::slots * kKeysPerWarp <= 32 && kKeysPerWarp * kWindow == 32,
              "a ring of at least one group; one validity bit per ring record; whole "
              "groups per index window");

// ------------------------------------------------------------- tcgen05 / mbarrier PTX

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// True once the phase with the given parity has completed.  A thread whose phase is not
// complete is suspended until it completes or kSuspendNs have passed: a waiting warp then
// takes no issue slots from the warps that work (spinning without the hint cost ~2 % of
// the sparse logits).
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0u;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase with the given parity to complete; false once kWaitNs have passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's shared-memory stores visible to the tensor cores (async proxy).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulator; one thread.  A sits in
// tensor memory with row i in lane i and its K values two to a 32-bit column (the lower
// half holds the even k), so the K = 16 of one instruction span 8 columns.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the mbarrier once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}
// 16 consecutive fp32 accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's lane (tcgen05.wait::st before handing
// them to the tensor cores).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint4 (&v)[4]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y),
        "r"(v[1].z), "r"(v[1].w), "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w),
        "r"(v[3].x), "r"(v[3].y), "r"(v[3].z), "r"(v[3].w)
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A and B
// (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (static_cast<uint32_t>(kN >> 3) << 17) |
                            (static_cast<uint32_t>(kM >> 4) << 24);

// Shared-memory matrix descriptor of the K-major B operand with the 128-byte swizzle: start
// address >> 4 (bits 0-13), leading offset (unused by this layout; 1) at bits 16-29,
// stride between 8-row groups (1024 bytes) >> 4 at bits 32-45, descriptor version 1 at
// bits 46-47, swizzle mode 128B (2) at bits 61-63.  The operand's rows are 128 bytes (64
// bf16 of K); row r of an 8-row group sits at r * 128 in its 1024-byte group, and its
// 16-byte piece c at position c ^ r.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Byte offset of the 16-byte piece holding dims [8c, 8c+8) of K block kb (dims 64kb..) of
// row r in an operand of `rows` rows: K blocks of rows x 128 bytes, 8-row swizzle groups.
__device__ __forceinline__ uint32_t sw128_offset(int rows, int r, int kb, int c) {
    return static_cast<uint32_t>(kb * rows * kRowBytes + (r >> 3) * 1024 + (r & 7) * kRowBytes +
                                 ((c ^ (r & 7)) << 4));
}

// Lane L's piece of half h of a 512-dim row (dims [256h + 8L, 256h + 8L + 8)) into row r of
// a swizzled half-K operand of kN rows: K block L / 8 (of 64 dims), 16-byte piece L % 8.
__device__ __forceinline__ void store_piece(uint8_t* op, int r, int lane, uint4 v) {
    *reinterpret_cast<uint4*>(op + sw128_offset(kN, r, lane >> 3, lane & 7)) = v;
}

// A CTA (one per SM) takes a contiguous run of work items (query, chunk of kChunk keys)
// in query-major order, so A changes only when its run moves to the next query.
struct alignas(8) Barriers {
    uint64_t full[kStages];      // producers -> MMA: B stage holds its half-group
    uint64_t empty[kStages];     // MMA -> producers: the stage's products are done
    uint64_t acc_full[2];        // MMA -> epilogue: an item's accumulator is complete
    uint64_t acc_empty[2];       // epilogue -> MMA: the accumulator has been read
    uint64_t a_ready[2];         // epilogue -> MMA: A's low / high half of K holds the
                                 // next query
    uint32_t tmem_base;
    int32_t timed_out;
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{\n .reg .b64 state;\n mbarrier.arrive.shared::cta.b64 state, [%0];\n}\n" ::"r"(bar)
        : "memory");
}

// A wait that records a timeout instead of hanging: after the first failure the thread
// stops waiting (its results are discarded, see GKR_ERR_TIMEOUT).
__device__ __forceinline__ void wait_or_flag(uint32_t bar, uint32_t parity, bool& ok) {
    if (ok) ok = mbar_wait(bar, parity);
}

// The same for a whole warp: lane 0 waits, the warp follows it (__syncwarp orders the
// lanes' later accesses after lane 0's acquire); every lane gets the outcome.
__device__ __forceinline__ void warp_wait_or_flag(uint32_t bar, uint32_t parity, bool& ok,
                                                  int lane) {
    if (lane == 0) wait_or_flag(bar, parity, ok);
    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
    __syncwarp();
}

// One arrival for a whole warp: every lane's earlier shared-memory writes (each lane has
// fenced them for the async proxy) are ordered before lane 0's arrive by __syncwarp.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Prefetch `bytes` (a multiple of 16) from a 16-byte aligned address into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// TMA store (async proxy) of a 32 x 32 fp32 box from shared memory to the logits at
// (entry x, head y, query z), in this thread's bulk group; entries past topk and heads past
// num_heads are not written.  The tile holds row r (head y + r) at r * 128 bytes, its
// 16-byte piece c at position c ^ (r % 8) (the map's 128-byte swizzle).
__device__ __forceinline__ void tma_store_tile(const CUtensorMap* map, const void* tile, int32_t x,
                                               int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_addr(tile))
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until none of this thread's bulk groups still reads its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st_shared16(void* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
}
// Four logits: sm_scale * accumulator for a record (bit i of recs), -inf otherwise.
__device__ __forceinline__ float4 logit4(const float* v, uint32_t recs, float sm_scale) {
    return make_float4(recs & 1u ? __fmul_rn(v[0], sm_scale) : -INFINITY,
                       recs & 2u ? __fmul_rn(v[1], sm_scale) : -INFINITY,
                       recs & 4u ? __fmul_rn(v[2], sm_scale) : -INFINITY,
                       recs & 8u ? __fmul_rn(v[3], sm_scale) : -INFINITY);
}

// Decode index idx into the record's byte offsets (off = -1: not a record -- index -1,
// out of range (bad = 1), or a bad fp8 scale).
template <int kRecord>
__device__ __forceinline__ void key_offsets(const LogitsParams& p, int32_t idx, bool scale_bad,
                                            int64_t& off, int64_t& soff, uint32_t& bad) {
    using R = Fmt<kRecord>;
    off = -1;
    soff = 0;
    if (scale_bad) return;
    if (idx >= 0 && idx < p.num_slots) {
        const uint32_t s = static_cast<uint32_t>(idx);
        const uint32_t bs = static_cast<uint32_t>(p.block_size);
        uint32_t page, row;
        page_row(s, bs, page, row);
        const int64_t pbase = static_cast<int64_t>(page) * p.page_stride;
        off = pbase + row * R::D;
        soff = pbase + bs * R::D + row * R::S;
    } else if (idx != -1) {
        bad = 1u;
    }
}

// One record's cp.async copies into its ring place, spread over the warp (data rows and
// V4.1 scale rows are 16-byte aligned in every valid cache, V4 scale rows 8-byte).
template <int kRecord>
__device__ __forceinline__ void copy_record(uint8_t* dst, const uint8_t* cache, int64_t off,
                                            int64_t soff, int lane) {
    cp_async16(dst + 16 * lane, cache + off + 16 * lane);
    if constexpr (kRecord == 1024) cp_async16(dst + 512 + 16 * lane, cache + off + 512 + 16 * lane);
    if constexpr (kRecord == 528) {
        if (lane == 0) cp_async16(dst + 512, cache + soff);
    }
    if constexpr (kRecord == 584) {
        if (lane < 4) cp_async16(dst + 512 + 16 * lane, cache + off + 512 + 16 * lane);
        if (lane == 0) cp_async8(dst + 576, cache + soff);
    }
}

// Lane L's piece of half h of a ring record, dequantised to bf16 exactly as kv_gather
// does (zeros for an invalid record): dims [256h + 8L, 256h + 8L + 8), from the e4m3 codes
// and the scale byte of their 32-dim (V4.1) or 64-dim (V4) group; the V4 rotated tail
// (dims 448..511, lanes 24..31 of the high half) and bf16 rows are copied.
template <int kRecord>
__device__ __forceinline__ uint4 convert_half(const uint8_t* src, bool valid, int lane, int h,
                                              float scale) {
    if (!valid) return make_uint4(0u, 0u, 0u, 0u);
    if constexpr (kRecord == 1024) {
        return lds16(src + 512 * h + 16 * lane);
    } else if constexpr (kRecord == 512) {
        return dequant8_scaled(lds8(src + 256 * h + 8 * lane), scale);
    } else if constexpr (kRecord == 528) {
        return dequant8(lds8(src + 256 * h + 8 * lane), src[512 + 8 * h + (lane >> 2)]);
    } else {   // 584: data 0..575 (bf16 tail at 448), scale bytes at 576
        if (h == 1 && lane >= 24) return lds16(src + 448 + 16 * (lane - 24));
        return dequant8(lds8(src + 256 * h + 8 * lane), src[576 + 4 * h + (lane >> 3)]);
    }
}

// The epilogue warp's quarter of A: lane L writes row h0 + L = head h0 + L of query qi
// (zeros past num_heads) into tensor memory at `dst` (its lanes, A's first column), 16
// columns (32 bf16) a step, the next step's loads in flight during each store (a deeper
// register ring spills at the call).
// After the first 8 steps (dims 0..255, the low half of K) it makes them visible to the
// tensor cores and arrives on `ready_lo`, so that the products of a low-half stage may
// start while the high half is loaded; after the last, on `ready_hi`.  Kept out of line:
// its registers would otherwise add to the drain loop's.
__device__ __noinline__ void load_a(const uint8_t* qbase, int64_t qi, int32_t num_heads, int h0,
                                    int lane, bool live, uint32_t dst, uint32_t ready_lo,
                                    uint32_t ready_hi) {
    const uint4* const row =
        reinterpret_cast<const uint4*>(qbase + (qi * num_heads + h0 + lane) * 1024);
    uint4 cur[4], nxt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) cur[i] = live ? __ldg(row + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        if (b < 15) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                nxt[i] = live ? __ldg(row + 4 * (b + 1) + i) : make_uint4(0u, 0u, 0u, 0u);
        }
        tmem_st16(dst + 16 * b, cur);
        if (b == 7) {
            tmem_st_wait();
            tc_fence_before_sync();
            warp_arrive(ready_lo, lane);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
    }
    tmem_st_wait();
    tc_fence_before_sync();
    warp_arrive(ready_hi, lane);
}

template <int kRecord>
__global__ void __launch_bounds__(kLogitThreads, 1)
    sparse_logits_kernel(const LogitsParams p, const __grid_constant__ CUtensorMap out_map) {
    using RawRing = Raw<kRecord>;
    constexpr int kSlots = RawRing::slots;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzle groups
    uint8_t* const base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* const sB = base;                                   // kStages B stages
    uint8_t* const sRaw = sB + kStages * kBBytes;               // the producers' rings
    uint8_t* const sTile = base + RawRing::tile_off;            // drain tiles
    Barriers* const bars = reinterpret_cast<Barriers*>(sTile + kTileBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t items = p.num_queries * p.chunks;
    const int64_t i0 = items * blockIdx.x / gridDim.x;
    const int64_t i1 = items * (blockIdx.x + 1) / gridDim.x;

    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&bars->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&bars->full[s]), kProducerWarps);
            mbar_init(smem_addr(&bars->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&bars->acc_full[a]), 1);
            mbar_init(smem_addr(&bars->acc_empty[a]), kEpilogueWarps);
        }
        mbar_init(smem_addr(&bars->a_ready[0]), kEpilogueWarps);
        mbar_init(smem_addr(&bars->a_ready[1]), kEpilogueWarps);
        bars->timed_out = 0;
        mbar_init_fence();
    }
    pdl_wait_previous();   // q, the cache and the indices may come from the kernel ahead
    pdl_release_next();
    if (threadIdx.x == 0 && i0 < i1) {   // the run's query tiles into L2 for the A loads
        for (int64_t qi = i0 / p.chunks; qi <= (i1 - 1) / p.chunks; ++qi)
            prefetch_l2_bulk(static_cast<const uint8_t*>(p.q) + qi * p.num_heads * 1024,
                             static_cast<uint32_t>(p.num_heads) * 1024);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    bool ok = true;

    if (warp < kProducerWarps) {
        // ------------------------------------------------------------- producers
        const int pw = warp;
        float scale = 1.0f;
        bool scale_bad = false;
        if constexpr (kRecord == 512) {
            scale = __ldg(p.fp8_scale);
            scale_bad = !scale_ok(scale);
            if (scale_bad && pw == 0 && lane == 0 && i0 < i1) report(p.err, kErrScale);
        }
        uint8_t* const ring = sRaw + pw * kSlots * kKeysPerWarp * RawRing::stride;
        const uint32_t groups = static_cast<uint32_t>(i1 - i0) * kGroups;
        uint32_t bad = 0;
        // The CTA's groups g = 0, 1, ... (item i0 + g / kGroups, keys (g % kGroups) * kN ..
        // of its chunk); this warp's keys of a group are kKeysPerWarp * pw + i.  Lane L of
        // window w decodes key i = L % kKeysPerWarp of group w * kWindow + L / kKeysPerWarp
        // into its record's offsets (off = -1: not a record -- past the CTA's groups, past
        // topk, index -1 or out of range, or a bad fp8 scale).
        struct Window {
            int64_t off, soff;
        };
        auto window = [&](uint32_t w) -> Window {
            Window r{-1, 0};
            const uint32_t g = w * kWindow + lane / kKeysPerWarp;
            if (g >= groups) return r;
            const int64_t item = i0 + g / kGroups;
            const int64_t qi = item / p.chunks;
            const int64_t k = (item % p.chunks) * kChunk + (g % kGroups) * kN +
                              kKeysPerWarp * pw + lane % kKeysPerWarp;
            if (k < p.topk)
                key_offsets<kRecord>(p, __ldg(p.indices + qi * p.topk + k), scale_bad, r.off,
                                     r.soff, bad);
            return r;
        };
        Window win_cur = window(0), win_nxt = window(1);
        uint32_t vmask = 0;   // bit slot * kKeysPerWarp + i: that ring record is valid
        // start the copies of group g into ring slot g % kSlots (groups are issued in order)
        auto issue = [&](uint32_t g) {
            if (g >= groups) return;
            if (g % kWindow == 0 && g > 0) {
                win_cur = win_nxt;
                win_nxt = window(g / kWindow + 1);
            }
            const int slot = static_cast<int>(g % kSlots);
#pragma unroll
            for (int i = 0; i < kKeysPerWarp; ++i) {
                const int src = static_cast<int>(g % kWindow) * kKeysPerWarp + i;
                const int64_t off = __shfl_sync(kFull, win_cur.off, src);
                const int64_t soff = __shfl_sync(kFull, win_cur.soff, src);
                const uint32_t bit = 1u << (slot * kKeysPerWarp + i);
                vmask = off >= 0 ? (vmask | bit) : (vmask & ~bit);
                if (off >= 0)
                    copy_record<kRecord>(ring + (slot * kKeysPerWarp + i) * RawRing::stride,
                                         p.cache, off, soff, lane);
            }
        };
#pragma unroll 1
        for (int t = 0; t < kSlots - 1; ++t) {
            issue(static_cast<uint32_t>(t));
            cp_async_commit();
        }
#pragma unroll 1
        for (uint32_t g = 0; g < groups; ++g) {
            __syncwarp();                  // every lane has read slot (g - 1) % kSlots
            issue(g + kSlots - 1);         // ... which now takes group g + kSlots - 1
            cp_async_commit();
            cp_async_wait<kSlots - 1>();   // this lane's copies of group g have landed
            __syncwarp();                  // ... and every lane's
            const uint8_t* const grp = ring + static_cast<int>(g % kSlots) * kKeysPerWarp *
                                                  RawRing::stride;
            const uint32_t valid = vmask >> (static_cast<int>(g % kSlots) * kKeysPerWarp);
            // the group's low half (dims 0..255), then its high half, each into a B stage
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t j = 2 * g + h;
                const int s = static_cast<int>(j % kStages);
                if (j >= kStages)
                    warp_wait_or_flag(smem_addr(&bars->empty[s]), ((j / kStages) - 1) & 1, ok,
                                      lane);
                uint8_t* const B = sB + s * kBBytes;
#pragma unroll
                for (int i = 0; i < kKeysPerWarp; ++i)
                    store_piece(B, kKeysPerWarp * pw + i, lane,
                                convert_half<kRecord>(grp + i * RawRing::stride,
                                                      ((valid >> i) & 1u) != 0u, lane, h, scale));
                fence_async_smem();
                warp_arrive(smem_addr(&bars->full[s]), lane);
            }
        }
        cp_async_wait<0>();
        if (__any_sync(kFull, bad != 0u) && lane == 0) report(p.err, kErrIndex);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            uint32_t j = 0, loads = 0;
            // the item's chunk within its query, counted rather than divided per item (a
            // 64-bit division costs this warp, which shares its scheduler with four producers,
            // more issue slots than the item's products)
            int64_t chunk = i0 % p.chunks;
            for (int64_t item = i0; item < i1; ++item, ++chunk) {
                const int64_t u = item - i0;
                const int a = static_cast<int>(u & 1);
                if (u >= 2) wait_or_flag(smem_addr(&bars->acc_empty[a]), ((u >> 1) - 1) & 1, ok);
                if (chunk == p.chunks) chunk = 0;
                // A is rewritten for each new query of the run: the item's first stage of
                // each half of K waits for that half of A
                uint32_t need = (u == 0 || chunk == 0) ? 3u : 0u;
                for (int t = 0; t < kTiles; ++t, ++j) {
                    const int s = static_cast<int>(j % kStages);
                    const int h = t & 1;   // half of K: the group's products accumulate both
                    if ((need >> h) & 1u) {
                        wait_or_flag(smem_addr(&bars->a_ready[h]), loads & 1, ok);
                        need &= ~(1u << h);
                        if (h == 1) ++loads;
                    }
                    wait_or_flag(smem_addr(&bars->full[s]), (j / kStages) & 1, ok);
                    tc_fence_after_sync();
                    const uint32_t d = tmem + a * kChunk + (t >> 1) * kN;
                    // the stage's descriptor once; each K step adds its offset / 16 to the
                    // start-address field (bits 0-13), which cannot carry: every stage lies
                    // below 227 KB, so address / 16 < 2^14
                    const uint64_t desc0 = sw128_desc(smem_addr(sB + s * kBBytes));
                    const uint32_t lo = static_cast<uint32_t>(desc0);
                    const uint32_t hi = static_cast<uint32_t>(desc0 >> 32);
                    const uint32_t a0 = tmem + kACol + (kHalfK / 2) * h;
#pragma unroll
                    for (int k = 0; k < kHalfK / 16; ++k) {   // K = 16 per instruction
                        const uint32_t step = ((k >> 2) * kN * kRowBytes + (k & 3) * 32) >> 4;
                        mma_bf16_ts(d, a0 + 8 * k,
                                    (static_cast<uint64_t>(hi) << 32) | (lo + step), kIdesc,
                                    (h | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(smem_addr(&bars->empty[s]));
                }
                mma_commit(smem_addr(&bars->acc_full[a]));
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- epilogue
        // Warp w owns tensor-memory lanes h0 .. h0 + 31, h0 = 32 (w % 4): the heads it
        // writes into A and whose accumulator rows it drains, 32 columns (entries) at a
        // time: each lane puts its head's 32 logits into the warp's swizzled tile and one
        // lane hands the tile to the TMA (entries that are not records: -inf).
        const int h0 = 32 * (warp & 3);
        const uint32_t lanes = static_cast<uint32_t>(h0) << 16;
        uint8_t* const tile = sTile + (warp - kFirstEpilogue) * kTileWarpBytes;
        uint8_t* const trow = tile + lane * 128;   // this lane's row
        bool scale_bad = false;
        if constexpr (kRecord == 512) scale_bad = !scale_ok(__ldg(p.fp8_scale));
        const uint8_t* const qbase = static_cast<const uint8_t*>(p.q);
        const bool live = h0 + lane < p.num_heads;   // this lane's head exists
        const bool stores = h0 < p.num_heads;        // this warp has heads to store
        const uint32_t a_lo = smem_addr(&bars->a_ready[0]), a_hi = smem_addr(&bars->a_ready[1]);
        const uint32_t a_dst = tmem + lanes + kACol;
        if (i0 < i1) load_a(qbase, i0 / p.chunks, p.num_heads, h0, lane, live, a_dst, a_lo, a_hi);
        int64_t qi = i0 / p.chunks, chunk = i0 - qi * p.chunks;   // counted, not divided, per item
        for (int64_t item = i0; item < i1; ++item, ++chunk) {
            const int64_t v = item - i0;
            const int a = static_cast<int>(v & 1);
            if (chunk == p.chunks) {
                chunk = 0;
                ++qi;
            }
            const int64_t k0 = chunk * kChunk;
            const bool next_query = item + 1 < i1 && chunk + 1 == p.chunks;
            if (next_query && live) {   // warm L2 with the next query's rows
                const uint8_t* const nrow = qbase + ((qi + 1) * p.num_heads + h0 + lane) * 1024;
#pragma unroll
                for (int i = 0; i < 8; ++i) prefetch_l2(nrow + 128 * i);
            }
            // the item's indices (lane L: entries k0 + L, k0 + 32 + L, ...), read before the
            // wait so that no drain step waits on a load
            int32_t idx[kChunk / kTileCols];
#pragma unroll
            for (int c = 0; c < kChunk / kTileCols; ++c) {
                const int64_t k = k0 + c * kTileCols + lane;
                idx[c] = k < p.topk ? __ldg(p.indices + qi * p.topk + k) : -1;
            }
            warp_wait_or_flag(smem_addr(&bars->acc_full[a]), (v >> 1) & 1, ok, lane);
            tc_fence_after_sync();
            // every product of this item is done, so A may take the next query now
            if (next_query) load_a(qbase, qi + 1, p.num_heads, h0, lane, live, a_dst, a_lo, a_hi);
#pragma unroll 1
            for (int c = 0; c < kChunk; c += kTileCols) {
                // bit j: entry k0 + c + j is a record (lane j read its index)
                const uint32_t recs =
                    __ballot_sync(kFull, !scale_bad && idx[0] >= 0 && idx[0] < p.num_slots);
#pragma unroll
                for (int i = 0; i + 1 < kChunk / kTileCols; ++i) idx[i] = idx[i + 1];
                float v0[16], v1[16];
                tmem_ld16(tmem + lanes + a * kChunk + c, v0);
                tmem_ld16(tmem + lanes + a * kChunk + c + 16, v1);
                if (lane == 0) bulk_wait_read_all();   // the last store has read the tile
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    st_shared16(trow + ((j ^ (lane & 7)) << 4), logit4(v0 + 4 * j, recs >> (4 * j), p.sm_scale));
                    st_shared16(trow + (((4 + j) ^ (lane & 7)) << 4),
                                logit4(v1 + 4 * j, recs >> (16 + 4 * j), p.sm_scale));
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0 && ok && stores) {
                    tma_store_tile(&out_map, tile, static_cast<int32_t>(k0 + c), h0,
                                   static_cast<int32_t>(qi));
                    bulk_commit();
                }
            }
            tc_fence_before_sync();
            warp_arrive(smem_addr(&bars->acc_empty[a]), lane);
        }
        if (lane == 0) bulk_wait_all();   // every logits store has completed
        __syncwarp();
    }
    if (!ok) atomicOr(&bars->timed_out, 1);
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && bars->timed_out != 0) report(p.err, kErrTimeout);
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to the driver
// library); null when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// The logits [num_queries, num_heads, topk] fp32 as a 3-D tensor map with 32 x 32 x 1 boxes
// and the 128-byte swizzle (topk % 4 == 0 and a 16-byte aligned base make the strides legal).
cudaError_t out_tensor_map(const LogitsParams& p, CUtensorMap* map) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.topk),
                                static_cast<cuuint64_t>(p.num_heads),
                                static_cast<cuuint64_t>(p.num_queries)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.topk) * 4,
                                   static_cast<cuuint64_t>(p.topk) * 4 * p.num_heads};
    const cuuint32_t box[3] = {kTileCols, 32, 1};
    const cuuint32_t step[3] = {1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.out, dims, strides, box,
                              step, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int kRecord>
cudaError_t launch(const LogitsParams& p, cudaStream_t stream) {
    const size_t smem = Raw<kRecord>::smem + sizeof(Barriers);
    static_assert(Raw<kRecord>::smem + sizeof(Barriers) <= kSmemLimit,
                  "the CTA's shared memory fits");
    CUtensorMap map;
    cudaError_t e = out_tensor_map(p, &map);
    if (e != cudaSuccess) return e;
    int64_t warps = 0;   // raises the kernel's dynamic shared-memory limit (once per device)
    e = resident_warps(reinterpret_cast<const void*>(sparse_logits_kernel<kRecord>), kLogitThreads,
                       smem, &warps);
    if (e != cudaSuccess) return e;
    const int64_t ctas = warps / (kLogitThreads / 32);        // one CTA per SM
    const int64_t items = p.num_queries * p.chunks;
    const int64_t blocks = items < ctas ? items : ctas;
    return launch_kernel(sparse_logits_kernel<kRecord>, blocks, kLogitThreads, smem, stream, p.pdl,
                         p, map);
}

}  // namespace

int32_t logits_chunk_keys(int32_t) { return kChunk; }
int32_t logits_max_heads() { return kM; }

cudaError_t launch_sparse_logits(int32_t record, const LogitsParams& p, cudaStream_t stream) {
    switch (record) {
        case 528: return launch<528>(p, stream);
        case 584: return launch<584>(p, stream);
        case 512: return launch<512>(p, stream);
        default: return launch<1024>(p, stream);
    }
}

}  // namespace gkr
