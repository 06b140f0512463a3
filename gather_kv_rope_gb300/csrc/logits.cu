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
// Launch shape (sm_103a, 5th-generation tensor cores): a persistent kernel, one CTA of 9
// warps per SM, each CTA taking a contiguous run of work items (query, chunk of 256 keys)
// in query-major order.
//   * A: the query's heads (up to 128, zero-padded) in shared memory as the MMA's A
//     operand (M = 128 x K = 512, bf16, K-major, 128-byte swizzle), copied with cp.async
//     when the run reaches a new query, after the last product that read the old one.
//   * 8 producer warps gather and dequantise the keys of a 32-key stage (4 each) into one
//     of 3 B tiles (N = 32 x K = 512, same layout); a ring of registers keeps the record
//     loads of the next 3 stages in flight while one is converted.
//   * one warp, once all producers have filled a stage, issues its 32 tcgen05.mma
//     (kind::f16, K = 16 each) into that stage's 32 columns of one of two 256-column TMEM
//     accumulators and commits them to the stage's mbarrier (the stage may then be
//     refilled); after an item's last stage it commits the accumulator.
//   * after producing an item the producers drain the accumulator of the item before (the
//     tensor cores are then on the new item, in the other accumulator): each reads a slice
//     of 32 lanes x 128 columns (tcgen05.ld), masks the entries that are not records (a
//     ballot over the indices) and streams the fp32 logits.
// Every wait on an mbarrier is bounded (20 ms of %globaltimer): past it the CTA sets
// GKR_ERR_TIMEOUT, stops waiting, still frees its tensor memory and returns.
#include <type_traits>

#include "decode.cuh"
#include "device.cuh"
#include "launch.h"

namespace gkr {

namespace {

constexpr int kM = 128;                  // heads per tile (MMA rows)
constexpr int kN = 32;                   // keys per B stage (MMA columns)
// Per record format: the producers' register ring (while one stage is converted, the
// record loads of the next ahead - 1 stages are in flight) and, from it, the work item
// (two turns of the ring: tiles stages of 32 keys).  Three slots for the records a lane
// holds 8 bytes of per chunk (V4.1, fp8 rows), two where it holds 16-byte pieces (the V4
// bf16 tail, bf16 rows), the most that fit the 168 registers without spilling.
template <int kRecord>
struct Shape {
    static constexpr int ahead = kRecord == 528 || kRecord == 512 ? 3 : 2;
    static constexpr int tiles = 2 * ahead;
    static constexpr int chunk = tiles * kN;                 // keys per work item
    static constexpr int drain_cols = chunk / (8 / 4);       // accumulator columns a producer
};                                                           // warp drains
constexpr int kStages = 3;               // B ring depth
constexpr int kProducerWarps = 8;        // warps 0..7: gather + dequantise, and drain the
                                         // accumulator of the item before
constexpr int kMmaWarp = kProducerWarps; // warp 8: tcgen05.mma issue; allocates and frees
                                         // TMEM too
constexpr int kKeysPerWarp = kN / kProducerWarps;           // keys of a stage per producer
constexpr int kLogitThreads = (kMmaWarp + 1) * 32;          // 9 warps: up to 168 registers
constexpr int kRowBytes = 128;           // one swizzle row: 64 bf16 of K
constexpr int kABytes = kM * 1024;       // 128 KB
constexpr int kBBytes = kN * 1024;       // 32 KB per stage
constexpr uint32_t kTmemCols = 512;      // two fp32 accumulators of kChunk columns
constexpr int32_t kErrIndex = 4;
constexpr int32_t kErrTimeout = 16;
constexpr uint64_t kWaitNs = 20000000;    // a wait gives up after 20 ms (a normal one takes us)

static_assert(kProducerWarps == 8, "two producer warps drain each quarter of the lanes");
static_assert(kKeysPerWarp * Shape<528>::tiles <= 32 && kKeysPerWarp * Shape<584>::tiles <= 32,
              "a producer lane holds the index of one (tile, key) pair of an item");
static_assert(2 * Shape<528>::chunk <= static_cast<int>(kTmemCols) &&
                  Shape<528>::drain_cols % 32 == 0 && Shape<584>::drain_cols % 32 == 0,
              "two accumulators fit; a producer drains whole 32-column index blocks");

// ------------------------------------------------------------- tcgen05 / mbarrier PTX

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
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
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator; one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the mbarrier once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}
// 32 consecutive fp32 accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
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

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A and B
// (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (static_cast<uint32_t>(kN >> 3) << 17) |
                            (static_cast<uint32_t>(kM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand with the 128-byte swizzle: start
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

// Lane L's two pieces of a 512-dim row (dims [8L, 8L+8) and [256+8L, 256+8L+8)) into
// row r of a swizzled operand of `rows` rows.
__device__ __forceinline__ void store_row_pieces(uint8_t* op, int rows, int r, int lane, uint4 a,
                                                 uint4 b) {
    *reinterpret_cast<uint4*>(op + sw128_offset(rows, r, lane >> 3, lane & 7)) = a;
    *reinterpret_cast<uint4*>(op + sw128_offset(rows, r, 4 + (lane >> 3), lane & 7)) = b;
}

// One work item = (query, chunk of kChunk keys).  A CTA (one per SM) takes a contiguous
// run of items in query-major order, so it reloads the query tile A only when its run
// moves to the next query.
struct alignas(8) Barriers {
    uint64_t full[kStages];      // producers -> MMA: B stage holds its 32 keys
    uint64_t empty[kStages];     // MMA -> producers: the stage's products are done
    uint64_t acc_full[2];        // MMA -> producers: an item's accumulator is complete
    uint64_t acc_empty[2];       // producers -> MMA: the accumulator has been read
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

// Decode key k of query row idx_row into the record's byte offsets (off = -1: not a
// record: past topk, index -1, out of range (bad = 1), or a bad fp8 scale).
template <int kRecord>
__device__ __forceinline__ void key_offsets(const LogitsParams& p, int32_t idx, bool in_range,
                                            bool scale_bad, int64_t& off, int64_t& soff,
                                            uint32_t& bad) {
    using R = Fmt<kRecord>;
    off = -1;
    soff = 0;
    if (!in_range || scale_bad) return;
    if (idx >= 0 && idx < p.num_slots) {
        const uint32_t s = static_cast<uint32_t>(idx);
        const uint32_t bs = static_cast<uint32_t>(p.block_size);
        const uint32_t page = s / bs, row = s - page * bs;
        const int64_t pbase = static_cast<int64_t>(page) * p.page_stride;
        off = pbase + row * R::D;
        soff = pbase + bs * R::D + row * R::S;
    } else if (idx != -1) {
        bad = 1u;
    }
}

template <int kRecord>
__global__ void __launch_bounds__(kLogitThreads, 1) sparse_logits_kernel(const LogitsParams p) {
    constexpr int kAhead = Shape<kRecord>::ahead;
    constexpr int kTiles = Shape<kRecord>::tiles;
    constexpr int kChunk = Shape<kRecord>::chunk;
    constexpr int kDrainCols = Shape<kRecord>::drain_cols;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzle groups
    uint8_t* const base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* const sA = base;
    uint8_t* const sB = base + kABytes;                               // kStages buffers
    Barriers* const bars = reinterpret_cast<Barriers*>(sB + kStages * kBBytes);

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
            mbar_init(smem_addr(&bars->acc_empty[a]), kProducerWarps);
        }
        bars->timed_out = 0;
        mbar_init_fence();
    }
    pdl_wait_previous();   // q, the cache and the indices may come from the kernel ahead
    pdl_release_next();
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
        LaneBases lb;
        lb.a = p.cache + Fmt<kRecord>::kLaneBytes * lane;
        lb.tail = p.cache + 448 + 16 * (lane >= 24 ? lane - 24 : 0);
        lb.s = p.cache + (kRecord == 528 ? (lane >> 2) : (lane >> 3));
        uint32_t bad = 0;
        // lane L < kTiles * kKeysPerWarp holds the index of this warp's key
        // (L / kKeysPerWarp, L % kKeysPerWarp) = tile L / kKeysPerWarp, key
        // kKeysPerWarp * pw + L % kKeysPerWarp of an item
        auto load_indices = [&](int64_t item, int32_t& idx, bool& in_range) {
            idx = -1;
            in_range = false;
            if (item >= i1 || lane >= kTiles * kKeysPerWarp) return;
            const int64_t qi = item / p.chunks;
            const int64_t k = (item % p.chunks) * kChunk + (lane / kKeysPerWarp) * kN +
                              kKeysPerWarp * pw + (lane % kKeysPerWarp);
            in_range = k < p.topk;
            if (in_range) idx = __ldg(p.indices + qi * p.topk + k);
        };
        // the records of tile t of an item whose indices are in idx_all
        auto load_tile = [&](int t, int32_t idx_all, bool rng_all, Loaded<kRecord> (&r)[kKeysPerWarp]) {
#pragma unroll
            for (int i = 0; i < kKeysPerWarp; ++i) {
                const int src = t * kKeysPerWarp + i;
                const int32_t idx = __shfl_sync(kFull, idx_all, src);
                const bool rg = __shfl_sync(kFull, rng_all ? 1 : 0, src) != 0;
                int64_t off, soff;
                key_offsets<kRecord>(p, idx, rg, scale_bad, off, soff, bad);
                load_record<kRecord>(off, soff, lb, lane, r[i]);
            }
        };
        // idx_cur: the indices of the item being converted; idx_nxt: of the next one
        int32_t idx_cur, idx_nxt;
        bool rng_cur, rng_nxt;
        load_indices(i0, idx_cur, rng_cur);
        load_indices(i0 + 1, idx_nxt, rng_nxt);
        // register ring over the CTA's stages g = 0, 1, ...: stage g (item g / kTiles, tile
        // g % kTiles) lives in slot g % kAhead; while it is converted the loads of stages
        // g + 1 .. g + kAhead - 1 (of this item or the next) are in flight
        Loaded<kRecord> ring[kAhead][kKeysPerWarp];
#pragma unroll
        for (int t = 0; t < kAhead - 1; ++t) load_tile(t, idx_cur, rng_cur, ring[t]);
        const uint32_t stages = static_cast<uint32_t>(i1 - i0) * kTiles;
        int64_t cur_q = -1;
        // Read this warp's slice of item v's accumulator -- lanes 32 (pw % 4) .. +31 (heads),
        // columns (pw / 4) * kDrainCols .. +kDrainCols-1 (entries) -- and write the logits;
        // which entries are records comes from the indices (lane l reads the index of
        // column c + l of each 32-column block, a ballot gives the block's mask).
        auto drain = [&](int64_t v) {
            const int a = static_cast<int>(v & 1);
            const int64_t item = i0 + v;
            const int64_t qi = item / p.chunks;
            const int col0 = (pw >> 2) * kDrainCols;
            const int64_t k0 = (item % p.chunks) * kChunk + col0;
            int32_t idx[kDrainCols / 32];
#pragma unroll
            for (int c = 0; c < kDrainCols / 32; ++c) {
                const int64_t k = k0 + 32 * c + lane;
                idx[c] = k < p.topk ? __ldg(p.indices + qi * p.topk + k) : -1;
            }
            warp_wait_or_flag(smem_addr(&bars->acc_full[a]), (v >> 1) & 1, ok, lane);
            tc_fence_after_sync();
            const int h = 32 * (pw & 3) + lane;
            float* const orow = p.out + (qi * p.num_heads + h) * p.topk + k0;
#pragma unroll 1
            for (int c = 0; c < kDrainCols / 16; ++c) {   // 16 columns at a time
                const uint32_t mask =
                    __ballot_sync(kFull, !scale_bad && idx[c >> 1] >= 0 && idx[c >> 1] < p.num_slots) >>
                    (16 * (c & 1));
                float val[16];
                tmem_ld16(tmem + (static_cast<uint32_t>(32 * (pw & 3)) << 16) + a * kChunk + col0 +
                              16 * c,
                          val);
                if (h < p.num_heads && ok) {
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 4) {
                        if (k0 + 16 * c + jj >= p.topk) break;   // topk is a multiple of 4
                        float4 o;
                        o.x = (mask >> jj) & 1u ? __fmul_rn(val[jj], p.sm_scale) : -INFINITY;
                        o.y = (mask >> (jj + 1)) & 1u ? __fmul_rn(val[jj + 1], p.sm_scale) : -INFINITY;
                        o.z = (mask >> (jj + 2)) & 1u ? __fmul_rn(val[jj + 2], p.sm_scale) : -INFINITY;
                        o.w = (mask >> (jj + 3)) & 1u ? __fmul_rn(val[jj + 3], p.sm_scale) : -INFINITY;
                        __stcs(reinterpret_cast<float4*>(orow + 16 * c + jj), o);
                    }
                }
            }
            tc_fence_before_sync();
            warp_arrive(smem_addr(&bars->acc_empty[a]), lane);
        };
        // one stage: slot R of the ring (static), stage number g
        auto stage = [&](auto slot_c, uint32_t g) {
            constexpr int R = decltype(slot_c)::value;
            const int t = static_cast<int>(g % kTiles);
            const int64_t u = g / kTiles;
            const int64_t item = i0 + u;
            if (t == 0) {
                if (u > 0) {              // the next item's indices become current
                    idx_cur = idx_nxt;
                    rng_cur = rng_nxt;
                    load_indices(item + 1, idx_nxt, rng_nxt);
                }
                const int64_t qi = item / p.chunks;
                if (qi != cur_q) {
                    // the query tile changes: every product that read the old one must be
                    // done; then all of its rows' copies in flight at once (cp.async into
                    // the swizzled places), one wait; rows past num_heads are zero
                    if (u > 0)
                        warp_wait_or_flag(smem_addr(&bars->acc_full[(u - 1) & 1]),
                                          ((u - 1) >> 1) & 1, ok, lane);
                    const uint8_t* const qrow =
                        static_cast<const uint8_t*>(p.q) + qi * p.num_heads * 1024;
                    for (int h = pw; h < kM; h += kProducerWarps) {
                        if (h < p.num_heads) {
                            cp_async16(sA + sw128_offset(kM, h, lane >> 3, lane & 7),
                                       qrow + h * 1024 + 16 * lane);
                            cp_async16(sA + sw128_offset(kM, h, 4 + (lane >> 3), lane & 7),
                                       qrow + h * 1024 + 512 + 16 * lane);
                        } else {
                            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                            store_row_pieces(sA, kM, h, lane, z, z);
                        }
                    }
                    cp_async_commit();
                    cp_async_wait<0>();
                    cur_q = qi;
                }
            }
            // start the loads of stage g + kAhead - 1
            {
                constexpr int RP = (R + kAhead - 1) % kAhead;
                const uint32_t gp = g + kAhead - 1;
                if (gp < stages) {
                    const int tp = static_cast<int>(gp % kTiles);
                    if (gp / kTiles == static_cast<uint32_t>(u)) load_tile(tp, idx_cur, rng_cur, ring[RP]);
                    else load_tile(tp, idx_nxt, rng_nxt, ring[RP]);
                }
            }
            const int s = static_cast<int>(g % kStages);
            if (g >= kStages)
                warp_wait_or_flag(smem_addr(&bars->empty[s]), ((g / kStages) - 1) & 1, ok, lane);
            uint8_t* const B = sB + s * kBBytes;
#pragma unroll
            for (int i = 0; i < kKeysPerWarp; ++i) {
                uint4 oa, ob;
                convert<kRecord>(ring[R][i], lane, scale, oa, ob);
                store_row_pieces(B, kN, kKeysPerWarp * pw + i, lane, oa, ob);
            }
            fence_async_smem();
            warp_arrive(smem_addr(&bars->full[s]), lane);
        };
        for (uint32_t g = 0; g < stages; g += kTiles) {    // one item; kTiles = 2 * kAhead
#pragma unroll 1
            for (uint32_t h = 0; h < kTiles; h += kAhead) {
                stage(std::integral_constant<int, 0>{}, g + h);
                stage(std::integral_constant<int, 1>{}, g + h + 1);
                if constexpr (kAhead > 2) stage(std::integral_constant<int, 2>{}, g + h + 2);
            }
            // then drain the item before (the tensor cores are on this item's stages, in the
            // other accumulator)
            if (g > 0) drain(g / kTiles - 1);
        }
        if (i1 > i0) drain(i1 - i0 - 1);
        if (__any_sync(kFull, bad != 0u) && lane == 0) report(p.err, kErrIndex);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            uint32_t j = 0;
            for (int64_t item = i0; item < i1; ++item) {
                const int64_t u = item - i0;
                const int a = static_cast<int>(u & 1);
                if (u >= 2) wait_or_flag(smem_addr(&bars->acc_empty[a]), ((u >> 1) - 1) & 1, ok);
                tc_fence_after_sync();
                const uint32_t d0 = tmem + a * kChunk;
                for (int t = 0; t < kTiles; ++t, ++j) {
                    const int s = static_cast<int>(j % kStages);
                    wait_or_flag(smem_addr(&bars->full[s]), (j / kStages) & 1, ok);
                    tc_fence_after_sync();
                    const uint32_t a0 = smem_addr(sA), b0 = smem_addr(sB + s * kBBytes);
#pragma unroll
                    for (int k = 0; k < 512 / 16; ++k) {   // K = 16 per instruction
                        const uint32_t koff = (k & 3) * 32;
                        mma_bf16(d0 + t * kN, sw128_desc(a0 + (k >> 2) * kM * kRowBytes + koff),
                                 sw128_desc(b0 + (k >> 2) * kN * kRowBytes + koff), kIdesc,
                                 k > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_addr(&bars->empty[s]));
                }
                mma_commit(smem_addr(&bars->acc_full[a]));
            }
        }
        __syncwarp();
    }
    if (!ok) atomicOr(&bars->timed_out, 1);
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && bars->timed_out != 0) report(p.err, kErrTimeout);
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int kRecord>
cudaError_t launch(const LogitsParams& p, cudaStream_t stream) {
    const size_t smem = kABytes + kStages * kBBytes + 1024 + sizeof(Barriers);
    int64_t warps = 0;   // raises the kernel's dynamic shared-memory limit (once per device)
    cudaError_t e = resident_warps(reinterpret_cast<const void*>(sparse_logits_kernel<kRecord>),
                                   kLogitThreads, smem, &warps);
    if (e != cudaSuccess) return e;
    const int64_t ctas = warps / (kLogitThreads / 32);        // one CTA per SM
    const int64_t items = p.num_queries * p.chunks;
    const int64_t blocks = items < ctas ? items : ctas;
    return launch_kernel(sparse_logits_kernel<kRecord>, blocks, kLogitThreads, smem, stream, p.pdl,
                         p);
}

}  // namespace

int32_t logits_chunk_keys(int32_t record) {
    return record == 528 || record == 512 ? Shape<528>::chunk : Shape<584>::chunk;
}
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
