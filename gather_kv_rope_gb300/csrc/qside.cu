// The fused attention write: query-side norm and rotation beside the KV insert, in one
// launch.
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "实现拆解" item 3 and the attention.py listing: one op takes q, the
// KV row, the cache, slots, positions, the cos/sin table, the padded head count and eps;
// page "PR #56441 [Perf][DSpark] KV-only context insertion across V4.1 cache formats",
// section "实现拆解" item 1: the KV-only insert is that op without q_in, q_head_padded,
// eps and apply_q_norm).  Per token t, with position p = positions[t]:
//   query heads h < H: x = q_in[t, h, :] in fp32; with the norm, x /= sqrt(mean(x^2) + eps)
//     (an RMS norm without a weight: the pages print neither the norm nor the q layout,
//     this is the reading the library takes); dims 448..511 rotated in adjacent pairs
//     with cos/sin row p, exactly as the KV row; q_out[t, h, :] = bf16(x), or with a query
//     scale the e4m3 codes of RN32(x / q_scale) (the fp8 cache's cast of its rows);
//   heads H .. Hp-1 of q_out: +0;  a position outside the table: every head of the
//     token +0 and GKR_ERR_POS;
//   the KV row: as gkr_kv_insert (slot -1 skips it).
//
// Launch shape: two block ranges.  The first covers rows of 512 dims, one warp per row at
// a time and two rows per warp (the lane layout of device.cuh).  Token t owns rows
// t*(H+1) .. t*(H+1)+H: first its KV row, then its H query heads, so a warp's rows are
// consecutive in q_in / q_out.  Lanes 0..1 decode their row (token, kind, slot,
// position) in parallel; every row's loads are issued before the first is converted.
// The second range writes the padded heads H .. Hp-1, which are zeros whatever the
// inputs: one contiguous span of (Hp - H) rows per token in q_out, cut into 512-byte
// pieces (16 bytes per lane), 16 consecutive pieces per warp.  A padded head thus costs
// one or two store instructions, not a warp of its own.
#include "device.cuh"
#include "encode.cuh"
#include "launch.h"

namespace gkr {

namespace {

constexpr int kRowsPerWarp = 2;
constexpr int kZeroPieces = 16;   // 512-byte pieces of padded heads per warp

#ifndef GKR_QSIDE_MIN_BLOCKS
#define GKR_QSIDE_MIN_BLOCKS 4
#endif

enum RowKind : int32_t { kNone = 0, kKvRow = 1, kQHead = 2, kZeroHead = 3 };

// One query head on one warp: chunks A and B of the head (16 bf16 per lane) -> normed
// (optionally) and rotated -> 16 fp32 values per lane.  The sum of squares is taken per
// lane in two fp32 accumulators (the lane's even and odd dims) by fused multiply-adds,
// two per instruction, then the two are added and summed over the warp by a butterfly
// (every lane ends with the same sum); mean = sum * 2^-9 (exact); factor = the correctly
// rounded 1/sqrt(mean + eps); each value times the factor is one rounded product, two per
// instruction.  Every sum of squares so formed goes through at most 14 roundings, and the
// results stay within the fp32-evaluation range of the exact values.
__device__ __forceinline__ void q_head(const uint4 ta, const uint4 tb, const float4 c,
                                       const float4 s, bool norm, float eps, int lane,
                                       float (&a)[8], float (&b)[8]) {
    unpack_bf16x8(ta, a);
    unpack_bf16x8(tb, b);
    if (norm) {
        uint64_t acc = mul_f32x2(f32x2(a[0], a[1]), f32x2(a[0], a[1]));
#pragma unroll
        for (int i = 2; i < 8; i += 2) {
            const uint64_t x = f32x2(a[i], a[i + 1]);
            acc = fma_f32x2(x, x, acc);
        }
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint64_t x = f32x2(b[i], b[i + 1]);
            acc = fma_f32x2(x, x, acc);
        }
        float even, odd;
        f32x2_split(acc, even, odd);
        float ss = __fadd_rn(even, odd);
#pragma unroll
        for (int x = 16; x >= 1; x >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, x));
        const float r = __frsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / 512.0f), eps));
        const uint64_t r2 = f32x2(r, r);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            f32x2_split(mul_f32x2(f32x2(a[i], a[i + 1]), r2), a[i], a[i + 1]);
            f32x2_split(mul_f32x2(f32x2(b[i], b[i + 1]), r2), b[i], b[i + 1]);
        }
    }
    if (lane >= 24) rope4(b, c, s);   // dims 448..511 = pairs 4(L-24) .. 4(L-24)+3
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2_rn(f[0], f[1]), pack_bf16x2_rn(f[2], f[3]),
                      pack_bf16x2_rn(f[4], f[5]), pack_bf16x2_rn(f[6], f[7]));
}

// Eight values -> e4m3(RN32(x / q_scale)), the cast the fp8 cache applies to its rows
// (the scale's reciprocal prepared as load_scale does).
__device__ __forceinline__ uint2 quantise_q(const float (&f)[8], const Scale& qs) {
    if (qs.y == 0.0f) return quantise8_ieee_div(f, qs.s);   // warp-uniform branches
    if (qs.pow2) return quantise8_pow2(f, qs.y);
    return quantise8_div(f, qs.s, qs.y);
}

__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
    __stcs(reinterpret_cast<uint2*>(p), v);
}

// 512-byte pieces of padded heads per token.
__host__ __device__ __forceinline__ int64_t zero_pieces_per_token(const QSideParams& qp,
                                                                   bool fp8q) {
    return static_cast<int64_t>(qp.num_heads_padded - qp.num_heads) * (fp8q ? 1 : 2);
}

// Heads H .. Hp-1 of every token (bytes [(t*Hp + H) * rb, (t*Hp + Hp) * rb) of q_out, rb
// the row's bytes): warp w of the range writes pieces 16w .. 16w+15 of the spans taken
// token after token, each piece 512 bytes at 16 per lane.
template <bool kFp8Q>
__device__ __forceinline__ void zero_padded_heads(const QSideParams& qp, int64_t num_tokens,
                                                  int64_t block, int lane) {
    constexpr int64_t kRowBytes = kFp8Q ? 512 : 1024;
    const int64_t per_token = zero_pieces_per_token(qp, kFp8Q);
    const int64_t total = num_tokens * per_token;
    const int64_t k0 = (block * kWarpsPerBlock + (threadIdx.x >> 5)) * kZeroPieces;
    if (k0 >= total) return;  // warp-uniform
    pdl_wait_previous();
    pdl_release_next();
    int64_t t = k0 / per_token;
    int64_t w = k0 - t * per_token;
    uint8_t* const out = static_cast<uint8_t*>(qp.q_out) + qp.num_heads * kRowBytes + 16 * lane;
    const int64_t n = total - k0;
#pragma unroll
    for (int i = 0; i < kZeroPieces; ++i) {
        if (i < n) st_stream16(out + t * qp.num_heads_padded * kRowBytes + w * 512,
                               make_uint4(0u, 0u, 0u, 0u));
        if (++w == per_token) {
            w = 0;
            ++t;
        }
    }
}

template <int kRecord, bool kFp8Q>
__global__ void __launch_bounds__(kThreads, GKR_QSIDE_MIN_BLOCKS)
    qnorm_rope_kv_insert_kernel(const InsertParams p, const QSideParams qp,
                                const int64_t blocks_of_rows, const uint64_t row_magic,
                                const uint32_t row_shift) {
    constexpr int U = kRowsPerWarp;
    constexpr uint32_t D = Fmt<kRecord>::D;
    constexpr uint32_t S = Fmt<kRecord>::S;
    const int lane = threadIdx.x & 31;
    if (blockIdx.x >= blocks_of_rows) {  // block-uniform: a block of padded heads
        zero_padded_heads<kFp8Q>(qp, p.num_tokens, blockIdx.x - blocks_of_rows, lane);
        return;
    }
    const int64_t per_token = static_cast<int64_t>(qp.num_heads) + 1;
    const int64_t n_rows = p.num_tokens * per_token;
    const int64_t r0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * U;
    if (r0 >= n_rows) return;  // warp-uniform

    // lane u < U decodes row r0 + u: its token and kind (j = 0: the KV row; 1..H: query
    // head j - 1)
    const bool mine = lane < U && r0 + lane < n_rows;
    int64_t t = 0;
    int32_t j = -1;
    if (mine) {
        if (row_magic != 0u) {  // uniform: rows < 2^31, a multiply and a shift (see the launch)
            const uint64_t r = static_cast<uint64_t>(r0 + lane);
            const uint64_t tt = (r * row_magic) >> row_shift;
            t = static_cast<int64_t>(tt);
            j = static_cast<int32_t>(r - tt * static_cast<uint64_t>(per_token));
        } else {
            t = (r0 + lane) / per_token;
            j = static_cast<int32_t>(r0 + lane - t * per_token);
        }
    }
    const bool reads_pos = mine;   // the KV row and the query heads
    int64_t slot = -1, q = 0;
    if (p.early_metadata != 0 && reads_pos) {
        if (j == 0) slot = __ldg(p.slots + t);
        q = __ldg(p.positions + t);
    }
    pdl_wait_previous();
    pdl_release_next();
    if (p.early_metadata == 0 && reads_pos) {
        if (j == 0) slot = __ldg(p.slots + t);
        q = __ldg(p.positions + t);
    }
    // the fp8 cache's scale, for warps with a KV row (a bad scale skips only KV rows)
    Scale scale{1.0f, 1.0f, false};
    bool scale_good = true;
    if (__ballot_sync(kFull, mine && j == 0) != 0u) scale_good = load_scale<kRecord>(p, lane, scale);

    int64_t off = -1, soff = 0;
    int32_t pos = 0, kind = kNone;
    uint32_t err = 0;
    if (mine) {
        if (j == 0) {
            if (scale_good) {
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
                        kind = kKvRow;
                    }
                }
            }
        } else if (q < 0 || q >= p.max_pos) {
            err = 2;
            kind = kZeroHead;
        } else {
            pos = static_cast<int32_t>(q);
            kind = kQHead;
        }
    }
    // the e4m3 query output's scale, read once by a warp with query heads; one that is not
    // a positive finite number turns them into zero heads
    Scale qs{1.0f, 1.0f, false};
    if constexpr (kFp8Q) {
        if (__ballot_sync(kFull, kind == kQHead) != 0u) {
            qs.s = __ldg(qp.q_scale);
            if (!scale_ok(qs.s)) {
                if (kind == kQHead) kind = kZeroHead;
                err |= static_cast<uint32_t>(kErrScale);
            } else {
                qs.pow2 = exact_power_of_two(qs.s);
                qs.y = qs.pow2 ? __frcp_rn(qs.s) : quotient_reciprocal(qs.s);
            }
        }
    }
    // every row's loads first: the KV row or the query head, and the cos/sin row
    const float* const csc_lane = p.csc + 4 * (lane >= 24 ? lane - 24 : 0);
    const uint8_t* const kv = static_cast<const uint8_t*>(p.kv);
    const uint8_t* const qin = static_cast<const uint8_t*>(qp.q_in);
    uint8_t* const qout = static_cast<uint8_t*>(qp.q_out);
    TokenLoads L[U];
    int32_t kinds[U];
    int64_t tok[U];
    int32_t head[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        kinds[u] = __shfl_sync(kFull, kind, u);
        tok[u] = __shfl_sync(kFull, t, u);
        head[u] = __shfl_sync(kFull, j, u) - 1;
        const int32_t pu = __shfl_sync(kFull, pos, u);
        if (kinds[u] == kKvRow || kinds[u] == kQHead) {   // warp-uniform
            const uint8_t* row = kinds[u] == kKvRow
                                     ? kv + tok[u] * 1024
                                     : qin + (tok[u] * qp.num_heads + head[u]) * 1024;
            L[u].a = ld_stream16(row + 16 * lane);
            L[u].b = ld_stream16(row + 512 + 16 * lane);
            if (lane >= 24) {
                const float* cs = csc_lane + static_cast<int64_t>(pu) * 64;
                L[u].c = ld_ro_f4(cs);
                L[u].s = ld_ro_f4(cs + 32);
            }
        }
    }
    // the error bits while the loads are in flight
    err = __reduce_or_sync(kFull, err);
    if (err != 0u && lane == 0) report(p.err, static_cast<int32_t>(err));
    uint8_t* const cache_a = p.cache + Fmt<kRecord>::kLaneBytes * lane;
    uint8_t* const cache_s = p.cache + ScaleRows<kRecord>::lane_byte(lane);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (kinds[u] == kKvRow) {
            const int64_t o = __shfl_sync(kFull, off, u);
            const int64_t so = __shfl_sync(kFull, soff, u);
            encode_store<kRecord>(L[u], cache_a + o, cache_s + so, lane, scale);
        } else if (kinds[u] == kQHead || kinds[u] == kZeroHead) {
            const int64_t row = tok[u] * qp.num_heads_padded + head[u];
            if constexpr (kFp8Q) {   // e4m3 codes: dims 8L.. at byte 8L, 256 + 8L.. at 256 + 8L
                uint2 ca = make_uint2(0u, 0u), cb = ca;
                if (kinds[u] == kQHead) {
                    float a[8], b[8];
                    q_head(L[u].a, L[u].b, L[u].c, L[u].s, qp.apply_norm != 0, qp.eps, lane, a, b);
                    ca = quantise_q(a, qs);
                    cb = quantise_q(b, qs);
                }
                uint8_t* dst = qout + row * 512 + 8 * lane;
                st_stream8(dst, ca);
                st_stream8(dst + 256, cb);
            } else {
                uint4 oa = make_uint4(0u, 0u, 0u, 0u), ob = oa;
                if (kinds[u] == kQHead) {
                    float a[8], b[8];
                    q_head(L[u].a, L[u].b, L[u].c, L[u].s, qp.apply_norm != 0, qp.eps, lane, a, b);
                    oa = pack_bf16x8(a);
                    ob = pack_bf16x8(b);
                }
                uint8_t* dst = qout + row * 1024 + 16 * lane;
                st_stream16(dst, oa);
                st_stream16(dst + 512, ob);
            }
        }
    }
}

template <int kRecord>
cudaError_t launch(const InsertParams& p, const QSideParams& qp, cudaStream_t stream) {
    if (p.num_tokens <= 0) return cudaSuccess;
    const int64_t rows = p.num_tokens * (static_cast<int64_t>(qp.num_heads) + 1);
    const int64_t per_block = static_cast<int64_t>(kWarpsPerBlock) * kRowsPerWarp;
    const int64_t pieces = p.num_tokens * zero_pieces_per_token(qp, qp.q_scale != nullptr);
    const int64_t zero_per_block = static_cast<int64_t>(kWarpsPerBlock) * kZeroPieces;
    const int64_t row_blocks = (rows + per_block - 1) / per_block;
    const int64_t blocks = row_blocks + (pieces + zero_per_block - 1) / zero_per_block;
    // row r's token r / d (d = H + 1 rows per token) as (r * M) >> S with S = 32 + ceil(log2 d)
    // and M = ceil(2^S / d): exact for every r < 2^31 (the error n (M d - 2^S) / (d 2^S) stays
    // below 1 / d), and r * M < 2^64 since M <= 2^33.  M = 0 (more rows): a division.
    uint64_t magic = 0;
    uint32_t shift = 0;
    const uint64_t d = static_cast<uint64_t>(qp.num_heads) + 1;
    if (rows < (INT64_C(1) << 31)) {
        uint32_t lg = 0;
        while ((UINT64_C(1) << lg) < d) ++lg;
        shift = 32 + lg;
        magic = ((UINT64_C(1) << shift) + d - 1) / d;
    }
    return qp.q_scale != nullptr
               ? launch_kernel(qnorm_rope_kv_insert_kernel<kRecord, true>, blocks, kThreads, 0,
                               stream, p.pdl, p, qp, row_blocks, magic, shift)
               : launch_kernel(qnorm_rope_kv_insert_kernel<kRecord, false>, blocks, kThreads, 0,
                               stream, p.pdl, p, qp, row_blocks, magic, shift);
}

}  // namespace

cudaError_t launch_qnorm_rope_kv_insert(int32_t record, const InsertParams& p,
                                        const QSideParams& qp, cudaStream_t stream) {
    switch (record) {
        case 528: return launch<528>(p, qp, stream);
        case 584: return launch<584>(p, qp, stream);
        case 512: return launch<512>(p, qp, stream);
        default: return launch<1024>(p, qp, stream);
    }
}

}  // namespace gkr
