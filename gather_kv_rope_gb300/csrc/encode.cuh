// Row encoders shared by the insert kernels (insert.cu) and the fused query + KV write
// (qside.cu): one warp encodes one token's 512-dim row into a cache row, with the lane
// layout of device.cuh (lane L owns dims [8L, 8L+8) and [256+8L, 256+8L+8)).
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "关键源码片段", the insert kernel of fused_compress_quant_cache.py,
// and section "功能与动机" for the legacy record; page "PR #56441 [Perf][DSpark] KV-only
// context insertion across V4.1 cache formats", section "实现拆解" item 1, for the
// plain bf16 and fp8 caches): rotate adjacent pairs of dims 448..511 with the
// position's cos/sin row; pick one UE8M0 scale per block (32 dims for V4.1 after
// rotation, 64 NoPE dims for V4); store e4m3 codes in the page's data region and the
// scale bytes in its scale region (or the rotated row as bf16 / as e4m3 of x / scale).
#pragma once

#include "device.cuh"
#include "launch.h"

namespace gkr {
namespace {

struct TokenLoads {
    uint4 a, b;       // bf16 chunks A and B
    float4 c, s;      // cos / sin of the 4 pairs in chunk B (lanes 24..31 only)
};

// The encoders write a token's scale bytes through `sl`, this lane's first byte of the
// token's scale row: the row in the cache itself, or the token's staging row in the
// warp's shared memory when a batch of rows is stored together (ScaleRows below).

// V4.1: 16 blocks of 32 dims.  Chunk A of lane L is in block L/4, chunk B in 8 + L/4.
// `da` = data row + 8L (chunk B's codes go to da + 256); `sl` = scale row + L/4.
// kSanitize: NaN -> +0 over the whole rotated row before the block maxima.  kPackedQ:
// quantise8's two-wide products (see there).
template <bool kSanitize = false, bool kPackedQ = true>
__device__ __forceinline__ void encode_store_v41(const TokenLoads& L, uint8_t* da, uint8_t* sl,
                                                 int lane) {
    float a[8], b[8];
    unpack_bf16x8(L.a, a);
    unpack_bf16x8(L.b, b);
    if (lane >= 24) rope4(b, L.c, L.s);  // dims 448..511 = pairs 4(L-24) .. 4(L-24)+3
    if (kSanitize) {
        zero_nans8(a);
        zero_nans8(b);
    }

    float ma = amax8(a), mb = amax8(b);
    ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, 1));
    mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 1));
    ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 2));
    const uint32_t ba = ue8m0_byte(ma), bb = ue8m0_byte(mb);

    st8(da, quantise8<kPackedQ>(a, ba));
    st8(da + 256, quantise8<kPackedQ>(b, bb));
    if ((lane & 3) == 0) {
        sl[0] = static_cast<uint8_t>(ba);
        sl[8] = static_cast<uint8_t>(bb);
    }
}

// V4: 7 blocks of 64 NoPE dims (chunk A of lane L in block L/8; chunk B of lanes 0..23
// in block 4 + L/8), rotated dims 448..511 (chunk B of lanes 24..31) stored as bf16.
// `da` = data row + 8L; `sl` = scale row + L/8 (all 8 bytes of the row are written,
// the pad byte 7 by lane 24).
template <bool kSanitize = false, bool kPackedQ = true>
__device__ __forceinline__ void encode_store_v4(const TokenLoads& L, uint8_t* da, uint8_t* sl,
                                                int lane) {
    float a[8], b[8];
    unpack_bf16x8(L.a, a);
    unpack_bf16x8(L.b, b);
    const bool rope_lane = lane >= 24;
    if (rope_lane) rope4(b, L.c, L.s);
    if (kSanitize) {
        zero_nans8(a);
        zero_nans8(b);
    }

    float ma = amax8(a), mb = rope_lane ? 0.0f : amax8(b);
#pragma unroll
    for (int x = 1; x <= 4; x <<= 1) {
        ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, x));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, x));
    }
    const uint32_t ba = ue8m0_byte(ma), bb = ue8m0_byte(mb);

    st8(da, quantise8<kPackedQ>(a, ba));
    if (!rope_lane) {
        st8(da + 256, quantise8<kPackedQ>(b, bb));
    } else {  // dims 448 + 8(L-24) .. as bf16 at data + 448 + 16(L-24) = da + 64 + 8L
        st16(da + 64 + 8 * lane,
             make_uint4(pack_bf16x2_rn(b[0], b[1]), pack_bf16x2_rn(b[2], b[3]),
                        pack_bf16x2_rn(b[4], b[5]), pack_bf16x2_rn(b[6], b[7])));
    }
    if ((lane & 7) == 0) {
        sl[0] = static_cast<uint8_t>(ba);                 // blocks 0..3
        if (!rope_lane) sl[4] = static_cast<uint8_t>(bb);  // blocks 4..6
        else sl[4] = 0;                                    // lane 24: L/8 = 3, byte 7 = pad
    }
}

// bf16 cache row (1024 B): the row with dims 448..511 rotated, rounded to bf16.  Lane L
// owns bytes [16L, 16L+16) (chunk A, copied) and [512+16L, 512+16L+16) (chunk B,
// rotated on lanes 24..31).  `da` = row + 16L.
__device__ __forceinline__ void encode_store_bf16(const TokenLoads& L, uint8_t* da, int lane) {
    st16(da, L.a);
    if (lane < 24) {
        st16(da + 512, L.b);
    } else {
        float b[8];
        unpack_bf16x8(L.b, b);
        rope4(b, L.c, L.s);
        st16(da + 512, make_uint4(pack_bf16x2_rn(b[0], b[1]), pack_bf16x2_rn(b[2], b[3]),
                                  pack_bf16x2_rn(b[4], b[5]), pack_bf16x2_rn(b[6], b[7])));
    }
}

// The fp8 cache's scale s and y = RN(1/s) for the corrected quotient (0: divide);
// pow2: s is a power of two in [2^-126, 2^126], so y = 1/s exactly and |x| * y is the
// quotient itself.
struct Scale {
    float s, y;
    bool pow2;
};

// fp8 row by IEEE divisions: the rare path (a scale outside [2^-64, 2^64]), kept out of
// line so that the common path keeps its registers.
__device__ __noinline__ void encode_store_fp8_ieee(uint4 ta, uint4 tb, float4 c, float4 sn,
                                                   uint8_t* da, int lane, float scale) {
    float a[8], b[8];
    unpack_bf16x8(ta, a);
    unpack_bf16x8(tb, b);
    if (lane >= 24) rope4(b, c, sn);
    st8(da, quantise8_ieee_div(a, scale));
    st8(da + 256, quantise8_ieee_div(b, scale));
}

// fp8 cache row (512 B): e4m3(x / scale) of the rotated row.  `da` = row + 8L.
__device__ __forceinline__ void encode_store_fp8(const TokenLoads& L, uint8_t* da, int lane,
                                                 Scale sc) {
    if (sc.y == 0.0f) {  // warp-uniform
        encode_store_fp8_ieee(L.a, L.b, L.c, L.s, da, lane, sc.s);
        return;
    }
    if (sc.pow2) {  // warp-uniform; each branch holds the whole row, so neither is predicated
        float a[8], b[8];
        unpack_bf16x8(L.a, a);
        unpack_bf16x8(L.b, b);
        if (lane >= 24) rope4(b, L.c, L.s);
        st8(da, quantise8_pow2(a, sc.y));
        st8(da + 256, quantise8_pow2(b, sc.y));
        return;
    }
    float a[8], b[8];
    unpack_bf16x8(L.a, a);
    unpack_bf16x8(L.b, b);
    if (lane >= 24) rope4(b, L.c, L.s);
    st8(da, quantise8_div(a, sc.s, sc.y));
    st8(da + 256, quantise8_div(b, sc.s, sc.y));
}

template <int kRecord, bool kSanitize = false, bool kPackedQ = true>
__device__ __forceinline__ void encode_store(const TokenLoads& L, uint8_t* da, uint8_t* sl,
                                             int lane, Scale sc) {
    if constexpr (kRecord == 528) encode_store_v41<kSanitize, kPackedQ>(L, da, sl, lane);
    else if constexpr (kRecord == 584) encode_store_v4<kSanitize, kPackedQ>(L, da, sl, lane);
    else if constexpr (kRecord == 1024) encode_store_bf16(L, da, lane);
    else encode_store_fp8(L, da, lane, sc);
}

// Scale rows of a batch of tokens, staged in the warp's shared memory (used by the
// streaming insert, whose warps write runs of consecutive tokens).  A V4.1 scale row is
// 16 bytes and a V4 row 8, so 8 (16) rows of consecutive slots fill one 128-byte line of
// the page's scale region.  Each lane's encoder writes its block's bytes into the
// token's staging row (two 1-byte shared stores from 8 or 4 lanes); `store` then writes
// the batch with one instruction: lane l stores row l (16 or 8 bytes) to the cache when
// its token was written.  Rows of consecutive slots thus leave as whole 32-byte sectors
// (whole lines for a batch starting on a line) instead of 8-byte pieces.  Kernels whose
// warps write scattered slots store each token's row straight from the encoders
// (lane_byte): there no batch can fill a sector, and the staging round trip measured
// slower.  The plain caches have no scale rows (kRows = 0).
template <int kRecord>
struct ScaleRows {
    static constexpr int S = static_cast<int>(Fmt<kRecord>::S);
    static constexpr int kRows = S == 0 ? 0 : 128 / S;   // rows per 128-byte line
    static constexpr int kBytes = S == 0 ? 16 : 128;     // staging bytes per warp

    // This lane's first byte within a scale row (block L/4 for V4.1, L/8 for V4).
    __device__ __forceinline__ static int lane_byte(int lane) {
        return kRecord == 528 ? (lane >> 2) : (lane >> 3);
    }

    // Staging row of batch row r, offset to this lane's first byte (block L/4 or L/8).
    __device__ __forceinline__ static uint8_t* row(uint8_t* warp_rows, int r, int lane) {
        return warp_rows + r * S + lane_byte(lane);
    }

    // Store batch rows 0 .. n-1: lane l < n stores row l at cache + soff when `mine`
    // (its token was encoded).  Call from all 32 lanes.
    __device__ __forceinline__ static void store(const uint8_t* warp_rows, uint8_t* cache,
                                                 int64_t soff, bool mine, int n, int lane) {
        if constexpr (S != 0) {
            __syncwarp();                              // the encoders' bytes are visible
            if (lane < n && mine) {
                if constexpr (S == 16) st16(cache + soff, lds16(warp_rows + 16 * lane));
                else st8(cache + soff, lds8(warp_rows + 8 * lane));
            }
            __syncwarp();                              // the rows may be reused
        }
    }
};

// The fp8 cache's scale (read once per warp) and its reciprocal; unused for the other
// formats.  Returns false -- after setting the error bit from lane 0 -- when an fp8 scale
// is not a positive finite number: the warp then writes nothing.
template <int kRecord>
__device__ __forceinline__ bool load_scale(const InsertParams& p, int lane, Scale& sc) {
    sc.s = 1.0f;
    sc.y = 1.0f;
    sc.pow2 = false;
    if constexpr (kRecord == 512) {
        sc.s = __ldg(p.fp8_scale);
        if (!scale_ok(sc.s)) {
            if (lane == 0) report(p.err, kErrScale);
            return false;
        }
        sc.pow2 = exact_power_of_two(sc.s);
        sc.y = sc.pow2 ? __frcp_rn(sc.s) : quotient_reciprocal(sc.s);
    }
    return true;
}

}  // namespace
}  // namespace gkr
