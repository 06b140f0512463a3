// Record decode of the gather (gather.cu): one warp loads one cache record (any of the
// four formats) with the lane layout of device.cuh and dequantises it to the bf16 row
// kv_gather returns.
//
// Operation (page "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1
// record)", section "实现拆解" item 4: the gather reads a record by its width and
// dequantises e4m3 * 2^(scale - 127) per group -- 512 dims in 32-dim groups for V4.1,
// 448 dims in 64-dim groups plus a copied bf16 tail for V4; the plain caches copy bf16
// rows or multiply e4m3 rows by the cache's scale).
#pragma once

#include <type_traits>

#include "device.cuh"
#include "launch.h"

namespace gkr {
namespace {

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

// The bytes one lane holds of a record: its 8-dim chunks A (dims [8L, 8L+8)) and B (dims
// [256+8L, 256+8L+8)) -- 8 e4m3 codes each, or 8 bf16 values for bf16 rows and for the V4
// rotated tail on lanes 24..31 -- and, for the packed records, the two chunks' scale bytes
// (A's in bits 0..7, B's in bits 8..15).  Sized per format, so a kernel that keeps several
// records in flight per lane holds no unused register.
template <int kRecord>
struct Loaded {
    using PieceA = typename std::conditional<kRecord == 1024, uint4, uint2>::type;
    using PieceB = typename std::conditional<kRecord == 1024 || kRecord == 584, uint4, uint2>::type;
    PieceA a;
    PieceB b;
    uint32_t s;
    bool valid;
};

// Per-lane base pointers: every load of a record is one 64-bit add away.
struct LaneBases {
    const uint8_t* a;      // cache + 8L (16L for bf16 rows): chunk A (chunk B at +256 / +512)
    const uint8_t* tail;   // V4, lanes 24..31: cache + 448 + 16 (L - 24)
    const uint8_t* s;      // cache + scale byte of chunk A (chunk B's at +8 / +4)
};

template <int kRecord>
__device__ __forceinline__ void load_record(int64_t off, int64_t soff, const LaneBases& lb,
                                            int lane, Loaded<kRecord>& r) {
    r.valid = off >= 0;
    if (!r.valid) return;
    if constexpr (kRecord == 1024) {
        r.a = ldg_na16(lb.a + off);
        r.b = ldg_na16(lb.a + off + 512);
    } else if constexpr (kRecord == 512) {
        r.a = ldg_na8(lb.a + off);
        r.b = ldg_na8(lb.a + off + 256);
    } else if constexpr (kRecord == 528) {
        r.a = ldg_na8(lb.a + off);
        r.b = ldg_na8(lb.a + off + 256);
        r.s = ldg_u8(lb.s + soff) | (ldg_u8(lb.s + soff + 8) << 8);
    } else {   // 584
        r.a = ldg_na8(lb.a + off);
        if (lane < 24) {
            const uint2 t = ldg_na8(lb.a + off + 256);
            r.b = make_uint4(t.x, t.y, 0u, 0u);
            r.s = ldg_u8(lb.s + soff) | (ldg_u8(lb.s + soff + 4) << 8);
        } else {
            r.b = ldg_na16(lb.tail + off);
            r.s = ldg_u8(lb.s + soff);
        }
    }
}

// Dequantise a loaded record into this lane's two 16-byte pieces of the bf16 row (chunk
// A = dims [8L, 8L+8), chunk B = dims [256+8L, 256+8L+8)); an invalid record gives zeros.
template <int kRecord>
__device__ __forceinline__ void convert(const Loaded<kRecord>& r, int lane, float scale,
                                        uint4& oa, uint4& ob) {
    oa = make_uint4(0u, 0u, 0u, 0u);
    ob = oa;
    if (r.valid) {
        if constexpr (kRecord == 1024) {
            oa = r.a;
            ob = r.b;
        } else if constexpr (kRecord == 512) {
            oa = dequant8_scaled(r.a, scale);
            ob = dequant8_scaled(r.b, scale);
        } else if constexpr (kRecord == 528) {
            oa = dequant8(r.a, r.s & 0xFFu);
            ob = dequant8(r.b, r.s >> 8);
        } else {
            oa = dequant8(r.a, r.s & 0xFFu);
            if (lane < 24) ob = dequant8(make_uint2(r.b.x, r.b.y), r.s >> 8);
            else ob = r.b;
        }
    }
}

}  // namespace
}  // namespace gkr
