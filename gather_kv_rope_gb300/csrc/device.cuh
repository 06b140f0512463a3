// Device helpers shared by the insert and gather kernels (sm_103a).
//
// Lane layout used by every kernel: one warp owns one 512-dim row (token or gather
// index) at a time.  Lane L holds two 8-dim chunks, A = dims [8L, 8L+8) and
// B = dims [256+8L, 256+8L+8), so every warp-wide access -- 16-byte bf16 pieces or
// 8-byte e4m3 pieces -- covers one contiguous 512-byte (256-byte) span: whole
// 128-byte lines per instruction for loads and stores.  A 32-dim V4.1 scale block is
// four consecutive lanes; a 64-dim V4 block eight.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace gkr {

#ifndef GKR_WARPS_PER_BLOCK
#define GKR_WARPS_PER_BLOCK 8
#endif
#ifndef GKR_MIN_BLOCKS
#define GKR_MIN_BLOCKS 4      // resident blocks per SM the register budget is sized for
#endif
constexpr int kWarpsPerBlock = GKR_WARPS_PER_BLOCK;
constexpr int kThreads = kWarpsPerBlock * 32;
constexpr unsigned kFull = 0xFFFFFFFFu;

// ---------------------------------------------------------------- memory access

// Streaming 16-byte load (read once: evict-first in L1 and L2).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
// Read-only 16-byte load through the non-coherent path.
__device__ __forceinline__ float4 ld_ro_f4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ void st8(void* p, uint2 v) { *reinterpret_cast<uint2*>(p) = v; }
// Streaming 16-byte store (written once, not re-read by this kernel).
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// ---------------------------------------------------------------- slot decode

// Page and row of slot s in pages of bs slots.  A power-of-two block size (the usual case)
// takes a shift and a mask; any other size, a 32-bit division.
__device__ __forceinline__ void page_row(uint32_t s, uint32_t bs, uint32_t& page, uint32_t& row) {
    if ((bs & (bs - 1u)) == 0u) {
        page = s >> (__ffs(static_cast<int>(bs)) - 1);
        row = s & (bs - 1u);
    } else {
        page = s / bs;
        row = s - page * bs;
    }
}

// ---------------------------------------------------------------- bf16 <-> fp32

// Eight bf16 values packed in a uint4 -> fp32 (exact: bf16 is the top half of fp32).
__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float* f) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Two fp32 -> packed bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- RoPE

// Rotate four adjacent pairs (f[0], f[1]) .. (f[6], f[7]) by (c[i], s[i]):
// even' = e*c - o*s, odd' = o*c + e*s; every product and sum is a separately
// rounded fp32 operation (the _rn intrinsics are never contracted into FMA).
__device__ __forceinline__ void rope4(float* f, const float4 c, const float4 s) {
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float e = f[2 * i], o = f[2 * i + 1];
        f[2 * i] = __fsub_rn(__fmul_rn(e, cc[i]), __fmul_rn(o, ss[i]));
        f[2 * i + 1] = __fadd_rn(__fmul_rn(o, cc[i]), __fmul_rn(e, ss[i]));
    }
}

// ---------------------------------------------------------------- MXFP8 encode

__device__ __forceinline__ float amax8(const float* f) {
    float m = fabsf(f[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    return m;
}

// UE8M0 scale byte for a block maximum: clamp(ceil(log2(amax / 448)), -127, 127) + 127,
// computed exactly from the fp32 fields of amax.  With amax = (1 + M/2^23) * 2^(E-127)
// and 448 = 1.75 * 2^8: amax / 448 = ((1 + M/2^23) / 1.75) * 2^(E-135), and the ratio
// in brackets lies in [0.57, 1.15), so the ceiling is E - 135 plus one exactly when
// 1 + M/2^23 > 1.75, i.e. M > 0x600000.  Adding the bias 127 gives E - 8 + [M > 0x600000];
// zero and subnormal maxima fall below the clamp and give byte 0.  Finite inputs never
// exceed byte 247; an infinite maximum (E = 255) is the clamp's upper end, exponent 127,
// byte 254.  The byte is a non-decreasing function of amax, so the byte of a block is
// the maximum of the bytes of its parts.
__device__ __forceinline__ uint32_t ue8m0_byte(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const uint32_t E = b >> 23;                    // amax >= 0
    const int e = int(E) - 8 + int((b & 0x7FFFFFu) > 0x600000u);
    return E == 255u ? 254u : (e > 0 ? uint32_t(e) : 0u);
}

// 2^(127 - byte) as fp32, exact: a normal number for byte <= 253, the subnormal 2^-127
// (bit 22) for byte 254.
__device__ __forceinline__ float inv_scale(uint32_t byte) {
    return __uint_as_float(byte < 254u ? (254u - byte) << 23 : 0x00400000u);
}

// NaN -> +0 in place (every other value unchanged).
__device__ __forceinline__ void zero_nans8(float* f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] == f[i] ? f[i] : 0.0f;
}

// Four fp32 values (already divided by the block scale) -> four e4m3 bytes,
// round to nearest even with saturation to +-448, first value in the low byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// (quantise8, the MXFP8 block quantiser, follows the two-wide fp32 helpers below.)

// ---------------------------------------------------------------- MXFP8 decode

// d = a * b on packed bf16x2, rounded to nearest even (subnormals kept).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

constexpr uint32_t kBf16NaN = 0x7FC0u;

// Eight e4m3 codes -> eight bf16 values e4m3 * 2^(byte - 127), exactly rounded.
//
// An e4m3 byte s.EEEE.MMM moved to bf16 bit positions s.0000EEEE.MMM0000 reads as
// (1 + M/8) * 2^(E-127) (E >= 1) or M * 2^-129 (E = 0): in both cases the e4m3 value
// times 2^-120.  One bf16 multiply by 2^(byte - 7) then gives the result, rounded once
// to nearest even (subnormals kept).  2^(byte - 7) is a normal bf16 for byte <= 134;
// above that the factor is split into 2^127 (exact step) and 2^(byte - 134).  The
// e4m3 NaN codes (0x7F, 0xFF) and the UE8M0 NaN byte 255 give the bf16 NaN 0x7FC0.
struct Dequant {
    uint32_t m1, m2;   // packed bf16x2 factors; m2 used only when split
    bool split, nan_scale;
};

__device__ __forceinline__ Dequant make_dequant(uint32_t byte) {
    Dequant d;
    d.nan_scale = byte == 255u;
    d.split = byte > 134u;
    // bf16 bits of 2^(min(byte,134) - 7) in both halves: biased exponent min(byte,134) + 120
    d.m1 = (min(byte, 134u) + 120u) * 0x00800080u;
    d.m2 = (byte - 7u) * 0x00800080u;                // 2^(byte - 134), used when split
    return d;
}

// Four codes of one word -> two packed bf16x2 words (codes 0,1 and 2,3).
__device__ __forceinline__ void dequant4(uint32_t w, const Dequant& d, uint32_t& o01,
                                         uint32_t& o23) {
    const uint32_t x = w & 0x7F7F7F7Fu;               // magnitudes
    const uint32_t sg = w & 0x80808080u;              // signs
    // magnitudes to bytes 0 and 2 (x16 puts them at bits 4..10 / 20..26), signs to
    // bytes 1 and 3 (bit 15 / 31)
    uint32_t a = __byte_perm(x, 0u, 0x4140u) * 16u + __byte_perm(sg, 0u, 0x1404u);
    uint32_t b = __byte_perm(x, 0u, 0x4342u) * 16u + __byte_perm(sg, 0u, 0x3424u);
    o01 = bf16x2_mul(a, d.m1);
    o23 = bf16x2_mul(b, d.m1);
}

// Bytes of w whose low 7 bits are all ones (the e4m3 NaN codes) -> 0x80 in that byte.
__device__ __forceinline__ uint32_t e4m3_nan_bytes(uint32_t w) {
    return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}

// Replace the bf16 halves of o01 / o23 (codes 0..3 of a word) flagged in nanmask by NaN.
__device__ __forceinline__ void patch_nan(uint32_t nanmask, uint32_t& o01, uint32_t& o23) {
    if (nanmask & 0x00000080u) o01 = (o01 & 0xFFFF0000u) | kBf16NaN;
    if (nanmask & 0x00008000u) o01 = (o01 & 0x0000FFFFu) | (kBf16NaN << 16);
    if (nanmask & 0x00800000u) o23 = (o23 & 0xFFFF0000u) | kBf16NaN;
    if (nanmask & 0x80000000u) o23 = (o23 & 0x0000FFFFu) | (kBf16NaN << 16);
}

// General path of dequant8: any scale byte (two multiplies above 134, NaN for 255)
// and NaN codes.  Inlined behind a branch marked unlikely: the common path handles bytes
// <= 134 without NaN codes with one multiply per pair and a single test (an out-of-line
// version made the gather spill).
__device__ __forceinline__ uint4 dequant8_general(uint2 c, uint32_t byte) {
    const uint32_t n = kBf16NaN | (kBf16NaN << 16);
    if (byte == 255u) return make_uint4(n, n, n, n);
    const Dequant d = make_dequant(byte);
    uint4 o;
    dequant4(c.x, d, o.x, o.y);
    dequant4(c.y, d, o.z, o.w);
    if (d.split) {
        o.x = bf16x2_mul(o.x, d.m2);
        o.y = bf16x2_mul(o.y, d.m2);
        o.z = bf16x2_mul(o.z, d.m2);
        o.w = bf16x2_mul(o.w, d.m2);
    }
    patch_nan(e4m3_nan_bytes(c.x), o.x, o.y);
    patch_nan(e4m3_nan_bytes(c.y), o.z, o.w);
    return o;
}

// 8 e4m3 codes (2 words) with one UE8M0 scale byte -> 8 bf16 (uint4).
__device__ __forceinline__ uint4 dequant8(const uint2 c, uint32_t byte) {
    // bit 7 of a byte of acc is set iff that code is a NaN (low 7 bits all ones)
    const uint32_t acc = ((c.x & 0x7F7F7F7Fu) + 0x01010101u) | ((c.y & 0x7F7F7F7Fu) + 0x01010101u);
    if (__builtin_expect((acc & 0x80808080u) != 0u || byte > 134u, 0))
        return dequant8_general(c, byte);
    const uint32_t m = (byte + 120u) * 0x00800080u;   // bf16 2^(byte - 7), both halves
    const Dequant d = {m, 0u, false, false};
    uint4 o;
    dequant4(c.x, d, o.x, o.y);
    dequant4(c.y, d, o.z, o.w);
    return o;
}

// ---------------------------------------------------------------- fp8 rows with one scale

// Error bit for an fp8 cache scale that is not a positive finite number.
constexpr int32_t kErrScale = 8;

__device__ __forceinline__ bool scale_ok(float s) { return s > 0.0f && s <= 3.40282347e38f; }

// The quotient x / s for the fp8 cache, as the e4m3 cast sees it.  With y = RN(1/s) (the
// correctly rounded reciprocal, computed once per warp) the quotient of |x| is the
// product |x| * y refined by two correction steps q' = RN(q + RN(|x| - q s) * y), each a
// fused multiply-add: Markstein's iteration ("Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  After the first step q
// is a faithful rounding of |x|/s, so the second returns RN(|x|/s) whenever the residual
// |x| - q s is exact, i.e. away from underflow.  For s in [2^-64, 2^64] an inexact
// residual needs |x| < 2^-102 and then |x|/s < 2^-38, far below the smallest e4m3 value,
// so the e4m3 code always equals that of the IEEE quotient.  Outside that range (and for
// y == 0) the callers use the IEEE division instead.  The sign is carried separately so
// that -0 and negative underflow keep it, as the division does.
__device__ __forceinline__ float quotient(float x, float s, float y) {
    const float a = fabsf(x);
    const float q0 = __fmul_rn(a, y);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, a), y, q0);
    const float q2 = __fmaf_rn(__fmaf_rn(-q1, s, a), y, q1);
    const float q = q0 <= 3.40282347e38f ? q2 : q0;  // q0 = inf: the quotient overflows
    return copysignf(q, x);
}

// 1/s for the corrected quotient, or 0 (use the IEEE division) when s is outside
// [2^-64, 2^64].
__device__ __forceinline__ float quotient_reciprocal(float s) {
    return (s >= 5.42101086e-20f && s <= 1.84467441e19f) ? __frcp_rn(s) : 0.0f;
}

// Eight values -> e4m3(x / scale) by quotient() one value at a time.
__device__ __forceinline__ uint2 quantise8_div_exact(const float* f, float scale, float y) {
    uint2 q;
    q.x = e4m3x4(quotient(f[0], scale, y), quotient(f[1], scale, y), quotient(f[2], scale, y),
                 quotient(f[3], scale, y));
    q.y = e4m3x4(quotient(f[4], scale, y), quotient(f[5], scale, y), quotient(f[6], scale, y),
                 quotient(f[7], scale, y));
    return q;
}

// ---------------------------------------------------------------- two-wide fp32

// Two fp32 values in one 64-bit register pair (lo in the low half), for the two-wide
// fp32 multiply and fused multiply-add: one instruction rounds each half to nearest
// even exactly as the scalar instruction would, subnormals kept.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// MXFP8 encode: 8 values with their block's scale byte -> 8 e4m3 bytes.  Each value times
// the exact power of two 2^(127 - byte), one rounded product, then the saturating
// nearest-even cast.  kPacked: two products per instruction (the same results); the scalar form
// is for kernels at a tight register budget, where the register pairs cost a spill.
template <bool kPacked = true>
__device__ __forceinline__ uint2 quantise8(const float* f, uint32_t byte) {
    const float k = inv_scale(byte);
    float p[8];
    if constexpr (kPacked) {
        const uint64_t k2 = f32x2(k, k);
#pragma unroll
        for (int i = 0; i < 8; i += 2)
            f32x2_split(mul_f32x2(f32x2(f[i], f[i + 1]), k2), p[i], p[i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = __fmul_rn(f[i], k);
    }
    uint2 q;
    q.x = e4m3x4(p[0], p[1], p[2], p[3]);
    q.y = e4m3x4(p[4], p[5], p[6], p[7]);
    return q;
}

// ---------------------------------------------------------------- fp8 rows, two values per instruction

// True when one of the eight codes is an e4m3 NaN (low seven bits all ones): adding 1 to
// each byte's low seven bits carries into its bit 7 only then, and never into the next
// byte.
__device__ __forceinline__ bool any_nan_code(uint2 q) {
    const uint32_t a = (q.x & 0x7F7F7F7Fu) + 0x01010101u;
    const uint32_t b = (q.y & 0x7F7F7F7Fu) + 0x01010101u;
    return ((a | b) & 0x80808080u) != 0u;
}

// Eight values -> e4m3(x / scale): the IEEE fp32 quotient (nearest even) by the corrected
// reciprocal y, then the saturating nearest-even e4m3 cast.  The steps of quotient() run
// on the signed values with the negated reciprocal -y, two values per instruction:
// p0 = RN(x (-y)), p' = RN(p + RN(x + p s) (-y)).  Nearest-even rounding is symmetric,
// so every p is the exact negation of quotient()'s step for x, and flipping the sign
// bit of each code gives the code of x / s.  Zeros come out with the sign opposite to
// x's (+0 gives -0 at every step, -0 gives +0), so the flip gives them x's sign, as the
// division does.  An input that is not finite, or a product x y that overflows, leaves
// a NaN code; those eight values go through quotient() instead.
__device__ __forceinline__ uint2 quantise8_div(const float* f, float scale, float y) {
    const uint64_t s2 = f32x2(scale, scale);
    const uint64_t n2 = f32x2(-y, -y);
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint64_t x = f32x2(f[i], f[i + 1]);
        const uint64_t p0 = mul_f32x2(x, n2);
        const uint64_t p1 = fma_f32x2(fma_f32x2(p0, s2, x), n2, p0);
        const uint64_t p2 = fma_f32x2(fma_f32x2(p1, s2, x), n2, p1);
        f32x2_split(p2, p[i], p[i + 1]);
    }
    uint2 q;
    q.x = e4m3x4(p[0], p[1], p[2], p[3]) ^ 0x80808080u;
    q.y = e4m3x4(p[4], p[5], p[6], p[7]) ^ 0x80808080u;
    if (any_nan_code(q)) q = quantise8_div_exact(f, scale, y);
    return q;
}

// True for a power of two in [2^-126, 2^126] (a normal number with a zero mantissa,
// whose reciprocal is a normal power of two too).
__device__ __forceinline__ bool exact_power_of_two(float s) {
    const uint32_t b = __float_as_uint(s);
    const uint32_t E = b >> 23;                    // s > 0
    return (b & 0x7FFFFFu) == 0u && E >= 1u && E <= 253u;
}

// Eight values -> e4m3(x / scale) for a power-of-two scale: with y = 1/scale exact, the
// rounded product |x| * y is the rounded quotient, so one multiply per value replaces
// the corrected reciprocal; the sign is carried as in quotient().
__device__ __forceinline__ uint2 quantise8_pow2_exact(const float* f, float y) {
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = copysignf(__fmul_rn(fabsf(f[i]), y), f[i]);
    uint2 r;
    r.x = e4m3x4(q[0], q[1], q[2], q[3]);
    r.y = e4m3x4(q[4], q[5], q[6], q[7]);
    return r;
}

// The same two products per instruction: as in quantise8_div, each product is taken with
// -y and each code's sign bit flipped, which gives zeros and underflows x's sign.  An
// infinite product saturates to the largest code either way; a NaN input (a NaN code)
// sends the eight values through the form above, whose NaN codes carry the input's sign.
__device__ __forceinline__ uint2 quantise8_pow2(const float* f, float y) {
    const uint64_t n2 = f32x2(-y, -y);
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) f32x2_split(mul_f32x2(f32x2(f[i], f[i + 1]), n2), p[i], p[i + 1]);
    uint2 q;
    q.x = e4m3x4(p[0], p[1], p[2], p[3]) ^ 0x80808080u;
    q.y = e4m3x4(p[4], p[5], p[6], p[7]) ^ 0x80808080u;
    if (any_nan_code(q)) q = quantise8_pow2_exact(f, y);
    return q;
}

// The same with one IEEE division per value (scales outside [2^-64, 2^64]).
__device__ __forceinline__ uint2 quantise8_ieee_div(const float* f, float scale) {
    uint2 q;
    q.x = e4m3x4(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale), __fdiv_rn(f[2], scale),
                 __fdiv_rn(f[3], scale));
    q.y = e4m3x4(__fdiv_rn(f[4], scale), __fdiv_rn(f[5], scale), __fdiv_rn(f[6], scale),
                 __fdiv_rn(f[7], scale));
    return q;
}

// Two e4m3 codes (low 16 bits of w >> shift) -> bf16x2 of fl32(e4m3 * scale), nearest even.
// e4m3 -> f16 -> f32 is exact for every finite code.
__device__ __forceinline__ uint32_t fp8x2_scaled_bf16x2(uint32_t w16, float scale) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w16),
                                                     __NV_E4M3);
    const float2 f = __half22float2(__half2(h));
    return pack_bf16x2_rn(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
}

// Eight e4m3 codes with one fp32 scale -> eight bf16; NaN codes give 0x7FC0.
__device__ __forceinline__ uint4 dequant8_scaled(const uint2 c, float scale) {
    uint4 o;
    o.x = fp8x2_scaled_bf16x2(c.x & 0xFFFFu, scale);
    o.y = fp8x2_scaled_bf16x2(c.x >> 16, scale);
    o.z = fp8x2_scaled_bf16x2(c.y & 0xFFFFu, scale);
    o.w = fp8x2_scaled_bf16x2(c.y >> 16, scale);
    patch_nan(e4m3_nan_bytes(c.x), o.x, o.y);
    patch_nan(e4m3_nan_bytes(c.y), o.z, o.w);
    return o;
}

__device__ __forceinline__ void report(int32_t* err, int32_t bits) {
    if (err != nullptr) atomicOr(err, bits);
}

// ---------------------------------------------------------------- async copies (LDGSTS)
//
// Each lane copies the bytes it will itself consume (or the warp synchronises
// before reading bytes copied by other lanes), one commit group per staged item,
// so a per-warp ring of S items keeps S items in flight per warp without holding
// them in registers.  The waits are hardware group counters: nothing spins.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(smem)), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_addr(smem)), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds8(const void* p) { return *reinterpret_cast<const uint2*>(p); }

// ---------------------------------------------------------------- programmatic dependent launch
//
// With the programmatic-stream-serialisation launch attribute, a kernel may be
// scheduled while the previous kernel in the stream is finishing.  Every kernel
// here waits for the previous grid's completion (and memory flush) before its
// first global access, then lets the next grid start scheduling.  Without the
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait_previous() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_release_next() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

}  // namespace gkr
