/*
 * Plain CPU oracle for the DeepSeek-V4.1 / V4 paged KV-cache hot path:
 * RoPE + MXFP8 quantise + paged insert, and dequantise-gather.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA library.
 *
 * Written to be read against the pages, not to be fast:
 *   - number formats are decoded from their definitions and encoded by
 *     "round the exact value to the format's grid, ties to even";
 *   - the UE8M0 scale is the smallest power of two 2^e with 448 * 2^e >= amax,
 *     found by walking e upwards (the definition of ceil(log2(amax / 448)));
 *   - RoPE is four separately rounded fp32 products and two fp32 sums.
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (no FMA contraction, no
 * flush-to-zero), so every float operation below is one IEEE-754 binary32
 * operation rounded to nearest even.
 *
 * Sources (page title, section):
 *   [P1] "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1 record)":
 *        section "功能与动机" (record contents: 528 B = 512 B e4m3 + 16 UE8M0 scales
 *        over 32-dim blocks; legacy 584 B = 448 B e4m3 NoPE + 128 B bf16 RoPE +
 *        7 UE8M0 scales over 64-dim blocks + 1 pad; page strides 512 / 576);
 *        section "关键源码片段", fused_compress_quant_cache.py kernel text
 *        (slot < 0 skips; page = slot // block, row = slot % block; data region
 *        then scale region in a page; adjacent-pair rotation of dims 448..511
 *        with cos = row[pair], sin = row[32 + pair]; per-32-block amax, scale
 *        2^ceil(log2(amax / 448)), biased exponent byte; clamp to +-448 and cast
 *        to e4m3);
 *        section "实现拆解" item 4 (gather dequantises fp8 * 2^(scale - 127)
 *        per group; the same gather serves 448/64 and 512/32 with a bf16 tail).
 *        The same kernel text also fixes the compressed-KV variant: a token is
 *        written only when (position + 1) % COMPRESS_RATIO == 0, rotated with the
 *        cos/sin row position // COMPRESS_RATIO * COMPRESS_RATIO, and with
 *        SANITIZE_CACHE_NANS every NaN of the rotated row becomes 0 before the
 *        block maxima are taken (the scale byte then never exceeds 254).
 *   [P2] "PR #56441 [Perf][DSpark] KV-only context insertion across V4.1 cache
 *        formats", section "实现拆解" item 1 (input contract).
 *   [P4] FlashMLA overview, DSA section (index -1 marks an invalid entry).
 *   [P2] section "实现拆解" item 1 also names the two other KV-only cache formats:
 *        a bf16 cache and a plain fp8 e4m3fn cache with one fp32 scale, rows of 512
 *        elements in pages whose stride may be padded.  The same item says the
 *        KV-only op is the attention write op with its query inputs (q_in,
 *        q_head_padded, eps, apply_q_norm) removed; [P1] section "实现拆解" item 3
 *        and the attention.py listing call that op with q, the padded head count
 *        and eps beside the KV insert arguments.
 *        The optional e4m3 query output casts each head as the plain fp8 cache
 *        casts its rows; the pages name a query scale for the fp8 path but not its
 *        meaning, so "one fp32 divisor per call" is a reading (parity unpinned
 *        against the pages for the scale).
 * Readings where the pages are silent (exact scale rule, amax 0 -> byte 0,
 * RNE + saturation, fp32 RoPE op order, V4 page layout, pad byte 0, NaN
 * output pattern, out-of-range handling) are listed in the design notes.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

/* Error bits reported by insert / gather for entries outside the cache. */
#define ORACLE_ERR_SLOT 1     /* slot >= num_pages * block_size          */
#define ORACLE_ERR_POS 2      /* position outside [0, max_pos)           */
#define ORACLE_ERR_INDEX 4    /* gather index < -1 or >= num_pages * bs  */
#define ORACLE_ERR_SCALE 8    /* fp8 scale not a positive finite number  */

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities; exponent 1111 with mantissa 111 is NaN.  Exponent field 0
 * holds subnormals M * 2^-9; otherwise the value is (1 + M/8) * 2^(E-7). */
ORACLE_EXPORT double oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int E = (code >> 3) & 15;
    int M = code & 7;
    double mag;
    if (E == 15 && M == 7)
        return NAN;
    if (E == 0)
        mag = ldexp((double)M, -9);
    else
        mag = ldexp(1.0 + M / 8.0, E - 7);
    return sign ? -mag : mag;
}

/* Round y to the nearest e4m3 value, ties to even, saturating at +-448
 * (the largest finite e4m3 value).  The sign is kept, so -0 and negative
 * values that round to zero give 0x80. */
ORACLE_EXPORT uint8_t oracle_e4m3_encode(double y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    double quantum, v;
    int k, code;

    if (isnan(y))
        return (uint8_t)(sign | 0x7F);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* In the binade [2^k, 2^(k+1)) e4m3 has 8 values, spaced 2^(k-3); below
     * 2^-6 (the smallest normal) the spacing is the subnormal step 2^-9. */
    if (a == 0.0) {
        k = -6;
    } else {
        (void)frexp(a, &k); /* a = f * 2^k with f in [0.5, 1) */
        k -= 1;             /* now a in [2^k, 2^(k+1))          */
        if (k < -6)
            k = -6;
    }
    quantum = ldexp(1.0, k - 3);
    v = nearbyint(a / quantum) * quantum; /* a / quantum is exact; RNE */
    /* Find the code whose value is v (values of codes 0x00..0x7E, decoded once). */
    {
        static double value_of[0x7F];
        static int filled = 0;
        if (!filled) {
            for (code = 0; code <= 0x7E; code++)
                value_of[code] = oracle_e4m3_value((uint8_t)code);
            filled = 1;
        }
        for (code = 0; code <= 0x7E; code++)
            if (value_of[code] == v)
                return (uint8_t)(sign | code);
    }
    return (uint8_t)(sign | 0x7F); /* unreachable for |y| < 448 */
}

/* bfloat16: sign, 8 exponent bits with bias 127, 7 mantissa bits. */
ORACLE_EXPORT double oracle_bf16_value(uint16_t bits)
{
    int sign = bits >> 15;
    int E = (bits >> 7) & 0xFF;
    int M = bits & 0x7F;
    double mag;
    if (E == 0xFF)
        return M ? NAN : (sign ? -INFINITY : INFINITY);
    if (E == 0)
        mag = ldexp((double)M, -133);
    else
        mag = ldexp(1.0 + M / 128.0, E - 127);
    return sign ? -mag : mag;
}

/* Round y to the nearest bfloat16, ties to even; values that round past the
 * largest finite bf16 become infinity.  Every NaN becomes 0x7FC0. */
ORACLE_EXPORT uint16_t oracle_bf16_encode(double y)
{
    uint16_t sign = signbit(y) ? 0x8000 : 0x0000;
    double a = fabs(y);
    double quantum, v, f;
    int k, e;

    if (isnan(y))
        return 0x7FC0;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    if (a == 0.0)
        return sign;
    (void)frexp(a, &k);
    k -= 1; /* a in [2^k, 2^(k+1)) */
    if (k < -126)
        k = -126; /* subnormal range: spacing 2^-133 */
    quantum = ldexp(1.0, k - 7);
    v = nearbyint(a / quantum) * quantum;
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    if (v < ldexp(1.0, -126)) /* subnormal (or zero): M = v / 2^-133 */
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -133)));
    f = frexp(v, &e); /* v = f * 2^e, f in [0.5, 1): value = (1 + M/128) * 2^(e-1) */
    return (uint16_t)(sign | (uint16_t)((e - 1 + 127) << 7) |
                      (uint16_t)((f * 2.0 - 1.0) * 128.0));
}

/* ------------------------------------------------------------------------ */
/* Method steps                                                              */
/* ------------------------------------------------------------------------ */

/* UE8M0 scale byte for a block whose largest magnitude is amax: the smallest
 * e in [-127, 127] with 448 * 2^e >= amax (that is ceil(log2(amax / 448))
 * clamped to [-127, 127]), stored as e + 127.  amax = 0 gives byte 0. */
ORACLE_EXPORT uint8_t oracle_ue8m0_byte(float amax)
{
    int e = -127;
    while (e < 127 && ldexp(448.0, e) < (double)amax)
        e++;
    return (uint8_t)(e + 127);
}

/* One adjacent-pair rotation in fp32: even' = e*c - o*s, odd' = o*c + e*s,
 * each product and each sum rounded separately. */
ORACLE_EXPORT void oracle_rope_pair(float e, float o, float c, float s,
                                    float *e_out, float *o_out)
{
    float t1 = e * c;
    float t2 = o * s;
    float t3 = o * c;
    float t4 = e * s;
    *e_out = t1 - t2;
    *o_out = t3 + t4;
}

/* Widen one token's 512 bf16 values to fp32 and rotate dims 448..511 with the
 * cos/sin row csc[0..31] = cos, csc[32..63] = sin: pair j covers dims
 * 448 + 2j and 449 + 2j.  With sanitize, every NaN of the rotated row (all 512
 * dims) is replaced by +0. */
static void load_and_rotate(const uint16_t *kv_row, const float *csc_row,
                            int sanitize, float x[512])
{
    int d, j;
    for (d = 0; d < 512; d++)
        x[d] = (float)oracle_bf16_value(kv_row[d]);
    for (j = 0; j < 32; j++) {
        float e = x[448 + 2 * j];
        float o = x[449 + 2 * j];
        oracle_rope_pair(e, o, csc_row[j], csc_row[32 + j], &x[448 + 2 * j],
                         &x[449 + 2 * j]);
    }
    if (sanitize)
        for (d = 0; d < 512; d++)
            if (isnan(x[d]))
                x[d] = 0.0f;
}

static float block_amax(const float *x, int n)
{
    float m = 0.0f;
    int i;
    for (i = 0; i < n; i++)
        if (fabsf(x[i]) > m)
            m = fabsf(x[i]);
    return m;
}

/* Quantise n values of one block with scale byte b: e4m3(x / 2^(b - 127)). */
static void quantise_block(const float *x, int n, uint8_t b, uint8_t *q)
{
    int i;
    for (i = 0; i < n; i++)
        q[i] = oracle_e4m3_encode(ldexp((double)x[i], 127 - (int)b));
}

/* V4.1 record of one token: 512 e4m3 bytes (all dims, rotated) and 16 scale
 * bytes, one per 32-dim block. */
static void encode_v41(const uint16_t *kv_row, const float *csc_row, int sanitize,
                       uint8_t data[512], uint8_t scales[16])
{
    float x[512];
    int b;
    load_and_rotate(kv_row, csc_row, sanitize, x);
    for (b = 0; b < 16; b++) {
        scales[b] = oracle_ue8m0_byte(block_amax(x + 32 * b, 32));
        quantise_block(x + 32 * b, 32, scales[b], data + 32 * b);
    }
}

/* V4 (legacy) record of one token: 448 e4m3 bytes for the NoPE dims in seven
 * 64-dim blocks, then the 64 rotated RoPE dims as little-endian bf16 (128 B);
 * scale row = 7 bytes + one pad byte 0x00. */
static void encode_v4(const uint16_t *kv_row, const float *csc_row, int sanitize,
                      uint8_t data[576], uint8_t scales[8])
{
    float x[512];
    int b, k;
    load_and_rotate(kv_row, csc_row, sanitize, x);
    for (b = 0; b < 7; b++) {
        scales[b] = oracle_ue8m0_byte(block_amax(x + 64 * b, 64));
        quantise_block(x + 64 * b, 64, scales[b], data + 64 * b);
    }
    scales[7] = 0x00;
    for (k = 0; k < 64; k++) {
        uint16_t h = oracle_bf16_encode((double)x[448 + k]);
        data[448 + 2 * k] = (uint8_t)(h & 0xFF);
        data[449 + 2 * k] = (uint8_t)(h >> 8);
    }
}

ORACLE_EXPORT void oracle_encode_v41(const uint16_t *kv_row, const float *csc_row,
                                     uint8_t data[512], uint8_t scales[16])
{
    encode_v41(kv_row, csc_row, 0, data, scales);
}

ORACLE_EXPORT void oracle_encode_v4(const uint16_t *kv_row, const float *csc_row,
                                    uint8_t data[576], uint8_t scales[8])
{
    encode_v4(kv_row, csc_row, 0, data, scales);
}

/* bf16 cache row of one token: the rotated row rounded to bf16 (nearest even),
 * 512 little-endian values.  Dims 0..447 come back unchanged (bf16 -> fp32 -> bf16
 * is exact). */
static void encode_bf16_row(const uint16_t *kv_row, const float *csc_row, uint8_t row[1024])
{
    float x[512];
    int d;
    load_and_rotate(kv_row, csc_row, 0, x);
    for (d = 0; d < 512; d++) {
        uint16_t h = oracle_bf16_encode((double)x[d]);
        row[2 * d] = (uint8_t)(h & 0xFF);
        row[2 * d + 1] = (uint8_t)(h >> 8);
    }
}

/* fp8 cache row of one token: e4m3(x / scale) per dim, the quotient one fp32
 * division (nearest even), then rounded to e4m3 (nearest even, saturating). */
static void encode_fp8_row(const uint16_t *kv_row, const float *csc_row, float scale,
                           uint8_t row[512])
{
    float x[512];
    int d;
    load_and_rotate(kv_row, csc_row, 0, x);
    for (d = 0; d < 512; d++) {
        float y = x[d] / scale;
        row[d] = oracle_e4m3_encode((double)y);
    }
}

/* Row sizes of a cache format: data row D bytes, scale row S bytes.  528 and 584
 * are the packed MXFP8 records; 512 is the fp8 e4m3 cache (512 codes, one scale
 * for the whole cache), 1024 the bf16 cache. */
static int record_rows(int record, int *D, int *S)
{
    if (record == 528) {
        *D = 512;
        *S = 16;
        return 0;
    }
    if (record == 584) {
        *D = 576;
        *S = 8;
        return 0;
    }
    if (record == 512 || record == 1024) {
        *D = record;
        *S = 0;
        return 0;
    }
    return -1;
}

static int scale_ok(float scale)
{
    return scale > 0.0f && isfinite(scale);
}

/* Compressed-KV insert of T tokens into a paged cache (host memory).  A page
 * starts at page * page_stride and holds the data region (block_size rows of D
 * bytes) followed by the scale region (block_size rows of S bytes).  Per token,
 * in this order:
 *   1. slot < 0: skip;
 *   2. slot >= num_pages * block_size: error bit ORACLE_ERR_SLOT, skip;
 *   3. position < 0: error bit ORACLE_ERR_POS, skip;
 *   4. (position + 1) % compress_ratio != 0: skip (not a group boundary);
 *   5. cos/sin row r = position // compress_ratio * compress_ratio; r >= max_pos:
 *      error bit ORACLE_ERR_POS, skip;
 *   6. rotate with row r, replace NaN by 0 when sanitize is set, encode, store.
 * Steps 1, 4, 5 (the table row) and 6 are the pages'; the error handling in 2, 3
 * and 5 is this library's.  compress_ratio 1 without sanitize is the plain insert.
 * Returns the OR of the error bits, or -1 for an unknown record width or a
 * compress_ratio below 1. */
static int insert_general(const uint16_t *kv, int64_t num_tokens, uint8_t *cache,
                          int record, int block_size, int64_t num_pages,
                          int64_t page_stride, const int64_t *slots,
                          const int64_t *positions, const float *csc, int64_t max_pos,
                          int64_t compress_ratio, int sanitize, float fp8_scale)
{
    int D, S, err = 0;
    int64_t t;
    if (record_rows(record, &D, &S) || compress_ratio < 1)
        return -1;
    if (record == 512 && !scale_ok(fp8_scale))
        return ORACLE_ERR_SCALE; /* nothing is written */
    for (t = 0; t < num_tokens; t++) {
        int64_t slot = slots[t], pos = positions[t], page, row, r;
        uint8_t *base;
        if (slot < 0)
            continue;
        if (slot >= num_pages * block_size) {
            err |= ORACLE_ERR_SLOT;
            continue;
        }
        if (pos < 0) {
            err |= ORACLE_ERR_POS;
            continue;
        }
        if ((pos + 1) % compress_ratio != 0)
            continue;
        r = pos / compress_ratio * compress_ratio;
        if (r >= max_pos) {
            err |= ORACLE_ERR_POS;
            continue;
        }
        page = slot / block_size;
        row = slot % block_size;
        base = cache + page * page_stride;
        if (record == 528)
            encode_v41(kv + t * 512, csc + r * 64, sanitize, base + row * D,
                       base + (int64_t)block_size * D + row * S);
        else if (record == 584)
            encode_v4(kv + t * 512, csc + r * 64, sanitize, base + row * D,
                      base + (int64_t)block_size * D + row * S);
        else if (record == 1024)
            encode_bf16_row(kv + t * 512, csc + r * 64, base + row * D);
        else
            encode_fp8_row(kv + t * 512, csc + r * 64, fp8_scale, base + row * D);
    }
    return err;
}

ORACLE_EXPORT int oracle_rope_quant_insert(const uint16_t *kv, int64_t num_tokens,
                                           uint8_t *cache, int record, int block_size,
                                           int64_t num_pages, int64_t page_stride,
                                           const int64_t *slots, const int64_t *positions,
                                           const float *csc, int64_t max_pos,
                                           int64_t compress_ratio, int sanitize)
{
    if (record != 528 && record != 584)
        return -1; /* the compressed insert writes the packed records only */
    return insert_general(kv, num_tokens, cache, record, block_size, num_pages, page_stride,
                          slots, positions, csc, max_pos, compress_ratio, sanitize, 1.0f);
}

/* Plain insert into any of the four cache formats; fp8_scale is used by the fp8
 * cache (record 512) only, and must there be a positive finite number, otherwise
 * nothing is written and ORACLE_ERR_SCALE is returned. */
ORACLE_EXPORT int oracle_kv_insert(const uint16_t *kv, int64_t num_tokens, uint8_t *cache,
                                   int record, int block_size, int64_t num_pages,
                                   int64_t page_stride, const int64_t *slots,
                                   const int64_t *positions, const float *csc,
                                   int64_t max_pos, float fp8_scale)
{
    return insert_general(kv, num_tokens, cache, record, block_size, num_pages, page_stride,
                          slots, positions, csc, max_pos, 1, 0, fp8_scale);
}

/* Plain insert: every token with a valid slot is written, rotated with the cos/sin
 * row of its own position. */
ORACLE_EXPORT int oracle_insert(const uint16_t *kv, int64_t num_tokens,
                                uint8_t *cache, int record, int block_size,
                                int64_t num_pages, int64_t page_stride,
                                const int64_t *slots, const int64_t *positions,
                                const float *csc, int64_t max_pos)
{
    if (record != 528 && record != 584)
        return -1;
    return insert_general(kv, num_tokens, cache, record, block_size, num_pages, page_stride,
                          slots, positions, csc, max_pos, 1, 0, 1.0f);
}

/* Dequantise one stored record into 512 bf16 values.
 * V4.1: out[d] = bf16(e4m3(data[d]) * 2^(scale[d/32] - 127)).
 * V4:   d < 448 as above with scale[d/64]; d >= 448 copies the stored bf16.
 * A scale byte of 255 is the UE8M0 NaN; NaN results are written as 0x7FC0. */
ORACLE_EXPORT void oracle_decode(const uint8_t *data, const uint8_t *scales,
                                 int record, uint16_t out[512])
{
    int d;
    for (d = 0; d < 512; d++) {
        int block;
        double scale, v;
        if (record == 584 && d >= 448) {
            out[d] = (uint16_t)(data[448 + 2 * (d - 448)] |
                                (data[449 + 2 * (d - 448)] << 8));
            continue;
        }
        block = (record == 528) ? d / 32 : d / 64;
        scale = (scales[block] == 255) ? NAN : ldexp(1.0, (int)scales[block] - 127);
        v = oracle_e4m3_value(data[d]) * scale; /* exact in double */
        out[d] = oracle_bf16_encode(v);
    }
}

/* bf16 cache row -> the stored values unchanged. */
static void decode_bf16_row(const uint8_t *row, uint16_t out[512])
{
    int d;
    for (d = 0; d < 512; d++)
        out[d] = (uint16_t)(row[2 * d] | (row[2 * d + 1] << 8));
}

/* fp8 cache row -> bf16(e4m3 * scale): the product is one fp32 multiplication
 * (nearest even), then rounded to bf16 (nearest even). */
static void decode_fp8_row(const uint8_t *row, float scale, uint16_t out[512])
{
    int d;
    for (d = 0; d < 512; d++) {
        float v = (float)oracle_e4m3_value(row[d]) * scale;
        out[d] = oracle_bf16_encode((double)v);
    }
}

/* Gather: for each index, -1 emits 512 bf16 zeros; any other index is a slot
 * number (page = index / block_size, row = index % block_size) whose record is
 * dequantised.  Indices < -1 or past the cache emit zeros and set an error bit.
 * Returns the OR of the error bits, or -1 for an unknown record width. */
static int gather_general(const uint8_t *cache, int record, int block_size,
                          int64_t num_pages, int64_t page_stride, const int32_t *indices,
                          int64_t num_indices, float fp8_scale, uint16_t *out)
{
    int D, S, err = 0;
    int64_t i;
    if (record_rows(record, &D, &S))
        return -1;
    if (record == 512 && !scale_ok(fp8_scale)) {
        memset(out, 0, (size_t)num_indices * 512 * sizeof(uint16_t));
        return ORACLE_ERR_SCALE;
    }
    for (i = 0; i < num_indices; i++) {
        int64_t idx = indices[i], page, row;
        const uint8_t *base;
        if (idx < 0 || idx >= num_pages * block_size) {
            if (idx != -1)
                err |= ORACLE_ERR_INDEX;
            memset(out + i * 512, 0, 512 * sizeof(uint16_t));
            continue;
        }
        page = idx / block_size;
        row = idx % block_size;
        base = cache + page * page_stride;
        if (record == 1024)
            decode_bf16_row(base + row * D, out + i * 512);
        else if (record == 512)
            decode_fp8_row(base + row * D, fp8_scale, out + i * 512);
        else
            oracle_decode(base + row * D, base + (int64_t)block_size * D + row * S,
                          record, out + i * 512);
    }
    return err;
}

ORACLE_EXPORT int oracle_gather(const uint8_t *cache, int record, int block_size,
                                int64_t num_pages, int64_t page_stride,
                                const int32_t *indices, int64_t num_indices,
                                uint16_t *out)
{
    if (record != 528 && record != 584)
        return -1;
    return gather_general(cache, record, block_size, num_pages, page_stride, indices,
                          num_indices, 1.0f, out);
}

/* Gather from any of the four cache formats (fp8_scale used by record 512 only;
 * not a positive finite number -> every row zero and ORACLE_ERR_SCALE). */
ORACLE_EXPORT int oracle_kv_gather(const uint8_t *cache, int record, int block_size,
                                   int64_t num_pages, int64_t page_stride,
                                   const int32_t *indices, int64_t num_indices,
                                   float fp8_scale, uint16_t *out)
{
    return gather_general(cache, record, block_size, num_pages, page_stride, indices,
                          num_indices, fp8_scale, out);
}

/* ------------------------------------------------------------------------ */
/* Fused query-side write ([P1] "实现拆解" item 3; [P2] "实现拆解" item 1)      */
/* ------------------------------------------------------------------------ */

/* The pages name the op (q norm, q rotation, the KV insert in one call) and its
 * arguments (q, the padded head count, eps, apply_q_norm) but print neither the
 * norm nor the q layout.  Reading taken here: q is bf16 [T, H, 512]; each head's
 * 512 values x are divided by sqrt(mean(x^2) + eps) (an RMS norm without a weight)
 * when apply_q_norm is set; dims 448..511 are then rotated in adjacent pairs with
 * the token's cos/sin row, as for the KV row; the result is written as bf16 to
 * q_out [T, Hp, 512]; heads H .. Hp-1 of q_out are written as +0.  The arithmetic
 * order inside the norm is not fixed by anything, so the oracle evaluates the
 * definition in double (every step exact or correctly rounded in binary64) and gives,
 * beside the exact value and its nearest bf16, the range of bf16 values that an fp32
 * evaluation in any order may round to: [RD(y - delta), RU(y + delta)] with
 * delta = 2^-19 * |y| for dims 0..447 and delta = 2^-19 * (|e c| + |o s|) (resp.
 * |o c| + |e s|) for a rotated pair, e and o the normed values.  2^-19 bounds, with a
 * factor 2 to spare, the fp32 errors of the sum of squares (at most 21 roundings on a
 * positive sum), the added eps, the reciprocal square root, the scaling, and the two
 * rounded products and the sum or difference of the rotation; the rotated dims take
 * the size of the products, not of the result, because e c - o s can cancel. */

/* The bf16 value next to `rn` in the direction of y (rn itself when it equals y).
 * rn is the nearest-even bf16 of y. */
static uint16_t bf16_toward(uint16_t rn, double y)
{
    double v = oracle_bf16_value(rn);
    int neg = rn >> 15;
    int zero = (rn & 0x7FFF) == 0;
    if (isnan(y) || v == y)
        return rn;
    if (v < y) /* the smallest bf16 above v */
        return zero ? (uint16_t)0x0001 : (uint16_t)(neg ? rn - 1 : rn + 1);
    return zero ? (uint16_t)0x8001 : (uint16_t)(neg ? rn + 1 : rn - 1);
}

/* The largest bf16 not above y, and the smallest not below it. */
static uint16_t bf16_down(double y)
{
    uint16_t b = oracle_bf16_encode(y);
    return oracle_bf16_value(b) > y ? bf16_toward(b, -INFINITY) : b;
}

static uint16_t bf16_up(double y)
{
    uint16_t b = oracle_bf16_encode(y);
    return oracle_bf16_value(b) < y ? bf16_toward(b, INFINITY) : b;
}

/* The normed (when apply_norm) and rotated values of one query head in double, and
 * the size each one's fp32 evaluation error scales with (see above). */
static void q_head_values(const uint16_t *q_row, const float *csc_row, double eps,
                          int apply_norm, double x[512], double size[512])
{
    double r = 1.0, ss = 0.0;
    int d, j;
    for (d = 0; d < 512; d++)
        x[d] = oracle_bf16_value(q_row[d]);
    if (apply_norm) {
        for (d = 0; d < 512; d++)
            ss += x[d] * x[d];
        r = 1.0 / sqrt(ss / 512.0 + eps);
        for (d = 0; d < 512; d++)
            x[d] *= r;
    }
    for (d = 0; d < 448; d++)
        size[d] = fabs(x[d]);
    for (j = 0; j < 32; j++) {
        double e = x[448 + 2 * j], o = x[449 + 2 * j];
        double c = csc_row[j], s = csc_row[32 + j];
        x[448 + 2 * j] = e * c - o * s;
        x[449 + 2 * j] = o * c + e * s;
        size[448 + 2 * j] = fabs(e * c) + fabs(o * s);
        size[449 + 2 * j] = fabs(o * c) + fabs(e * s);
    }
}

/* One query head: exact[d] = the normed and rotated value of dim d (double);
 * rn[d] = its nearest-even bf16, alt[d] = the other faithful bf16 (== rn when the
 * value is a bf16); lo[d] .. hi[d] = the bf16 values an fp32 evaluation may give (see
 * above).  eps >= 0; a zero row with eps = 0 is outside the contract. */
ORACLE_EXPORT void oracle_q_head(const uint16_t *q_row, const float *csc_row, double eps,
                                 int apply_norm, double exact[512], uint16_t rn[512],
                                 uint16_t alt[512], uint16_t lo[512], uint16_t hi[512])
{
    double x[512], size[512];
    const double rel = ldexp(1.0, -19);
    int d;
    q_head_values(q_row, csc_row, eps, apply_norm, x, size);
    for (d = 0; d < 512; d++) {
        exact[d] = x[d];
        rn[d] = oracle_bf16_encode(x[d]);
        alt[d] = bf16_toward(rn[d], x[d]);
        lo[d] = bf16_down(x[d] - rel * size[d]);
        hi[d] = bf16_up(x[d] + rel * size[d]);
    }
}

/* The largest fp32 not above v, and the smallest not below it. */
static float f32_down(double v)
{
    float f = (float)v;
    return (double)f > v ? nextafterf(f, -INFINITY) : f;
}

static float f32_up(double v)
{
    float f = (float)v;
    return (double)f < v ? nextafterf(f, INFINITY) : f;
}

/* One query head cast to e4m3 with the fp32 scale q_scale (a positive finite number),
 * as the fp8 cache casts its rows: code = e4m3(RN32(x / q_scale)), x the head's fp32
 * value.  rn[d] takes x = RN32(exact); lo[d] .. hi[d] (by value) are the codes of the
 * smallest and the largest fp32 x within the range of oracle_q_head (the quotient and
 * the cast are monotone, so every fp32 evaluation gives a code between them). */
ORACLE_EXPORT void oracle_q_head_fp8(const uint16_t *q_row, const float *csc_row, double eps,
                                     int apply_norm, float q_scale, uint8_t rn[512],
                                     uint8_t lo[512], uint8_t hi[512])
{
    double x[512], size[512];
    const double rel = ldexp(1.0, -19);
    int d;
    q_head_values(q_row, csc_row, eps, apply_norm, x, size);
    for (d = 0; d < 512; d++) {
        float q;
        q = (float)x[d] / q_scale;
        rn[d] = oracle_e4m3_encode((double)q);
        q = f32_down(x[d] - rel * size[d]) / q_scale;
        lo[d] = oracle_e4m3_encode((double)q);
        q = f32_up(x[d] + rel * size[d]) / q_scale;
        hi[d] = oracle_e4m3_encode((double)q);
    }
}

/* The query side of the fused op with an e4m3 output (q_out [T, Hp, 512] codes): heads
 * h < num_heads of a token whose position is in [0, max_pos) by oracle_q_head_fp8, every
 * other head (padded, or a bad position: ORACLE_ERR_POS) +0 (code 0).  A q_scale that is
 * not a positive finite number writes every head as +0, and returns ORACLE_ERR_SCALE
 * when there is a head to cast (num_heads > 0 and a token with its position in the
 * table).  The KV side is oracle_kv_insert's.  Returns the error bits. */
ORACLE_EXPORT int oracle_qnorm_rope_fp8q(const uint16_t *q_in, int num_heads,
                                         int num_heads_padded, double eps, int apply_norm,
                                         float q_scale, int64_t num_tokens,
                                         const int64_t *positions, const float *csc,
                                         int64_t max_pos, uint8_t *q_rn, uint8_t *q_lo,
                                         uint8_t *q_hi)
{
    int64_t t;
    int h, err = 0;
    int good = scale_ok(q_scale);
    for (t = 0; t < num_tokens; t++) {
        int64_t pos = positions[t];
        if (!good && num_heads > 0 && pos >= 0 && pos < max_pos)
            err |= ORACLE_ERR_SCALE;
        for (h = 0; h < num_heads_padded; h++) {
            int64_t at = (t * num_heads_padded + h) * 512;
            if (!good || h >= num_heads || pos < 0 || pos >= max_pos) {
                memset(q_rn + at, 0, 512);
                memset(q_lo + at, 0, 512);
                memset(q_hi + at, 0, 512);
                continue;
            }
            oracle_q_head_fp8(q_in + (t * num_heads + h) * 512, csc + pos * 64, eps, apply_norm,
                              q_scale, q_rn + at, q_lo + at, q_hi + at);
        }
        if (num_heads > 0 && (pos < 0 || pos >= max_pos))
            err |= ORACLE_ERR_POS;
    }
    return err;
}

/* The fused op: for every token t (slot and position checks as the KV insert, but the
 * query side needs only the position):
 *   position outside [0, max_pos): ORACLE_ERR_POS; the token's query heads are
 *     written as +0 (rn = alt = 0) and its KV row is not inserted;
 *   otherwise heads h < num_heads are written by oracle_q_head, heads
 *     num_heads .. num_heads_padded - 1 as +0;
 *   the KV row is inserted exactly as oracle_kv_insert does (slot < 0 skips it).
 * q_rn / q_alt / q_lo / q_hi: uint16 [T, num_heads_padded, 512] (see oracle_q_head;
 * zero heads give 0 in all four).  Returns the error bits, or -1 for an unknown record
 * width. */
ORACLE_EXPORT int oracle_qnorm_rope_kv_insert(const uint16_t *q_in, int num_heads,
                                              int num_heads_padded, double eps,
                                              int apply_norm, uint16_t *q_rn,
                                              uint16_t *q_alt, uint16_t *q_lo,
                                              uint16_t *q_hi, const uint16_t *kv,
                                              int64_t num_tokens, uint8_t *cache, int record,
                                              int block_size, int64_t num_pages,
                                              int64_t page_stride, const int64_t *slots,
                                              const int64_t *positions, const float *csc,
                                              int64_t max_pos, float fp8_scale)
{
    int64_t t;
    int h, err;
    double exact[512];
    uint16_t *out[4];
    err = insert_general(kv, num_tokens, cache, record, block_size, num_pages, page_stride,
                         slots, positions, csc, max_pos, 1, 0, fp8_scale);
    if (err < 0)
        return err;
    for (t = 0; t < num_tokens; t++) {
        int64_t pos = positions[t];
        for (h = 0; h < num_heads_padded; h++) {
            int64_t at = (t * num_heads_padded + h) * 512;
            int k;
            out[0] = q_rn + at;
            out[1] = q_alt + at;
            out[2] = q_lo + at;
            out[3] = q_hi + at;
            if (h >= num_heads || pos < 0 || pos >= max_pos) {
                for (k = 0; k < 4; k++)
                    memset(out[k], 0, 512 * sizeof(uint16_t));
                continue;
            }
            oracle_q_head(q_in + (t * num_heads + h) * 512, csc + pos * 64, eps, apply_norm,
                          exact, out[0], out[1], out[2], out[3]);
        }
        if (num_heads > 0 && (pos < 0 || pos >= max_pos))
            err |= ORACLE_ERR_POS;
    }
    return err;
}
