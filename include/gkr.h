/*
 * gkr.h -- C ABI of libgkr.so: the DeepSeek-V4.1 / V4 paged KV-cache hot path
 * on NVIDIA GB300 (sm_103a).
 *
 *   gkr_kv_insert: bf16 latent [T, 512] -> RoPE on dims 448..511 -> MXFP8
 *                  (e4m3 + UE8M0) encode -> scatter into a paged cache (or
 *                  into a plain bf16 / fp8 e4m3 cache);
 *   gkr_kv_gather: the inverse: dequantise listed slots back to bf16 [N, 512];
 *   gkr_rope_quant_insert: the compressed-KV insert (one record per group of
 *                  compress_ratio positions, optional NaN sanitising);
 *   gkr_qnorm_rope_kv_insert: the fused attention write: query heads normed and
 *                  rotated (bf16 out, padded heads zeroed) beside the KV insert, in one
 *                  launch;
 *   gkr_sparse_logits: the dequant-gather fused into its consumer: sparse decode
 *                  logits q . k over each query's top-k records, dequantised on chip.
 *
 * Operations follow these passages (page title, section):
 *   "PR #56893 [DSv4.1] Store the whole KV in MXFP8 (FlashMLA V4.1 record)",
 *     section "功能与动机" (the two records and their page alignment), section
 *     "关键源码片段" (the fused_compress_quant_cache.py insert kernel: skip on
 *     slot < 0, page/row addressing, rotation, block scale, e4m3 cast), section
 *     "实现拆解" item 4 (the dequant-gather parameterised by record);
 *   "PR #56441 [Perf][DSpark] KV-only context insertion across V4.1 cache
 *     formats", section "实现拆解" items 1-2 (the KV-only insert contract:
 *     kv bf16 [tokens, 512], int64 slots and positions, fp32 cos_sin_cache
 *     [max_pos, 64], paged cache written in place);
 *   FlashMLA overview page, DSA section (index -1 marks an invalid entry);
 *   "PR #56441 ...", section "实现拆解" item 1 also names the two plain KV-only
 *     caches (bf16; fp8 e4m3fn with a required fp32 scalar scale).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device;
 *     the caller owns and allocates all memory.  The library allocates no
 *     device memory and never synchronises the stream; the only state it keeps
 *     is the process-wide default launch policy (gkr_set_*), which a call's
 *     gkr_launch_opts overrides, and a per-device cache of occupancy queries.
 *     Calls may be captured into CUDA graphs.
 *   - Work is enqueued on `stream` (0 = the legacy default stream); results
 *     are visible after the stream's work completes.
 *   - Host-side argument checks run before anything is enqueued; on failure
 *     nothing is enqueued and a non-zero gkr_status is returned.  No C++
 *     exception crosses this boundary.
 *   - Out-of-range data found on the device (a slot past the cache, a
 *     position outside the cos/sin table, an index < -1 or past the cache) is
 *     never dereferenced: the token is skipped / the output row is zeroed, and
 *     the matching GKR_ERR_* bit is OR-ed into *err_flag when err_flag is not
 *     NULL.  The kernels never trap.
 */
#ifndef GKR_H
#define GKR_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GKR_API __attribute__((visibility("default")))
#else
#define GKR_API
#endif

typedef enum gkr_status {
    GKR_OK = 0,
    GKR_EINVAL = 1,               /* null pointer, negative count, bad block size, ... */
    GKR_EUNSUPPORTED_RECORD = 2,  /* record width not 528, 584, 512 or 1024             */
    GKR_EBAD_PAGE_GEOMETRY = 3,   /* page stride too small or not a multiple of align   */
    GKR_EALIGN = 4,               /* a pointer is not aligned as documented             */
    GKR_ECUDA = 5                 /* the launch failed; see gkr_last_cuda_error()       */
} gkr_status;

/* Bits OR-ed into *err_flag by the kernels. */
#define GKR_ERR_SLOT 1   /* insert: slot >= num_pages * block_size (token skipped)      */
#define GKR_ERR_POS 2    /* insert: position < 0 or >= max_pos (token skipped)           */
#define GKR_ERR_INDEX 4  /* gather: index < -1 or >= num_pages * block_size (row zeroed) */
#define GKR_ERR_SCALE 8  /* fp8 cache: *fp8_scale not a positive finite number (nothing
                            written by the insert; every gathered row zeroed)           */
#define GKR_ERR_TIMEOUT 16 /* sparse logits: a bounded wait for the tensor cores gave up
                              (the launch's logits are not written); not expected      */

/*
 * Paged cache geometry.  The cache is num_pages pages, page p starting at byte
 * p * page_stride.  A page holds a data region (block_size rows of D bytes)
 * followed by a scale region (block_size rows of S bytes); the remaining
 * page_stride - block_size * record bytes are padding and are never touched.
 *   record 528 (V4.1): D = 512 (e4m3 of dims 0..511), S = 16 (one UE8M0 byte
 *                      per 32-dim block); page alignment 512.
 *   record 584 (V4):   D = 576 (448 e4m3 bytes for dims 0..447, then dims
 *                      448..511 as little-endian bf16), S = 8 (7 UE8M0 bytes
 *                      per 64-dim block + 1 pad byte 0x00); page alignment 576.
 *   record 512 (fp8):  D = 512 e4m3 codes of x / scale, S = 0; the scale is one
 *                      fp32 for the whole cache, passed as fp8_scale; align 512.
 *   record 1024 (bf16): D = 1024 (512 little-endian bf16), S = 0; align 512.
 * A slot s lives in page s / block_size, row s % block_size.
 * Requirements: record in {528, 584, 512, 1024}; block_size > 0, and a multiple
 * of 32 for 528 / 584; num_pages > 0; page_stride >= block_size * record and a
 * multiple of the record's page alignment; num_pages * block_size < 2^31.
 */
typedef struct gkr_cache_desc {
    int32_t record;
    int32_t block_size;
    int64_t num_pages;
    int64_t page_stride;
} gkr_cache_desc;

/*
 * Launch options of one call (every entry point that launches takes a nullable
 * `const gkr_launch_opts *opts`).  A field of -1, or a NULL opts, takes the
 * process-wide default set by the matching gkr_set_* call; GKR_EINVAL for any other
 * negative value or a flag other than -1, 0, 1.  Options apply to the launch of that
 * call only, so threads or libraries that share the process can each use their own.
 *   pdl                1: launch with programmatic dependent launch (see gkr_set_pdl)
 *   early_metadata     1: read slots / positions / indices before waiting for the kernel
 *                      ahead (see gkr_set_early_metadata for when this is safe)
 *   insert_staged_min  token count from which gkr_kv_insert stages rows in shared memory
 *   insert_stream_min  token count from which gkr_kv_insert streams (see
 *                      gkr_set_insert_stream_min)
 */
typedef struct gkr_launch_opts {
    int32_t pdl;
    int32_t early_metadata;
    int64_t insert_staged_min;
    int64_t insert_stream_min;
} gkr_launch_opts;

/* Every field "take the process default". */
#define GKR_LAUNCH_OPTS_INIT {-1, -1, -1, -1}

/*
 * Smallest valid page stride: block_size * record rounded up to the record's
 * page alignment (576 for 584, 512 otherwise).  Returns -1 for an unsupported
 * record or block_size.
 */
GKR_API int64_t gkr_page_stride(int32_t record, int32_t block_size);

/*
 * Row sizes of a record: data row bytes, scale row bytes and page alignment.
 * Any output pointer may be NULL.  GKR_EUNSUPPORTED_RECORD for other widths.
 */
GKR_API gkr_status gkr_record_rows(int32_t record, int32_t *data_row_bytes,
                                   int32_t *scale_row_bytes, int32_t *page_align);

/*
 * kv_insert: for each token t in [0, num_tokens):
 *   s = slot_mapping[t]; s < 0 -> skip the token (nothing read or written);
 *   x = kv[t, 0..511] widened to fp32;
 *   for pair j = 0..31 with c = cos_sin_cache[positions[t], j] and
 *   n = cos_sin_cache[positions[t], 32 + j]:
 *       x[448+2j], x[449+2j] = x[448+2j]*c - x[449+2j]*n, x[449+2j]*c + x[448+2j]*n
 *     (fp32, each product and sum rounded to nearest even, no fused multiply-add);
 *   each block (32 dims for 528, 64 NoPE dims for 584) gets the scale byte
 *     b = clamp(ceil(log2(amax / 448)), -127, 127) + 127 (amax 0 -> b = 0),
 *     and each value is stored as e4m3(x / 2^(b - 127)), round to nearest even,
 *     saturating at +-448 (an infinite amax gives b = 254 and +-inf -> +-448);
 *   for 584 the rotated dims 448..511 are stored as bf16 (round to nearest even);
 *   record 1024 stores the rotated row as bf16 (dims 0..447 unchanged);
 *   record 512 stores e4m3(fl32(x / *fp8_scale)) for all 512 dims (one IEEE fp32
 *     division, then the saturating nearest-even cast).
 *   NaN inputs, and non-finite inputs in dims 448..511 (whose rotation can give
 *   NaN, e.g. inf * 0), are outside the contract here (see gkr_rope_quant_insert).
 *
 * kv             device, bf16 [num_tokens, 512] row-major, 16-byte aligned; read only.
 * num_tokens     >= 0; 0 enqueues nothing: *cache is still validated, every other
 *                argument is ignored (pointers may be NULL, max_pos any value).
 * k_cache        device, the cache described by *cache, 16-byte aligned; only the
 *                data and scale rows of the slots written are modified.
 * cache          host pointer to the geometry (read during the call only).
 * slot_mapping   device, int64 [num_tokens]; slots must be distinct (duplicate
 *                non-negative slots race and are outside the contract).
 * positions      device, int64 [num_tokens]; row of cos_sin_cache for each token.
 * cos_sin_cache  device, fp32 [max_pos, 64] row-major (cos 0..31 | sin 0..31),
 *                16-byte aligned.
 * max_pos        rows in cos_sin_cache, 0 < max_pos < 2^31.
 * fp8_scale      device pointer to one fp32 (4-byte aligned): required for record
 *                512 (GKR_EINVAL if NULL), ignored otherwise (may be NULL).
 * err_flag       device int32 or NULL; GKR_ERR_SLOT / GKR_ERR_POS / GKR_ERR_SCALE
 *                bits are OR-ed in.
 * opts           host pointer to this call's launch options, or NULL (defaults).
 * stream         CUDA stream to enqueue on.
 */
GKR_API gkr_status gkr_kv_insert(const void *kv, int64_t num_tokens, void *k_cache,
                                 const gkr_cache_desc *cache, const int64_t *slot_mapping,
                                 const int64_t *positions, const float *cos_sin_cache,
                                 int64_t max_pos, const float *fp8_scale, int32_t *err_flag,
                                 const gkr_launch_opts *opts, cudaStream_t stream);

/*
 * rope_quant_insert: the compressed-KV insert ("PR #56893 [DSv4.1] Store the whole
 * KV in MXFP8 (FlashMLA V4.1 record)", section "关键源码片段": the kernel text of
 * fused_compress_quant_cache.py with COMPRESS_RATIO and SANITIZE_CACHE_NANS).  Per
 * token t, with s = slot_mapping[t], q = positions[t], R = compress_ratio:
 *   s < 0 -> skip;  s past the cache -> GKR_ERR_SLOT, skip;  q < 0 -> GKR_ERR_POS, skip;
 *   (q + 1) % R != 0 -> skip (only the last position of each group is written);
 *   r = q // R * R (the group's first position); r >= max_pos -> GKR_ERR_POS, skip;
 *   otherwise the record is encoded exactly as in gkr_kv_insert but rotated with
 *   cos/sin row r, and with sanitize_nans every NaN of the rotated row (all 512
 *   dims) is replaced by +0 before the block maxima are taken; scale bytes are then
 *   at most 254 (the UE8M0 NaN 255 is never written).
 * R = 1 without sanitising is gkr_kv_insert.  Records 528 and 584 only
 * (GKR_EUNSUPPORTED_RECORD otherwise).  Arguments as for gkr_kv_insert, plus
 * compress_ratio  >= 1 (GKR_EINVAL otherwise);
 * sanitize_nans   0 or 1 (GKR_EINVAL otherwise).
 * Without sanitising, NaN inputs and non-finite inputs in dims 448..511 are outside
 * the contract (as for gkr_kv_insert); with it every input value is.
 */
GKR_API gkr_status gkr_rope_quant_insert(const void *kv, int64_t num_tokens, void *k_cache,
                                         const gkr_cache_desc *cache,
                                         const int64_t *slot_mapping, const int64_t *positions,
                                         const float *cos_sin_cache, int64_t max_pos,
                                         int32_t compress_ratio, int32_t sanitize_nans,
                                         int32_t *err_flag, const gkr_launch_opts *opts,
                                         cudaStream_t stream);

/*
 * qnorm_rope_kv_insert: the fused attention write ("PR #56893 [DSv4.1] Store the whole
 * KV in MXFP8 (FlashMLA V4.1 record)", section "实现拆解" item 3 and the attention.py
 * listing: one op takes q, the KV row, the cache, slots, positions, the cos/sin table,
 * the padded head count and eps; "PR #56441 [Perf][DSpark] KV-only context insertion
 * across V4.1 cache formats", section "实现拆解" item 1: gkr_kv_insert is this op with
 * q_in, the padded head count, eps and apply_q_norm removed).  The pages print neither
 * the norm nor the q layout; this library's reading, per token t at position p:
 *   query head h < num_heads: x = q_in[t, h, 0..511] in fp32; with apply_q_norm,
 *     x = x * 1/sqrt(mean(x^2) + eps) (an RMS norm over the head's 512 dims, no
 *     weight); dims 448..511 rotated in adjacent pairs with cos/sin row p exactly as
 *     the KV row is; q_out[t, h, :] = bf16(x), round to nearest even;
 *   heads num_heads .. num_heads_padded - 1 of q_out: +0;
 *   p outside [0, max_pos) (with num_heads > 0): every head of q_out[t] is +0 and
 *     GKR_ERR_POS is set;
 *   the KV row: exactly gkr_kv_insert (slot -1 skips it; the query heads are written
 *     whatever the slot).
 * With q_scale (an extension reading the pages' fp8 query scale like the fp8 cache's
 * scale; its meaning is not on the pages), q_out holds e4m3 codes instead of bf16:
 * q_out[t, h, d] = e4m3(RN32(x_d / q_scale)), saturating, nearest even, x_d the fp32
 * value whose bf16 rounding is the bf16 output -- the cast the fp8 cache applies to its
 * rows.  A q_scale that is not a positive finite number writes every query head as +0
 * and sets GKR_ERR_SCALE (when there is a query head to cast: num_heads > 0 and a token
 * whose position is in the table); the KV rows are not affected.
 * Accuracy: the norm's arithmetic order is the kernel's (per-lane sums, a warp
 * butterfly, a correctly rounded reciprocal square root), so each q_out value is one of
 * the two bf16 values around the exact result (a faithful rounding; nearest in all but
 * rare ties of the fp32 error), while the KV record is bit-exact.  The contract needs
 * sum(x^2) < 2^128 and mean(x^2) + eps >= 2^-126 per head (eps = 0 with a zero head is
 * outside it).  num_heads_padded == 0 is exactly gkr_kv_insert (q pointers ignored).
 *
 * q_in              device, bf16 [num_tokens, num_heads, 512] row-major, 16-byte
 *                   aligned; read only (may be NULL when num_heads == 0).
 * num_heads         >= 0.
 * num_heads_padded  num_heads <= num_heads_padded <= 4096.
 * q_out             device, bf16 [num_tokens, num_heads_padded, 512] (uint8 e4m3 codes of
 *                   the same shape with q_scale), 16-byte aligned.  Without q_scale it
 *                   may be q_in itself when num_heads_padded == num_heads (in place);
 *                   with q_scale any overlap with q_in is rejected (GKR_EINVAL); any
 *                   other overlap with an input races.
 * q_scale           device, one fp32, 4-byte aligned, read by the kernel; or NULL for a
 *                   bf16 q_out.
 * eps               finite, >= 0.
 * apply_q_norm      0 or 1.
 * The other arguments are gkr_kv_insert's, for the KV row (any of the four records).
 */
GKR_API gkr_status gkr_qnorm_rope_kv_insert(const void *q_in, int32_t num_heads,
                                            int32_t num_heads_padded, void *q_out,
                                            const float *q_scale, float eps,
                                            int32_t apply_q_norm, const void *kv,
                                            int64_t num_tokens, void *k_cache,
                                            const gkr_cache_desc *cache,
                                            const int64_t *slot_mapping,
                                            const int64_t *positions,
                                            const float *cos_sin_cache, int64_t max_pos,
                                            const float *fp8_scale, int32_t *err_flag,
                                            const gkr_launch_opts *opts, cudaStream_t stream);

/*
 * kv_gather: for each i in [0, num_indices):
 *   indices[i] == -1 -> out[i, :] = +0 (bf16 0x0000);
 *   otherwise slot s = indices[i]:
 *     528: out[i, d] = bf16(e4m3(data[d]) * 2^(scale[d / 32] - 127));
 *     584: d < 448 as above with scale[d / 64]; d >= 448 copies the stored bf16.
 *     1024: out[i, :] = the stored bf16 row;
 *     512: out[i, d] = bf16(fl32(e4m3(data[d]) * *fp8_scale)).
 *   For 528 / 584 the product is exact in fp32 and rounded once to bf16 (nearest
 *   even, subnormals kept).  An e4m3 NaN code (0x7F / 0xFF) or scale byte 255 (the
 *   UE8M0 NaN) yields the bf16 NaN 0x7FC0.
 *
 * k_cache      device, the cache described by *cache, 16-byte aligned; read only.
 * cache        host pointer to the geometry.
 * indices      device, int32 [num_indices].
 * num_indices  >= 0; 0 enqueues nothing: *cache is still validated, every other
 *              argument is ignored (pointers may be NULL).
 * out          device, bf16 [num_indices, 512] row-major, 16-byte aligned.
 * fp8_scale    device pointer to one fp32: required for record 512, else ignored.
 * err_flag     device int32 or NULL; GKR_ERR_INDEX / GKR_ERR_SCALE are OR-ed in.
 * opts         host pointer to this call's launch options, or NULL (defaults).
 * stream       CUDA stream to enqueue on.
 */
GKR_API gkr_status gkr_kv_gather(const void *k_cache, const gkr_cache_desc *cache,
                                 const int32_t *indices, int64_t num_indices, void *out,
                                 const float *fp8_scale, int32_t *err_flag,
                                 const gkr_launch_opts *opts, cudaStream_t stream);

/*
 * sparse_logits: the dequant-gather fused into its consumer (FlashMLA overview page, DSA
 * section: a decode query attends to the top-k cache entries its index row lists, -1
 * marking an invalid entry, and FP8 entries are dequantised to bf16 for the matrix
 * product).  For query i, head h < num_heads and entry k < topk:
 *   out[i, h, k] = fl32(sm_scale * sum_d q[i, h, d] * K[d])
 * where K = the bf16 row gkr_kv_gather returns for indices[i, k] (any of the four
 * records); indices[i, k] == -1 gives -inf, an index < -1 or past the cache gives -inf
 * and sets GKR_ERR_INDEX; an fp8 cache whose scale is not a positive finite number gives
 * -inf everywhere and GKR_ERR_SCALE.  The gathered rows stay on chip (shared memory) and
 * the products run on the tensor cores (bf16 x bf16, fp32 accumulation over the 512
 * dims in the hardware's order), so each value is within 2^-13 * |sm_scale| *
 * sum_d |q[i, h, d] * K[d]| of the exact sum times sm_scale (a bound on fp32
 * accumulation of 512 exact products, whatever its order).
 *
 * q            device, bf16 [num_queries, num_heads, 512] row-major, 16-byte aligned.
 * num_heads    1 .. 128.
 * k_cache      device, the cache described by *cache, 16-byte aligned; read only.
 * indices      device, int32 [num_queries, topk] row-major.
 * num_queries  >= 0; topk >= 0 and a multiple of 4 (0 of either enqueues nothing).
 * sm_scale     finite; the logits' scale (e.g. the softmax scale).
 * fp8_scale    as for gkr_kv_gather.
 * out          device, fp32 [num_queries, num_heads, topk] row-major, 16-byte aligned.
 * err_flag     device int32 or NULL; GKR_ERR_INDEX / GKR_ERR_SCALE / GKR_ERR_TIMEOUT.
 * opts, stream as for the other entry points.
 */
GKR_API gkr_status gkr_sparse_logits(const void *q, int32_t num_heads, const void *k_cache,
                                     const gkr_cache_desc *cache, const int32_t *indices,
                                     int64_t num_queries, int64_t topk, float sm_scale,
                                     const float *fp8_scale, float *out, int32_t *err_flag,
                                     const gkr_launch_opts *opts, cudaStream_t stream);

/*
 * Process-wide defaults of the launch options (gkr_launch_opts fields left at -1 take
 * them).  Setting them while another thread launches is safe (atomics) but changes that
 * thread's later calls too; per-call options do not.
 *
 * Programmatic dependent launch (default on).  When on, kernels are
 * launched with the programmatic-stream-serialisation attribute: a launch may be
 * scheduled while the previous kernel in the stream drains, and waits for that
 * kernel's completion and memory flush before its first global memory access, so
 * stream order semantics are unchanged.  The setting applies to launches made
 * after the call (including launches recorded into CUDA graphs by stream capture).
 */
GKR_API void gkr_set_pdl(int32_t enable);
GKR_API int32_t gkr_get_pdl(void);

/*
 * Early metadata reads (process-wide, default off; takes effect only with programmatic
 * dependent launch on).  When set, the insert kernels may read slot_mapping and
 * positions, and the gather kernel may read indices, before waiting for the kernel
 * launched ahead of them in the stream; every other read (kv, cos_sin_cache, the
 * cache, fp8_scale) and every write still waits.  This hides one memory round trip per
 * launch (measured on GB300: 4-5 % on the 16384-token insert and gather).  Set it only
 * when the kernel ahead of an insert or gather in its stream never writes those arrays
 * -- for instance when they are filled by host copies or earlier kernels -- and not when
 * the gather's indices come straight from a preceding top-k kernel: with the setting on,
 * a kernel that writes them just ahead races with the read.  This is an extension of
 * the library; the pages have no counterpart.  Applies to launches made after the call.
 */
GKR_API void gkr_set_early_metadata(int32_t enable);
GKR_API int32_t gkr_get_early_metadata(void);

/*
 * Insert launch policy (process-wide; gkr_kv_insert only).  Three kernels write
 * identical bytes and differ only in how they hide memory latency:
 *   T < staged_min (and < stream_min): short-lived warps of two tokens, loads to
 *                                      registers;
 *   staged_min <= T < stream_min:      short-lived warps of 1-3 tokens staged in
 *                                      shared memory with cp.async;
 *   T >= stream_min:                   warps streaming runs of up to 16 tokens through a
 *                                      4-deep shared-memory ring.
 * Defaults: staged_min 24576, stream_min 131072 (measured crossovers on GB300).  A
 * negative value restores the default.
 */
GKR_API void gkr_set_insert_stream_min(int64_t tokens);
GKR_API int64_t gkr_get_insert_stream_min(void);
GKR_API void gkr_set_insert_staged_min(int64_t tokens);
GKR_API int64_t gkr_get_insert_staged_min(void);

/* Static, NUL-terminated description of a status code. */
GKR_API const char *gkr_status_string(gkr_status status);

/* The cudaError_t of the last GKR_ECUDA returned on this host thread (0 if none). */
GKR_API int32_t gkr_last_cuda_error(void);

/* ABI version: major * 10000 + minor * 100 + patch.  2.0.0: gkr_kv_insert and
 * gkr_kv_gather take fp8_scale (the plain fp8 / bf16 caches); gkr_rope_quant_insert and
 * gkr_set_insert_staged_min / gkr_get_insert_staged_min were added.  2.1.0:
 * gkr_set_early_metadata / gkr_get_early_metadata.  3.0.0: every launching entry point
 * takes a gkr_launch_opts pointer before the stream; gkr_qnorm_rope_kv_insert.
 * 3.1.0: gkr_sparse_logits.  3.2.0: gkr_qnorm_rope_kv_insert takes q_scale (an e4m3
 * query output). */
GKR_API int32_t gkr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GKR_H */
