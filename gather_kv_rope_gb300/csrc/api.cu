// Host side of the C ABI declared in include/gkr.h: argument checks, geometry
// and kernel dispatch.  No allocation, no synchronisation, no exceptions.
#include "gkr.h"
#include "launch.h"

#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

namespace {

thread_local int32_t g_last_cuda_error = 0;
std::atomic<int> g_pdl{1};
std::atomic<int> g_early_metadata{0};
constexpr int64_t kDefaultStagedMin = 24576;
constexpr int64_t kDefaultStreamMin = 131072;
constexpr int32_t kMaxQHeads = 4096;   // query heads per token (padded) at most
std::atomic<int64_t> g_staged_min{kDefaultStagedMin};
std::atomic<int64_t> g_stream_min{kDefaultStreamMin};

struct OccEntry {
    int device;
    const void* func;
    size_t smem;
    int threads;
    int64_t warps;
};
std::mutex g_occ_mutex;
std::vector<OccEntry> g_occ;

struct RecordRows {
    int32_t data, scale, align;
};

bool record_rows(int32_t record, RecordRows* r) {
    // V4.1: 512 B e4m3 + 16 UE8M0; V4: 448 B e4m3 + 128 B bf16 + 7 UE8M0 + 1 pad.
    // Pages align to 512 B (V4.1) and 576 B (V4) ("PR #56893 [DSv4.1] Store the whole
    // KV in MXFP8 (FlashMLA V4.1 record)", section "功能与动机").  The plain KV-only
    // caches keep 512 elements a row: fp8 e4m3 (512 B) or bf16 (1024 B), pages aligned
    // to 512 B ("PR #56441 [Perf][DSpark] KV-only context insertion across V4.1 cache
    // formats", section "实现拆解" item 1).
    if (record == 528) { *r = {512, 16, 512}; return true; }
    if (record == 584) { *r = {576, 8, 576}; return true; }
    if (record == 512) { *r = {512, 0, 512}; return true; }
    if (record == 1024) { *r = {1024, 0, 512}; return true; }
    return false;
}

bool packed(int32_t record) { return record == 528 || record == 584; }

// Packed records need block_size % 32 == 0 (the page geometry of the pages); the
// plain caches take any block_size >= 1.
bool block_size_ok(int32_t record, int32_t bs) {
    return bs > 0 && (!packed(record) || bs % 32 == 0);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

gkr_status check_cache(const gkr_cache_desc* c, RecordRows* rows) {
    if (c == nullptr) return GKR_EINVAL;
    if (!record_rows(c->record, rows)) return GKR_EUNSUPPORTED_RECORD;
    if (!block_size_ok(c->record, c->block_size)) return GKR_EINVAL;
    if (c->num_pages <= 0) return GKR_EINVAL;
    if (c->num_pages > (INT64_C(0x7FFFFFFF) / c->block_size)) return GKR_EINVAL;  // slots < 2^31
    const int64_t need = static_cast<int64_t>(c->block_size) * c->record;
    if (need > INT64_C(0x7FFFFFFF)) return GKR_EINVAL;                             // page < 2^31 B
    if (c->page_stride < need || c->page_stride % rows->align != 0) return GKR_EBAD_PAGE_GEOMETRY;
    if (c->page_stride > INT64_MAX / c->num_pages) return GKR_EBAD_PAGE_GEOMETRY;
    return GKR_OK;
}

gkr_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GKR_OK;
    g_last_cuda_error = static_cast<int32_t>(e);
    return GKR_ECUDA;
}

// The launch policy of one call: the process-wide defaults (gkr_set_*), overridden by
// the fields of `o` that are not -1.  GKR_EINVAL for any other negative value, or a
// flag other than -1, 0 or 1.
struct Policy {
    int32_t pdl, early_metadata;
    int64_t staged_min, stream_min;
};

gkr_status resolve_policy(const gkr_launch_opts* o, Policy* out) {
    out->pdl = g_pdl.load(std::memory_order_relaxed);
    out->early_metadata = g_early_metadata.load(std::memory_order_relaxed);
    out->staged_min = g_staged_min.load(std::memory_order_relaxed);
    out->stream_min = g_stream_min.load(std::memory_order_relaxed);
    if (o == nullptr) return GKR_OK;
    if (o->pdl < -1 || o->pdl > 1 || o->early_metadata < -1 || o->early_metadata > 1 ||
        o->insert_staged_min < -1 || o->insert_stream_min < -1)
        return GKR_EINVAL;
    if (o->pdl >= 0) out->pdl = o->pdl;
    if (o->early_metadata >= 0) out->early_metadata = o->early_metadata;
    if (o->insert_staged_min >= 0) out->staged_min = o->insert_staged_min;
    if (o->insert_stream_min >= 0) out->stream_min = o->insert_stream_min;
    return GKR_OK;
}

}  // namespace

namespace gkr {

cudaError_t resident_warps(const void* func, int threads, size_t smem, int64_t* warps) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (const OccEntry& o : g_occ) {
        if (o.device == dev && o.func == func && o.smem == smem && o.threads == threads) {
            *warps = o.warps;
            return cudaSuccess;
        }
    }
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t w = static_cast<int64_t>(sms) * per_sm * (threads / 32);
    g_occ.push_back({dev, func, smem, threads, w});
    *warps = w;
    return cudaSuccess;
}

}  // namespace gkr

extern "C" {

GKR_API void gkr_set_pdl(int32_t enable) { g_pdl.store(enable ? 1 : 0); }

GKR_API int32_t gkr_get_pdl(void) { return g_pdl.load() ? 1 : 0; }

GKR_API void gkr_set_early_metadata(int32_t enable) { g_early_metadata.store(enable ? 1 : 0); }

GKR_API int32_t gkr_get_early_metadata(void) { return g_early_metadata.load() ? 1 : 0; }

GKR_API void gkr_set_insert_stream_min(int64_t tokens) {
    g_stream_min.store(tokens < 0 ? kDefaultStreamMin : tokens);
}

GKR_API int64_t gkr_get_insert_stream_min(void) { return g_stream_min.load(); }

GKR_API void gkr_set_insert_staged_min(int64_t tokens) {
    g_staged_min.store(tokens < 0 ? kDefaultStagedMin : tokens);
}

GKR_API int64_t gkr_get_insert_staged_min(void) { return g_staged_min.load(); }

GKR_API int64_t gkr_page_stride(int32_t record, int32_t block_size) {
    RecordRows r;
    if (!record_rows(record, &r) || !block_size_ok(record, block_size)) return -1;
    const int64_t need = static_cast<int64_t>(block_size) * record;
    return (need + r.align - 1) / r.align * r.align;
}

GKR_API gkr_status gkr_record_rows(int32_t record, int32_t* data_row_bytes,
                                   int32_t* scale_row_bytes, int32_t* page_align) {
    RecordRows r;
    if (!record_rows(record, &r)) return GKR_EUNSUPPORTED_RECORD;
    if (data_row_bytes) *data_row_bytes = r.data;
    if (scale_row_bytes) *scale_row_bytes = r.scale;
    if (page_align) *page_align = r.align;
    return GKR_OK;
}

}  // extern "C"

namespace {

// Checks shared by the insert entry points; fills `p` on success.  A GKR_OK status
// with p.num_tokens == 0 means there is nothing to launch.
gkr_status prepare_insert(const void* kv, int64_t num_tokens, void* k_cache,
                          const gkr_cache_desc* cache, const int64_t* slot_mapping,
                          const int64_t* positions, const float* cos_sin_cache, int64_t max_pos,
                          const float* fp8_scale, int32_t* err_flag,
                          const gkr_launch_opts* opts, gkr::InsertParams* p) {
    RecordRows rows;
    gkr_status st = check_cache(cache, &rows);
    if (st != GKR_OK) return st;
    Policy pol;
    st = resolve_policy(opts, &pol);
    if (st != GKR_OK) return st;
    if (num_tokens < 0) return GKR_EINVAL;
    p->num_tokens = num_tokens;
    if (num_tokens == 0) return GKR_OK;  // the descriptor is checked; nothing else is read
    if (max_pos <= 0 || max_pos > INT64_C(0x7FFFFFFF)) return GKR_EINVAL;
    if (!kv || !k_cache || !slot_mapping || !positions || !cos_sin_cache) return GKR_EINVAL;
    const bool fp8 = cache->record == 512;  // fp8_scale is read for fp8 rows only
    if (fp8 && !fp8_scale) return GKR_EINVAL;
    if (!aligned(kv, 16) || !aligned(k_cache, 16) || !aligned(cos_sin_cache, 16) ||
        !aligned(slot_mapping, 8) || !aligned(positions, 8) || !aligned(err_flag, 4) ||
        (fp8 && !aligned(fp8_scale, 4)))
        return GKR_EALIGN;
    p->kv = kv;
    p->cache = static_cast<uint8_t*>(k_cache);
    p->page_stride = cache->page_stride;
    p->block_size = cache->block_size;
    p->num_slots = static_cast<int32_t>(cache->num_pages * cache->block_size);
    p->slots = slot_mapping;
    p->positions = positions;
    p->csc = cos_sin_cache;
    p->max_pos = max_pos;
    p->ratio = 1;
    p->fp8_scale = cache->record == 512 ? fp8_scale : nullptr;
    p->err = err_flag;
    p->early_metadata = pol.early_metadata;
    p->pdl = pol.pdl;
    p->staged_min = pol.staged_min;
    p->stream_min = pol.stream_min;
    return GKR_OK;
}

cudaError_t launch_insert(int32_t record, const gkr::InsertParams& p, cudaStream_t stream) {
    switch (record) {
        case 528: return gkr::launch_insert_v41(p, stream);
        case 584: return gkr::launch_insert_v4(p, stream);
        case 512: return gkr::launch_insert_fp8(p, stream);
        default: return gkr::launch_insert_bf16(p, stream);
    }
}

cudaError_t launch_gather(int32_t record, const gkr::GatherParams& p, cudaStream_t stream) {
    switch (record) {
        case 528: return gkr::launch_gather_v41(p, stream);
        case 584: return gkr::launch_gather_v4(p, stream);
        case 512: return gkr::launch_gather_fp8(p, stream);
        default: return gkr::launch_gather_bf16(p, stream);
    }
}

}  // namespace

extern "C" {

GKR_API gkr_status gkr_kv_insert(const void* kv, int64_t num_tokens, void* k_cache,
                                 const gkr_cache_desc* cache, const int64_t* slot_mapping,
                                 const int64_t* positions, const float* cos_sin_cache,
                                 int64_t max_pos, const float* fp8_scale, int32_t* err_flag,
                                 const gkr_launch_opts* opts, cudaStream_t stream) {
    gkr::InsertParams p;
    const gkr_status st = prepare_insert(kv, num_tokens, k_cache, cache, slot_mapping,
                                         positions, cos_sin_cache, max_pos, fp8_scale, err_flag,
                                         opts, &p);
    if (st != GKR_OK || p.num_tokens == 0) return st;
    return cuda_status(launch_insert(cache->record, p, stream));
}

GKR_API gkr_status gkr_rope_quant_insert(const void* kv, int64_t num_tokens, void* k_cache,
                                         const gkr_cache_desc* cache,
                                         const int64_t* slot_mapping, const int64_t* positions,
                                         const float* cos_sin_cache, int64_t max_pos,
                                         int32_t compress_ratio, int32_t sanitize_nans,
                                         int32_t* err_flag, const gkr_launch_opts* opts,
                                         cudaStream_t stream) {
    if (compress_ratio < 1 || (sanitize_nans != 0 && sanitize_nans != 1)) return GKR_EINVAL;
    if (cache != nullptr && !packed(cache->record)) return GKR_EUNSUPPORTED_RECORD;
    gkr::InsertParams p;
    const gkr_status st = prepare_insert(kv, num_tokens, k_cache, cache, slot_mapping,
                                         positions, cos_sin_cache, max_pos, nullptr, err_flag,
                                         opts, &p);
    if (st != GKR_OK || p.num_tokens == 0) return st;
    p.ratio = compress_ratio;
    const bool san = sanitize_nans != 0;
    return cuda_status(cache->record == 528 ? gkr::launch_rope_quant_insert_v41(p, san, stream)
                                            : gkr::launch_rope_quant_insert_v4(p, san, stream));
}

GKR_API gkr_status gkr_kv_gather(const void* k_cache, const gkr_cache_desc* cache,
                                 const int32_t* indices, int64_t num_indices, void* out,
                                 const float* fp8_scale, int32_t* err_flag,
                                 const gkr_launch_opts* opts, cudaStream_t stream) {
    RecordRows rows;
    gkr_status st = check_cache(cache, &rows);
    if (st != GKR_OK) return st;
    Policy pol;
    st = resolve_policy(opts, &pol);
    if (st != GKR_OK) return st;
    if (num_indices < 0) return GKR_EINVAL;
    if (num_indices == 0) return GKR_OK;
    if (!k_cache || !indices || !out) return GKR_EINVAL;
    const bool fp8 = cache->record == 512;  // fp8_scale is read for fp8 rows only
    if (fp8 && !fp8_scale) return GKR_EINVAL;
    if (!aligned(k_cache, 16) || !aligned(out, 16) || !aligned(indices, 4) ||
        !aligned(err_flag, 4) || (fp8 && !aligned(fp8_scale, 4)))
        return GKR_EALIGN;

    gkr::GatherParams p;
    p.cache = static_cast<const uint8_t*>(k_cache);
    p.page_stride = cache->page_stride;
    p.block_size = cache->block_size;
    p.num_slots = static_cast<int32_t>(cache->num_pages * cache->block_size);
    p.indices = indices;
    p.num_indices = num_indices;
    p.out = out;
    p.fp8_scale = cache->record == 512 ? fp8_scale : nullptr;
    p.err = err_flag;
    p.early_metadata = pol.early_metadata;
    p.pdl = pol.pdl;
    return cuda_status(launch_gather(cache->record, p, stream));
}

GKR_API gkr_status gkr_qnorm_rope_kv_insert(const void* q_in, int32_t num_heads,
                                            int32_t num_heads_padded, void* q_out,
                                            const float* q_scale, float eps,
                                            int32_t apply_q_norm, const void* kv,
                                            int64_t num_tokens, void* k_cache,
                                            const gkr_cache_desc* cache,
                                            const int64_t* slot_mapping,
                                            const int64_t* positions,
                                            const float* cos_sin_cache, int64_t max_pos,
                                            const float* fp8_scale, int32_t* err_flag,
                                            const gkr_launch_opts* opts,
                                            cudaStream_t stream) {
    if (num_heads < 0 || num_heads_padded < num_heads || num_heads_padded > kMaxQHeads ||
        (apply_q_norm != 0 && apply_q_norm != 1) || !(eps >= 0.0f && eps <= 3.40282347e38f))
        return GKR_EINVAL;
    gkr::InsertParams p;
    const gkr_status st = prepare_insert(kv, num_tokens, k_cache, cache, slot_mapping,
                                         positions, cos_sin_cache, max_pos, fp8_scale, err_flag,
                                         opts, &p);
    if (st != GKR_OK || p.num_tokens == 0) return st;
    if (num_heads_padded == 0) return cuda_status(launch_insert(cache->record, p, stream));
    if ((num_heads > 0 && q_in == nullptr) || q_out == nullptr) return GKR_EINVAL;
    if ((num_heads > 0 && !aligned(q_in, 16)) || !aligned(q_out, 16) ||
        (q_scale != nullptr && !aligned(q_scale, 4)))
        return GKR_EALIGN;
    if (q_scale != nullptr && num_heads > 0) {   // e4m3 rows of 512 B must not overlap q_in
        const uintptr_t in0 = reinterpret_cast<uintptr_t>(q_in);
        const uintptr_t out0 = reinterpret_cast<uintptr_t>(q_out);
        const uintptr_t in1 = in0 + static_cast<uintptr_t>(p.num_tokens) * num_heads * 1024;
        const uintptr_t out1 = out0 + static_cast<uintptr_t>(p.num_tokens) * num_heads_padded * 512;
        if (out0 < in1 && in0 < out1) return GKR_EINVAL;
    }
    gkr::QSideParams qp;
    qp.q_in = q_in;
    qp.q_out = q_out;
    qp.q_scale = q_scale;
    qp.num_heads = num_heads;
    qp.num_heads_padded = num_heads_padded;
    qp.eps = eps;
    qp.apply_norm = apply_q_norm;
    return cuda_status(gkr::launch_qnorm_rope_kv_insert(cache->record, p, qp, stream));
}

GKR_API gkr_status gkr_sparse_logits(const void* q, int32_t num_heads, const void* k_cache,
                                     const gkr_cache_desc* cache, const int32_t* indices,
                                     int64_t num_queries, int64_t topk, float sm_scale,
                                     const float* fp8_scale, float* out, int32_t* err_flag,
                                     const gkr_launch_opts* opts, cudaStream_t stream) {
    RecordRows rows;
    gkr_status st = check_cache(cache, &rows);
    if (st != GKR_OK) return st;
    Policy pol;
    st = resolve_policy(opts, &pol);
    if (st != GKR_OK) return st;
    if (num_queries < 0 || topk < 0 || topk % 4 != 0 || topk > INT64_C(0x7FFFFFFF) ||
        num_heads < 1 || num_heads > gkr::logits_max_heads() ||
        !(sm_scale >= -3.40282347e38f && sm_scale <= 3.40282347e38f))
        return GKR_EINVAL;
    if (num_queries == 0 || topk == 0) return GKR_OK;
    if (!q || !k_cache || !indices || !out) return GKR_EINVAL;
    const bool fp8 = cache->record == 512;
    if (fp8 && !fp8_scale) return GKR_EINVAL;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(out, 16) || !aligned(indices, 4) ||
        !aligned(err_flag, 4) || (fp8 && !aligned(fp8_scale, 4)))
        return GKR_EALIGN;
    gkr::LogitsParams p;
    p.q = q;
    p.num_heads = num_heads;
    p.cache = static_cast<const uint8_t*>(k_cache);
    p.page_stride = cache->page_stride;
    p.block_size = cache->block_size;
    p.num_slots = static_cast<int32_t>(cache->num_pages * cache->block_size);
    p.indices = indices;
    p.num_queries = num_queries;
    p.topk = topk;
    const int64_t chunk = gkr::logits_chunk_keys(cache->record);
    p.chunks = (topk + chunk - 1) / chunk;
    if (num_queries > INT64_C(0x7FFFFFFF) / p.chunks) return GKR_EINVAL;   // grid < 2^31
    p.sm_scale = sm_scale;
    p.fp8_scale = fp8 ? fp8_scale : nullptr;
    p.out = out;
    p.err = err_flag;
    p.pdl = pol.pdl;
    return cuda_status(gkr::launch_sparse_logits(cache->record, p, stream));
}

GKR_API const char* gkr_status_string(gkr_status status) {
    switch (status) {
        case GKR_OK: return "ok";
        case GKR_EINVAL: return "invalid argument";
        case GKR_EUNSUPPORTED_RECORD:
            return "unsupported record width (expected 528 or 584, or 512 / 1024 for the fp8 "
                   "and bf16 caches; the compressed insert writes 528 / 584 only)";
        case GKR_EBAD_PAGE_GEOMETRY:
            return "bad page geometry (page_stride below block_size * record or not a "
                   "multiple of the record's page alignment: 576 for 584, else 512)";
        case GKR_EALIGN: return "misaligned pointer";
        case GKR_ECUDA: return "CUDA launch error";
    }
    return "unknown status";
}

GKR_API int32_t gkr_last_cuda_error(void) { return g_last_cuda_error; }

GKR_API int32_t gkr_version(void) { return 30200; }

}  // extern "C"
