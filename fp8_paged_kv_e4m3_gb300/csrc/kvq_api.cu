// kvq_api.cu -- the extern "C" entry points declared in include/kvq.h:
// argument validation (fail closed, before any launch), workspace layout,
// split-count choice, and the launches.
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "kvq.h"
#include "kvq_internal.h"

namespace kvq {

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static inline bool good_scale(float s) { return std::isfinite(s) && s > 0.0f; }

static inline size_t round256(size_t x) { return (x + 255u) & ~size_t(255u); }

WorkspaceLayout workspace_layout(int64_t rows_total, int32_t num_splits, int32_t head_dim)
{
    WorkspaceLayout w;
    const size_t units = size_t(rows_total) * size_t(num_splits);
    w.o_off = 0;
    w.m_off = round256(units * size_t(head_dim) * sizeof(float));
    w.l_off = w.m_off + round256(units * sizeof(float));
    w.total = w.l_off + round256(units * sizeof(float));
    return w;
}

int device_sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

// Fewest fixed-size splits that give every page and list entry a split.
static int64_t splits_to_cover(const kvq_attn_params *p)
{
    const int64_t sp = p->split_pages;
    int64_t s = (int64_t(p->max_pages_per_seq) + sp - 1) / sp;
    const int64_t t = (int64_t(p->max_topk) + 4 * sp - 1) / (4 * sp);
    return s > t ? s : t;
}

// shape checks shared by every attention entry point; KVQ_OK or an error
static int check_params(const kvq_attn_params *p)
{
    if (!p) return KVQ_ERR_INVALID_ARG;
    if (p->batch < 0 || p->q_len < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1 ||
        p->num_splits < 0 || p->max_pages_per_seq < 1 || p->max_topk < 0 || p->split_pages < 0)
        return KVQ_ERR_INVALID_ARG;
    if (p->flags & ~int32_t(KVQ_ATTN_BITCAST_DECODE | KVQ_ATTN_MMA_SYNC | KVQ_ATTN_FP8_QK | KVQ_ATTN_STRICT_ORDER |
                            KVQ_ATTN_LONGEST_FIRST))
        return KVQ_ERR_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
    if (!std::isfinite(p->sm_scale) || p->sm_scale < 0.0f) return KVQ_ERR_INVALID_ARG;
    if (p->head_dim != 64 && p->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
    if (p->q_len > 4) return KVQ_ERR_UNSUPPORTED;
    const int64_t rows = int64_t(p->num_q_heads / p->num_kv_heads) * p->q_len;
    if (rows > 64) return KVQ_ERR_UNSUPPORTED;
    if (p->batch > 65535 || p->num_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (int64_t(p->max_pages_per_seq) * 4 > INT32_MAX) return KVQ_ERR_UNSUPPORTED;
    // fixed-size splits must give every page and list entry a split
    if (p->split_pages > 0 && p->num_splits > 0 && splits_to_cover(p) > p->num_splits)
        return KVQ_ERR_INVALID_ARG;
    if (p->split_pages > 0 && p->num_splits == 0 && splits_to_cover(p) > 65535)
        return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

static int32_t resolve_splits(const kvq_attn_params *p)
{
    if (p->num_splits > 0) return p->num_splits;
    if (p->split_pages > 0) {
        const int64_t s = splits_to_cover(p);   // <= 65535 (checked)
        return int32_t(s < 1 ? 1 : s);
    }
    const int64_t pairs = int64_t(p->batch > 0 ? p->batch : 1) * p->num_kv_heads;
    const int64_t sms = device_sm_count();
    const int64_t rows = int64_t(p->num_q_heads / p->num_kv_heads) * p->q_len;
    const bool tc = p->head_dim == 128 && rows > 8 && rows <= 64 &&
                    !(p->flags & (KVQ_ATTN_MMA_SYNC | KVQ_ATTN_BITCAST_DECODE));
    int64_t s, cap;
    if (tc) {
        // tcgen05 kernel (two CTAs per SM): about three and a half waves of its
        // resident CTAs, so that long and short sequences pack; no split shorter
        // than 16 pages
        s = (sms * 6 + pairs - 1) / pairs;
        cap = (int64_t(p->max_pages_per_seq) + 15) / 16;
        if (p->max_topk > 0) cap = cap > (p->max_topk + 31) / 32 ? cap : (p->max_topk + 31) / 32;
    } else {
        // split kernel (up to four CTAs per SM): the most splits that fit the
        // (sequence, kv head) pairs in two waves of resident CTAs -- two and a
        // half for batches whose lengths vary (longest-first order), which pack
        // better in smaller pieces -- but no split shorter than 256 pages (or
        // 1024 list entries), whose fixed cost per CTA would dominate
        const int64_t slots = sms * 4;
        s = (p->flags & KVQ_ATTN_LONGEST_FIRST) ? (slots * 5 / 2) / pairs : (slots * 2) / pairs;
        cap = (int64_t(p->max_pages_per_seq) + 255) / 256;
        if (p->max_topk > 0) cap = cap > (p->max_topk + 1023) / 1024 ? cap : (p->max_topk + 1023) / 1024;
    }
    if (s > cap) s = cap;
    if (s < 1) s = 1;
    if (s > 1024) s = 1024;
    return int32_t(s);
}

struct AttnCall {
    bool e4m3;
    const void *q, *k_cache, *v_cache;
    int64_t num_pages;
    const int32_t *block_tables, *context_lens;
    float k_scale, v_scale;
    const int32_t *topk_idx, *topk_lens;
    float *workspace;
    size_t workspace_bytes;
    void *out;          // null for the partial-only entry points
    const kvq_attn_params *p;
    int32_t *err_flag;
    void *stream;
    const void *k_new = nullptr;   // fused step: this step's new rows (fp16), appended in the launch
    const void *v_new = nullptr;
};

static int run_attention(const AttnCall &c, bool with_combine)
{
    int st = check_params(c.p);
    if (st != KVQ_OK) return st;
    const kvq_attn_params &p = *c.p;
    if (p.batch == 0) return KVQ_OK;   // nothing to read or write
    if (!c.q || !c.k_cache || !c.v_cache || !c.block_tables || !c.context_lens)
        return KVQ_ERR_INVALID_ARG;
    if (with_combine && !c.out) return KVQ_ERR_INVALID_ARG;
    if (c.num_pages < 1) return KVQ_ERR_INVALID_ARG;
    if ((c.topk_idx == nullptr) != (c.topk_lens == nullptr)) return KVQ_ERR_INVALID_ARG;
    if (c.topk_idx && p.max_topk < 1) return KVQ_ERR_INVALID_ARG;
    if (c.e4m3 && (!good_scale(c.k_scale) || !good_scale(c.v_scale))) return KVQ_ERR_BAD_SCALE;
    // the FP8 scores exist on the tcgen05 kernel over E4M3 pools only
    if ((p.flags & KVQ_ATTN_FP8_QK) &&
        (!c.e4m3 || (p.flags & (KVQ_ATTN_BITCAST_DECODE | KVQ_ATTN_MMA_SYNC)) ||
         !tc_supported(p.head_dim, (p.num_q_heads / p.num_kv_heads) * p.q_len)))
        return KVQ_ERR_UNSUPPORTED;
    // the fused step appends this step's rows of each sequence; with a top-k
    // list another split's CTA could read them, so it has no top-k form
    if ((c.k_new == nullptr) != (c.v_new == nullptr)) return KVQ_ERR_INVALID_ARG;
    if (c.k_new && c.topk_idx) return KVQ_ERR_UNSUPPORTED;
    // its instances use the hardware E4M3 conversion and fp16 scores
    if (c.k_new && (p.flags & (KVQ_ATTN_BITCAST_DECODE | KVQ_ATTN_FP8_QK))) return KVQ_ERR_UNSUPPORTED;
    if (!aligned16(c.q) || !aligned16(c.k_cache) || !aligned16(c.v_cache) ||
        (c.out && !aligned16(c.out)) || !aligned16(c.workspace) || (c.k_new && !aligned16(c.k_new)) ||
        (c.v_new && !aligned16(c.v_new)))
        return KVQ_ERR_ALIGNMENT;
    const int32_t S = resolve_splits(&p);
    const int64_t rows_total = int64_t(p.batch) * p.num_q_heads * p.q_len;
    if (rows_total * S > INT32_MAX) return KVQ_ERR_UNSUPPORTED;   // partials are indexed in 32 bits
    const WorkspaceLayout wl = workspace_layout(rows_total, S, p.head_dim);
    if (!c.workspace || c.workspace_bytes < wl.total) return KVQ_ERR_WORKSPACE;
    if (p.batch == 0) return KVQ_OK;

    const int G = p.num_q_heads / p.num_kv_heads;
    const double sm = p.sm_scale > 0.0f ? double(p.sm_scale) : 1.0 / std::sqrt(double(p.head_dim));
    const double log2e = 1.4426950408889634;
    AttnArgs a;
    a.q = c.q;
    a.k_cache = c.k_cache;
    a.v_cache = c.v_cache;
    a.num_pages = c.num_pages;
    a.block_tables = c.block_tables;
    a.context_lens = c.context_lens;
    a.topk_idx = c.topk_idx;
    a.topk_lens = c.topk_lens;
    auto *ws = reinterpret_cast<uint8_t *>(c.workspace);
    a.ws_o = reinterpret_cast<float *>(ws + wl.o_off);
    a.ws_m = reinterpret_cast<float *>(ws + wl.m_off);
    a.ws_l = reinterpret_cast<float *>(ws + wl.l_off);
    a.err_flag = c.err_flag;
    a.batch = p.batch;
    a.q_len = p.q_len;
    a.num_q_heads = p.num_q_heads;
    a.num_kv_heads = p.num_kv_heads;
    a.group = G;
    a.rows = G * p.q_len;
    a.num_splits = S;
    a.split_pages = p.split_pages;
    a.max_pages = p.max_pages_per_seq;
    a.max_topk = c.topk_idx ? p.max_topk : 0;
    // hoisted per-layer scales (the kernel folds any decoder factor itself)
    const double kfold = c.e4m3 ? double(c.k_scale) : 1.0;
    const double vfold = c.e4m3 ? double(c.v_scale) : 1.0;
    a.qk_scale_log2 = float(sm * log2e * kfold);
    a.out_scale = float(vfold);
    a.bitcast_decode = (p.flags & KVQ_ATTN_BITCAST_DECODE) != 0;
    a.mma_sync = (p.flags & KVQ_ATTN_MMA_SYNC) != 0;
    a.fp8_qk = (p.flags & KVQ_ATTN_FP8_QK) != 0;
    a.early_pages = (p.flags & KVQ_ATTN_STRICT_ORDER) == 0;
    a.longest_first = (p.flags & KVQ_ATTN_LONGEST_FIRST) != 0;
    a.k_new = c.k_new;
    a.v_new = c.v_new;
    a.k_scale = c.e4m3 ? c.k_scale : 1.0f;
    a.v_scale = c.e4m3 ? c.v_scale : 1.0f;

    a.out = with_combine ? c.out : nullptr;

    cudaStream_t stream = static_cast<cudaStream_t>(c.stream);
    bool merged = false;
    if (launch_attention(c.e4m3, p.head_dim, a, stream, &merged) != cudaSuccess) return KVQ_ERR_CUDA;
    if (with_combine && !merged &&
        launch_combine(a.ws_o, a.ws_m, a.ws_l, c.out, p.batch, p.q_len, p.num_q_heads, p.head_dim, S,
                       stream) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

static int run_append(bool e4m3, const void *k_new, const void *v_new, const int32_t *slot_mapping,
                      int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim, void *k_cache,
                      void *v_cache, int64_t num_pages, float k_scale, float v_scale,
                      int32_t *err_flag, void *stream)
{
    if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || num_pages < 1)
        return KVQ_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return KVQ_ERR_UNSUPPORTED;
    if (e4m3 && (!good_scale(k_scale) || !good_scale(v_scale))) return KVQ_ERR_BAD_SCALE;
    if (num_tokens == 0) return KVQ_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return KVQ_ERR_ALIGNMENT;
    const cudaError_t e = launch_append(e4m3, k_new, v_new, slot_mapping, num_tokens, num_kv_heads,
                                        head_dim, k_cache, v_cache, num_pages, k_scale, v_scale,
                                        err_flag, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// shape checks of the prefill entry points; KVQ_OK or an error
static int check_prefill_params(const kvq_prefill_params *p)
{
    if (!p) return KVQ_ERR_INVALID_ARG;
    if (p->batch < 0 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->max_pages_per_seq < 1 ||
        p->max_q_len < 1 || p->total_q < 0 || p->flags != 0)
        return KVQ_ERR_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
    if (!std::isfinite(p->sm_scale) || p->sm_scale < 0.0f) return KVQ_ERR_INVALID_ARG;
    if (p->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
    if (p->batch > 65535 || p->num_q_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (int64_t(p->max_pages_per_seq) * 4 > INT32_MAX) return KVQ_ERR_UNSUPPORTED;
    if (p->max_q_len > p->max_pages_per_seq * int64_t(4)) return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

static int run_prefill(bool e4m3, const void *q, const void *k_cache, const void *v_cache,
                       int64_t num_pages, const int32_t *block_tables, const int32_t *context_lens,
                       const int32_t *q_start, float k_scale, float v_scale, void *workspace,
                       size_t workspace_bytes, void *out, const kvq_prefill_params *p,
                       int32_t *err_flag, void *stream)
{
    const int st = check_prefill_params(p);
    if (st != KVQ_OK) return st;
    if (p->batch == 0) return KVQ_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !q_start || !out)
        return KVQ_ERR_INVALID_ARG;
    if (num_pages < 1) return KVQ_ERR_INVALID_ARG;
    if (e4m3 && (!good_scale(k_scale) || !good_scale(v_scale))) return KVQ_ERR_BAD_SCALE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        !aligned16(workspace))
        return KVQ_ERR_ALIGNMENT;
    const int32_t max_tiles = prefill_max_tiles(p->max_pages_per_seq);
    if (!workspace || workspace_bytes < prefill_tiles_bytes(p->batch, p->num_kv_heads, max_tiles))
        return KVQ_ERR_WORKSPACE;
    const double sm = p->sm_scale > 0.0f ? double(p->sm_scale) : 1.0 / std::sqrt(double(p->head_dim));
    const double log2e = 1.4426950408889634;
    PrefillArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_pages = num_pages;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.q_start = q_start;
    a.out = out;
    a.tiles = static_cast<uint8_t *>(workspace);
    a.tile_mask = reinterpret_cast<uint32_t *>(a.tiles + prefill_mask_offset(p->batch, p->num_kv_heads, max_tiles));
    a.err_flag = err_flag;
    a.batch = p->batch;
    a.num_q_heads = p->num_q_heads;
    a.num_kv_heads = p->num_kv_heads;
    a.group = p->num_q_heads / p->num_kv_heads;
    a.max_pages = p->max_pages_per_seq;
    a.max_q_len = p->max_q_len;
    a.max_tiles = max_tiles;
    a.total_q = p->total_q;
    a.qk_scale_log2 = float(sm * log2e * (e4m3 ? double(k_scale) : 1.0));
    a.out_scale = e4m3 ? v_scale : 1.0f;
    return launch_prefill(e4m3, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

int kvq_version(void) { return KVQ_VERSION; }

const char *kvq_status_string(int status)
{
    switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_BAD_SCALE: return "K/V scale is not finite and positive";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    default: return "unknown status";
    }
}

int kvq_validate_scales(const float *k_scales, const float *v_scales, int32_t num_layers)
{
    if (!k_scales || !v_scales || num_layers < 1) return KVQ_ERR_INVALID_ARG;
    for (int32_t i = 0; i < num_layers; ++i)
        if (!good_scale(k_scales[i]) || !good_scale(v_scales[i])) return KVQ_ERR_BAD_SCALE;
    return KVQ_OK;
}

int kvq_amax_f16(const void *x, int64_t n, float *amax_out, void *stream)
{
    if (!x || !amax_out || n < 1) return KVQ_ERR_INVALID_ARG;
    return launch_amax(x, n, amax_out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVQ_OK
               : KVQ_ERR_CUDA;
}

float kvq_scale_from_amax(float amax)
{
    if (!std::isfinite(amax) || !(amax > 0.0f)) return 0.0f;
    return amax / 448.0f;   // one binary32 division, as the method defines
}

int kv_append_e4m3(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim, uint8_t *k_cache,
                   uint8_t *v_cache, int64_t num_pages, float k_scale, float v_scale,
                   int32_t *err_flag, void *stream)
{
    return run_append(true, k_new, v_new, slot_mapping, num_tokens, num_kv_heads, head_dim, k_cache,
                      v_cache, num_pages, k_scale, v_scale, err_flag, stream);
}

int kv_append_fp16(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim, void *k_cache,
                   void *v_cache, int64_t num_pages, int32_t *err_flag, void *stream)
{
    return run_append(false, k_new, v_new, slot_mapping, num_tokens, num_kv_heads, head_dim,
                      k_cache, v_cache, num_pages, 1.0f, 1.0f, err_flag, stream);
}

int32_t kvq_attn_num_splits(const kvq_attn_params *p)
{
    const int st = check_params(p);
    if (st != KVQ_OK) return st;
    return resolve_splits(p);
}

int32_t kvq_attn_launches(const kvq_attn_params *p, int32_t e4m3, int32_t fused_step)
{
    const int st = check_params(p);
    if (st != KVQ_OK) return st;
    if (p->batch == 0) return 0;
    const int32_t S = resolve_splits(p);
    const int rows = (p->num_q_heads / p->num_kv_heads) * p->q_len;
    const bool tc = !(p->flags & KVQ_ATTN_MMA_SYNC) && tc_supported(p->head_dim, rows);
    if (tc) return fused_step ? 3 : 2;   // [the append by block table,] attention, combine
    const bool bitcast = e4m3 && (p->flags & KVQ_ATTN_BITCAST_DECODE);
    const bool lpt = (p->flags & KVQ_ATTN_LONGEST_FIRST) != 0;
    return cluster_merge_applies(e4m3 != 0, p->batch, p->num_kv_heads, rows, S, bitcast, lpt) ? 1 : 2;
}

size_t kvq_attn_workspace_bytes(const kvq_attn_params *p)
{
    if (check_params(p) != KVQ_OK) return 0;
    const int64_t rows = int64_t(p->batch) * p->num_q_heads * p->q_len;
    return workspace_layout(rows, resolve_splits(p), p->head_dim).total;
}

int paged_decode_attn_e4m3(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                           int64_t num_pages, const int32_t *block_tables,
                           const int32_t *context_lens, float k_scale, float v_scale,
                           const int32_t *topk_idx, const int32_t *topk_lens, float *workspace,
                           size_t workspace_bytes, void *out, const kvq_attn_params *p,
                           int32_t *err_flag, void *stream)
{
    const AttnCall c{true, q, k_cache, v_cache, num_pages, block_tables, context_lens, k_scale,
                     v_scale, topk_idx, topk_lens, workspace, workspace_bytes, out, p, err_flag,
                     stream};
    return run_attention(c, true);
}

int paged_decode_attn_fp16(const void *q, const void *k_cache, const void *v_cache,
                           int64_t num_pages, const int32_t *block_tables,
                           const int32_t *context_lens, const int32_t *topk_idx,
                           const int32_t *topk_lens, float *workspace, size_t workspace_bytes,
                           void *out, const kvq_attn_params *p, int32_t *err_flag, void *stream)
{
    const AttnCall c{false, q, k_cache, v_cache, num_pages, block_tables, context_lens, 1.0f, 1.0f,
                     topk_idx, topk_lens, workspace, workspace_bytes, out, p, err_flag, stream};
    return run_attention(c, true);
}

int paged_decode_attn_e4m3_partial(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                   int64_t num_pages, const int32_t *block_tables,
                                   const int32_t *context_lens, float k_scale, float v_scale,
                                   const int32_t *topk_idx, const int32_t *topk_lens,
                                   float *workspace, size_t workspace_bytes,
                                   const kvq_attn_params *p, int32_t *err_flag, void *stream)
{
    const AttnCall c{true, q, k_cache, v_cache, num_pages, block_tables, context_lens, k_scale,
                     v_scale, topk_idx, topk_lens, workspace, workspace_bytes, nullptr, p,
                     err_flag, stream};
    return run_attention(c, false);
}

int paged_decode_attn_fp16_partial(const void *q, const void *k_cache, const void *v_cache,
                                   int64_t num_pages, const int32_t *block_tables,
                                   const int32_t *context_lens, const int32_t *topk_idx,
                                   const int32_t *topk_lens, float *workspace,
                                   size_t workspace_bytes, const kvq_attn_params *p,
                                   int32_t *err_flag, void *stream)
{
    const AttnCall c{false, q, k_cache, v_cache, num_pages, block_tables, context_lens, 1.0f, 1.0f,
                     topk_idx, topk_lens, workspace, workspace_bytes, nullptr, p, err_flag, stream};
    return run_attention(c, false);
}

int paged_decode_step_e4m3(const void *q, const void *k_new, const void *v_new, uint8_t *k_cache,
                           uint8_t *v_cache, int64_t num_pages, const int32_t *block_tables,
                           const int32_t *context_lens, float k_scale, float v_scale, float *workspace,
                           size_t workspace_bytes, void *out, const kvq_attn_params *p, int32_t *err_flag,
                           void *stream)
{
    if (!k_new || !v_new) return KVQ_ERR_INVALID_ARG;
    AttnCall c{true, q, k_cache, v_cache, num_pages, block_tables, context_lens, k_scale, v_scale,
               nullptr, nullptr, workspace, workspace_bytes, out, p, err_flag, stream};
    c.k_new = k_new;
    c.v_new = v_new;
    return run_attention(c, true);
}

int paged_decode_step_fp16(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           int64_t num_pages, const int32_t *block_tables, const int32_t *context_lens,
                           float *workspace, size_t workspace_bytes, void *out, const kvq_attn_params *p,
                           int32_t *err_flag, void *stream)
{
    if (!k_new || !v_new) return KVQ_ERR_INVALID_ARG;
    AttnCall c{false, q, k_cache, v_cache, num_pages, block_tables, context_lens, 1.0f, 1.0f,
               nullptr, nullptr, workspace, workspace_bytes, out, p, err_flag, stream};
    c.k_new = k_new;
    c.v_new = v_new;
    return run_attention(c, true);
}

int kvq_lse_combine(const float *workspace, size_t workspace_bytes, void *out,
                    const kvq_attn_params *p, void *stream)
{
    const int st = check_params(p);
    if (st != KVQ_OK) return st;
    if (!workspace || !out) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(workspace) || !aligned16(out)) return KVQ_ERR_ALIGNMENT;
    const int32_t S = resolve_splits(p);
    const int64_t rows = int64_t(p->batch) * p->num_q_heads * p->q_len;
    const WorkspaceLayout wl = workspace_layout(rows, S, p->head_dim);
    if (workspace_bytes < wl.total) return KVQ_ERR_WORKSPACE;
    const auto *ws = reinterpret_cast<const uint8_t *>(workspace);
    const cudaError_t e = launch_combine(reinterpret_cast<const float *>(ws + wl.o_off),
                                         reinterpret_cast<const float *>(ws + wl.m_off),
                                         reinterpret_cast<const float *>(ws + wl.l_off), out,
                                         p->batch, p->q_len, p->num_q_heads, p->head_dim, S,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

size_t kvq_prefill_workspace_bytes(const kvq_prefill_params *p)
{
    if (check_prefill_params(p) != KVQ_OK) return 0;
    return prefill_tiles_bytes(p->batch, p->num_kv_heads, prefill_max_tiles(p->max_pages_per_seq));
}

int paged_prefill_attn_e4m3(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                            int64_t num_pages, const int32_t *block_tables, const int32_t *context_lens,
                            const int32_t *q_start, float k_scale, float v_scale, void *workspace,
                            size_t workspace_bytes, void *out, const kvq_prefill_params *p,
                            int32_t *err_flag, void *stream)
{
    return run_prefill(true, q, k_cache, v_cache, num_pages, block_tables, context_lens, q_start, k_scale,
                       v_scale, workspace, workspace_bytes, out, p, err_flag, stream);
}

int paged_prefill_attn_fp16(const void *q, const void *k_cache, const void *v_cache, int64_t num_pages,
                            const int32_t *block_tables, const int32_t *context_lens, const int32_t *q_start,
                            void *workspace, size_t workspace_bytes, void *out, const kvq_prefill_params *p,
                            int32_t *err_flag, void *stream)
{
    return run_prefill(false, q, k_cache, v_cache, num_pages, block_tables, context_lens, q_start, 1.0f, 1.0f,
                       workspace, workspace_bytes, out, p, err_flag, stream);
}

}  // extern "C"
