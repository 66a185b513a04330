/*
 * kvq.h -- C ABI of the GB300 (sm_103a) calibrated E4M3 paged KV cache.
 *
 * The operations follow three pull-request pages that describe the method:
 *   [P1] "[Model][SM70] Calibrated E4M3 KV cache for Qwen4Exp QSA with MTP"
 *   [P2] "[Model][SM70][FP8] Integrate calibrated E4M3 QSA KV capacity path"
 *   [P3] "[Experiment][SM70] Qualify E4M3 KV with MTP3"
 * Each declaration below cites the section that defines what it computes.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers marked "device" are CUDA device (or managed) memory on the
 *    current device; pointers marked "host" are ordinary host memory.  The
 *    caller owns every buffer.  The library allocates nothing, keeps no
 *    pointer after a call returns and holds no global state, so calls are
 *    reentrant (the one exception, paged_decode_attn_e4m3_noalloc at the
 *    end of this file, uses a scratch buffer the library keeps itself).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every GPU call is asynchronous and stream-ordered; none
 *    synchronises the host, so the calls can be captured in a CUDA graph.
 *  - The kernels use programmatic dependent launch: a call's kernel may
 *    start while the preceding kernel in the stream still runs, when that
 *    kernel allows it (griddepcontrol.launch_dependents; the library's own
 *    kernels do), and waits for it before reading what it may write.  One
 *    relaxation, on the decode attention calls without a top-k list (unless
 *    KVQ_ATTN_STRICT_ORDER is set): block tables, context lengths and the
 *    cache pages that hold only positions below L - q_len may be read
 *    before that wait.  The append of the step writes only positions
 *    L - q_len and later, so append then attention is safe; a preceding
 *    kernel of the caller's that allows early launch must not write those
 *    inputs, or the call must set KVQ_ATTN_STRICT_ORDER.  Kernels that do
 *    not allow early launch, and copies, order fully as usual.
 *  - Return value: KVQ_OK, or a negative kvq_status.  Errors that the host
 *    can see (bad sizes, bad scales, misaligned pointers, a short workspace)
 *    are returned BEFORE anything is launched: the call fails closed and
 *    leaves every buffer untouched.  A launch failure returns KVQ_ERR_CUDA.
 *  - `err_flag` (device int32, nullable): errors only the GPU can see -- an
 *    out-of-range block-table entry, slot or top-k index, or an invalid
 *    context length -- OR a KVQ_DEV_* bit into *err_flag; the offending
 *    token is skipped (treated as absent), nothing faults and nothing
 *    traps.  The caller clears the flag.
 *  - Page size is 4 tokens ("page4" routes, [P2] Changes).  A K or V pool is
 *    [num_pages][num_kv_heads][4][head_dim]: one page of one KV head is
 *    4 * head_dim contiguous elements.  E4M3 pools hold one byte per
 *    element, fp16 pools two.
 *  - head_dim is 64 or 128; query rows per KV head (q_len * Hq / Hkv) are
 *    at most 64; q_len is 1 .. 4 (decode, or MTP verify with 1 + 3 drafts,
 *    [P1] Purpose).  Other shapes return KVQ_ERR_UNSUPPORTED, and so does a
 *    call whose split partials (batch * Hq * q_len * splits) exceed INT32_MAX.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_PAGE_SIZE 4
#define KVQ_VERSION 1

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = -1,  /* null pointer, negative or inconsistent size   */
    KVQ_ERR_BAD_SCALE = -2,    /* a K or V scale that is not finite and > 0      */
    KVQ_ERR_WORKSPACE = -3,    /* workspace missing or smaller than required     */
    KVQ_ERR_UNSUPPORTED = -4,  /* head_dim / q_len / group shape not supported   */
    KVQ_ERR_CUDA = -5,         /* a CUDA launch or runtime call failed           */
    KVQ_ERR_ALIGNMENT = -6     /* a pointer is not 16-byte aligned               */
} kvq_status;

/* bits OR-ed into *err_flag by the kernels */
enum {
    KVQ_DEV_BAD_PAGE = 1,   /* block-table entry outside [0, num_pages): page skipped   */
    KVQ_DEV_BAD_SLOT = 2,   /* append slot beyond the pool: token not written           */
    KVQ_DEV_BAD_TOPK = 4,   /* top-k index outside [0, context_len): entry skipped      */
    KVQ_DEV_BAD_LEN = 8,    /* context_len < q_len or > 4 * max_pages_per_seq: row = 0   */
    KVQ_DEV_TIMEOUT = 16    /* an internal pipeline wait gave up (~2 s): results invalid;
                               the CTA that gave up drained its copies, wrote its split
                               partials as empty (m = -inf, l = 0) and exited            */
};

/* Library version (KVQ_VERSION) and a static string for a status code. */
int kvq_version(void);
const char *kvq_status_string(int status);

/* ------------------------------------------------------------------------
 * Scale gate.  [P2] Changes: the E4M3 mode starts only when every layer
 * (24 of 24 on the pages' model) has a K and a V scale that is finite and
 * positive; a missing or partial set stops start-up.  [P2] Validation
 * boundary: a scale is never replaced by a default such as 1.
 *   k_scales, v_scales : host float[num_layers]
 * Returns KVQ_OK when every entry is finite and > 0, KVQ_ERR_BAD_SCALE when
 * any is not, KVQ_ERR_INVALID_ARG for a null array or num_layers < 1.
 * There is no default: a caller without calibrated scales cannot proceed.
 */
int kvq_validate_scales(const float *k_scales, const float *v_scales, int32_t num_layers);

/* ------------------------------------------------------------------------
 * Calibration.  [P2] Changes: the scales are produced offline by a
 * calibration pass; the calibrated scale is amax / 448 (448 = largest
 * finite E4M3 value) for one layer's K or V, amax being the largest |x| of
 * a calibration draw.
 *
 * kvq_amax_f16: amax over n fp16 values.
 *   x        : device fp16[n] (any alignment)
 *   amax_out : device float[1]; overwritten (not accumulated) with max |x|
 *              (NaN if any input is NaN, +inf if any is infinite)
 *   Launches one reduction kernel on `stream`.
 * kvq_scale_from_amax: host helper, returns amax / 448 in binary32, or 0
 *   (an invalid scale that kvq_validate_scales refuses) when amax is not
 *   finite and > 0.
 */
int kvq_amax_f16(const void *x, int64_t n, float *amax_out, void *stream);
float kvq_scale_from_amax(float amax);

/* ------------------------------------------------------------------------
 * Quantise-on-append.  [P2] Changes: only the main K/V cache is stored in
 * calibrated E4M3, in page-4 pools; [P2] Changes "mixed catch-up/decode
 * batches" append prefill chunks and decode tokens alike.
 *
 * For every token t with slot_mapping[t] >= 0, page = slot / 4 and
 * offset = slot % 4, and for every head g and channel d:
 *     k_cache[page][g][offset][d] = E4M3(fp32(k_new[t][g][d]) / k_scale)
 *     v_cache[page][g][offset][d] = E4M3(fp32(v_new[t][g][d]) / v_scale)
 * where "/" is one IEEE binary32 division and E4M3() rounds to nearest
 * even, saturates finite overflow to +-448 and maps NaN to a NaN code.
 *   k_new, v_new   : device fp16 [num_tokens][num_kv_heads][head_dim], 16-B aligned
 *   slot_mapping   : device int32 [num_tokens]; -1 = skip the token;
 *                    slots >= 4 * num_pages set KVQ_DEV_BAD_SLOT and are skipped
 *   k_cache, v_cache : device uint8 pools (see conventions), 16-B aligned
 *   k_scale, v_scale : the layer's calibrated scales (finite, > 0)
 * Bad scale -> KVQ_ERR_BAD_SCALE; head_dim not a multiple of 8 ->
 * KVQ_ERR_UNSUPPORTED.  num_tokens == 0 is a no-op.
 */
int kv_append_e4m3(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                   uint8_t *k_cache, uint8_t *v_cache, int64_t num_pages,
                   float k_scale, float v_scale, int32_t *err_flag, void *stream);

/* fp16-KV twin ([P1] Validation: the comparison arm differs only in the KV
 * cache dtype): the same slots, values copied unchanged into fp16 pools. */
int kv_append_fp16(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                   void *k_cache, void *v_cache, int64_t num_pages,
                   int32_t *err_flag, void *stream);

/* ------------------------------------------------------------------------
 * Decode / MTP-verify attention over the paged cache.
 *
 * For sequence b with context length L (which INCLUDES the q_len tokens
 * appended this step), query position i (0 <= i < q_len) and query head h,
 * KV head g = h / (Hq / Hkv) (contiguous grouping, "grouped page4" route,
 * [P2] Changes):
 *     keys  J = { j : 0 <= j <= L - q_len + i }                     (dense)
 *        or J = { j in topk_idx[b][g][0 : topk_lens[b]] : j <= L - q_len + i }
 *     s_j   = sm_scale * sum_d q[b][i][h][d] * K^_j[d]
 *     out   = sum_{j in J} exp(s_j - max s) V^_j / sum_{j in J} exp(s_j - max s)
 * with K^ = decode(k byte) * k_scale and V^ = decode(v byte) * v_scale
 * (E4M3), or the fp16 values themselves (fp16 twin).  The window of q_len
 * rows is causal inside itself: MTP3 verifies one target token and three
 * drafts in one pass ([P1] Purpose).  An empty J gives a zero row.
 *
 * Split-K: the work of each (b, g) is cut into num_splits parts whose
 * partial results go to an FP32 workspace ([P1] Status and history and
 * [P3] Problem: the page-4 route's temporary output must be FP32) and are
 * merged by a log-sum-exp combine.  Split s covers
 *   split_pages == 0 (equal division of each sequence):
 *     logical pages [s*c, (s+1)*c), c = ceil(ceil(L/4) / num_splits), or
 *     top-k list entries [s*c, (s+1)*c), c = ceil(topk_lens[b] / num_splits);
 *   split_pages  > 0 (fixed-size splits, for batches of mixed lengths):
 *     logical pages [s*split_pages, (s+1)*split_pages), or top-k list entries
 *     [s*4*split_pages, (s+1)*4*split_pages); splits past a sequence's end
 *     are empty, so a short sequence uses few splits and a long one many,
 *     and every split does about the same work.
 * The pages leave the partition open; any partition gives the same result
 * up to rounding.
 */
typedef struct {
    int32_t batch;             /* B: sequences in the call                            */
    int32_t q_len;             /* 1 (decode) .. 4 (MTP3 verify)                       */
    int32_t num_q_heads;       /* Hq                                                   */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0                                   */
    int32_t head_dim;          /* 64 or 128                                            */
    int32_t num_splits;        /* S >= 1, or 0 = let the library choose (see below)    */
    int32_t max_pages_per_seq; /* row stride of block_tables                           */
    int32_t max_topk;          /* row length of topk_idx; 0 when no top-k list is used */
    float sm_scale;            /* softmax temperature; 0 = 1/sqrt(head_dim)            */
    int32_t split_pages;       /* 0 = equal division; > 0 = pages per split (above).
                                  Needs num_splits * split_pages >= max_pages_per_seq
                                  and num_splits * 4 * split_pages >= max_topk, so
                                  that every page and list entry has a split;
                                  otherwise the call returns KVQ_ERR_INVALID_ARG */
    int32_t flags;             /* KVQ_ATTN_* bits below; other bits are refused     */
} kvq_attn_params;

/* E4M3 decoder of the attention kernels.  Default: the hardware conversion
 * (cvt.rn.f16x2.e4m3x2), exact.  KVQ_ATTN_BITCAST_DECODE: the bitcast decoder
 * of [P2] Changes (the E4M3 sign, exponent and mantissa bits placed into the
 * fp16 bit pattern, which is the value times 2^-8, exact; the 2^8 is folded
 * into the hoisted scales).  Both decode every byte to the same value up to
 * that power of two.  On the mma.sync kernel the outputs are identical; on
 * the tcgen05 kernel the bitcast decoder pairs channels 4i, 4i + 2 and
 * 4i + 1, 4i + 3 (the query tile takes the same order), so Q K^T sums its
 * products in another order and the outputs agree within rounding.  Ignored
 * for the fp16 twins. */
#define KVQ_ATTN_BITCAST_DECODE 1

/* Kernel choice for more than 8 query rows per KV head (G * q_len > 8, e.g.
 * MTP verify) at head_dim 128: by default the tcgen05 kernel (tensor-memory
 * accumulators, M = 128 tokens per MMA); KVQ_ATTN_MMA_SYNC keeps such calls
 * on the mma.sync kernel that serves every shape.  Both compute the same
 * partials up to rounding.  Either E4M3 decoder runs on either kernel. */
#define KVQ_ATTN_MMA_SYNC 2

/* FP8 scores (E4M3 pools, the tcgen05 kernel's shapes: head_dim 128 and
 * 8 < G * q_len <= 64; other calls with this bit, or with it together with
 * KVQ_ATTN_BITCAST_DECODE or KVQ_ATTN_MMA_SYNC, return KVQ_ERR_UNSUPPORTED
 * before any launch).  Not on the pages, which keep q in fp16: the query
 * rows of each (sequence, kv head) are quantised to E4M3 with one scale
 * amax / 448 over those rows (1 for an all-zero group; binary32 division,
 * round to nearest even, finite overflow saturated, like a cache element),
 * and q k^T is computed on E4M3 x E4M3 tensor-core instructions with the
 * query scale folded into the hoisted score scale.  P V, the workspace and
 * the combine are unchanged.  The result is the attention of the quantised
 * query, which is not the fp16-query attention: where q and k share large
 * outlier channels the scores are large and the query's rounding moves
 * them visibly. */
#define KVQ_ATTN_FP8_QK 4

/* Strict ordering: the attention kernel reads no input before the preceding
 * kernel in the stream has completed (see the conventions at the top).
 * Without it, decode attention without a top-k list starts copying the
 * cache pages of positions below L - q_len while the preceding kernel (for
 * example this step's append) finishes. */
#define KVQ_ATTN_STRICT_ORDER 8

/* Longest first: the split kernel's CTAs take the sequences in decreasing
 * order of work (context length, or top-k list length) instead of index
 * order, so that on a grid of several waves the long sequences start first
 * and the short ones fill the gaps at the end.  Each CTA then classifies
 * every sequence in its prologue, which costs a little when all lengths are
 * equal (1 to 3 us per call on the uniform workloads measured) and pays when
 * they vary (the mixed-length batch: step 137 -> 120 us).  A scheduling
 * choice only: the outputs are bit-identical.  The tcgen05 kernel always
 * orders its sequences this way. */
#define KVQ_ATTN_LONGEST_FIRST 32

/* The split count a call with these parameters uses: p->num_splits if > 0;
 * else, with split_pages > 0, the fewest splits that cover max_pages_per_seq
 * pages and max_topk list entries; else a count chosen from the shape and
 * the current device's SM count.
 * Returns a value >= 1, or a negative kvq_status for invalid parameters. */
int32_t kvq_attn_num_splits(const kvq_attn_params *p);

/* The number of kernels paged_decode_attn_e4m3 (e4m3 != 0) or _fp16 launches
 * with these parameters on the current device -- fused_step != 0: the
 * paged_decode_step_* call -- or a negative kvq_status for invalid
 * parameters.  Host only: it launches nothing.  The full call launches the
 * attention kernel and the log-sum-exp combine, except that with up to 8
 * query rows per KV head and up to 8 splits, on a grid resident in one wave
 * (the hardware decoder, index order), the splits of each (sequence, KV head)
 * run as one thread-block cluster and merge into `out` themselves (the
 * combine's arithmetic: the same bits), so one kernel.  On the tcgen05
 * kernel's shapes the fused step launches its append first. */
int32_t kvq_attn_launches(const kvq_attn_params *p, int32_t e4m3, int32_t fused_step);

/* Bytes of FP32 workspace the call needs, 0 for invalid parameters.
 * Workspace layout (float32, each part starting on a 256-byte boundary):
 *   tmp_out [B][Hq][q_len][S][head_dim]  partial output of each split,
 *                                        normalised by its own l
 *   tmp_max [B][Hq][q_len][S]            m = max score of the split
 *                                        (natural-log units, -inf if empty)
 *   tmp_sum [B][Hq][q_len][S]            l = sum of exp(s - m) (0 if empty)
 * Entries of empty splits (l == 0) leave tmp_out unwritten. */
size_t kvq_attn_workspace_bytes(const kvq_attn_params *p);

/* Full decode / verify attention: split partials, then the combine.
 *   q            : device fp16 [B][q_len][Hq][head_dim], 16-B aligned
 *   k_cache, v_cache : device pools (uint8 E4M3), 16-B aligned
 *   num_pages    : pool size P
 *   block_tables : device int32 [B][max_pages_per_seq]; entries past the
 *                  sequence's last page are not read
 *   context_lens : device int32 [B] (includes this step's q_len tokens)
 *   k_scale, v_scale : the layer's calibrated scales (finite, > 0)
 *   topk_idx     : device int32 [B][Hkv][max_topk] or NULL; per (sequence,
 *                  KV head) token positions, ascending ([P2] Changes: the
 *                  shared QSA top-k index workspace)
 *   topk_lens    : device int32 [B] or NULL; 0 = dense for that sequence
 *   workspace    : device float32, >= kvq_attn_workspace_bytes(p) bytes,
 *                  256-B aligned.  FP32 by contract: there is no fp16 form.
 *   out          : device fp16 [B][q_len][Hq][head_dim], 16-B aligned
 * Launches two kernels (attention, combine) on `stream`, or one (see
 * kvq_attn_launches).
 */
int paged_decode_attn_e4m3(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                           int64_t num_pages, const int32_t *block_tables,
                           const int32_t *context_lens, float k_scale, float v_scale,
                           const int32_t *topk_idx, const int32_t *topk_lens,
                           float *workspace, size_t workspace_bytes, void *out,
                           const kvq_attn_params *p, int32_t *err_flag, void *stream);

/* fp16-KV twin: the same computation over fp16 pools, without scales. */
int paged_decode_attn_fp16(const void *q, const void *k_cache, const void *v_cache,
                           int64_t num_pages, const int32_t *block_tables,
                           const int32_t *context_lens,
                           const int32_t *topk_idx, const int32_t *topk_lens,
                           float *workspace, size_t workspace_bytes, void *out,
                           const kvq_attn_params *p, int32_t *err_flag, void *stream);

/* Fused decode / verify step: this step's append and the attention over the
 * updated cache, in fewer launches than kv_append_* followed by
 * paged_decode_attn_*.  On the split kernel's shapes the attention launch
 * appends the new rows itself (and where the cluster merge applies, see
 * kvq_attn_launches, it also merges the partials: one kernel); on the
 * tcgen05 kernel's shapes a small append by block table precedes the
 * attention.  [P2] Changes: the main K/V cache is written in calibrated E4M3
 * as tokens are appended, and decode reads it through the page4 route.
 *
 * Sequence b appends its q_len new tokens at positions L - q_len + i
 * (0 <= i < q_len), L = context_lens[b] (which includes them), into the page
 * slots its block table names:
 *     slot = block_tables[b][pos / 4] * 4 + pos % 4,  pos = L - q_len + i
 *     k_cache[slot / 4][g][slot % 4][d] = E4M3(fp32(k_new[b][i][g][d]) / k_scale)
 * (v likewise), exactly as kv_append_e4m3 with that slot mapping would, and
 * the attention is then the one defined above over the cache including them.
 * Pools and outputs are identical to the two separate calls.
 *   k_new, v_new : device fp16 [B][q_len][Hkv][head_dim], 16-B aligned
 *   k_cache, v_cache : written (the new rows) and read
 * Every other argument as for paged_decode_attn_e4m3.  There is no top-k
 * form: with a list, tokens of one sequence may be read by several of its
 * split CTAs, so the append must complete first (use the separate calls).
 * The fused kernels decode with the hardware conversion and compute fp16
 * scores: KVQ_ATTN_BITCAST_DECODE and KVQ_ATTN_FP8_QK return
 * KVQ_ERR_UNSUPPORTED before any launch; KVQ_ATTN_LONGEST_FIRST does not
 * reorder the split kernel's fused instances (a scheduling choice only).
 * A sequence with an invalid context length (KVQ_DEV_BAD_LEN) appends
 * nothing; a new row whose block-table entry is out of range is skipped
 * (KVQ_DEV_BAD_PAGE).  The new tokens' pages must belong to their sequence
 * alone (no other sequence in the call may map them), as for any append.
 * The preceding kernel may write k_new and v_new: they are read after the
 * dependency wait.  Early reads (see the conventions) cover only the pages
 * holding positions below L - q_len - 4, so that the previous step's fused
 * call, which may run as the directly preceding kernel and wrote its up to
 * 4 rows just below this step's window, is never read early.  Launches the
 * kernels kvq_attn_launches(p, e4m3, 1) counts. */
int paged_decode_step_e4m3(const void *q, const void *k_new, const void *v_new,
                           uint8_t *k_cache, uint8_t *v_cache, int64_t num_pages,
                           const int32_t *block_tables, const int32_t *context_lens,
                           float k_scale, float v_scale, float *workspace,
                           size_t workspace_bytes, void *out, const kvq_attn_params *p,
                           int32_t *err_flag, void *stream);

/* fp16-KV twin: the new rows are copied unchanged into fp16 pools. */
int paged_decode_step_fp16(const void *q, const void *k_new, const void *v_new,
                           void *k_cache, void *v_cache, int64_t num_pages,
                           const int32_t *block_tables, const int32_t *context_lens,
                           float *workspace, size_t workspace_bytes, void *out,
                           const kvq_attn_params *p, int32_t *err_flag, void *stream);

/* The two halves of the calls above, for callers that merge partials from
 * several sources (for example partials computed on different devices over
 * different token ranges) or time the halves separately.
 * *_partial: the split-K attention kernel alone; fills the workspace.
 * kvq_lse_combine: the combine alone; reads the workspace, writes `out`:
 *     M = max_s m_s, w_s = l_s * exp(m_s - M),
 *     out = sum_s w_s tmp_out_s / sum_s w_s  (0 when every l_s == 0). */
int paged_decode_attn_e4m3_partial(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                   int64_t num_pages, const int32_t *block_tables,
                                   const int32_t *context_lens, float k_scale, float v_scale,
                                   const int32_t *topk_idx, const int32_t *topk_lens,
                                   float *workspace, size_t workspace_bytes,
                                   const kvq_attn_params *p, int32_t *err_flag, void *stream);
int paged_decode_attn_fp16_partial(const void *q, const void *k_cache, const void *v_cache,
                                   int64_t num_pages, const int32_t *block_tables,
                                   const int32_t *context_lens,
                                   const int32_t *topk_idx, const int32_t *topk_lens,
                                   float *workspace, size_t workspace_bytes,
                                   const kvq_attn_params *p, int32_t *err_flag, void *stream);
int kvq_lse_combine(const float *workspace, size_t workspace_bytes, void *out,
                    const kvq_attn_params *p, void *stream);

/* ------------------------------------------------------------------------
 * Chunked-prefill attention over the paged cache.  [P2] Changes: mixed
 * catch-up/decode batches append prefill chunks to the same page-4 cache;
 * this call attends those chunks.  It is the attention defined above with
 * q_len = the chunk length: sequence b has context length L_b, which
 * includes its chunk of n_b = q_start[b+1] - q_start[b] query tokens, the
 * last n_b positions of the context.  Query token i (0 <= i < n_b) sits at
 * position L_b - n_b + i and, for query head h (KV head h / (Hq / Hkv)),
 * attends the dense keys 0 .. L_b - n_b + i (causal inside the chunk).
 * There is no top-k form and no split partial: the output is written
 * directly.
 *   q            : device fp16 [q_start[B]][Hq][head_dim], the chunks packed
 *                  in sequence order, 16-B aligned
 *   k_cache, v_cache, num_pages, block_tables, k_scale, v_scale : as for
 *                  paged_decode_attn_e4m3
 *   context_lens : device int32 [B] (includes the chunk)
 *   q_start      : device int32 [B + 1], q_start[0] = 0, non-decreasing.
 *                  n_b = 0 leaves the sequence out.  A sequence with
 *                  n_b > max_q_len, n_b > L_b, n_b < 0, L_b outside
 *                  [0, 4 * max_pages_per_seq] or rows outside
 *                  [0, total_q) sets KVQ_DEV_BAD_LEN and its output rows
 *                  are not written.
 *   workspace    : device memory of at least kvq_prefill_workspace_bytes(p)
 *                  bytes, 16-B aligned: the call writes the attended keys and
 *                  values there as fp16 tiles (the E4M3 bytes decoded exactly,
 *                  scales not applied) before it reads them back.
 *   out          : device fp16 [q_start[B]][Hq][head_dim], 16-B aligned
 * head_dim must be 128 (otherwise KVQ_ERR_UNSUPPORTED).  A block-table
 * entry outside the pool sets KVQ_DEV_BAD_PAGE and that key is left out.
 * Launches two kernels on `stream`: the gather/decode of the pages into the
 * workspace, then the attention.
 */
typedef struct {
    int32_t batch;             /* B                                                   */
    int32_t num_q_heads;       /* Hq                                                  */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0                                  */
    int32_t head_dim;          /* 128                                                 */
    int32_t max_pages_per_seq; /* row stride of block_tables                          */
    int32_t max_q_len;         /* bound on every n_b (<= 4 * max_pages_per_seq)        */
    int32_t total_q;           /* rows of q and out; every chunk must lie inside them  */
    float sm_scale;            /* softmax temperature; 0 = 1/sqrt(head_dim)           */
    int32_t flags;             /* must be 0                                           */
} kvq_prefill_params;

/* Workspace bytes of a prefill call: B * Hkv * ceil(4 * max_pages_per_seq / 128)
 * tiles of 2 x 32 KiB (K and V, 128 keys x 128 channels of fp16 each) plus
 * 16 bytes per tile (a mask of keys with a bad page); 0 for invalid
 * parameters. */
size_t kvq_prefill_workspace_bytes(const kvq_prefill_params *p);

int paged_prefill_attn_e4m3(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                            int64_t num_pages, const int32_t *block_tables,
                            const int32_t *context_lens, const int32_t *q_start,
                            float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                            void *out, const kvq_prefill_params *p, int32_t *err_flag, void *stream);

/* fp16-KV twin: the same computation over fp16 pools, without scales. */
int paged_prefill_attn_fp16(const void *q, const void *k_cache, const void *v_cache,
                            int64_t num_pages, const int32_t *block_tables,
                            const int32_t *context_lens, const int32_t *q_start,
                            void *workspace, size_t workspace_bytes, void *out,
                            const kvq_prefill_params *p, int32_t *err_flag, void *stream);

/* ------------------------------------------------------------------------
 * Allocation-free variant for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot provide a workspace -- code running under another framework's
 * memory pool that forbids outside cudaMalloc calls, plugins inside a
 * process whose allocator they do not control, or latency-critical paths
 * that ban allocation after start-up.
 *
 * Same computation, arguments and errors as paged_decode_attn_e4m3, minus
 * the workspace: the FP32 split partials go to a scratch buffer of
 * KVQ_NOALLOC_SCRATCH_BYTES that the library keeps in its own device memory
 * (a file-scope __device__ array, present on every GPU that loads the
 * library until the process exits).  The call allocates nothing.
 *  - A problem whose workspace (kvq_attn_workspace_bytes) exceeds
 *    KVQ_NOALLOC_SCRATCH_BYTES returns KVQ_ERR_WORKSPACE before any launch;
 *    use paged_decode_attn_e4m3 with your own workspace for those.
 *  - The first call on a device looks up the buffer's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address belongs to the device's
 *    context: after a device reset (cudaDeviceReset) the next call looks it
 *    up again, so make that call before any capture too.  A failed lookup
 *    returns KVQ_ERR_CUDA.
 *  - Every call on a device shares the one buffer, and it keeps the last
 *    call's contents (nothing in it has to start at zero).  Calls whose GPU
 *    work overlaps -- e.g. issued on two streams without ordering -- race
 *    on it and give undefined results: order them.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

int paged_decode_attn_e4m3_noalloc(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                   int64_t num_pages, const int32_t *block_tables,
                                   const int32_t *context_lens, float k_scale, float v_scale,
                                   const int32_t *topk_idx, const int32_t *topk_lens, void *out,
                                   const kvq_attn_params *p, int32_t *err_flag, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
