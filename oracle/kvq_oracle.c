/*
 * kvq_oracle.c -- plain, slow CPU oracle for the calibrated E4M3 paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant generator
 * with the CUDA library; it has its own binary16 and E4M3 arithmetic, its own
 * page addressing and its own attention loop, all written from the
 * definitions.
 *
 * Source pages (cited by page title and section):
 *   [P1] "[Model][SM70] Calibrated E4M3 KV cache for Qwen4Exp QSA with MTP",
 *        sections Purpose, Status and history.
 *   [P2] "[Model][SM70][FP8] Integrate calibrated E4M3 QSA KV capacity path",
 *        sections Changes, Validation boundary.
 *   [P3] "[Experiment][SM70] Qualify E4M3 KV with MTP3", section Problem and
 *        resulting behavior.
 * The pages describe the method in prose only (E4M3 storage of the main K/V
 * cache, one calibrated finite positive scale per layer for K and one for V,
 * page-4 routes, an FP32 split workspace, MTP verify windows, a top-k token
 * workspace).  The numeric details they leave open are fixed as follows, and
 * each function says which reading it follows:
 *   - E4M3 is the OCP 8-bit floating point "E4M3FN" format: bias 7, no
 *     infinities, 0x7F/0xFF are NaN, largest finite 448.
 *   - quantisation divides in IEEE binary32, then rounds to E4M3 with
 *     round-to-nearest-even and saturates finite overflow at +-448;
 *   - the calibrated scale is amax / 448 in binary32;
 *   - attention is the plain softmax(q k^T * sm_scale) v over the dequantised
 *     values, in binary64, with the verify window causal inside itself;
 *   - the FP8 score variant (not on the pages) replaces q in the scores by
 *     its E4M3 quantisation with one amax / 448 scale per (sequence, kv
 *     head) group of query rows, quantised like a cache element.
 *
 * Precision: binary64 for attention, binary32 exactly where the method's
 * quantisation is defined in binary32.  Build with -O2 -fno-fast-math
 * -ffp-contract=off so that every binary32 operation is a single IEEE
 * operation.
 *
 * Parity pins: every function here is checked in tests/ against something
 * other than itself (exhaustive library conversions, closed forms,
 * invariants, brute force); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)

/* error bits reported by the attention and append oracles (skipped inputs) */
#define ORACLE_BAD_PAGE 1
#define ORACLE_BAD_SLOT 2
#define ORACLE_BAD_TOPK 4
#define ORACLE_BAD_LEN 8

/* ------------------------------------------------------------------------ */
/* IEEE binary16 -> binary64, written from the IEEE 754 binary16 definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0x1F)
        v = (f == 0) ? INFINITY : NAN;
    else if (e == 0)
        v = ldexp((double)f, -24);             /* subnormal: f * 2^-24 */
    else
        v = ldexp(1.0 + f / 1024.0, e - 15);   /* normal */
    return s ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* OCP E4M3 (E4M3FN) decode.  Byte c = s eeee mmm.
 *   e == 0          : (-1)^s * m * 2^-9            (subnormals, +-0)
 *   e == 15, m == 7 : NaN                          (0x7F, 0xFF)
 *   otherwise       : (-1)^s * (1 + m/8) * 2^(e-7)
 * [P2] Changes: the main K/V cache is stored in E4M3. */
double oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* round-to-nearest-even of sig / 2^sh for an integer sig < 2^25 */
static uint32_t rne_shift(uint32_t sig, int sh)
{
    uint32_t q, rem, half;
    if (sh <= 0)
        return sig << (-sh);
    if (sh > 26)
        return 0; /* sig / 2^sh < 2^-1, below half of one unit */
    q = sig >> sh;
    rem = sig & ((1u << sh) - 1u);
    half = 1u << (sh - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q += 1u;
    return q;
}

/* OCP E4M3 encode of a binary32 value with round-to-nearest-even and
 * saturation of finite overflow (and of infinities) to +-448; NaN -> 0x7F.
 * Integer guard/sticky rounding on the binary32 bit pattern, so the result
 * does not depend on the FPU rounding mode.  The sign of zero is kept. */
uint8_t oracle_e4m3_encode_f32(float v)
{
    uint32_t u, ex, man, sig;
    uint8_t sign;
    int E;
    memcpy(&u, &v, sizeof u);
    sign = (u >> 31) ? 0x80 : 0x00;
    ex = (u >> 23) & 0xFFu;
    man = u & 0x7FFFFFu;
    if (ex == 0xFFu)
        return man ? 0x7F : (uint8_t)(sign | 0x7E); /* NaN ; +-inf saturates */
    if (ex == 0)
        return sign; /* zero or binary32 subnormal (< 2^-126): rounds to +-0 */
    E = (int)ex - 127;
    sig = man | 0x800000u; /* 24-bit significand, value = sig * 2^(E-23) */
    /* |v| >= 448 = 1.75 * 2^8 saturates */
    if (E > 8 || (E == 8 && man >= 0x600000u))
        return (uint8_t)(sign | 0x7E);
    if (E < -6) {
        /* E4M3 subnormal range: k = RNE(|v| * 2^9), k in [0, 8];
         * k == 8 is the smallest normal, code 0x08, so no special case. */
        uint32_t k = rne_shift(sig, 23 - (E + 9));
        return (uint8_t)(sign | k);
    } else {
        /* normal: keep 1 + 3 fraction bits, round the other 20 bits */
        uint32_t q = rne_shift(sig, 20); /* in [8, 16] */
        int e = E;
        if (q == 16u) {
            q = 8u;
            e += 1;
        }
        return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | (int)(q - 8u)));
    }
}

/* The method's quantiser: code = E4M3_RNE_sat(fp32(x) / scale), the division
 * being one IEEE binary32 division ([P2] Changes: calibrated E4M3 K/V with a
 * per-layer scale). */
uint8_t oracle_quantize(uint16_t x, float scale)
{
    float xf = (float)oracle_f16_to_f64(x); /* exact: binary16 is a subset of binary32 */
    float q = xf / scale;                    /* single binary32 division, RNE */
    return oracle_e4m3_encode_f32(q);
}

void oracle_quantize_array(const uint16_t *x, int64_t n, float scale, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_quantize(x[i], scale);
}

/* Calibration ([P2] Changes: offline calibration; one finite positive scale
 * per layer for K and one for V): amax = max |x| over the whole calibration
 * tensor, scale = amax / 448 in binary32.  Returns 0 when amax is 0 or not
 * finite (an invalid scale that the scale gate must refuse). */
float oracle_calibrate_scale(const uint16_t *x, int64_t n)
{
    double amax = 0.0;
    int64_t i;
    for (i = 0; i < n; ++i) {
        double a = fabs(oracle_f16_to_f64(x[i]));
        if (a != a)
            return 0.0f;
        if (a > amax)
            amax = a;
    }
    if (isinf(amax))
        return 0.0f;
    return (float)amax / 448.0f;
}

/* Query quantisation of the FP8 tensor-core score variant.  The pages store
 * only K and V in E4M3 and keep q in fp16; this variant is not on them, and
 * its reading is the plainest one that puts q into the same format as the
 * cache.  Per (sequence b, kv head g), the G * q_len query rows that attend
 * kv head g (heads g*G .. g*G+G-1, contiguous grouping, every row of the
 * verify window) share one scale:
 *   amax  = max |q| over those rows and all channels,
 *   scale = amax / 448 in binary32, or 1 when amax is 0 (an all-zero group),
 * and each element is quantised like a cache element (binary32 division by
 * the scale, then RNE to E4M3 with finite overflow saturated).  Writes codes
 * [B][q_len][Hq][D] and scales [B][Hkv]; returns ORACLE_OK or
 * ORACLE_BAD_ARG.  The query must be finite. */
int oracle_quantize_q_groups(const uint16_t *q, int B, int q_len, int Hq, int Hkv, int D,
                             uint8_t *codes, float *scales)
{
    int G, b, g, i, h, d;
    if (!q || !codes || !scales || B < 0 || q_len < 1 || Hkv < 1 || Hq < 1 || Hq % Hkv != 0 || D < 1)
        return ORACLE_BAD_ARG;
    G = Hq / Hkv;
    for (b = 0; b < B; ++b)
        for (g = 0; g < Hkv; ++g) {
            double amax = 0.0;
            float qs;
            for (i = 0; i < q_len; ++i)
                for (h = g * G; h < (g + 1) * G; ++h)
                    for (d = 0; d < D; ++d) {
                        double a = fabs(oracle_f16_to_f64(q[(((int64_t)b * q_len + i) * Hq + h) * D + d]));
                        if (a > amax)
                            amax = a;
                    }
            qs = amax > 0.0 ? (float)amax / 448.0f : 1.0f;
            scales[(int64_t)b * Hkv + g] = qs;
            for (i = 0; i < q_len; ++i)
                for (h = g * G; h < (g + 1) * G; ++h)
                    for (d = 0; d < D; ++d) {
                        int64_t idx = (((int64_t)b * q_len + i) * Hq + h) * D + d;
                        codes[idx] = oracle_quantize(q[idx], qs);
                    }
        }
    return ORACLE_OK;
}

/* Scale gate ([P2] Changes: every layer needs a finite, positive K and V
 * scale before the E4M3 mode starts; [P2] Validation boundary: a default
 * scale never replaces a missing one).  Returns the number of bad entries. */
int oracle_count_bad_scales(const float *k_scales, const float *v_scales, int n)
{
    int i, bad = 0;
    if (!k_scales || !v_scales || n <= 0)
        return -1;
    for (i = 0; i < n; ++i) {
        float a = k_scales[i], b = v_scales[i];
        if (!(a > 0.0f) || isinf(a) || !(b > 0.0f) || isinf(b))
            ++bad;
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Page-4 pool addressing.  Pool layout [page][kv_head][slot(4)][head_dim]
 * (the pages fix the page size, 4 tokens, and the per-sequence block table,
 * [P2] Changes "grouped page4"; the order of the inner dimensions is this
 * library's choice).  Element (page, g, slot, d) of a pool with Hkv heads. */
static int64_t pool_index(int64_t page, int g, int slot, int d, int Hkv, int D)
{
    return (((page * Hkv + g) * 4 + slot) * (int64_t)D) + d;
}

/* Quantise-on-append: token t of the step goes to slot_mapping[t] =
 * page * 4 + offset; a negative entry means "do not write".  Entries whose
 * page is outside the pool are skipped and reported. */
int oracle_append_e4m3(const uint16_t *k_new, const uint16_t *v_new,
                       const int32_t *slot_mapping, int32_t T, int32_t Hkv, int32_t D,
                       uint8_t *k_cache, uint8_t *v_cache, int64_t P,
                       float k_scale, float v_scale)
{
    int flags = 0;
    int32_t t;
    for (t = 0; t < T; ++t) {
        int32_t slot = slot_mapping[t];
        int64_t page;
        int g, d;
        if (slot < 0)
            continue;
        page = slot / 4;
        if (page >= P) {
            flags |= ORACLE_BAD_SLOT;
            continue;
        }
        for (g = 0; g < Hkv; ++g)
            for (d = 0; d < D; ++d) {
                int64_t src = ((int64_t)t * Hkv + g) * D + d;
                int64_t dst = pool_index(page, g, slot % 4, d, Hkv, D);
                k_cache[dst] = oracle_quantize(k_new[src], k_scale);
                v_cache[dst] = oracle_quantize(v_new[src], v_scale);
            }
    }
    return flags;
}

/* fp16-KV comparison arm ([P1] Validation: the only difference between the
 * arms is the KV cache dtype): the same slots, values stored unchanged. */
int oracle_append_fp16(const uint16_t *k_new, const uint16_t *v_new,
                       const int32_t *slot_mapping, int32_t T, int32_t Hkv, int32_t D,
                       uint16_t *k_cache, uint16_t *v_cache, int64_t P)
{
    int flags = 0;
    int32_t t;
    for (t = 0; t < T; ++t) {
        int32_t slot = slot_mapping[t];
        int64_t page;
        int g, d;
        if (slot < 0)
            continue;
        page = slot / 4;
        if (page >= P) {
            flags |= ORACLE_BAD_SLOT;
            continue;
        }
        for (g = 0; g < Hkv; ++g)
            for (d = 0; d < D; ++d) {
                int64_t src = ((int64_t)t * Hkv + g) * D + d;
                int64_t dst = pool_index(page, g, slot % 4, d, Hkv, D);
                k_cache[dst] = k_new[src];
                v_cache[dst] = v_new[src];
            }
    }
    return flags;
}

/* ------------------------------------------------------------------------ */
/* Attention.  One problem description shared by the E4M3 and fp16 arms. */
typedef struct {
    const uint16_t *q;            /* fp16 [B][q_len][Hq][D] */
    const void *k_cache;          /* E4M3 bytes or fp16, [P][Hkv][4][D] */
    const void *v_cache;
    int is_e4m3;
    int64_t P;
    const int32_t *block_tables;  /* [B][max_pages] */
    const int32_t *context_lens;  /* [B], includes the q_len tokens of this step */
    double k_scale, v_scale;      /* E4M3 arm only */
    const int32_t *topk_idx;      /* nullable, [B][Hkv][max_topk] */
    const int32_t *topk_lens;     /* nullable, [B]; 0 = dense */
    int B, q_len, Hq, Hkv, D, max_pages, max_topk;
    double sm_scale;
    /* nullable: the query quantised to E4M3 (codes [B][q_len][Hq][D], one
     * scale per (sequence, kv head) in q_scales [B][Hkv]); NULL = fp16 q */
    const uint8_t *q_codes;
    const float *q_scales;
} oracle_problem;

/* dequantised K or V element j (token position) of sequence b, head g, channel d;
 * returns 0 and sets *ok = 0 when the block-table entry is out of range */
static double kv_value(const oracle_problem *pr, int is_k, int b, int g, int j, int d, int *ok)
{
    int32_t page = pr->block_tables[(int64_t)b * pr->max_pages + j / 4];
    int64_t idx;
    if (page < 0 || page >= pr->P) {
        *ok = 0;
        return 0.0;
    }
    *ok = 1;
    idx = pool_index(page, g, j % 4, d, pr->Hkv, pr->D);
    if (pr->is_e4m3) {
        const uint8_t *c = (const uint8_t *)(is_k ? pr->k_cache : pr->v_cache);
        return oracle_e4m3_decode(c[idx]) * (is_k ? pr->k_scale : pr->v_scale);
    } else {
        const uint16_t *c = (const uint16_t *)(is_k ? pr->k_cache : pr->v_cache);
        return oracle_f16_to_f64(c[idx]);
    }
}

/* The key set of query row i of sequence b (kv head g), in order.  Dense:
 * positions 0 .. L-q_len+i (causal inside the verify window, [P1] Purpose:
 * MTP3, one target token plus three drafts checked in one pass).  Top-k:
 * the caller's listed positions that are <= that bound ([P2] Changes: the
 * QSA top-k index workspace).  Listed positions outside [0, L) are skipped
 * and reported.  Returns the count written to keys[]. */
static int key_set(const oracle_problem *pr, int b, int g, int i, int32_t *keys, int *flags)
{
    int L = pr->context_lens[b];
    int pos = L - pr->q_len + i;
    int n = 0, j;
    int use_topk = pr->topk_idx && pr->topk_lens && pr->topk_lens[b] > 0;
    if (L < pr->q_len || L > pr->max_pages * 4) {
        *flags |= ORACLE_BAD_LEN;
        return 0;
    }
    if (!use_topk) {
        for (j = 0; j <= pos; ++j)
            keys[n++] = j;
    } else {
        int cnt = pr->topk_lens[b];
        const int32_t *list = pr->topk_idx + ((int64_t)b * pr->Hkv + g) * pr->max_topk;
        if (cnt > pr->max_topk) {
            *flags |= ORACLE_BAD_TOPK;
            cnt = pr->max_topk;
        }
        for (j = 0; j < cnt; ++j) {
            int32_t t = list[j];
            if (t < 0 || t >= L) {
                *flags |= ORACLE_BAD_TOPK;
                continue;
            }
            if (t <= pos)
                keys[n++] = t;
        }
    }
    return n;
}

/* softmax-weighted sum over an explicit key list, binary64.  Writes out[D]
 * and returns through *m_out and *l_out the maximum score and the sum of
 * exp(s - m) (m = -inf, l = 0, out = 0 for an empty list). */
static int attend_keys(const oracle_problem *pr, int b, int h, int i, const int32_t *keys, int n,
                       double *out, double *m_out, double *l_out, double *scores)
{
    int G = pr->Hq / pr->Hkv;
    int g = h / G; /* contiguous grouping of query heads onto kv heads */
    int D = pr->D, k, d, ok, flags = 0;
    const uint16_t *qrow = pr->q + (((int64_t)b * pr->q_len + i) * pr->Hq + h) * D;
    const uint8_t *qcode = pr->q_codes ? pr->q_codes + (qrow - pr->q) : NULL;
    double qscale = pr->q_codes ? (double)pr->q_scales[(int64_t)b * pr->Hkv + g] : 0.0;
    double m = -INFINITY, l = 0.0;
    for (d = 0; d < D; ++d)
        out[d] = 0.0;
    for (k = 0; k < n; ++k) {
        double s = 0.0;
        for (d = 0; d < D; ++d) {
            double kv = kv_value(pr, 1, b, g, keys[k], d, &ok);
            if (!ok)
                break;
            if (qcode)
                s += oracle_e4m3_decode(qcode[d]) * qscale * kv;
            else
                s += oracle_f16_to_f64(qrow[d]) * kv;
        }
        if (!ok) {
            flags |= ORACLE_BAD_PAGE;
            scores[k] = -INFINITY;
            continue;
        }
        scores[k] = s * pr->sm_scale;
        if (scores[k] > m)
            m = scores[k];
    }
    if (m == -INFINITY) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return flags;
    }
    for (k = 0; k < n; ++k) {
        double p;
        if (scores[k] == -INFINITY)
            continue;
        p = exp(scores[k] - m);
        l += p;
        for (d = 0; d < D; ++d)
            out[d] += p * kv_value(pr, 0, b, g, keys[k], d, &ok);
    }
    for (d = 0; d < D; ++d)
        out[d] /= l;
    *m_out = m;
    *l_out = l;
    return flags;
}

static int check_problem(const oracle_problem *pr)
{
    if (!pr->q || !pr->k_cache || !pr->v_cache || !pr->block_tables || !pr->context_lens)
        return 0;
    if (pr->B < 0 || pr->q_len < 1 || pr->Hq < 1 || pr->Hkv < 1 || pr->D < 1)
        return 0;
    if (pr->Hq % pr->Hkv != 0 || pr->max_pages < 0)
        return 0;
    if (pr->q_codes && !pr->q_scales)
        return 0;
    return 1;
}

/* Full attention: out [B][q_len][Hq][D] in binary64 and, if lse is not
 * NULL, lse [B][q_len][Hq] = m + ln(l) (-inf for an empty key set).
 * Returns the OR of the error bits, or ORACLE_BAD_ARG. */
static int oracle_attention(const oracle_problem *pr, double *out, double *lse)
{
    int b, h, i, flags = 0;
    int32_t *keys;
    double *scores;
    int cap = pr->max_pages * 4 + pr->max_topk + 1;
    if (!check_problem(pr))
        return ORACLE_BAD_ARG;
    keys = (int32_t *)malloc(sizeof(int32_t) * cap);
    scores = (double *)malloc(sizeof(double) * cap);
    if (!keys || !scores) {
        free(keys);
        free(scores);
        return ORACLE_BAD_ARG;
    }
    for (b = 0; b < pr->B; ++b)
        for (i = 0; i < pr->q_len; ++i)
            for (h = 0; h < pr->Hq; ++h) {
                int g = h / (pr->Hq / pr->Hkv);
                int64_t row = ((int64_t)b * pr->q_len + i) * pr->Hq + h;
                double m, l;
                int n = key_set(pr, b, g, i, keys, &flags);
                flags |= attend_keys(pr, b, h, i, keys, n, out + row * pr->D, &m, &l, scores);
                if (lse)
                    lse[row] = (l > 0.0) ? m + log(l) : -INFINITY;
            }
    free(keys);
    free(scores);
    return flags;
}

/* Split partials, for checking the FP32 split workspace ([P1] Status and
 * history / [P3] Problem: the page-4 route writes an FP32 temporary output).
 * The pages leave the partition open; two readings are implemented.  With
 * split_pages == 0, split s of a sequence covers logical pages
 * [s*c, (s+1)*c) with c = ceil(npages / S) (dense), or list entries
 * [s*c, (s+1)*c) with c = ceil(topk_len / S) (top-k).  With split_pages > 0,
 * c = split_pages pages (dense) or 4 * split_pages list entries (top-k), the
 * same for every sequence.  Per (b, h, i, s): o normalised by its own l,
 * m = max score, l = sum exp(s - m).  Layout o [B][Hq][q_len][S][D],
 * m and l [B][Hq][q_len][S]. */
static int oracle_partials(const oracle_problem *pr, int S, int split_pages, double *o, double *m,
                           double *l)
{
    int b, h, i, s, flags = 0;
    int32_t *keys, *sub;
    double *scores;
    int cap = pr->max_pages * 4 + pr->max_topk + 1;
    if (!check_problem(pr) || S < 1 || split_pages < 0)
        return ORACLE_BAD_ARG;
    keys = (int32_t *)malloc(sizeof(int32_t) * cap);
    sub = (int32_t *)malloc(sizeof(int32_t) * cap);
    scores = (double *)malloc(sizeof(double) * cap);
    if (!keys || !sub || !scores) {
        free(keys);
        free(sub);
        free(scores);
        return ORACLE_BAD_ARG;
    }
    for (b = 0; b < pr->B; ++b) {
        int L = pr->context_lens[b];
        int use_topk = pr->topk_idx && pr->topk_lens && pr->topk_lens[b] > 0;
        for (h = 0; h < pr->Hq; ++h) {
            int g = h / (pr->Hq / pr->Hkv);
            for (i = 0; i < pr->q_len; ++i) {
                int n, k;
                n = key_set(pr, b, g, i, keys, &flags);
                for (s = 0; s < S; ++s) {
                    int64_t unit = (((int64_t)b * pr->Hq + h) * pr->q_len + i) * S + s;
                    int ns = 0;
                    if (!use_topk) {
                        int npages = (L + 3) / 4;
                        int64_t c = split_pages > 0 ? split_pages : (npages + S - 1) / S;
                        int64_t lo = s * c * 4, hi = (s + 1) * c * 4;
                        for (k = 0; k < n; ++k)
                            if (keys[k] >= lo && keys[k] < hi)
                                sub[ns++] = keys[k];
                    } else {
                        /* split by list entry, then keep the causal/valid ones */
                        int cnt = pr->topk_lens[b] < pr->max_topk ? pr->topk_lens[b] : pr->max_topk;
                        int64_t c = split_pages > 0 ? 4 * (int64_t)split_pages : (cnt + S - 1) / S;
                        int64_t lo = s * c, hi = (s + 1) * c, e;
                        const int32_t *list = pr->topk_idx + ((int64_t)b * pr->Hkv + g) * pr->max_topk;
                        int pos = L - pr->q_len + i;
                        for (e = lo; e < hi && e < cnt; ++e) {
                            int32_t t = list[e];
                            if (t >= 0 && t < L && t <= pos)
                                sub[ns++] = t;
                        }
                    }
                    flags |= attend_keys(pr, b, h, i, sub, ns, o + unit * pr->D, &m[unit], &l[unit], scores);
                }
            }
        }
    }
    free(keys);
    free(sub);
    free(scores);
    return flags;
}

/* Log-sum-exp combine of split partials: M = max_s m_s, w_s = l_s exp(m_s - M),
 * out = sum_s w_s o_s / sum_s w_s; a row whose splits are all empty gives 0.
 * o [rows][S][D], m and l [rows][S] -> out [rows][D]. */
void oracle_combine(const double *o, const double *m, const double *l, int64_t rows, int S, int D,
                    double *out)
{
    int64_t r;
    int s, d;
    for (r = 0; r < rows; ++r) {
        double M = -INFINITY, W = 0.0;
        for (s = 0; s < S; ++s)
            if (l[r * S + s] > 0.0 && m[r * S + s] > M)
                M = m[r * S + s];
        for (d = 0; d < D; ++d)
            out[r * D + d] = 0.0;
        if (M == -INFINITY)
            continue;
        for (s = 0; s < S; ++s) {
            double w;
            if (!(l[r * S + s] > 0.0))
                continue;
            w = l[r * S + s] * exp(m[r * S + s] - M);
            W += w;
            for (d = 0; d < D; ++d)
                out[r * D + d] += w * o[(r * S + s) * D + d];
        }
        for (d = 0; d < D; ++d)
            out[r * D + d] /= W;
    }
}

/* ------------------------------------------------------------------------ */
/* Flat entry points for the ctypes wrapper. */
int oracle_attn(const uint16_t *q, const void *k_cache, const void *v_cache, int is_e4m3, int64_t P,
                const int32_t *block_tables, const int32_t *context_lens, double k_scale,
                double v_scale, const int32_t *topk_idx, const int32_t *topk_lens, int B,
                int q_len, int Hq, int Hkv, int D, int max_pages, int max_topk, double sm_scale,
                const uint8_t *q_codes, const float *q_scales, double *out, double *lse)
{
    oracle_problem pr;
    pr.q = q;
    pr.k_cache = k_cache;
    pr.v_cache = v_cache;
    pr.is_e4m3 = is_e4m3;
    pr.P = P;
    pr.block_tables = block_tables;
    pr.context_lens = context_lens;
    pr.k_scale = k_scale;
    pr.v_scale = v_scale;
    pr.topk_idx = topk_idx;
    pr.topk_lens = topk_lens;
    pr.B = B;
    pr.q_len = q_len;
    pr.Hq = Hq;
    pr.Hkv = Hkv;
    pr.D = D;
    pr.max_pages = max_pages;
    pr.max_topk = topk_idx ? max_topk : 0;
    pr.sm_scale = sm_scale;
    pr.q_codes = q_codes;
    pr.q_scales = q_codes ? q_scales : NULL;
    return oracle_attention(&pr, out, lse);
}

int oracle_attn_partials(const uint16_t *q, const void *k_cache, const void *v_cache, int is_e4m3,
                         int64_t P, const int32_t *block_tables, const int32_t *context_lens,
                         double k_scale, double v_scale, const int32_t *topk_idx,
                         const int32_t *topk_lens, int B, int q_len, int Hq, int Hkv, int D,
                         int max_pages, int max_topk, double sm_scale, const uint8_t *q_codes,
                         const float *q_scales, int S, int split_pages, double *o, double *m,
                         double *l)
{
    oracle_problem pr;
    pr.q = q;
    pr.k_cache = k_cache;
    pr.v_cache = v_cache;
    pr.is_e4m3 = is_e4m3;
    pr.P = P;
    pr.block_tables = block_tables;
    pr.context_lens = context_lens;
    pr.k_scale = k_scale;
    pr.v_scale = v_scale;
    pr.topk_idx = topk_idx;
    pr.topk_lens = topk_lens;
    pr.B = B;
    pr.q_len = q_len;
    pr.Hq = Hq;
    pr.Hkv = Hkv;
    pr.D = D;
    pr.max_pages = max_pages;
    pr.max_topk = topk_idx ? max_topk : 0;
    pr.sm_scale = sm_scale;
    pr.q_codes = q_codes;
    pr.q_scales = q_codes ? q_scales : NULL;
    return oracle_partials(&pr, S, split_pages, o, m, l);
}
