// kvq_attn_kernel.cuh -- the split-K paged decode / MTP-verify attention
// kernel over E4M3 or fp16 page-4 pools, and its launchers.  kvq_attn.cu
// instantiates it with the hardware E4M3 conversion (and for fp16 pools),
// kvq_attn_bitcast.cu with the bitcast decoder.
//
// What is computed (PR "[Model][SM70][FP8] Integrate calibrated E4M3 QSA KV
// capacity path", section Changes; PR "[Model][SM70] Calibrated E4M3 KV cache
// for Qwen4Exp QSA with MTP", sections Purpose and Status and history):
// grouped-query attention of q_len = 1 (decode) or 1 + 3 (MTP verify, causal
// inside the window) query rows over a page-4 cache whose K/V are stored in
// calibrated E4M3, decoded exactly to fp16 with the per-layer scales hoisted
// out of the inner loop, split over the token axis into an FP32 workspace,
// and merged by a log-sum-exp combine.
//
// GB300 design (one CTA per (split, kv head, sequence), 4 consumer warps and
// 2 producer warps):
//  * Two producer warps walk the split's pages one stage at a time (16 pages
//    for one query-row group, 8 otherwise), read the block table a batch
//    ahead, and issue one 1-D bulk TMA copy per page -- one warp for K, the
//    other for V (a page of one kv head = 4 * head_dim contiguous elements)
//    -- into a ring of about 50 KB of shared memory, each stage completing
//    on its own mbarrier.  A single warp issues bulk copies at a limited
//    rate (about 27 million per second measured on GB300, whatever their
//    size), so splitting K and V doubles the CTA's copy rate.  In top-k mode
//    a stage is 4 tokens per page slot, each fetched as one row.
//  * Every consumer warp takes part in every stage: warp w owns one (or, for
//    64 query rows, two) 16-token tiles of the stage and one group of query
//    rows.  Each warp therefore waits on every phase of every ring slot in
//    order, and a slot is refilled only after all four warps released it.
//  * Per 16-token tile: K via ldmatrix, E4M3 -> fp16 by the hardware
//    conversion (exact), S^T = K Q^T on tensor cores (mma.sync m16n8k16,
//    tokens on M, query rows on N: the 8 heads of a GQA group fill N
//    exactly); online softmax in the log2 domain with k_scale * sm_scale *
//    log2(e) folded into one multiplier; P transposed in registers by
//    movmatrix; V^T via ldmatrix.trans, decoded (byte permute + conversion,
//    or the bitcast decoder), O^T += V^T P^T.  v_scale is applied once per
//    output row.
//  * Page chunks sit 16 bytes further apart than their size in shared
//    memory, so the eight rows an ldmatrix reads (one slot of eight pages)
//    fall in distinct banks.
//  * Every wait is bounded (about 2 s); on expiry the kernel reports
//    KVQ_DEV_TIMEOUT, drains its own copies, gives its rows zero weight in
//    the workspace (m = -inf, l = 0) and exits.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_merge.cuh"

namespace kvq {

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarps = 2;   // K pages and V pages
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLn2 = 0.69314718055994530942f;

// Work split of the 4 consumer warps: RW warps share the same tokens and
// split the query rows (NT 8-row tiles each); 4/RW warps split the tokens.
template <int NT, int RW>
struct Split {
    static constexpr int kRowWarps = RW;
    static constexpr int kTokWarps = kConsumerWarps / RW;
    static constexpr int kTilesPerWarp = (RW == kConsumerWarps) ? 2 : 1;    // 16-token tiles
    static constexpr int kTilesPerStage = kTokWarps * kTilesPerWarp;
    static constexpr int kPagesPerStage = 4 * kTilesPerStage;             // 16 or 8
    static constexpr int kRowsPad = RW * NT * 8;
};

// MIN_STAGES: a consumer that waits on one stage out of several in flight
// (the tcgen05 kernel's workers) needs the ring to hold all of them, or its
// wait could see the phase parity of the slot's previous use.
template <bool E4M3, int D, int PPS, int MIN_STAGES = 2>
struct Geometry {
    static constexpr int kD = D;
    static constexpr int kElem = E4M3 ? 1 : 2;
    static constexpr int kRowBytes = D * kElem;           // one token of one kv head
    static constexpr int kChunk = 4 * kRowBytes;          // one page of one kv head
    static constexpr int kPageStride = kChunk + 16;       // bank-skewed page placement
    static constexpr int kRegion = PPS * kPageStride;     // K (or V) part of a stage
    static constexpr int kStageBytes = 2 * kRegion;
    static constexpr int kStagesRaw = 50688 / kStageBytes;   // ~50 KB of ring
    static constexpr int kStagesClamped = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kStages = kStagesClamped < MIN_STAGES ? MIN_STAGES : kStagesClamped;
    static constexpr int kX4 = kRowBytes / 32;            // ldmatrix.x4 per 16-token tile
    static constexpr int kKSteps = D / 16;                // QK mma k-steps
    static constexpr int kPVTiles = D / 16;               // PV mma m-tiles (16 channels)
    static constexpr int kTokPerStage = 4 * PPS;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kTokPosOff = kRingBytes;
    static constexpr int kBarOff = kTokPosOff + kStages * kTokPerStage * 4;
    // abort flag, sticky bad-stage flag, and the stages each producer issued
    static constexpr int kAbortOff = kBarOff + 2 * kStages * 8;
    static constexpr int kAppBarOff = kAbortOff + 16;     // fused step, consumer append: the new rows are in the pool
    static constexpr int kBytes = kAbortOff + 24;
    static_assert(kPageStride % 128 == 16, "page skew must be 16 bytes mod 128");
    static_assert(kBarOff % 8 == 0, "mbarriers need 8-byte alignment");
};

template <bool E4M3, int D, int NT, int RW>
constexpr int smem_bytes()
{
    using W = Split<NT, RW>;
    using G = Geometry<E4M3, D, W::kPagesPerStage>;
    constexpr int merge = (W::kTokWarps * W::kRowsPad * (D + 2) + W::kRowsPad * W::kTokWarps) * 4;
    return G::kBytes > merge ? G::kBytes : merge;
}

// channel of the O^T accumulator row held by this thread for PV tile `pv`
// (first = fragment row gid, second = fragment row gid + 8)
template <bool BYTE_PAIRS>
__device__ __forceinline__ int2 pv_channels(int pv, int gid)
{
    if (BYTE_PAIRS) return make_int2(16 * pv + 2 * gid, 16 * pv + 2 * gid + 1);
    return make_int2(16 * pv + gid, 16 * pv + 8 + gid);
}

// First logical page of split s's speculative block-table read (the same for
// every sequence: equal division assumes a full block-table row).
__device__ __forceinline__ int split_spec0(const AttnArgs &a, int s)
{
    const int64_t spec_per = a.split_pages > 0 ? (int64_t)a.split_pages
                                               : (int64_t)(a.max_pages + a.num_splits - 1) / a.num_splits;
    return (int)min((int64_t)s * spec_per, (int64_t)a.max_pages);
}

// The split's share of one (sequence, kv head): the context length, the
// mode, and the items (logical pages, or top-k list entries) it covers --
// split s covers items [s * per, (s + 1) * per): an equal share of this
// sequence, or a fixed number of pages (4 list entries per page).
struct SplitRange {
    const int32_t *bt_row;
    int L, item0, item1, spec0;
    bool len_ok, topk;
};

// L = context_lens[b], topk_len = topk_lens[b] (0 without a top-k list).
__device__ __forceinline__ SplitRange split_range(const AttnArgs &a, int s, int b, int L, int topk_len)
{
    SplitRange r;
    r.bt_row = a.block_tables + (int64_t)b * a.max_pages;
    r.spec0 = split_spec0(a, s);
    r.L = L;
    r.len_ok = (r.L >= a.q_len) && (r.L <= a.max_pages * 4);
    int topk_n = topk_len;
    r.topk = r.len_ok && topk_n > 0;
    if (r.topk && topk_n > a.max_topk) topk_n = a.max_topk;
    const int n_items = !r.len_ok ? 0 : (r.topk ? topk_n : (r.L + 3) / 4);
    const int64_t per = a.split_pages > 0 ? (r.topk ? 4 * (int64_t)a.split_pages : (int64_t)a.split_pages)
                                          : (int64_t)(n_items + a.num_splits - 1) / a.num_splits;
    r.item0 = (int)min((int64_t)s * per, (int64_t)n_items);
    r.item1 = (int)min(r.item0 + per, (int64_t)n_items);
    return r;
}

// Longest-first order of the sequences.  The CTAs of blockIdx.z = z attend
// the sequence of rank z when the sequences are ordered by the work they
// attend -- context length, or top-k list length -- in classes of a quarter
// octave, longest class first and by index inside a class.  The block
// scheduler hands out CTAs roughly in index order, so the long sequences
// start first and the short ones fill the gaps at the end of the grid.  When
// every sequence falls in one class the order is the identity, found after a
// barrier that the CTA's setup needs anyway.  A scheduling choice only:
// which (sequence, split) a CTA computes does not change any result.
//
// Use, by every thread of the CTA after grid_dependency_wait:
//     SeqPick p = seq_identity(a, z);
//     const bool keep = lpt_classify(a, scratch, scratch_bytes);
//     if (!__syncthreads_and(keep)) p = lpt_pick(a, z, scratch);
// `scratch` is `scratch_bytes` of shared memory that nothing else uses
// meanwhile; a batch too large for it keeps the identity order.
constexpr int kWorkClasses = 128;
constexpr int kLptScratchFixed = (kWorkClasses + 4) * 4;

__device__ __forceinline__ int work_class(const AttnArgs &a, int L, int topk_len)
{
    int n = 0;   // items attended; an invalid length attends none
    if (L >= a.q_len && L <= a.max_pages * 4) n = topk_len > 0 ? min(topk_len, a.max_topk) : L;
    if (n <= 0) return 0;
    const int e = 31 - __clz(n);                                         // octave
    const int quarter = (e >= 2 ? (n >> (e - 2)) : (n << (2 - e))) & 3;   // two bits below the leading one
    return 1 + 4 * e + quarter;                                          // <= 124
}

struct SeqPick {
    int b, L, topk_len;
};

__device__ __forceinline__ SeqPick seq_identity(const AttnArgs &a, int z)
{
    SeqPick p;
    p.b = z;
    p.L = __ldg(a.context_lens + z);
    p.topk_len = (a.topk_idx && a.topk_lens) ? __ldg(a.topk_lens + z) : 0;
    return p;
}

// Each sequence's class into scratch; true when the identity order stands
// (one class, or a batch too large for the scratch).
__device__ __forceinline__ bool lpt_classify(const AttnArgs &a, uint8_t *scratch, int scratch_bytes)
{
    const int B = a.batch;
    if (B + kLptScratchFixed > scratch_bytes) return true;
    const bool with_topk = a.topk_idx && a.topk_lens;
    int *hist = reinterpret_cast<int *>(scratch);                  // [kWorkClasses]
    uint8_t *cls = scratch + kLptScratchFixed;                     // [B]
    for (int i = threadIdx.x; i < kWorkClasses; i += blockDim.x) hist[i] = 0;
    const int c0 = work_class(a, __ldg(a.context_lens), with_topk ? __ldg(a.topk_lens) : 0);
    bool one_class = true;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        const int c = work_class(a, __ldg(a.context_lens + i), with_topk ? __ldg(a.topk_lens + i) : 0);
        cls[i] = (uint8_t)c;
        one_class &= c == c0;
    }
    return one_class;
}

// The sequence of rank z, after lpt_classify and a barrier.
__device__ __forceinline__ SeqPick lpt_pick(const AttnArgs &a, int z, uint8_t *scratch)
{
    const int B = a.batch;
    int *hist = reinterpret_cast<int *>(scratch);
    int *sel = hist + kWorkClasses;
    const uint8_t *cls = scratch + kLptScratchFixed;
    for (int i = threadIdx.x; i < B; i += blockDim.x) atomicAdd(&hist[cls[i]], 1);
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        // lane l holds classes 127 - 4l .. 124 - 4l (descending); exclusive scan of their counts
        int cnt[4], tot = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            cnt[k] = hist[kWorkClasses - 1 - 4 * lane - k];
            tot += cnt[k];
        }
        int incl = tot;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += v;
        }
        const int start = incl - tot;
        const unsigned hit = __ballot_sync(kFull, z >= start && z < incl);
        const int owner = __ffs(hit) - 1;                          // z < B = sum of all counts
        int c_sel = 0, idx = 0;
        if (lane == owner) {
            int acc = start;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (z >= acc && z < acc + cnt[k]) {
                    c_sel = kWorkClasses - 1 - 4 * lane - k;
                    idx = z - acc;
                }
                acc += cnt[k];
            }
        }
        c_sel = __shfl_sync(kFull, c_sel, owner);
        idx = __shfl_sync(kFull, idx, owner);
        // the idx-th sequence (by index) of class c_sel
        for (int base = 0; base < B; base += 32) {
            const bool mine = base + lane < B && cls[base + lane] == c_sel;
            const unsigned m = __ballot_sync(kFull, mine);
            const int n = __popc(m);
            if (idx < n) {
                if (mine && __popc(m & ((1u << lane) - 1u)) == idx) *sel = base + lane;
                break;
            }
            idx -= n;
        }
    }
    __syncthreads();
    const int b = *sel;
    __syncthreads();   // the scratch may be reused
    return seq_identity(a, b);
}

// ---------------------------------------------------------------------------
// Fused step: quantise-on-append inside the attention launch (PR "[Model]
// [SM70][FP8] Integrate calibrated E4M3 QSA KV capacity path", section
// Changes: the cache is written in calibrated E4M3 as tokens are appended).
//
// Two fp16 values (element 0 in the low half) to two E4M3 codes (element 0
// in the low byte): each divided by the layer's scale in IEEE binary32
// (round to nearest even), then the satfinite conversion (round to nearest
// even, finite overflow to +-448) -- the append kernel's two roundings.
__device__ __forceinline__ uint32_t quantize_pair(uint32_t h2, float scale)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
    return __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale)), __NV_SATFINITE,
                                    __NV_E4M3);
}

// Orders this thread's global stores (generic proxy) before bulk copies
// (async proxy) issued after a later synchronisation with the issuing thread.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The producer warp of one half (K when !is_v, V otherwise) writes this
// step's new rows of (sequence b, kv head g) -- positions L - q_len .. L - 1,
// input rows b * q_len + i -- whose pages lie in its split, into the page
// slots its block table names, and fences them for its bulk copies.  Only
// this CTA reads those pages (dense splits partition the pages of a
// (sequence, kv head)), so no other CTA can see them half-written.  Lane l
// takes channels [l * D / 32, (l + 1) * D / 32) of every row; every load
// (the rows' page entries and new values, q_len <= 4) is issued before any
// store, so that one memory round trip covers them.  A bad page is skipped
// here and reported when its copy is issued.
template <class G>
__device__ __forceinline__ void append_step_rows(const AttnArgs &a, const SplitRange &r, int b, int g, int lane,
                                                 bool is_v)
{
    constexpr int CPL = G::kD / 32;   // channels per lane: 4 or 2
    static_assert(CPL == 4 || CPL == 2, "head_dim 128 or 64");
    using Vec = typename std::conditional<CPL == 4, uint2, uint32_t>::type;   // CPL fp16 values
    const auto *src = static_cast<const uint8_t *>(is_v ? a.v_new : a.k_new) +
                      ((int64_t)b * a.q_len * a.num_kv_heads + g) * (G::kD * 2) + lane * (CPL * 2);
    auto *pool = static_cast<uint8_t *>(const_cast<void *>(is_v ? a.v_cache : a.k_cache)) +
                 (int64_t)g * 4 * G::kRowBytes + lane * (CPL * G::kElem);
    const float scale = is_v ? a.v_scale : a.k_scale;
    const int first = r.L - a.q_len;
    int phys[4];
    Vec h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int item = (first + i) >> 2;
        const bool mine = i < a.q_len && item >= r.item0 && item < r.item1;
        phys[i] = mine ? __ldg(r.bt_row + item) : -1;
        if (mine) h[i] = *reinterpret_cast<const Vec *>(src + (int64_t)i * a.num_kv_heads * (G::kD * 2));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (phys[i] < 0 || (int64_t)phys[i] >= a.num_pages) continue;
        uint8_t *dst = pool + ((int64_t)phys[i] * a.num_kv_heads * 4 + ((first + i) & 3)) * G::kRowBytes;
        const uint32_t *x = reinterpret_cast<const uint32_t *>(&h[i]);
        if (G::kElem == 2)
            *reinterpret_cast<Vec *>(dst) = h[i];
        else if (CPL == 4)
            *reinterpret_cast<uint32_t *>(dst) = quantize_pair(x[0], scale) | (quantize_pair(x[1], scale) << 16);
        else
            *reinterpret_cast<uint16_t *>(dst) = (uint16_t)quantize_pair(x[0], scale);
    }
    fence_proxy_async_global();
    __syncwarp();
}

// One producer warp (K pages when !is_v, V pages otherwise) walks the
// split's nst stages: it reads the block table a batch ahead, waits for the
// stage's ring slot to be released, records the token positions (K warp),
// and issues one 1-D bulk copy per page (dense) or per listed token row
// (top-k), completing on the slot's full mbarrier.  Returns the stages issued.
// clean_items >= 0: the caller has not yet waited for the preceding kernel,
// and the logical pages below clean_items (positions below L - q_len, which
// this step's append does not write) may be copied before that wait; the
// wait comes before the first stage that reaches past them.  -1: the caller
// has waited.
// FMODE, the fused step's instances (dense only):
//  1: a producer whose split holds some of this step's new rows first waits
//     for the preceding kernel (which may write them) and appends its half of
//     them, then walks its stages as the other instances do.  Its first
//     copies start a memory round trip later; the consumers, which wait for
//     the preceding kernel before reading q, start no earlier anyway.
//     Appending later inside the stage loop measured slower: that code in
//     the loop slowed every stage.
//  2: consumer warps append the rows (after their own dependency wait) while
//     the producers copy the earlier pages; a producer waits for them, on the
//     mbarrier at app_bar, before the first stage that holds a new row.  The
//     cluster-merge instances use it: their grid is resident in one wave, so
//     an appending CTA's late start lengthens the whole launch (decode step
//     27.75 -> 27.3 us); on longer launches the check in the loop costs more
//     (long context: +2.2 us).
template <class G, int PPS, int FMODE = 0>
__device__ __forceinline__ int produce_stages(const AttnArgs &a, const SplitRange &r, int nst, int b, int g,
                                              int lane, bool is_v, int bt_spec, uint32_t ring, uint32_t bar0,
                                              int32_t *tokpos, volatile int *abort_flag, volatile int *stage_bad,
                                              int clean_items = -1, uint32_t app_bar = 0)
{
    const int item0 = r.item0, item1 = r.item1, L = r.L, spec0 = r.spec0;
    const bool topk = r.topk;
    const int32_t *bt_row = r.bt_row;
    int issued = 0;
        const uint64_t pol = l2_policy_evict_first();
        const uint8_t *pool = static_cast<const uint8_t *>(is_v ? a.v_cache : a.k_cache);
        if (!topk) {
            constexpr int SPB = 32 / PPS;                 // stages per block-table batch
            auto load_bt = [&](int first) -> int {
                const int it = first + lane;
                return it < item1 ? __ldg(bt_row + it) : -1;
            };
            int bt_cur = (item0 == spec0) ? (item0 + lane < item1 ? bt_spec : -1) : load_bt(item0);
            int bt_nxt = load_bt(item0 + 32);
            const int p = lane % PPS;                      // page of the stage this lane copies
            const bool copier = lane < PPS;
            bool waited = clean_items < 0;
            int st_new = nst;   // FMODE 2: the first stage that holds a new row
            if constexpr (FMODE != 0) {
                const int first_new = max(L - a.q_len, 0) / 4;   // first page with a new row
                if constexpr (FMODE == 1) {
                    if (nst > 0 && first_new < item1) {
                        if (!waited) grid_dependency_wait();
                        waited = true;
                        append_step_rows<G>(a, r, b, g, lane, is_v);
                    }
                } else {
                    if (first_new < item1) st_new = first_new <= item0 ? 0 : (first_new - item0) / PPS;
                }
            }
            for (int st = 0; st < nst; ++st) {
                const int slot = st % G::kStages;
                if constexpr (FMODE == 2) {
                    if (st == st_new && !mbar_wait_bounded(app_bar, 0, abort_flag, a.err_flag)) break;
                }
                if (!waited && item0 + (st + 1) * PPS > clean_items) {
                    grid_dependency_wait();
                    waited = true;
                }
                if (st >= G::kStages &&
                    !mbar_wait_bounded(bar0 + 8 * (G::kStages + slot), ((st / G::kStages) + 1) & 1,
                                       abort_flag, a.err_flag))
                    break;
                if (st > 0 && st % SPB == 0) {
                    bt_cur = bt_nxt;
                    bt_nxt = load_bt(item0 + (st + SPB) * PPS);
                }
                const int item = item0 + st * PPS + p;
                const int phys = __shfl_sync(kFull, bt_cur, (st % SPB) * PPS + p);
                const bool exists = item < item1;
                const bool valid = exists && phys >= 0 && (int64_t)phys < a.num_pages;
                if (!is_v && lane < PPS) {
                    if (exists && !valid) {
                        report(a.err_flag, KVQ_DEV_BAD_PAGE);
                        *stage_bad = 1;
                    }
#pragma unroll
                    for (int sl = 0; sl < 4; ++sl) {
                        const int pos = item * 4 + sl;
                        tokpos[slot * G::kTokPerStage + p * 4 + sl] = (valid && pos < L) ? pos : -1;
                    }
                }
                const unsigned vmask = __ballot_sync(kFull, valid && copier);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(bar0 + 8 * slot, __popc(vmask) * G::kChunk);
                __syncwarp();
                if (copier && valid) {
                    const uint8_t *src = pool + ((int64_t)phys * a.num_kv_heads + g) * G::kChunk;
                    const uint32_t dst = ring + slot * G::kStageBytes + (is_v ? G::kRegion : 0) +
                                         p * G::kPageStride;
                    tma_load_1d(dst, src, G::kChunk, bar0 + 8 * slot, pol);
                }
                issued = st + 1;
            }
        } else {
            // top-k: kTokPerStage listed tokens per stage, R per lane
            constexpr int R = G::kTokPerStage / 32;
            const int32_t *list = a.topk_idx + ((int64_t)b * a.num_kv_heads + g) * a.max_topk;
            auto load_idx = [&](int st, int r) -> int {
                const int it = item0 + st * G::kTokPerStage + r * 32 + lane;
                return (st < nst && it < item1) ? __ldg(list + it) : -1;
            };
            auto load_page = [&](int idx) -> int {
                return (idx >= 0 && idx < L) ? __ldg(bt_row + (idx >> 2)) : -1;
            };
            int idx_cur[R], pg_cur[R], idx_nxt[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                idx_cur[r] = load_idx(0, r);
                pg_cur[r] = load_page(idx_cur[r]);
                idx_nxt[r] = load_idx(1, r);
            }
            for (int st = 0; st < nst; ++st) {
                const int slot = st % G::kStages;
                if (st >= G::kStages &&
                    !mbar_wait_bounded(bar0 + 8 * (G::kStages + slot), ((st / G::kStages) + 1) & 1,
                                       abort_flag, a.err_flag))
                    break;
                int pg_nxt[R], idx_nxt2[R];
                bool valid[R];
                int cnt = 0;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    pg_nxt[r] = load_page(idx_nxt[r]);
                    idx_nxt2[r] = load_idx(st + 2, r);
                    const int e = r * 32 + lane;                    // token of the stage
                    const bool exists = item0 + st * G::kTokPerStage + e < item1;
                    const bool idx_ok = exists && idx_cur[r] >= 0 && idx_cur[r] < L;
                    valid[r] = idx_ok && pg_cur[r] >= 0 && (int64_t)pg_cur[r] < a.num_pages;
                    if (!is_v) {
                        if (exists && !idx_ok) report(a.err_flag, KVQ_DEV_BAD_TOPK);
                        if (idx_ok && !valid[r]) report(a.err_flag, KVQ_DEV_BAD_PAGE);
                        tokpos[slot * G::kTokPerStage + e] = valid[r] ? idx_cur[r] : -1;
                    }
                    cnt += __popc(__ballot_sync(kFull, valid[r]));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(bar0 + 8 * slot, cnt * G::kRowBytes);
                __syncwarp();
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (valid[r]) {
                        const int e = r * 32 + lane;
                        const int64_t row =
                            ((int64_t)pg_cur[r] * a.num_kv_heads + g) * 4 + (idx_cur[r] & 3);
                        const uint32_t dst = ring + slot * G::kStageBytes + (is_v ? G::kRegion : 0) +
                                             (e >> 2) * G::kPageStride + (e & 3) * G::kRowBytes;
                        tma_load_1d(dst, pool + row * G::kRowBytes, G::kRowBytes, bar0 + 8 * slot, pol);
                    }
                    idx_cur[r] = idx_nxt[r];
                    pg_cur[r] = pg_nxt[r];
                    idx_nxt[r] = idx_nxt2[r];
                }
                issued = st + 1;
            }
        }
    return issued;
}

// ---------------------------------------------------------------------------
// Cluster merge (CMERGE instances): the S <= 8 splits of one (sequence, kv
// head) run as one thread-block cluster, split s as cluster rank s.  Every CTA
// writes its partials to the workspace as usual; after one cluster barrier
// (release, then acquire, at cluster scope: the other CTAs' workspace stores
// are visible), CTA s merges rows s, s + S, ... of the group, one warp per
// row, with the combine kernel's merge (the same function, hence the same
// bits), and writes them to `out`.  This replaces the combine launch and its
// wait for the whole grid by a wait for the group's own splits.  Every thread
// of every CTA passes the barrier exactly once, on the give-up path as well.
__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

template <int D>
__device__ __forceinline__ void cluster_merge(const AttnArgs &a, int b, int g, int s, int warp, int lane)
{
    cluster_barrier();
    const int S = a.num_splits;
    for (int lr = s + S * warp; lr < a.rows; lr += S * kThreads / 32) {
        const int i = lr / a.group, h = g * a.group + lr % a.group;
        const int64_t row = ((int64_t)b * a.num_q_heads + h) * a.q_len + i;
        float acc[D / 32];
        const float W = merge_splits<D>(a.ws_o + row * S * D, a.ws_m + row * S, a.ws_l + row * S, S, lane, 0, 1,
                                        acc);
        store_merged<D>(static_cast<__half *>(a.out), b, i, h, a.q_len, a.num_q_heads, lane, acc, W);
    }
}

// BITCAST selects the E4M3 decoder: false = the hardware conversion
// (cvt.rn.f16x2.e4m3x2, the value itself); true = the bitcast decoder of the
// source pages (E4M3 bits placed into fp16 bits, the value * 2^-8, exact),
// with the 2^8 folded into the hoisted scales.  Both give the same fp16
// values up to that power of two, so the outputs are identical.
template <bool E4M3, int D, int NT, int RW, bool BITCAST, bool LPT = false, bool FUSED = false, bool CMERGE = false>
__global__ void __launch_bounds__(kThreads, NT == 1 ? (E4M3 ? 4 : 2) : 1)
    attn_split_kernel(const AttnArgs a)
{
    static_assert(!CMERGE || (NT == 1 && RW == 1 && !LPT), "the cluster merge is for up to 8 rows in index order");
    using W = Split<NT, RW>;
    constexpr int PPS = W::kPagesPerStage;
    constexpr int MTW = W::kTilesPerWarp;
    using G = Geometry<E4M3, D, PPS>;
    extern __shared__ __align__(128) uint8_t smem[];

    const int s = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(smem);
    int32_t *tokpos = reinterpret_cast<int32_t *>(smem + G::kTokPosOff);
    const uint32_t bar0 = smem_u32(smem + G::kBarOff);   // full[k] = bar0 + 8k, empty[k] = bar0 + 8(S+k)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + G::kAbortOff);
    volatile int *stage_bad = abort_flag + 1;            // a bad entry was seen (sticky)

    // barriers first: this part reads no input and overlaps the previous kernel's tail
    if (threadIdx.x == 0) {
        for (int k = 0; k < G::kStages; ++k) {
            mbar_init(bar0 + 8 * k, kProducerWarps);   // one arrive.expect_tx per producer
            mbar_init(bar0 + 8 * (G::kStages + k), kConsumerWarps);
        }
        *abort_flag = 0;
        *stage_bad = 0;
        if constexpr (FUSED && CMERGE) mbar_init(smem_u32(smem + G::kAppBarOff), 2);   // K and V rows appended
        fence_mbar_init();
    }
    __syncthreads();
    // Inputs may come from the preceding kernel (e.g. the append).  Without a
    // top-k list, only q and the pages holding this step's positions (L -
    // q_len and later) can: block tables, context lengths and the earlier
    // pages are read before waiting for it (the producers start copying at
    // once; the consumers wait before reading q).  With a top-k list, whose
    // lists a preceding kernel may write, or with strict ordering, everything
    // waits here.  The fused step's preceding kernel may be the previous
    // step's fused launch (with the cluster merge nothing else runs between
    // them), which wrote its q_len <= 4 rows just below this step's window
    // (decode: position L - 2; verify: up to 4 positions below L - q_len), so
    // its instances copy early only the pages below position L - q_len - 4.
    const bool early = a.early_pages && a.topk_idx == nullptr;
    if (!early) grid_dependency_wait();
    launch_dependents();      // the combine may start launching; it waits for our completion

    // ---- work of this CTA --------------------------------------------------
    // The producers' first block-table batch is fetched speculatively for a
    // sequence that fills its block-table row, in parallel with the context
    // length; it is refetched below if the real split starts elsewhere.
    // Blocks take the sequences in index order, or (LPT, the instances that
    // KVQ_ATTN_LONGEST_FIRST selects) longest first: that pays a
    // classification of every sequence in each CTA's prologue, which returns
    // it only when lengths vary over a grid of several waves.
    SeqPick pick = seq_identity(a, blockIdx.z);
    if (LPT && !__syncthreads_and(lpt_classify(a, smem, G::kRingBytes))) pick = lpt_pick(a, blockIdx.z, smem);
    const int b = pick.b;
    const SplitRange sr = split_range(a, s, b, pick.L, pick.topk_len);
    const int L = sr.L, item0 = sr.item0, item1 = sr.item1;
    const bool len_ok = sr.len_ok, topk = sr.topk;
    int bt_spec = -1;
    if (warp >= kConsumerWarps && sr.spec0 + lane < a.max_pages) bt_spec = __ldg(sr.bt_row + sr.spec0 + lane);
    const int ipst = topk ? G::kTokPerStage : PPS;        // items per stage
    const int nst = (item1 - item0 + ipst - 1) / ipst;

    if (threadIdx.x == 0) {
        if (!len_ok) report(a.err_flag, KVQ_DEV_BAD_LEN);
        if (len_ok && pick.topk_len > a.max_topk)
            report(a.err_flag, KVQ_DEV_BAD_TOPK);
    }

    float o[NT][G::kPVTiles][4];
    float m_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int pv = 0; pv < G::kPVTiles; ++pv)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[j][pv][e] = 0.f;
        m_run[j][0] = m_run[j][1] = -INFINITY;
        l_run[j][0] = l_run[j][1] = 0.f;
    }
    const int gid = lane >> 2, t = lane & 3;
    const int rw = warp % RW, tw = warp / RW;
    int issued = 0;   // stages this producer has issued

    if (warp >= kConsumerWarps) {
        // ================= producers: the first moves K, the second V =================
        const bool is_v = warp == kConsumerWarps + 1;
        constexpr int kPrevRows = FUSED ? 4 : 0;   // rows a preceding fused step may have written below the window
        constexpr int kFmode = FUSED ? (CMERGE ? 2 : 1) : 0;
        issued = produce_stages<G, PPS, kFmode>(a, sr, nst, b, g, lane, is_v, bt_spec, ring, bar0, tokpos, abort_flag,
                                                stage_bad, early ? max(L - a.q_len - kPrevRows, 0) / 4 : -1,
                                                smem_u32(smem + G::kAppBarOff));
    } else {
        if (early) grid_dependency_wait();
        if constexpr (FUSED && CMERGE) {
            // consumer warps 0 (K) and 1 (V) append this split's new rows while the producers copy
            // the earlier pages; the producers copy the rows' pages after the arrival
            if (warp < 2 && nst > 0 && max(L - a.q_len, 0) / 4 < item1) {
                append_step_rows<G>(a, sr, b, g, lane, warp == 1);
                if (lane == 0) mbar_arrive(smem_u32(smem + G::kAppBarOff));
            }
        }
        int c_nst = nst;   // stages this consumer takes
#ifdef KVQ_TEST_STALL_CONSUMERS
        // Test builds only (never the library's default build): before their
        // first stage the consumers wait, with a bound of
        // KVQ_TEST_STALL_CONSUMERS nanoseconds, on slot 0's empty barrier,
        // which completes only after the consumers themselves release slot 0.
        // The wait therefore always gives up, and the give-up path below runs.
        if (!mbar_wait_bounded(bar0 + 8 * G::kStages, 0, abort_flag, a.err_flag, KVQ_TEST_STALL_CONSUMERS))
            c_nst = 0;
#endif
        // ================= consumers =================
        // Q as mma B fragments, one set per 8-row n-tile; k-step ks of this
        // lane covers channels 16ks + 4t .. +3 (E4M3: the pairs the hardware
        // conversion makes from adjacent K bytes) or 16ks + 2t, +1 and
        // 16ks + 8 + 2t, +1 (fp16).
        uint32_t qf[NT][G::kKSteps][2];
        int lim[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int row = (rw * NT + j) * 8 + gid;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int r = (rw * NT + j) * 8 + 2 * t + c;
                lim[j][c] = (r < a.rows) ? L - a.q_len + r / a.group : 0x7FFFFFFF;
            }
            if (row < a.rows) {
                const int i = row / a.group, h = g * a.group + row % a.group;
                const __half *qrow = static_cast<const __half *>(a.q) +
                                     (((int64_t)b * a.q_len + i) * a.num_q_heads + h) * D;
#pragma unroll
                for (int ks = 0; ks < G::kKSteps; ++ks) {
                    if (E4M3 && BITCAST) {
                        // the bitcast decoder pairs K bytes (0, 2) and (1, 3) of a word
                        const uint2 v = *reinterpret_cast<const uint2 *>(qrow + 16 * ks + 4 * t);
                        qf[j][ks][0] = __byte_perm(v.x, v.y, 0x5410);   // (d, d+2)
                        qf[j][ks][1] = __byte_perm(v.x, v.y, 0x7632);   // (d+1, d+3)
                    } else if (E4M3) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(qrow + 16 * ks + 4 * t);
                        qf[j][ks][0] = v.x;   // (d, d+1)
                        qf[j][ks][1] = v.y;   // (d+2, d+3)
                    } else {
                        qf[j][ks][0] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * t);
                        qf[j][ks][1] = *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 8 + 2 * t);
                    }
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < G::kKSteps; ++ks) qf[j][ks][0] = qf[j][ks][1] = 0u;
            }
        }
        // per-lane ldmatrix offset: matrix q = lane/8 reads row (page) lane%8,
        // token slot (q&1) of the tile's slot pair, 16-byte chunk (q>>1) of the pair
        const int mq = lane >> 3;
        const uint32_t lane_off = (lane & 7) * G::kPageStride + (mq & 1) * G::kRowBytes + (mq >> 1) * 16;
        // this warp's tiles: tile index tg -> page group tg/2, slot pair tg%2
        uint32_t tile_off[MTW];
        int tile_pg[MTW], tile_sp[MTW];
#pragma unroll
        for (int k = 0; k < MTW; ++k) {
            const int tg = tw * MTW + k;
            tile_pg[k] = tg >> 1;
            tile_sp[k] = tg & 1;
            tile_off[k] = tile_pg[k] * 8 * G::kPageStride + tile_sp[k] * 2 * G::kRowBytes + lane_off;
        }
        // the bitcast decoder yields K * 2^-8: its 2^8 joins the hoisted multiplier
        const float qk = a.qk_scale_log2 * (E4M3 && BITCAST ? 256.f : 1.f);
        const int first_masked = L - a.q_len + 1;   // positions >= this are masked for some row

        for (int st = 0; st < c_nst; ++st) {
            const int slot = st % G::kStages;
            if (!mbar_wait_bounded(bar0 + 8 * slot, (st / G::kStages) & 1, abort_flag, a.err_flag))
                break;
            const uint32_t sk = ring + slot * G::kStageBytes;
            const uint32_t sv = sk + G::kRegion;
            const int32_t *tp = tokpos + slot * G::kTokPerStage;
            // Mask when some slot of the stage may hold no valid token for some
            // row: top-k lists, bad pages, a stage with missing pages (their
            // slots keep whatever an earlier stage left there), or positions
            // inside the verify window / past the context end.
            const int stage_end = item0 + (st + 1) * PPS;
            const bool need_mask = topk || *stage_bad || stage_end > item1 ||
                                   stage_end * 4 - 1 >= first_masked;

            // ---- S^T = K Q^T, one 16-token tile at a time ----
            float sc[NT][MTW][4];
            float sc2[NT > 1 ? NT : 1][MTW][4];
#pragma unroll
            for (int k = 0; k < MTW; ++k) {
                uint32_t kr[G::kX4][4];
#pragma unroll
                for (int u = 0; u < G::kX4; ++u) ldsm_x4(kr[u], sk + tile_off[k] + u * 32);
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[j][k][e] = 0.f;
                if (NT > 1) {
#pragma unroll
                    for (int j = 0; j < (NT > 1 ? NT : 1); ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc2[j][k][e] = 0.f;
                }
#pragma unroll
                for (int ks = 0; ks < G::kKSteps; ++ks) {
                    uint32_t af[4];
                    if (E4M3) {
                        const uint32_t w0 = kr[ks >> 1][2 * (ks & 1)];
                        const uint32_t w1 = kr[ks >> 1][2 * (ks & 1) + 1];
                        if (BITCAST) {
                            af[0] = dec_lo(w0);
                            af[1] = dec_lo(w1);
                            af[2] = dec_hi(w0);
                            af[3] = dec_hi(w1);
                        } else {
                            af[0] = cvt_lo(w0);
                            af[1] = cvt_lo(w1);
                            af[2] = cvt_hi(w0);
                            af[3] = cvt_hi(w1);
                        }
                    } else {
                        af[0] = kr[ks][0];
                        af[1] = kr[ks][1];
                        af[2] = kr[ks][2];
                        af[3] = kr[ks][3];
                    }
                    // with several row tiles, odd k-steps accumulate separately:
                    // twice the independent MMA chains per warp
                    if (NT > 1 && (ks & 1)) {
#pragma unroll
                        for (int j = 0; j < NT; ++j) mma_16816(sc2[j][k], af, qf[j][ks][0], qf[j][ks][1]);
                    } else {
#pragma unroll
                        for (int j = 0; j < NT; ++j) mma_16816(sc[j][k], af, qf[j][ks][0], qf[j][ks][1]);
                    }
                }
                if (NT > 1) {
#pragma unroll
                    for (int j = 0; j < NT; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[j][k][e] += sc2[j][k][e];
                }
            }
            // ---- scores in the log2 domain, masking ----
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int k = 0; k < MTW; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[j][k][e] *= qk;
            if (need_mask) {
#pragma unroll
                for (int k = 0; k < MTW; ++k) {
                    const int pbase = (tile_pg[k] * 8 + gid) * 4 + 2 * tile_sp[k];
                    const int pa = tp[pbase], pb = tp[pbase + 1];
#pragma unroll
                    for (int j = 0; j < NT; ++j)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            if (!(pa >= 0 && pa <= lim[j][c])) sc[j][k][c] = -INFINITY;
                            if (!(pb >= 0 && pb <= lim[j][c])) sc[j][k][2 + c] = -INFINITY;
                        }
                }
            }
            // ---- online softmax (row max across the 8 lanes sharing t) ----
            // The O rescale is skipped while no row of the warp raised its
            // running max (a factor of exactly 1): after the first tiles a new
            // maximum is rare, and this saves 8 multiplies per row and tile.
            float corr[NT][2];
            bool raised = false;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float mx = fmaxf(sc[j][0][c], sc[j][0][c + 2]);
#pragma unroll
                    for (int k = 1; k < MTW; ++k) mx = fmaxf(mx, fmaxf(sc[j][k][c], sc[j][k][c + 2]));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                    const float m_new = fmaxf(m_run[j][c], mx);
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    const bool up = m_new != m_run[j][c];
                    corr[j][c] = up ? fast_exp2(m_run[j][c] - m_use) : 1.f;
                    raised |= up;
                    m_run[j][c] = m_new;
                    float lsum = l_run[j][c] * corr[j][c];
#pragma unroll
                    for (int k = 0; k < MTW; ++k) {
                        const float p0 = fast_exp2(sc[j][k][c] - m_use);
                        const float p1 = fast_exp2(sc[j][k][c + 2] - m_use);
                        sc[j][k][c] = p0;
                        sc[j][k][c + 2] = p1;
                        lsum += p0 + p1;
                    }
                    l_run[j][c] = lsum;
                }
            if (__any_sync(kFull, raised)) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int pv = 0; pv < G::kPVTiles; ++pv) {
                        o[j][pv][0] *= corr[j][0];
                        o[j][pv][2] *= corr[j][0];
                        o[j][pv][1] *= corr[j][1];
                        o[j][pv][3] *= corr[j][1];
                    }
            }
            // ---- P^T as mma B fragments: transpose the score tiles in registers ----
            uint32_t pf[NT][MTW][2];
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int k = 0; k < MTW; ++k) {
                    pf[j][k][0] = movmatrix_trans(pack_half2(sc[j][k][0], sc[j][k][1]));
                    pf[j][k][1] = movmatrix_trans(pack_half2(sc[j][k][2], sc[j][k][3]));
                }
            // ---- O^T += V^T P^T ----
#pragma unroll
            for (int k = 0; k < MTW; ++k) {
                uint32_t vr[G::kX4][4];
#pragma unroll
                for (int u = 0; u < G::kX4; ++u) ldsm_x4_trans(vr[u], sv + tile_off[k] + u * 32);
                if (need_mask) {
                    // Slots that hold no token may contain any bits -- fp16 NaN, or
                    // the E4M3 NaN codes 0x7F/0xFF, which the conversion turns into
                    // NaN -- so their V is zeroed (P = 0 alone would give 0 * NaN).
                    // Token (page 2t) sits in the low half of each word, (page 2t+1)
                    // in the high half, for both element sizes.
                    const int q0 = (tile_pg[k] * 8 + 2 * t) * 4 + 2 * tile_sp[k];
                    const uint32_t m0 = (tp[q0] >= 0 ? 0x0000FFFFu : 0u) |
                                        (tp[q0 + 4] >= 0 ? 0xFFFF0000u : 0u);
                    const uint32_t m1 = (tp[q0 + 1] >= 0 ? 0x0000FFFFu : 0u) |
                                        (tp[q0 + 5] >= 0 ? 0xFFFF0000u : 0u);
#pragma unroll
                    for (int u = 0; u < G::kX4; ++u) {
                        vr[u][0] &= m0;
                        vr[u][2] &= m0;
                        vr[u][1] &= m1;
                        vr[u][3] &= m1;
                    }
                }
#pragma unroll
                for (int pv = 0; pv < G::kPVTiles; ++pv) {
                    uint32_t af[4];
                    if (E4M3) {
                        // bytes of a word: (token A, d) (A, d+1) (B, d) (B, d+1)
                        const uint32_t h0 = vr[pv >> 1][2 * (pv & 1)];
                        const uint32_t h1 = vr[pv >> 1][2 * (pv & 1) + 1];
                        if (BITCAST) {
                            af[0] = dec_lo(h0);
                            af[1] = dec_hi(h0);
                            af[2] = dec_lo(h1);
                            af[3] = dec_hi(h1);
                        } else {
                            const uint32_t p0 = __byte_perm(h0, 0, 0x3120);
                            const uint32_t p1 = __byte_perm(h1, 0, 0x3120);
                            af[0] = cvt_lo(p0);
                            af[1] = cvt_hi(p0);
                            af[2] = cvt_lo(p1);
                            af[3] = cvt_hi(p1);
                        }
                    } else {
                        af[0] = vr[pv][0];
                        af[1] = vr[pv][2];
                        af[2] = vr[pv][1];
                        af[3] = vr[pv][3];
                    }
#pragma unroll
                    for (int j = 0; j < NT; ++j) mma_16816(o[j][pv], af, pf[j][k][0], pf[j][k][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * (G::kStages + slot));
        }
        // full row sums: add the partial sums of the 8 lanes sharing t
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v = l_run[j][c];
                v += __shfl_xor_sync(kFull, v, 4);
                v += __shfl_xor_sync(kFull, v, 8);
                v += __shfl_xor_sync(kFull, v, 16);
                l_run[j][c] = v;
            }
    }

    // ---- merge the token warps through shared memory, write the split partial ----
    volatile int *issued_by = abort_flag + 2;            // [2]: stages the K and V producers issued
    if (warp >= kConsumerWarps && lane == 0) issued_by[warp - kConsumerWarps] = issued;
    __syncthreads();
    if (*abort_flag) {
        // Something gave up.  Before the CTA's shared memory is released,
        // every bulk copy in flight must land.  A stage's full barrier counts
        // one arrival per producer, so a stage that only one producer issued
        // could never complete: the other producer arrives for it here
        // (without copies).  Neither producer is more than kStages stages
        // ahead of the other (a producer reuses a slot only after the
        // consumers released it, which needs both producers' copies of the
        // slot's previous stage), so the stages [hi - kStages, hi), hi = the
        // larger count, sit in distinct slots, every earlier stage has
        // completed, and each of them completes once its copies land.  The
        // waits are bounded all the same.  Then the CTA's rows get zero weight
        // in the workspace (m = -inf, l = 0), so that the combine ignores
        // this split, and the CTA leaves.  The error bit is already set.
        if (warp >= kConsumerWarps && lane == 0) {
            const int mine = issued, other = issued_by[kConsumerWarps + 1 - warp];
            for (int st = mine; st < other; ++st) mbar_arrive(bar0 + 8 * (st % G::kStages));
            const int hi = max(mine, other);
            for (int st = max(0, hi - G::kStages); st < hi; ++st)
                mbar_wait_bounded(bar0 + 8 * (st % G::kStages), (st / G::kStages) & 1, nullptr,
                                  a.err_flag, 100000000ull);
        }
        for (int row = threadIdx.x; row < a.rows; row += kThreads) {
            const int i = row / a.group, h = g * a.group + row % a.group;
            const int64_t unit = (((int64_t)b * a.num_q_heads + h) * a.q_len + i) * a.num_splits + s;
            a.ws_m[unit] = -INFINITY;
            a.ws_l[unit] = 0.f;
        }
        __syncthreads();
        if constexpr (CMERGE) cluster_merge<D>(a, b, g, s, warp, lane);
        return;
    }
    float *mbuf = reinterpret_cast<float *>(smem);    // [token warps][kRowsPad][D + 2]: m, l, o[D]
    constexpr int kRowF = D + 2;
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int row = (rw * NT + j) * 8 + 2 * t + c;
                float *dst = mbuf + (tw * W::kRowsPad + row) * kRowF;
                if (gid == 0) {
                    dst[0] = m_run[j][c];
                    dst[1] = l_run[j][c];
                }
#pragma unroll
                for (int pv = 0; pv < G::kPVTiles; ++pv) {
                    const int2 ch = pv_channels<E4M3>(pv, gid);
                    dst[2 + ch.x] = o[j][pv][c];
                    dst[2 + ch.y] = o[j][pv][c + 2];
                }
            }
    }
    __syncthreads();
    // Per row: the merge weights of the token warps (w_q / l, v_scale folded
    // in), and the split's m and l; an empty row gets m = -inf, l = 0 and no
    // output.
    constexpr int TW = W::kTokWarps;
    const int S = a.num_splits;
    // the bitcast decoder yields V * 2^-8; the hardware conversion V itself
    constexpr float kVFold = (E4M3 && BITCAST) ? 256.f : 1.f;
    float *coef = mbuf + TW * W::kRowsPad * kRowF;        // [kRowsPad][TW]
    for (int row = threadIdx.x; row < a.rows; row += kThreads) {
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < TW; ++q) M = fmaxf(M, mbuf[(q * W::kRowsPad + row) * kRowF]);
        const int i = row / a.group, h = g * a.group + row % a.group;
        const int64_t unit = (((int64_t)b * a.num_q_heads + h) * a.q_len + i) * S + s;
        float w[TW];
        float lsum = 0.f;
#pragma unroll
        for (int q = 0; q < TW; ++q) {
            const float *src = mbuf + (q * W::kRowsPad + row) * kRowF;
            w[q] = (M == -INFINITY) ? 0.f : fast_exp2(src[0] - M);
            lsum += w[q] * src[1];
        }
        const float inv = lsum > 0.f ? a.out_scale * kVFold / lsum : 0.f;
#pragma unroll
        for (int q = 0; q < TW; ++q) coef[row * TW + q] = w[q] * inv;
        a.ws_m[unit] = lsum > 0.f ? M * kLn2 : -INFINITY;
        a.ws_l[unit] = lsum;
    }
    __syncthreads();
    // o = sum_q coef_q * o_q, four channels per thread, stored as float4
    for (int idx = threadIdx.x * 4; idx < a.rows * D; idx += kThreads * 4) {
        const int row = idx / D, d = idx % D;
        const float *cf = coef + row * TW;
        bool any = false;
#pragma unroll
        for (int q = 0; q < TW; ++q) any |= cf[q] != 0.f;
        if (!any) continue;                        // empty row: tmp_out stays unwritten
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < TW; ++q) {
            const float c = cf[q];
            const float *src = mbuf + (q * W::kRowsPad + row) * kRowF + 2 + d;
            acc.x += c * src[0];
            acc.y += c * src[1];
            acc.z += c * src[2];
            acc.w += c * src[3];
        }
        const int i = row / a.group, h = g * a.group + row % a.group;
        const int64_t unit = (((int64_t)b * a.num_q_heads + h) * a.q_len + i) * S + s;
        *reinterpret_cast<float4 *>(a.ws_o + unit * D + d) = acc;
    }
    if constexpr (CMERGE) cluster_merge<D>(a, b, g, s, warp, lane);
}

// ---------------------------------------------------------------------------
// host launchers

template <bool E4M3, int D, int NT, int RW, bool BITCAST, bool LPT, bool FUSED, bool CMERGE = false>
static cudaError_t launch_one(const AttnArgs &a, cudaStream_t stream)
{
    constexpr int bytes = smem_bytes<E4M3, D, NT, RW>();
    static uint64_t configured = 0;   // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(attn_split_kernel<E4M3, D, NT, RW, BITCAST, LPT, FUSED, CMERGE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    const dim3 grid(a.num_splits, a.num_kv_heads, a.batch);
    if constexpr (CMERGE) {
        // one cluster per (sequence, kv head): its splits along x
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = bytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)a.num_splits;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, attn_split_kernel<E4M3, D, NT, RW, BITCAST, LPT, FUSED, CMERGE>, a);
    }
    return launch_pdl(attn_split_kernel<E4M3, D, NT, RW, BITCAST, LPT, FUSED>, grid, dim3(kThreads), bytes, stream,
                      a);
}

template <bool E4M3, int D, bool BITCAST, bool LPT = false, bool FUSED = false>
static cudaError_t launch_rows(const AttnArgs &a, cudaStream_t stream)
{
    const int tiles = (a.rows + 7) / 8;
    if (tiles <= 1) return launch_one<E4M3, D, 1, 1, BITCAST, LPT, FUSED>(a, stream);
    if (tiles <= 2) return launch_one<E4M3, D, 2, 1, BITCAST, LPT, FUSED>(a, stream);
    if (tiles <= 4) return launch_one<E4M3, D, 2, 2, BITCAST, LPT, FUSED>(a, stream);
    return launch_one<E4M3, D, 2, 4, BITCAST, LPT, FUSED>(a, stream);
}

}  // namespace kvq
