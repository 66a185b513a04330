// kvq_prefill.cu -- chunked-prefill attention over the paged cache.
//
// What is computed: the attention of the decode path with q_len = the chunk
// length -- PR "[Model][SM70][FP8] Integrate calibrated E4M3 QSA KV capacity
// path", section Changes (mixed catch-up/decode batches append prefill chunks
// to the same page-4 cache); PR "[Model][SM70] Calibrated E4M3 KV cache for
// Qwen4Exp QSA with MTP", section Purpose (causal inside the window of new
// tokens).  Query token i of a chunk of n tokens in a context of L tokens
// sits at position L - n + i and attends keys 0 .. L - n + i; the per-layer
// scales are hoisted (k_scale into the score multiplier, v_scale into the
// output normalisation).
//
// Design, two launches:
//  1. kv_tile_kernel gathers each (sequence, kv head)'s pages, decodes E4M3
//     to fp16 (exact: every E4M3 value is an fp16 value; the scales stay
//     out) and writes 128-key tiles in the tensor core's no-swizzle canonical
//     layout, with a 128-bit mask per tile of the keys whose block-table
//     entry is outside the pool.  A prefill chunk is re-read by every query
//     tile, so decoding once costs O(L) instead of O(L x query tiles).
//  2. prefill_attn_kernel, persistent: one CTA per SM (320 threads), which
//     takes work items -- (256 query tokens, query head, sequence), two
//     128-row query tiles A and B -- longest first, in rounds over the grid
//     in alternating direction.  The roles run through the CTA's items
//     independently, so that one item's tail overlaps the next item's start:
//     the tiles of the next item stream in behind the current ones, and each
//     softmax group writes its next Q tile (once the MMA thread has taken the
//     current one) before its epilogue, so that the next item's first
//     S = Q K^T runs during that epilogue.
//       warp 8: one thread streams the K and V tiles (one 32 KB 1-D bulk copy
//               each) through a 2-stage shared ring;
//       warp 9: allocates tensor memory; one thread issues the MMAs:
//               S_X = Q_X K^T (M = 128 rows, N = 128 keys, K = 16 per
//               instruction, both K-major in shared memory) and
//               O_X += P_X V (P from tensor memory, V MN-major in shared
//               memory), alternating between the tiles so that the tensor
//               core works on one tile while the other's softmax runs;
//       warps 0-3 (tile A) and 4-7 (tile B): thread r of a group owns row r
//               of its tile (tensor-memory lane r): reads its 128 scores,
//               masks the causal diagonal, and writes P (fp16) over the S it
//               read.  A row's reference moves only when a score rises more
//               than 2^8 above it (the O row is then rescaled in tensor
//               memory); the row sum stays in a register.
//     Every wait is bounded (about 2 s); on expiry the CTA reports
//     KVQ_DEV_TIMEOUT, lets its copies and MMAs drain, frees its tensor
//     memory and exits without writing.  Every tensor-memory load and store
//     and every barrier is reached by whole warps.
#include <algorithm>
#include <cstdint>
#include <type_traits>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tcgen05.cuh"

namespace kvq {

namespace {

constexpr int kPfTile = 128;                        // keys per KV tile = query rows per CTA
constexpr int kPfD = 128;                           // head_dim of this path
constexpr int kPfTileBytes = kPfTile * kPfD * 2;    // one fp16 tile: 32 KB
constexpr int kPfStages = 2;
constexpr int kPfThreads = 320;
constexpr int kPfSoftmaxWarps = 8;                  // two groups of 4, one per query tile
constexpr int kPfLoadWarp = 8;
constexpr int kPfMmaWarp = 9;
constexpr unsigned kPfFull = 0xFFFFFFFFu;

// shared memory: the two Q tiles, the ring of (K, V) tile pairs, mbarriers, tensor-memory slot
constexpr int kPfQ = 0;
constexpr int kPfRing = kPfQ + 2 * kPfTileBytes;
constexpr int kPfBar = kPfRing + kPfStages * 2 * kPfTileBytes;
// barriers: full[2], empty[2], q[2], q taken[2], s[2], p[2], pv[2], drain
constexpr int kPfNumBars = 2 * kPfStages + 2 + 2 + 2 + 2 + 2 + 1;
constexpr int kPfAbort = kPfBar + 8 * kPfNumBars;
constexpr int kPfTmemSlot = kPfAbort + 8;
constexpr int kPfSmemBytes = kPfTmemSlot + 8;
static_assert(kPfSmemBytes <= 232448, "prefill shared memory exceeds one CTA's limit");

// tensor-memory columns: S_A, S_B (P written over the first 64 columns of the
// S it came from), O_A, O_B
constexpr uint32_t kPfColS = 0, kPfColO = 2 * kPfTile, kPfCols = 512;

// Byte offset of element (row, col) of a 128 x 128 fp16 tile in the
// canonical no-swizzle layout: 8 x 16-byte core matrices, 8 rows of 8
// elements each, rows of a core matrix 16 bytes apart, core matrices 128
// bytes apart along the column direction and 2048 bytes apart along the
// row direction.  For K (row = key, col = channel) it is the K-major
// operand of S = Q K^T; for V (row = key, col = channel) the MN-major
// operand of O = P V; for Q (row = query row) the K-major A operand.
__device__ __forceinline__ uint32_t tile_off(int row, int col8)
{
    return (uint32_t)((row >> 3) * 2048 + col8 * 128 + (row & 7) * 16);
}

// a chunk that can be attended: non-empty, inside q / out, inside its context
__device__ __forceinline__ bool seq_ok(const PrefillArgs &a, int q0, int q1, int L)
{
    const int n = q1 - q0;
    return n >= 1 && n <= a.max_q_len && q0 >= 0 && q1 <= a.total_q && L >= n && L <= a.max_pages * 4;
}

}  // namespace

// ---------------------------------------------------------------------------
// 1. pages -> fp16 tiles

template <bool E4M3>
__global__ void __launch_bounds__(256) kv_tile_kernel(const PrefillArgs a)
{
    // four blocks per tile: K or V (kv), keys 0-63 or 64-127 (kh)
    const int j = blockIdx.x >> 2, kv = (blockIdx.x >> 1) & 1, kh = blockIdx.x & 1;
    const int g = blockIdx.y, b = blockIdx.z;
    grid_dependency_wait();
    launch_dependents();
    const int L = __ldg(a.context_lens + b);
    const int q0 = __ldg(a.q_start + b);
    if (!seq_ok(a, q0, __ldg(a.q_start + b + 1), L)) return;   // flagged by the attention kernel
    if (j * kPfTile >= L) return;
    const int32_t *bt_row = a.block_tables + (int64_t)b * a.max_pages;
    const int64_t tile = ((int64_t)b * a.num_kv_heads + g) * a.max_tiles + j;
    uint8_t *dst = a.tiles + tile * 2 * kPfTileBytes;
    constexpr int kElem = E4M3 ? 1 : 2;
    __shared__ uint32_t bad[2];   // this block's keys whose page is outside the pool (K blocks)
    if (threadIdx.x < 2) bad[threadIdx.x] = 0u;
    __syncthreads();
    // item = (key n8 group, 8-channel group c8, key n%8), key fastest: the 8
    // lanes of a quarter warp write one 128-byte core-matrix row block.  A
    // thread's KI items load their page entries, then their rows, before any
    // store, so that two memory round trips cover them.
    constexpr int kHalf = kPfTile / 2;
    constexpr int KI = kHalf * (kPfD / 8) / 256;   // items per thread (4)
    static_assert(KI * 256 == kHalf * (kPfD / 8), "the block's items divide evenly");
    const uint8_t *pool = static_cast<const uint8_t *>(kv ? a.v_cache : a.k_cache);
    int key[KI], c8[KI], page[KI];
    bool in_ctx[KI];
#pragma unroll
    for (int u = 0; u < KI; ++u) {
        const int r = threadIdx.x + 256 * u;
        key[u] = kh * kHalf + (r / (8 * (kPfD / 8))) * 8 + (r & 7);
        c8[u] = (r / 8) % (kPfD / 8);
        const int pos = j * kPfTile + key[u];
        in_ctx[u] = pos < L;
        page[u] = in_ctx[u] ? __ldg(bt_row + (pos >> 2)) : -1;
    }
    using Raw = typename std::conditional<E4M3, uint2, uint4>::type;
    Raw x[KI];
#pragma unroll
    for (int u = 0; u < KI; ++u) {
        const int pos = j * kPfTile + key[u];
        if (in_ctx[u] && page[u] >= 0 && page[u] < a.num_pages)
            x[u] = __ldg(reinterpret_cast<const Raw *>(
                pool + ((((int64_t)page[u] * a.num_kv_heads + g) * 4 + (pos & 3)) * kPfD + c8[u] * 8) * kElem));
    }
#pragma unroll
    for (int u = 0; u < KI; ++u) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);   // keys past the context: zero (and masked)
        if (in_ctx[u] && page[u] >= 0 && page[u] < a.num_pages) {
            if constexpr (E4M3)
                v = make_uint4(cvt_lo(x[u].x), cvt_hi(x[u].x), cvt_lo(x[u].y), cvt_hi(x[u].y));
            else
                v = x[u];
        } else if (in_ctx[u] && kv == 0 && c8[u] == 0) {
            report(a.err_flag, KVQ_DEV_BAD_PAGE);   // the row stays zero and its key is masked
            atomicOr(&bad[(key[u] - kh * kHalf) >> 5], 1u << (key[u] & 31));
        }
        *reinterpret_cast<uint4 *>(dst + kv * kPfTileBytes + tile_off(key[u], c8[u])) = v;
    }
    __syncthreads();
    if (kv == 0 && threadIdx.x < 2) a.tile_mask[tile * 4 + 2 * kh + threadIdx.x] = bad[threadIdx.x];
}

// ---------------------------------------------------------------------------
// 2. flash attention over the tiles

// Work items: (sequence b, query head h, pair of query tiles), longest first.
// Item i has rank r = i / (B Hq) from the top (pair = pairs(b) - 1 - r), and
// b = (i % (B Hq)) % B, h = (i % (B Hq)) / B.  An item whose sequence has
// fewer pairs, or is not a valid chunk, is empty (pair < 0).  Each CTA takes
// its items in rounds of gridDim.x, in alternating direction, so that the
// CTAs' shares of the descending sizes even out.
struct PfItem {
    int b, h, pair, q0, n, L;
};

__device__ __forceinline__ PfItem pf_item(const PrefillArgs &a, int i)
{
    PfItem it;
    const int per = a.batch * a.num_q_heads;
    const int rnk = i / per, rem = i - rnk * per;
    it.b = rem % a.batch;
    it.h = rem / a.batch;
    it.q0 = __ldg(a.q_start + it.b);
    const int q1 = __ldg(a.q_start + it.b + 1);
    it.n = q1 - it.q0;
    it.L = __ldg(a.context_lens + it.b);
    it.pair = seq_ok(a, it.q0, q1, it.L) ? (it.n + 2 * kPfTile - 1) / (2 * kPfTile) - 1 - rnk : -1;
    return it;
}

__device__ __forceinline__ int pf_item_index(int k)
{
    const int G = gridDim.x, c = blockIdx.x;
    return k * G + ((k & 1) ? G - 1 - c : c);
}

// key tiles a row of tile x of the item sees (0: no rows)
__device__ __forceinline__ int pf_tiles_of(const PfItem &it, int x)
{
    const int lo = it.pair * 2 * kPfTile + x * kPfTile;
    return lo < it.n ? (it.L - it.n + min(it.n, lo + kPfTile) - 1) / kPfTile + 1 : 0;
}

// this CTA's next non-empty item from position k on; false when none is left
__device__ __forceinline__ bool pf_next(const PrefillArgs &a, int total, int &k, PfItem &it)
{
    for (;; ++k) {
        const int i = pf_item_index(k);
        if (i >= total) return false;
        it = pf_item(a, i);
        if (it.pair >= 0) return true;
    }
}

template <bool E4M3>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_attn_kernel(const PrefillArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = ((a.max_q_len + 2 * kPfTile - 1) / (2 * kPfTile)) * a.batch * a.num_q_heads;

    // chunks that cannot be attended are flagged once per launch
    // (q_start and context_lens are read before grid_dependency_wait: the
    // previous kernel, the tile gather, does not write them)
    if (blockIdx.x == 0 && threadIdx.x == 0)
        for (int bb = 0; bb < a.batch; ++bb) {
            const int q0 = __ldg(a.q_start + bb), q1 = __ldg(a.q_start + bb + 1), L = __ldg(a.context_lens + bb);
            const int n = q1 - q0;
            const bool empty_ok = n == 0 && q0 >= 0 && q0 <= a.total_q && L >= 0 && L <= a.max_pages * 4;
            if (!seq_ok(a, q0, q1, L) && !empty_ok) report(a.err_flag, KVQ_DEV_BAD_LEN);
        }

    const uint32_t bar = smem_u32(smem + kPfBar);
    auto full = [&](int s) { return bar + 8 * s; };
    auto empty = [&](int s) { return bar + 8 * (kPfStages + s); };
    // per query tile X (at + 8 X): its Q written (softmax group -> MMA), its Q
    // taken (MMA -> softmax group), S ready, P ready, P V complete
    const uint32_t b_q0 = bar + 8 * (2 * kPfStages);
    const uint32_t b_qf0 = b_q0 + 16, b_s0 = b_q0 + 32, b_p0 = b_q0 + 48, b_pv0 = b_q0 + 64, b_drain = b_q0 + 80;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kPfAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kPfTmemSlot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(b_q0 + 8 * x, kPfSoftmaxWarps / 2);
            mbar_init(b_qf0 + 8 * x, 1);
            mbar_init(b_s0 + 8 * x, 1);
            mbar_init(b_p0 + 8 * x, kPfSoftmaxWarps / 2);
            mbar_init(b_pv0 + 8 * x, 1);
        }
        mbar_init(b_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kPfMmaWarp) tmem_alloc(smem_u32(tmem_slot), kPfCols);
    grid_dependency_wait();   // the tiles come from the previous kernel
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    launch_dependents();      // this CTA holds its tensor memory already
    const uint32_t tmem = *tmem_slot;
    int issued = 0;           // K/V tile pairs this CTA's load warp issued, over all its items

    if (warp == kPfLoadWarp) {
        // ================= tile loads: every item's key tiles, in order =================
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();   // every query tile of the group re-reads them
            bool ok = true;
            PfItem it;
            for (int k = 0; ok && pf_next(a, total, k, it); ++k) {
                const int ntiles = max(pf_tiles_of(it, 0), pf_tiles_of(it, 1));
                const uint8_t *src =
                    a.tiles + (((int64_t)it.b * a.num_kv_heads + it.h / a.group) * a.max_tiles) * 2 * kPfTileBytes;
                for (int t = 0; t < ntiles; ++t) {
                    const int T = issued, s = T % kPfStages;
                    if (T >= kPfStages &&
                        !mbar_wait_bounded(empty(s), ((T / kPfStages) - 1) & 1, abort_flag, a.err_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full(s), 2 * kPfTileBytes);
                    const uint32_t dst = smem_u32(smem + kPfRing + s * 2 * kPfTileBytes);
                    tma_load_1d(dst, src + (int64_t)t * 2 * kPfTileBytes, kPfTileBytes, full(s), pol);
                    tma_load_1d(dst + kPfTileBytes, src + ((int64_t)t * 2 + 1) * kPfTileBytes, kPfTileBytes,
                                full(s), pol);
                    ++issued;
                }
            }
        }
        __syncwarp();   // the whole warp reaches the teardown barrier together
    } else if (warp == kPfMmaWarp) {
        // ================= MMA issue (one thread) =================
        if (lane == 0) {
            const uint32_t id_qk = umma_idesc_f16(kPfTile, kPfTile, false, false);
            const uint32_t id_pv = umma_idesc_f16(kPfTile, kPfD, false, true);
            const uint32_t q_addr = smem_u32(smem + kPfQ);
            // S_X = Q_X K_T^T (T: the CTA's running tile count).  S_X last held P_X
            // of the previous tile, which the P V issued before this has read
            // (MMAs of one thread run in order).
            // descriptors built once per operand; a K step adds its byte offset / 16 to the
            // start-address field (bits 0..13), which the shared-memory addresses never overflow
            auto qk = [&](int x, int T) {
                const uint32_t k_addr = smem_u32(smem + kPfRing + (T % kPfStages) * 2 * kPfTileBytes);
                const uint64_t dq = umma_desc(q_addr + x * kPfTileBytes, 128, 2048);
                const uint64_t dk = umma_desc(k_addr, 128, 2048);
#pragma unroll
                for (int ks = 0; ks < kPfD / 16; ++ks)
                    umma_smem_a(tmem + kPfColS + x * kPfTile, dq + (uint64_t)(ks * 16), dk + (uint64_t)(ks * 16),
                                id_qk, ks > 0);
                umma_commit(b_s0 + 8 * x);
            };
            // O_X (+)= P_X V_T: A = P (tensor memory, two fp16 per column), B = V (MN-major)
            auto pv = [&](int x, int T, bool acc) {
                const uint32_t v_addr = smem_u32(smem + kPfRing + (T % kPfStages) * 2 * kPfTileBytes + kPfTileBytes);
                const uint64_t dv = umma_desc(v_addr, 2048, 128);
#pragma unroll
                for (int ks = 0; ks < kPfTile / 16; ++ks)
                    umma_tmem_a(tmem + kPfColO + x * kPfTile, tmem + kPfColS + x * kPfTile + ks * 8,
                                dv + (uint64_t)(ks * 256), id_pv, acc || ks > 0);
                umma_commit(b_pv0 + 8 * x);
            };
            auto wait_full = [&](int T) {
                if (!mbar_wait_bounded(full(T % kPfStages), (T / kPfStages) & 1, abort_flag, a.err_flag)) return false;
                tc_fence_after();
                return true;
            };
            int T0 = 0, ni = 0, np[2] = {0, 0};   // tiles before this item, items, P waits per tile
            bool ok = true;
            PfItem it;
            for (int k = 0; ok && pf_next(a, total, k, it); ++k, ++ni) {
                const int nt_a = pf_tiles_of(it, 0), nt_b = pf_tiles_of(it, 1);
                const int ntiles = max(nt_a, nt_b);
                // both query tiles of the item in shared memory; their groups may then write the next item's
                for (int x = 0; x < 2 && ok; ++x) {
                    ok = mbar_wait_bounded(b_q0 + 8 * x, ni & 1, abort_flag, a.err_flag);
                    mbar_arrive(b_qf0 + 8 * x);
                }
                tc_fence_after();
                if (!ok || !wait_full(T0)) {
                    ok = false;
                    break;
                }
                if (nt_a > 0) qk(0, T0);
                if (nt_b > 0) qk(1, T0);
                for (int t = 0; ok && t < ntiles; ++t) {
                    if (t < nt_a) {
                        if (!mbar_wait_bounded(b_p0, np[0]++ & 1, abort_flag, a.err_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        pv(0, T0 + t, t > 0);
                    }
                    const bool next = t + 1 < ntiles;
                    if (next && !wait_full(T0 + t + 1)) {
                        ok = false;
                        break;
                    }
                    if (t + 1 < nt_a) qk(0, T0 + t + 1);
                    if (t < nt_b) {
                        if (!mbar_wait_bounded(b_p0 + 8, np[1]++ & 1, abort_flag, a.err_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        pv(1, T0 + t, t > 0);
                    }
                    umma_commit(empty((T0 + t) % kPfStages));   // the stage's K and V are read once these complete
                    if (t + 1 < nt_b) qk(1, T0 + t + 1);
                }
                T0 += ntiles;
            }
            // every MMA issued so far completes before the tensor memory is freed
            umma_commit(b_drain);
            mbar_wait_bounded(b_drain, 0, nullptr, a.err_flag, 100000000ull);
        }
        __syncwarp();
    } else {
        // ================= softmax groups: thread r of group X owns row r of tile X =================
        const int x = warp >> 2;                                // query tile
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t b_q = b_q0 + 8 * x, b_qf = b_qf0 + 8 * x, b_s = b_s0 + 8 * x, b_p = b_p0 + 8 * x,
                       b_pv = b_pv0 + 8 * x;
        const uint32_t sb = tmem + lane_base + kPfColS + x * kPfTile;
        const uint32_t ob = tmem + lane_base + kPfColO + x * kPfTile;
        const float qk = a.qk_scale_log2;
        // this row's Q -> the K-major Q tile of tile X (rows past the chunk: zeros)
        auto load_q = [&](const PfItem &it) {
            const int i = it.pair * 2 * kPfTile + x * kPfTile + r;
            const bool row_ok = i < it.n;
            const __half *qrow = static_cast<const __half *>(a.q) +
                                 ((int64_t)(it.q0 + (row_ok ? i : 0)) * a.num_q_heads + it.h) * kPfD;
#pragma unroll
            for (int c8 = 0; c8 < kPfD / 8; ++c8) {
                const uint4 v = row_ok ? __ldg(reinterpret_cast<const uint4 *>(qrow) + c8) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(smem + kPfQ + x * kPfTileBytes + tile_off(r, c8)) = v;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_q);
        };
        int k = 0, ni = 0, ns = 0, npv = 0;   // item position, items, S waits and P V commits of tile X so far
        bool ok = true;                       // the same on every lane: tensor-memory loads and stores are warp-wide
        PfItem it;
        bool have = pf_next(a, total, k, it);
        if (have) load_q(it);
        while (have && ok) {
            const int h = it.h, g = h / a.group, q0 = it.q0, n = it.n;
            const int base = it.L - n;                              // position of query token 0
            const int i0 = it.pair * 2 * kPfTile;
            const int i = i0 + x * kPfTile + r;                     // query token of this row
            const bool row_ok = i < n;
            const int limit = row_ok ? base + i : -1;               // last key this row sees
            const int nt = pf_tiles_of(it, x);
            const int first_masked = (base + i0 + x * kPfTile) / kPfTile;   // tiles from here on need the causal mask
            const uint32_t *mask_row = a.tile_mask + (((int64_t)it.b * a.num_kv_heads + g) * a.max_tiles) * 4;
            float ref = -INFINITY;   // the row's reference (log2 units)
            float lsum = 0.f;        // sum of 2^(s - ref) over the keys so far
            for (int t = 0; t < nt; ++t) {
                // keys of this tile left out for a bad block-table entry (almost always none)
                const uint4 badk = __ldg(reinterpret_cast<const uint4 *>(mask_row) + t);
                if (!__all_sync(kPfFull, mbar_wait_bounded(b_s, (ns + t) & 1, abort_flag, a.err_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t xr[kPfTile / 16][16];   // the row's 128 scores, loaded together
#pragma unroll
                for (int c = 0; c < kPfTile / 16; ++c) tmem_ld16(sb + 16 * c, xr[c]);
                tmem_wait_ld();
                float xv[kPfTile];
#pragma unroll
                for (int c = 0; c < kPfTile / 16; ++c) {
                    tmem_regs_ready(xr[c]);
#pragma unroll
                    for (int e = 0; e < 16; ++e) xv[16 * c + e] = __uint_as_float(xr[c][e]);
                }
                if ((badk.x | badk.y | badk.z | badk.w) != 0u) {
                    const uint32_t bw[4] = {badk.x, badk.y, badk.z, badk.w};
#pragma unroll
                    for (int c = 0; c < kPfTile; ++c)
                        if ((bw[c >> 5] >> (c & 31)) & 1u) xv[c] = -INFINITY;
                }
                // the row maximum of the raw scores over 8 independent chains (the
                // log2-domain scale qk > 0 is applied after: max(s) * qk = max(s * qk))
                if (t >= first_masked) {
                    const int k0 = t * kPfTile;
#pragma unroll
                    for (int c = 0; c < kPfTile; ++c)
                        if (k0 + c > limit) xv[c] = -INFINITY;
                }
                // (chain u takes columns u, u + 8, ..., u + 120, two more per three-way maximum)
                static_assert(kPfTile == 128, "the maximum's chains cover 128 columns");
                float m8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    float m = fmax3(xv[u], xv[u + 8], xv[u + 16]);
#pragma unroll
                    for (int k = 3; k < 15; k += 2) m = fmax3(m, xv[u + 8 * k], xv[u + 8 * k + 8]);
                    m8[u] = fmaxf(m, xv[u + 120]);
                }
                const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * qk;
                // the reference moves when a score rises more than 2^8 above it; the
                // row's sum and (once PV(t-1) is complete) its O row are rescaled.  The
                // O pass is warp-wide; lanes whose reference stays scale by 1.
                const bool move = mx > ref + 8.f;
                const float corr = !move ? 1.f : (ref == -INFINITY ? 0.f : fast_exp2(ref - mx));
                if (move) {
                    lsum *= corr;
                    ref = mx;
                }
                if (t > 0 && __any_sync(kPfFull, move)) {
                    if (!__all_sync(kPfFull, mbar_wait_bounded(b_pv, (npv + t - 1) & 1, abort_flag, a.err_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kPfD; c += 16) {
                        uint32_t r16[16];
                        tmem_ld16(ob + c, r16);
                        tmem_wait_ld();
                        tmem_regs_ready(r16);
#pragma unroll
                        for (int e = 0; e < 16; ++e) r16[e] = __float_as_uint(__uint_as_float(r16[e]) * corr);
                        tmem_st16(ob + c, r16);
                    }
                }
                // P = 2^(s qk - ref) as fp16 pairs over the first 64 columns of S; the
                // exponents and the row sum two columns per instruction, the sum over
                // four independent pair chains
                const float rf = (ref == -INFINITY) ? 0.f : ref;   // a row with no key yet: P = 0
                const float2 qk2 = make_float2(qk, qk), nrf2 = make_float2(-rf, -rf);
                float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < kPfTile; c += 32) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 z = ffma2(make_float2(xv[c + 2 * e], xv[c + 2 * e + 1]), qk2, nrf2);
                        const float2 p = make_float2(fast_exp2(z.x), fast_exp2(z.y));
                        l4[e & 3] = fadd2(l4[e & 3], p);
                        w[e] = pack_half2(p.x, p.y);
                    }
                    tmem_st16(sb + c / 2, w);
                }
                lsum += ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_p);
            }
            ns += nt;
            // the next item's Q: this tile's last S = Q K^T has been read, and the MMA
            // thread has taken this item's Q (so that no Q arrival runs two items ahead)
            ++k;
            PfItem nxt;
            const bool have_next = ok && pf_next(a, total, k, nxt);
            if (have_next) {
                if (!__all_sync(kPfFull, mbar_wait_bounded(b_qf, ni & 1, abort_flag, a.err_flag))) ok = false;
                else load_q(nxt);
            }
            ++ni;
            // ---- epilogue: O / l * v_scale -> fp16 output row (every lane loads, valid rows store) ----
            if (nt > 0 && ok &&
                __all_sync(kPfFull, !*abort_flag && mbar_wait_bounded(b_pv, (npv + nt - 1) & 1, abort_flag, a.err_flag))) {
                tc_fence_after();
                const float coef = lsum > 0.f ? a.out_scale / lsum : 0.f;
                __half *orow = static_cast<__half *>(a.out) + ((int64_t)(q0 + (row_ok ? i : 0)) * a.num_q_heads + h) * kPfD;
                // the row's 128 output columns in one tensor-memory round trip
                uint32_t orr[kPfD / 16][16];
#pragma unroll
                for (int c = 0; c < kPfD / 16; ++c) tmem_ld16(ob + 16 * c, orr[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < kPfD / 16; ++c) {
                    uint32_t(&r16)[16] = orr[c];
                    tmem_regs_ready(r16);
                    uint4 o0, o1;
                    o0.x = pack_half2(__uint_as_float(r16[0]) * coef, __uint_as_float(r16[1]) * coef);
                    o0.y = pack_half2(__uint_as_float(r16[2]) * coef, __uint_as_float(r16[3]) * coef);
                    o0.z = pack_half2(__uint_as_float(r16[4]) * coef, __uint_as_float(r16[5]) * coef);
                    o0.w = pack_half2(__uint_as_float(r16[6]) * coef, __uint_as_float(r16[7]) * coef);
                    o1.x = pack_half2(__uint_as_float(r16[8]) * coef, __uint_as_float(r16[9]) * coef);
                    o1.y = pack_half2(__uint_as_float(r16[10]) * coef, __uint_as_float(r16[11]) * coef);
                    o1.z = pack_half2(__uint_as_float(r16[12]) * coef, __uint_as_float(r16[13]) * coef);
                    o1.w = pack_half2(__uint_as_float(r16[14]) * coef, __uint_as_float(r16[15]) * coef);
                    if (row_ok) {
                        *reinterpret_cast<uint4 *>(orow + 16 * c) = o0;
                        *reinterpret_cast<uint4 *>(orow + 16 * c + 8) = o1;
                    }
                }
            }
            npv += nt;
            it = nxt;
            have = have_next;
        }
    }

    // ---- teardown: copies drained, MMAs complete (the MMA thread waited), tensor memory freed ----
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == kPfLoadWarp) {
        if (lane == 0)
            for (int t = max(0, issued - kPfStages); t < issued; ++t)
                mbar_wait_bounded(full(t % kPfStages), (t / kPfStages) & 1, nullptr, a.err_flag, 100000000ull);
        __syncwarp();
    }
    tc_fence_after();
    __syncthreads();
    if (warp == kPfMmaWarp) tmem_dealloc(tmem, kPfCols);
}

// ---------------------------------------------------------------------------
// host side

size_t prefill_mask_offset(int32_t batch, int32_t num_kv_heads, int32_t max_tiles)
{
    return (size_t)batch * (size_t)num_kv_heads * (size_t)max_tiles * 2 * (size_t)kPfTileBytes;
}

size_t prefill_tiles_bytes(int32_t batch, int32_t num_kv_heads, int32_t max_tiles)
{
    // the K and V tiles, then a 16-byte key mask per tile
    return (size_t)batch * (size_t)num_kv_heads * (size_t)max_tiles * (2 * (size_t)kPfTileBytes + 16);
}

int32_t prefill_max_tiles(int32_t max_pages) { return (int32_t)(((int64_t)max_pages * 4 + kPfTile - 1) / kPfTile); }

template <bool E4M3>
static cudaError_t launch_prefill_t(const PrefillArgs &a, cudaStream_t stream)
{
    static uint64_t configured = 0;   // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(prefill_attn_kernel<E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPfSmemBytes);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    e = launch_pdl(kv_tile_kernel<E4M3>, dim3(4 * a.max_tiles, a.num_kv_heads, a.batch), dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
    // one CTA per SM, each taking its work items in turn
    const int64_t items = (int64_t)((a.max_q_len + 2 * kPfTile - 1) / (2 * kPfTile)) * a.batch * a.num_q_heads;
    if (items > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)std::min<int64_t>(items, device_sm_count()));
    return launch_pdl(prefill_attn_kernel<E4M3>, grid, dim3(kPfThreads), kPfSmemBytes, stream, a);
}

cudaError_t launch_prefill(bool e4m3, const PrefillArgs &a, cudaStream_t stream)
{
    if (a.batch == 0) return cudaSuccess;
    return e4m3 ? launch_prefill_t<true>(a, stream) : launch_prefill_t<false>(a, stream);
}

}  // namespace kvq
