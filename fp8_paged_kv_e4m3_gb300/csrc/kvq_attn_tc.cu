// kvq_attn_tc.cu -- split-K paged attention for many query rows per kv head
// (MTP verify: G heads x q_len rows, 16 < rows <= 64) on the fifth-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// What is computed is the same as attn_split_kernel -- PR "[Model][SM70][FP8]
// Integrate calibrated E4M3 QSA KV capacity path", section Changes; PR
// "[Model][SM70] Calibrated E4M3 KV cache for Qwen4Exp QSA with MTP", sections
// Purpose and Status and history: grouped-query attention of q_len rows,
// causal inside the verify window, over a page-4 E4M3 (or fp16) cache with the
// per-layer scales hoisted, split over the token axis into the same FP32
// workspace partials.
//
// Design (one CTA per (split, kv head, sequence); 7 warps):
//  * warps 4, 5: the producers of the split kernel -- 1-D bulk copies of K and
//    V pages (16 pages = 64 tokens per staging stage) into a shared ring.
//  * warps 0-3 ("workers", warp q owns tensor-memory lanes 32q..32q+31): per
//    tile of 128 tokens (two staging stages) each worker converts its 32
//    tokens -- K rows to fp16 straight into tensor memory (the A operand of
//    S^T = K Q^T, token t in lane t), V rows to fp16 in shared memory (the
//    MN-major A operand of O^T = V^T P^T) -- then reads S^T back (thread =
//    token, one column per query row), runs the online softmax in the log2
//    domain with the scores' scale hoisted, and writes P^T (fp16, MN-major)
//    to shared memory.  Row maxima and sums over the 128 tokens are reduced
//    across the lanes by a butterfly transpose and across the four workers
//    through shared memory.  The O^T accumulator (lane = channel, column =
//    query row) is rescaled in tensor memory only when a row's maximum rises
//    by more than 2^8 over the reference used so far; the exact maximum is
//    tracked apart and restored in the epilogue.
//  * warp 6: allocates tensor memory; one thread issues the MMAs (M = 128
//    tokens or channels, N = rows padded to 16/32/64, K = 16 per instruction)
//    and commits their completion to mbarriers.
//  * Every wait is bounded (about 2 s); on expiry the CTA reports
//    KVQ_DEV_TIMEOUT, lets its copies and MMAs drain, gives its rows zero
//    weight in the workspace (m = -inf, l = 0), frees its tensor memory and
//    exits.
//
// FP8 score variant (F8, E4M3 pools only; not on the pages): the workers
// quantise the CTA's query rows to E4M3 with one scale amax / 448 over them
// (the rows of one (sequence, kv head) group, so every split of the group
// takes the same codes), K rows go to tensor memory as their E4M3 bytes
// without conversion, and S^T = K Q^T runs as tcgen05.mma kind::f8f6f4
// (K = 32 per instruction); the query scale joins the hoisted score scale.
// P V is unchanged (fp16).
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kvq_attn_kernel.cuh"
#include "kvq_tcgen05.cuh"

namespace kvq {

constexpr int kTcWorkers = 4;
constexpr int kTcMmaWarp = kConsumerWarps + kProducerWarps;   // 6
constexpr int kTcThreads = 32 * (kTcMmaWarp + 1);             // 224
constexpr int kTcTile = 128;                                  // tokens per MMA tile
constexpr int kTcD = 128;                                     // head_dim of this kernel
// pages per staging stage: 16 (64 tokens) for E4M3, 8 (32 tokens) for fp16, so
// that the staging ring keeps two CTAs per SM for both element sizes
template <bool E4M3> __host__ __device__ constexpr int tc_pps() { return E4M3 ? 16 : 8; }
// staging stages per 128-token tile; the ring holds at least that many, since a
// worker waits only on its own stage of the tile, which must never be a slot's
// next-but-one phase
template <bool E4M3> __host__ __device__ constexpr int tc_spt() { return kTcTile / (4 * tc_pps<E4M3>()); }
template <bool E4M3> using TcGeometry = Geometry<E4M3, kTcD, tc_pps<E4M3>(), tc_spt<E4M3>()>;

// shared memory after the staging ring of Geometry<E4M3, 128, 16>
template <bool E4M3, int NR>
struct TcLayout {
    using G = TcGeometry<E4M3>;
    static constexpr int kQ = (G::kBytes + 1023) & ~1023;   // Q: NR x 128 fp16, K-major
    static constexpr int kV = kQ + NR * 256;                 // V^T: 128 ch x 128 tok fp16, MN-major
    static constexpr int kP = kV + kTcTile * kTcD * 2;       // P^T: NR x 128 tok fp16, MN-major
    static constexpr int kWmax = kP + NR * 256;              // [2][4][NR] float: per-worker row maxima
    static constexpr int kPriv = kWmax + 2 * 4 * NR * 4;     // [4][5][NR] float: per-worker reference,
                                                             //   correction, coefficient, reference in use,
                                                             //   reference + 8 (the band's top)
    static constexpr int kLsum = kPriv + 4 * 5 * NR * 4;     // [4][NR] float: per-worker row sums
    static constexpr int kMend = kLsum + 4 * NR * 4;         // [4][NR] float: per-worker final row maxima
    static constexpr int kFlag = kMend + 4 * NR * 4;         // [2][4] int: per-worker "left the band" flags
    static constexpr int kQmax = kFlag + 2 * 4 * 4;          // [2][4] float: per-worker max |q|, score
                                                             //   scale with the query's (FP8 scores)
    static constexpr int kBar = kQmax + 2 * 4 * 4;           // 8 mbarriers
    static constexpr int kBarV = kBar + 8 * 8;               // V staging: [full][kStages], [empty][kStages]
    static constexpr int kTmemSlot = kBarV + 2 * G::kStages * 8;
    static constexpr int kBytes = kTmemSlot + 16;
    // tensor-memory columns: K tile (64: 128 fp16 per lane), S^T (NR), O^T (NR), the row
    // sums L^T (NR, every lane the same: a ones tile times P^T), the ones tile (64)
    static constexpr int kColK = 0, kColS = 64, kColO = 64 + NR, kColL = 64 + 2 * NR, kColOnes = 64 + 3 * NR;
    static constexpr int kCols = (128 + 3 * NR) <= 128 ? 128 : ((128 + 3 * NR) <= 256 ? 256 : 512);
};

// two fp32 lanes per instruction (sm_100 and later): d = a - b and d = a * b,
// each lane rounded to nearest as its scalar form
__device__ __forceinline__ float2 fsub2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0 in
// bits 7-9 and 10-12), fp32 accumulator, M x N tile, both operands K-major.
__device__ __forceinline__ uint32_t umma_idesc_e4m3(int m, int n)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (tensor memory) (+)= A (tensor memory, 4 E4M3 per 32-bit column) x B (shared memory, E4M3)
__device__ __forceinline__ void umma_tmem_a_e4m3(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 bool accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
                 : "memory");
}

// four fp16 (two 32-bit words) -> four E4M3 bytes, element 0 in the lowest
// byte: binary32 division by the scale (round to nearest even), then the
// hardware satfinite E4M3 conversion (round to nearest even, finite overflow
// to +-448) -- the cache quantiser's two roundings
__device__ __forceinline__ uint32_t quantize_q4(uint32_t h01, uint32_t h23, float scale)
{
    const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
    const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(fa.x, scale), __fdiv_rn(fa.y, scale)),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(fb.x, scale), __fdiv_rn(fb.y, scale)),
                                                 __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ float absmax8(uint4 v)
{
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&v.z));
    const float2 d = __half22float2(*reinterpret_cast<const __half2 *>(&v.w));
    return fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))),
                 fmaxf(fmaxf(fabsf(c.x), fabsf(c.y)), fmaxf(fabsf(d.x), fabsf(d.y))));
}

// Lane r of the warp ends with the maximum (or sum) over the warp's 32 lanes
// of value v[r] (r < 32): a butterfly that halves the set each step.
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane)
{
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) {
        const bool hi = (lane & k) != 0;
#pragma unroll
        for (int i = 0; i < k; ++i) {
            const float send = hi ? v[i] : v[i + k];
            const float keep = hi ? v[i + k] : v[i];
            const float recv = __shfl_xor_sync(kFull, send, k);
            v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];   // row `lane`
}

// Two CTAs per SM when NR <= 32: the bound is stated for 256 threads so that
// registers stay at 128 per thread -- with 7 warps per CTA, two CTAs put four
// warps on some SM sub-partitions, whose register files hold 4 x 128 x 32.
template <bool E4M3, int NR, bool F8, bool BITCAST>
__global__ void __launch_bounds__(256, NR <= 32 ? 2 : 1) attn_tc_kernel(const AttnArgs a)
{
    static_assert(E4M3 || !F8, "FP8 scores need E4M3 pools");
    static_assert(!BITCAST || (E4M3 && !F8), "the bitcast decoder is for E4M3 pools with fp16 scores");
    constexpr int D = kTcD, PPS = tc_pps<E4M3>();
    using G = TcGeometry<E4M3>;
    constexpr int SPT = tc_spt<E4M3>();                       // staging stages per tile: 2 or 4
    static_assert(G::kStages >= SPT, "the ring must hold a whole tile's staging stages");
    constexpr int WPS = kTcWorkers / SPT;                     // workers per staging stage: 2 or 1
    using T = TcLayout<E4M3, NR>;
    constexpr int NH = NR <= 32 ? 1 : 2;                      // rows per lane after a transpose-reduce
    extern __shared__ __align__(128) uint8_t smem[];

    const int s = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(smem);
    int32_t *tokpos = reinterpret_cast<int32_t *>(smem + G::kTokPosOff);
    // staging barriers, one set per producer, so that a slot's K half refills as
    // soon as the workers hold its rows in tensor memory, before its V half is
    // converted: bar0 for K (the ring's own barriers), barv for V
    const uint32_t bar0 = smem_u32(smem + G::kBarOff);
    const uint32_t barv = smem_u32(smem + T::kBarV);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + G::kAbortOff);
    volatile int *stage_bad = abort_flag + 1;
    const uint32_t tb = smem_u32(smem + T::kBar);
    const uint32_t b_k = tb, b_s = tb + 8, b_p = tb + 16, b_pv = tb + 24, b_x = tb + 32, b_l = tb + 40,
                   b_drain = tb + 48, b_y = tb + 56;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + T::kTmemSlot);

    if (threadIdx.x == 0) {
        for (int k = 0; k < G::kStages; ++k) {
            mbar_init(bar0 + 8 * k, 1);                     // K copies landed
            mbar_init(bar0 + 8 * (G::kStages + k), WPS);   // K rows taken by the workers it feeds
            mbar_init(barv + 8 * k, 1);                     // V copies landed
            mbar_init(barv + 8 * (G::kStages + k), WPS);   // V rows taken
        }
        mbar_init(b_k, kTcWorkers);
        mbar_init(b_s, 1);
        mbar_init(b_p, kTcWorkers);
        mbar_init(b_pv, 1);
        mbar_init(b_x, kTcWorkers);
        mbar_init(b_l, kTcWorkers);
        mbar_init(b_drain, 1);
        mbar_init(b_y, kTcWorkers);
        *abort_flag = 0;
        *stage_bad = 0;
        fence_mbar_init();
    }
    if (warp == kTcMmaWarp) tmem_alloc(smem_u32(tmem_slot), T::kCols);
    grid_dependency_wait();   // inputs may come from the previous kernel (e.g. the append)

    // sequences longest first; the speculative block-table read (producers) is
    // issued for the identity order and repeated if another sequence is picked
    const int z = blockIdx.z;
    const int spec0 = split_spec0(a, s);
    const bool spec_lane = warp >= kConsumerWarps && warp < kTcMmaWarp && spec0 + lane < a.max_pages;
    int bt_spec = spec_lane ? __ldg(a.block_tables + (int64_t)z * a.max_pages + spec0 + lane) : -1;
    SeqPick pick = seq_identity(a, z);
    const bool keep_order = lpt_classify(a, smem, G::kRingBytes);
    tc_fence_before();
    if (!__syncthreads_and(keep_order)) {   // the setup barrier (mbarriers, tensor memory) as well
        pick = lpt_pick(a, z, smem);
        if (pick.b != z) bt_spec = spec_lane ? __ldg(a.block_tables + (int64_t)pick.b * a.max_pages + spec0 + lane) : -1;
    }
    tc_fence_after();
    const int b = pick.b;
    const SplitRange sr = split_range(a, s, b, pick.L, pick.topk_len);
    const int L = sr.L;
    const int ipst = sr.topk ? G::kTokPerStage : PPS;
    const int nst = (sr.item1 - sr.item0 + ipst - 1) / ipst;   // staging stages
    const int ntiles = (nst + SPT - 1) / SPT;
    if (threadIdx.x == 0) {
        if (!sr.len_ok) report(a.err_flag, KVQ_DEV_BAD_LEN);
        if (sr.len_ok && pick.topk_len > a.max_topk)
            report(a.err_flag, KVQ_DEV_BAD_TOPK);
    }
    // only now may a dependent grid start: this CTA already holds its tensor
    // memory, so a dependent CTA cannot take the columns it waits for
    launch_dependents();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;

    if (warp >= kConsumerWarps && warp < kTcMmaWarp) {
        // ================= producers =================
        const bool is_v = warp == kConsumerWarps + 1;
        issued = produce_stages<G, PPS>(a, sr, nst, b, g, lane, is_v, bt_spec, ring, is_v ? barv : bar0, tokpos,
                                        abort_flag, stage_bad);
    } else if (warp == kTcMmaWarp) {
        // ================= MMA issue (one thread) =================
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(smem + T::kQ), v_addr = smem_u32(smem + T::kV),
                           p_addr = smem_u32(smem + T::kP);
            const uint32_t id_qk = F8 ? umma_idesc_e4m3(kTcTile, NR) : umma_idesc_f16(kTcTile, NR, false, false);
            const uint32_t id_pv = umma_idesc_f16(kTcTile, NR, true, true);
            const uint32_t id_l = umma_idesc_f16(kTcTile, NR, false, true);
            for (int t = 0; t < ntiles; ++t) {
                if (!mbar_wait_bounded(b_k, t & 1, abort_flag, a.err_flag)) break;
                tc_fence_after();
                // S^T[tok][row] = sum_d K[tok][d] Q[row][d]: A = K tile (tensor memory), B = Q (K-major);
                // 8 tensor-memory columns and two 128-byte core-matrix columns of Q per instruction
                if constexpr (F8) {
#pragma unroll
                    for (int ks = 0; ks < D / 32; ++ks)
                        umma_tmem_a_e4m3(tmem + T::kColS, tmem + T::kColK + ks * 8,
                                         umma_desc(q_addr + ks * 256, 128, (D / 16) * 128), id_qk, ks > 0);
                } else {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma_tmem_a(tmem + T::kColS, tmem + T::kColK + ks * 8,
                                    umma_desc(q_addr + ks * 256, 128, (D / 8) * 128), id_qk, ks > 0);
                }
                umma_commit(b_s);
                if (!mbar_wait_bounded(b_p, t & 1, abort_flag, a.err_flag)) break;
                tc_fence_after();
                // O^T[ch][row] += sum_tok V[tok][ch] P[tok][row]: A = V^T, B = P^T, both MN-major;
                // L^T[lane][row] += sum_tok 1 * P[tok][row]: the row sums -- the two accumulation
                // chains interleaved
#pragma unroll
                for (int ks = 0; ks < kTcTile / 16; ++ks) {
                    umma_smem_a(tmem + T::kColO, umma_desc(v_addr + ks * 2 * (D / 8) * 128, (D / 8) * 128, 128),
                                umma_desc(p_addr + ks * 2 * NR * 16, NR * 16, 128), id_pv, t > 0 || ks > 0);
                    umma_tmem_a(tmem + T::kColL, tmem + T::kColOnes + ks * 8,
                                umma_desc(p_addr + ks * 2 * NR * 16, NR * 16, 128), id_l, t > 0 || ks > 0);
                }
                umma_commit(b_pv);
            }
            // every MMA issued so far completes before the tensor memory is freed
            umma_commit(b_drain);
            mbar_wait_bounded(b_drain, 0, nullptr, a.err_flag, 100000000ull);
        }
        __syncwarp();
    } else {
        // ================= workers: conversion, softmax, epilogue =================
        const int q = warp;                          // tensor-memory lane quadrant
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int tt = 32 * q + lane;                // token of the tile (S^T lane), channel of O^T
        const int win0 = L - a.q_len;                // row i sees positions <= win0 + i
        float *wmax = reinterpret_cast<float *>(smem + T::kWmax);
        // reference, corr, coef, reference in use, reference + 8
        float *priv = reinterpret_cast<float *>(smem + T::kPriv) + q * 5 * NR;
        float *lsum = reinterpret_cast<float *>(smem + T::kLsum);
        // the final maxima get a buffer of their own: a worker may still read the
        // last tile's exchange in wmax while another has reached the epilogue
        float *mend = reinterpret_cast<float *>(smem + T::kMend);

        // the score scale: hoisted in the arguments, or (FP8 scores) with the
        // query's scale in shared memory, read once per tile rather than held
        // in a register across the loop
        float *qk_f8 = reinterpret_cast<float *>(smem + T::kQmax) + 4 + q;
        if constexpr (F8) {
            // Q rows (padding rows zero) quantised into the K-major E4M3 Q tile:
            // element (r, d) at (r/8) * 1024 + (d/16) * 128 + (r%8) * 16 + d%16;
            // thread item = 16 channels of one row, the 8 lanes of a quarter
            // warp on 8 rows of one 16-byte column
            constexpr int QI = NR * (D / 16) / (32 * kTcWorkers);   // items per thread
            static_assert(QI * 32 * kTcWorkers == NR * (D / 16), "Q items must divide evenly");
            uint4 qv[QI][2];
            float mx = 0.f;
#pragma unroll
            for (int u = 0; u < QI; ++u) {
                const int idx = tt + u * 32 * kTcWorkers;
                const int r = (idx & 7) + 8 * (idx / (8 * (D / 16))), c = (idx / 8) % (D / 16);
                qv[u][0] = qv[u][1] = make_uint4(0u, 0u, 0u, 0u);
                if (r < a.rows) {
                    const int i = r / a.group, h = g * a.group + r % a.group;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        static_cast<const __half *>(a.q) + (((int64_t)b * a.q_len + i) * a.num_q_heads + h) * D +
                        16 * c);
                    qv[u][0] = src[0];
                    qv[u][1] = src[1];
                }
                mx = fmaxf(mx, fmaxf(absmax8(qv[u][0]), absmax8(qv[u][1])));
            }
            // the group's max |q| over the four workers
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
            float *qmax = reinterpret_cast<float *>(smem + T::kQmax);
            if (lane == 0) qmax[q] = mx;
            named_bar_sync(1, 32 * kTcWorkers);
            const float amax = fmaxf(fmaxf(qmax[0], qmax[1]), fmaxf(qmax[2], qmax[3]));
            const float q_scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
            if (lane == 0) *qk_f8 = a.qk_scale_log2 * q_scale;
#pragma unroll
            for (int u = 0; u < QI; ++u) {
                const int idx = tt + u * 32 * kTcWorkers;
                const int r = (idx & 7) + 8 * (idx / (8 * (D / 16))), c = (idx / 8) % (D / 16);
                uint4 v;
                v.x = quantize_q4(qv[u][0].x, qv[u][0].y, q_scale);
                v.y = quantize_q4(qv[u][0].z, qv[u][0].w, q_scale);
                v.z = quantize_q4(qv[u][1].x, qv[u][1].y, q_scale);
                v.w = quantize_q4(qv[u][1].z, qv[u][1].w, q_scale);
                *reinterpret_cast<uint4 *>(smem + T::kQ + (r >> 3) * 1024 + c * 128 + (r & 7) * 16) = v;
            }
        } else {
            // Q rows (padding rows zero) into the K-major Q tile: element (r, d) at
            // (r/8) * 2048 + (d/8) * 128 + (r%8) * 16 + (d%8) * 2; the 8 lanes of a
            // quarter warp take 8 rows of one 16-byte column, one 128-byte line
            for (int idx = tt; idx < NR * (D / 8); idx += 32 * kTcWorkers) {
                const int r = (idx & 7) + 8 * (idx / (8 * (D / 8))), c = (idx / 8) % (D / 8);
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < a.rows) {
                    const int i = r / a.group, h = g * a.group + r % a.group;
                    v = *reinterpret_cast<const uint4 *>(static_cast<const __half *>(a.q) +
                                                         (((int64_t)b * a.q_len + i) * a.num_q_heads + h) * D + 8 * c);
                    if (BITCAST) {
                        // channel order of the bitcast-decoded K rows: 0, 2, 1, 3 in each group of four
                        v = make_uint4(__byte_perm(v.x, v.y, 0x5410), __byte_perm(v.x, v.y, 0x7632),
                                       __byte_perm(v.z, v.w, 0x5410), __byte_perm(v.z, v.w, 0x7632));
                    }
                }
                *reinterpret_cast<uint4 *>(smem + T::kQ + (r >> 3) * 2048 + c * 128 + (r & 7) * 16) = v;
            }
        }
        fence_async_smem();   // the Q tile is read by the tensor core (async proxy)

        // Per row, the reference of the exponentials lives in the worker's private
        // shared copy (all four workers hold the same values): priv[r] (-inf while
        // the row has none), priv[3 NR + r] (the same, 0 while none), priv[4 NR + r]
        // (the reference + 8, the top of the row's band; -inf while none).  This
        // thread keeps, per row, the running maximum and the sum over its tokens.
        int *flag = reinterpret_cast<int *>(smem + T::kFlag);
#pragma unroll
        for (int h = 0; h < NH; ++h)
            if (32 * h + lane < NR) {
                priv[32 * h + lane] = -INFINITY;
                priv[3 * NR + 32 * h + lane] = 0.f;
                priv[4 * NR + 32 * h + lane] = -INFINITY;
            }
        __syncwarp();
        float mt[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) mt[r] = -INFINITY;
        {   // the ones tile (fp16 1.0 pairs), A operand of the row sums
            uint32_t ones[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) ones[e] = 0x3C003C00u;
#pragma unroll
            for (int c = 0; c < 64; c += 16) tmem_st16(tmem + lane_base + T::kColOnes + c, ones);
            tmem_wait_st();
        }
        int nband = 0;   // times a row left the band (the same count on every worker)
        bool ok = true;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int st = SPT * t + q / WPS;        // staging stage of this warp's 32 tokens
            // token of that stage: the 8 lanes of a quarter warp take the same slot of 8
            // different pages, whose 16-byte rows sit in distinct banks (page stride
            // = 16 mod 128); tile slot tt holds this token in S^T, V^T and P^T alike
            const int j = (q % WPS) * 32 + ((lane & 7) << 2) + (lane >> 3);
            const bool have = st < nst;
            const int slot = st % G::kStages;
            if (have && !__all_sync(kFull, mbar_wait_bounded(bar0 + 8 * slot, (st / G::kStages) & 1, abort_flag,
                                                             a.err_flag))) {
                ok = false;
                break;
            }
            const int pos = have ? tokpos[slot * G::kTokPerStage + j] : -1;
            const uint8_t *krow = smem + slot * G::kStageBytes + (j >> 2) * G::kPageStride + (j & 3) * G::kRowBytes;
            const uint8_t *vrow = krow + G::kRegion;
            // ---- K row -> fp16 in tensor memory (token tt in lane tt, channels 2c, 2c+1 in column c);
            // the K tile is free: the previous tile's S^T is complete ----
            // all of the row's loads first (krow is a ring address whether or not the slot
            // holds this tile's token; its scores are masked below), conversions after
            constexpr int kKV = E4M3 ? 8 : 16;        // 16-byte pieces of a K (or V) row
            uint4 kx[kKV];
#pragma unroll
            for (int u = 0; u < kKV; ++u) kx[u] = *reinterpret_cast<const uint4 *>(krow + 16 * u);
            if constexpr (F8) {
                // the E4M3 bytes themselves: channels 4c..4c+3 in column c, lowest byte first
#pragma unroll
                for (int h = 0; h < 2; ++h) {        // 16 columns = 64 channels per store
                    uint32_t w[16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 x = kx[4 * h + u];
                        w[4 * u + 0] = x.x;
                        w[4 * u + 1] = x.y;
                        w[4 * u + 2] = x.z;
                        w[4 * u + 3] = x.w;
                    }
                    tmem_st16(tmem + lane_base + T::kColK + 16 * h, w);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 4; ++h) {            // 16 columns = 32 channels per store
                    uint32_t w[16];
                    if (E4M3) {
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const uint4 x = kx[2 * h + u];
                            if (BITCAST) {
                                // channels 4i, 4i + 2 and 4i + 1, 4i + 3 of each word, times 2^-8
                                w[8 * u + 0] = dec_lo(x.x);
                                w[8 * u + 1] = dec_hi(x.x);
                                w[8 * u + 2] = dec_lo(x.y);
                                w[8 * u + 3] = dec_hi(x.y);
                                w[8 * u + 4] = dec_lo(x.z);
                                w[8 * u + 5] = dec_hi(x.z);
                                w[8 * u + 6] = dec_lo(x.w);
                                w[8 * u + 7] = dec_hi(x.w);
                            } else {
                                w[8 * u + 0] = cvt_lo(x.x);
                                w[8 * u + 1] = cvt_hi(x.x);
                                w[8 * u + 2] = cvt_lo(x.y);
                                w[8 * u + 3] = cvt_hi(x.y);
                                w[8 * u + 4] = cvt_lo(x.z);
                                w[8 * u + 5] = cvt_hi(x.z);
                                w[8 * u + 6] = cvt_lo(x.w);
                                w[8 * u + 7] = cvt_hi(x.w);
                            }
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint4 x = kx[4 * h + u];
                            w[4 * u + 0] = x.x;
                            w[4 * u + 1] = x.y;
                            w[4 * u + 2] = x.z;
                            w[4 * u + 3] = x.w;
                        }
                    }
                    tmem_st16(tmem + lane_base + T::kColK + 16 * h, w);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_k);           // S^T of this tile may start
            if (have && lane == 0) mbar_arrive(bar0 + 8 * (G::kStages + slot));   // K half of the slot free
            // ---- V row -> fp16 V^T tile (MN-major): (ch, tok) at (tok/8)*2048 + (ch/8)*128 + (tok%8)*16;
            // V^T and P^T are reused: the previous tile's PV must be complete ----
            if (t > 0 && !__all_sync(kFull, mbar_wait_bounded(b_pv, (t - 1) & 1, abort_flag, a.err_flag))) {
                ok = false;
                break;
            }
            if (have && !__all_sync(kFull, mbar_wait_bounded(barv + 8 * slot, (st / G::kStages) & 1, abort_flag,
                                                             a.err_flag))) {
                ok = false;
                break;
            }
            {
                // a slot without a token is zeroed: its bits may be NaN, and P = 0 alone leaves 0 * NaN
                uint8_t *vdst = smem + T::kV + (tt >> 3) * ((D / 8) * 128) + (tt & 7) * 16;
                const bool vok = have && pos >= 0;
                uint4 vx[kKV];
#pragma unroll
                for (int u = 0; u < kKV; ++u) vx[u] = *reinterpret_cast<const uint4 *>(vrow + 16 * u);
                const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {   // 16 channels per step
                    uint4 lo, hi;
                    if (E4M3 && BITCAST) {   // channel slots in the order 0, 2, 1, 3 per four, times 2^-8
                        const uint4 x = vx[c];
                        lo = make_uint4(dec_lo(x.x), dec_hi(x.x), dec_lo(x.y), dec_hi(x.y));
                        hi = make_uint4(dec_lo(x.z), dec_hi(x.z), dec_lo(x.w), dec_hi(x.w));
                    } else if (E4M3) {
                        const uint4 x = vx[c];
                        lo = make_uint4(cvt_lo(x.x), cvt_hi(x.x), cvt_lo(x.y), cvt_hi(x.y));
                        hi = make_uint4(cvt_lo(x.z), cvt_hi(x.z), cvt_lo(x.w), cvt_hi(x.w));
                    } else {
                        lo = vx[2 * c];
                        hi = vx[2 * c + 1];
                    }
                    *reinterpret_cast<uint4 *>(vdst + (2 * c) * 128) = vok ? lo : zero;
                    *reinterpret_cast<uint4 *>(vdst + (2 * c + 1) * 128) = vok ? hi : zero;
                }
            }
            __syncwarp();
            if (have && lane == 0) mbar_arrive(barv + 8 * (G::kStages + slot));   // V half of the slot free

            // ---- S^T of this warp's 32 tokens: one column per query row ----
            if (!__all_sync(kFull, mbar_wait_bounded(b_s, t & 1, abort_flag, a.err_flag))) { ok = false; break; }
            tc_fence_after();
            float x[NR];
#pragma unroll
            for (int c = 0; c < NR; c += 16) {
                uint32_t r16[16];
                tmem_ld16(tmem + lane_base + T::kColS + c, r16);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) x[c + e] = __uint_as_float(r16[e]);
            }
            // scores in the log2 domain; row r (window row r / G) sees positions <= win0 + r / G
            // (the bitcast decoder's K is K * 2^-8: its 2^8 joins the hoisted scale, exactly)
            const float qk = F8 ? *reinterpret_cast<volatile float *>(qk_f8) : a.qk_scale_log2 * (BITCAST ? 256.f : 1.f);
            const int rmin = pos < 0 ? NR : (pos > win0 ? a.group * (pos - win0) : 0);
            if (rmin == 0 && a.rows == NR) {
#pragma unroll
                for (int r = 0; r < NR; r += 2) {
                    const float2 y = fmul2(make_float2(x[r], x[r + 1]), make_float2(qk, qk));
                    x[r] = y.x;
                    x[r + 1] = y.y;
                }
            } else {
#pragma unroll
                for (int r = 0; r < NR; ++r) x[r] = (r >= rmin && r < a.rows) ? x[r] * qk : -INFINITY;
            }

            // ---- running maxima; does any score leave the band of 2^8 above its row's reference? ----
            // (a row without a reference has its band top at -inf: any finite score leaves it)
            bool over = false;
#pragma unroll
            for (int r = 0; r < NR; r += 4) {
                const float4 top = *reinterpret_cast<const float4 *>(priv + 4 * NR + r);
                mt[r] = fmaxf(mt[r], x[r]);
                mt[r + 1] = fmaxf(mt[r + 1], x[r + 1]);
                mt[r + 2] = fmaxf(mt[r + 2], x[r + 2]);
                mt[r + 3] = fmaxf(mt[r + 3], x[r + 3]);
                over |= (x[r] > top.x) | (x[r + 1] > top.y) | (x[r + 2] > top.z) | (x[r + 3] > top.w);
            }
            over = __any_sync(kFull, over);
            if (lane == 0) flag[(t & 1) * 4 + q] = over ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(b_x);
            if (!__all_sync(kFull, mbar_wait_bounded(b_x, t & 1, abort_flag, a.err_flag))) { ok = false; break; }
            const bool band = (flag[(t & 1) * 4 + 0] | flag[(t & 1) * 4 + 1] | flag[(t & 1) * 4 + 2] |
                               flag[(t & 1) * 4 + 3]) != 0;
            if (band) {
                // rare: the tile's exact row maxima, then new references where a maximum
                // rose more than 2^8 above the old one (the same decision on every worker)
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    float v[32];
#pragma unroll
                    for (int r = 0; r < 32; ++r) v[r] = (32 * h + r < NR) ? x[32 * h + r] : -INFINITY;
                    const float m = warp_transpose_reduce<true>(v, lane);
                    if (32 * h + lane < NR) wmax[q * NR + 32 * h + lane] = m;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(b_y);
                if (!__all_sync(kFull, mbar_wait_bounded(b_y, nband & 1, abort_flag, a.err_flag))) { ok = false; break; }
                ++nband;
                bool moved = false;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const int r = 32 * h + lane;
                    if (r >= NR) continue;
                    float mx = -INFINITY;
#pragma unroll
                    for (int w = 0; w < 4; ++w) mx = fmaxf(mx, wmax[w * NR + r]);
                    const float ref = priv[r];
                    float corr = 1.f;
                    if (mx > -INFINITY && (ref == -INFINITY || mx > ref + 8.f)) {
                        corr = (ref == -INFINITY) ? 0.f : fast_exp2(ref - mx);
                        priv[r] = mx;
                        priv[3 * NR + r] = mx;
                        priv[4 * NR + r] = mx + 8.f;
                        moved = true;
                    }
                    priv[NR + r] = corr;
                }
                moved = __any_sync(kFull, moved);
                __syncwarp();
                if (moved && t > 0) {
                    // O^T and L^T columns of the rows whose reference moved (the previous PV is complete)
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 2 * NR; c += 16) {   // O^T then L^T: adjacent columns
                        uint32_t r16[16];
                        tmem_ld16(tmem + lane_base + T::kColO + c, r16);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            r16[e] = __float_as_uint(__uint_as_float(r16[e]) * priv[NR + ((c + e) % NR)]);
                        tmem_st16(tmem + lane_base + T::kColO + c, r16);
                    }
                    tmem_wait_st();
                }
            }
            // ---- P = exp2(score - reference) ----
#pragma unroll
            for (int r = 0; r < NR; r += 4) {
                const float4 rf = *reinterpret_cast<const float4 *>(priv + 3 * NR + r);
                const float2 d0 = fsub2(make_float2(x[r], x[r + 1]), make_float2(rf.x, rf.y));
                const float2 d1 = fsub2(make_float2(x[r + 2], x[r + 3]), make_float2(rf.z, rf.w));
                x[r] = fast_exp2(d0.x);
                x[r + 1] = fast_exp2(d0.y);
                x[r + 2] = fast_exp2(d1.x);
                x[r + 3] = fast_exp2(d1.y);
            }
            // ---- P^T (fp16, MN-major): (row, tok) at (tok/8) * NR*16 + (row/8) * 128 + (tok%8) * 16 ----
            {
                uint8_t *pdst = smem + T::kP + (tt >> 3) * (NR * 16) + (tt & 7) * 16;
#pragma unroll
                for (int c = 0; c < NR / 8; ++c) {
                    uint4 v;
                    v.x = pack_half2(x[8 * c + 0], x[8 * c + 1]);
                    v.y = pack_half2(x[8 * c + 2], x[8 * c + 3]);
                    v.z = pack_half2(x[8 * c + 4], x[8 * c + 5]);
                    v.w = pack_half2(x[8 * c + 6], x[8 * c + 7]);
                    *reinterpret_cast<uint4 *>(pdst + c * 128) = v;
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_p);
        }
        // the warp's row maxima: lane r (and r + 32) ends with row r's over the warp's tokens
        float m_w[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            float v[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) v[r] = (32 * h + r < NR) ? mt[32 * h + r] : -INFINITY;
            m_w[h] = warp_transpose_reduce<true>(v, lane);
        }

        // ---- epilogue: the split's partial (o normalised, m, l) per row ----
        // (every branch below is taken by whole warps: tensor-memory loads are warp-wide)
        if (__all_sync(kFull, ok && !*abort_flag)) {
            bool have_o = ntiles > 0;
            if (have_o && !__all_sync(kFull, mbar_wait_bounded(b_pv, (ntiles - 1) & 1, abort_flag, a.err_flag)))
                have_o = false;
            tc_fence_after();
            // the row sums over all tiles, from L^T (every lane holds them)
            if (have_o) {
#pragma unroll
                for (int c = 0; c < NR; c += 16) {
                    uint32_t r16[16];
                    tmem_ld16(tmem + lane_base + T::kColL + c, r16);
                    tmem_wait_ld();
                    if (lane == 0)
#pragma unroll
                        for (int e = 0; e < 16; ++e) lsum[q * NR + c + e] = __uint_as_float(r16[e]);
                }
            } else if (lane == 0) {
#pragma unroll
                for (int r = 0; r < NR; ++r) lsum[q * NR + r] = 0.f;
            }
#pragma unroll
            for (int h = 0; h < NH; ++h)
                if (32 * h + lane < NR) mend[q * NR + 32 * h + lane] = m_w[h];
            __syncwarp();
            if (lane == 0) mbar_arrive(b_l);
            if (__all_sync(kFull, mbar_wait_bounded(b_l, 0, abort_flag, a.err_flag) && !*abort_flag)) {
                const int S = a.num_splits;
                // per row (lane r, and r + 32): its workspace unit, -1 for a padding row;
                // the stores below take it from that lane instead of dividing per row
                int unit_l[NH];
                // per row: total l (relative to the reference), the coefficient v_scale / l
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const int r = 32 * h + lane;
                    unit_l[h] = -1;
                    if (r >= NR) continue;
                    if (r < a.rows) {
                        const int i = r / a.group, hh = g * a.group + r % a.group;
                        unit_l[h] = ((b * a.num_q_heads + hh) * a.q_len + i) * S + s;
                    }
                    const float lt = lsum[q * NR + r];   // the whole tile set's sum (from L^T)
                    float mx = -INFINITY;
#pragma unroll
                    for (int w = 0; w < 4; ++w) mx = fmaxf(mx, mend[w * NR + r]);
                    // (the bitcast decoder's V is V * 2^-8: its 2^8 joins v_scale, exactly)
                    priv[2 * NR + r] = lt > 0.f ? (a.out_scale * (BITCAST ? 256.f : 1.f)) / lt : 0.f;
                    if (q == 0 && unit_l[h] >= 0) {
                        // the sum relative to the exact maximum, m in natural-log units
                        a.ws_m[unit_l[h]] = lt > 0.f ? mx * kLn2 : -INFINITY;
                        a.ws_l[unit_l[h]] = lt > 0.f ? lt * fast_exp2(priv[3 * NR + r] - mx) : 0.f;
                    }
                }
                __syncwarp();
                if (have_o) {
#pragma unroll
                    for (int c = 0; c < NR; c += 16) {
                        uint32_t r16[16];
                        tmem_ld16(tmem + lane_base + T::kColO + c, r16);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int r = c + e;
                            const int unit = __shfl_sync(kFull, unit_l[r / 32], r % 32);
                            const float coef = priv[2 * NR + r];
                            // O^T lane tt holds channel tt, or (bitcast decoder) channel tt with
                            // bits 0 and 1 swapped
                            const int ch = BITCAST ? ((tt & ~3) | ((tt & 1) << 1) | ((tt >> 1) & 1)) : tt;
                            if (unit >= 0 && coef != 0.f)
                                a.ws_o[(int64_t)unit * D + ch] = __uint_as_float(r16[e]) * coef;
                        }
                    }
                }
            }
        }
    }

    // ---- teardown: copies drained, MMAs complete (the MMA thread waited), tensor memory freed ----
    // On a give-up, each producer waits (bounded) for the copies of the stages it
    // issued: K and V stages complete on barriers of their own with one arrival
    // each, a producer reuses a slot only after its previous stage completed, so
    // the last kStages stages it issued sit in distinct slots and each completes
    // once its copies land.  The CTA's rows then get zero weight (m = -inf, l = 0).
    tc_fence_before();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (aborted && warp >= kConsumerWarps && warp < kTcMmaWarp) {
        if (lane == 0)
            for (int st = max(0, issued - G::kStages); st < issued; ++st)
                mbar_wait_bounded((warp == kConsumerWarps + 1 ? barv : bar0) + 8 * (st % G::kStages),
                                  (st / G::kStages) & 1, nullptr, a.err_flag, 100000000ull);
        __syncwarp();
    }
    if (aborted && warp < kTcWorkers) {
        for (int r = threadIdx.x; r < a.rows; r += 32 * kTcWorkers) {
            const int i = r / a.group, hh = g * a.group + r % a.group;
            const int64_t unit = (((int64_t)b * a.num_q_heads + hh) * a.q_len + i) * a.num_splits + s;
            a.ws_m[unit] = -INFINITY;
            a.ws_l[unit] = 0.f;
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == kTcMmaWarp) tmem_dealloc(tmem, T::kCols);
}

template <bool E4M3, int NR, bool F8 = false, bool BITCAST = false>
static cudaError_t launch_tc_one(const AttnArgs &a, cudaStream_t stream)
{
    constexpr int bytes = TcLayout<E4M3, NR>::kBytes;
    static uint64_t configured = 0;   // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(attn_tc_kernel<E4M3, NR, F8, BITCAST>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_tc_kernel<E4M3, NR, F8, BITCAST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    const dim3 grid(a.num_splits, a.num_kv_heads, a.batch);
    return launch_pdl(attn_tc_kernel<E4M3, NR, F8, BITCAST>, grid, dim3(kTcThreads), bytes, stream, a);
}

bool tc_supported(int head_dim, int rows) { return head_dim == kTcD && rows > 8 && rows <= 64; }

cudaError_t launch_attention_tc(bool e4m3, const AttnArgs &a, cudaStream_t stream)
{
    if (a.batch == 0) return cudaSuccess;
    if (e4m3 && a.fp8_qk) {
        if (a.rows <= 16) return launch_tc_one<true, 16, true>(a, stream);
        if (a.rows <= 32) return launch_tc_one<true, 32, true>(a, stream);
        return launch_tc_one<true, 64, true>(a, stream);
    }
    if (e4m3 && a.bitcast_decode) {
        if (a.rows <= 16) return launch_tc_one<true, 16, false, true>(a, stream);
        if (a.rows <= 32) return launch_tc_one<true, 32, false, true>(a, stream);
        return launch_tc_one<true, 64, false, true>(a, stream);
    }
    if (e4m3) {
        if (a.rows <= 16) return launch_tc_one<true, 16>(a, stream);
        if (a.rows <= 32) return launch_tc_one<true, 32>(a, stream);
        return launch_tc_one<true, 64>(a, stream);
    }
    if (a.rows <= 16) return launch_tc_one<false, 16>(a, stream);
    if (a.rows <= 32) return launch_tc_one<false, 32>(a, stream);
    return launch_tc_one<false, 64>(a, stream);
}

}  // namespace kvq
