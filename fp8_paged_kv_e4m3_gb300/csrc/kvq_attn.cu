// kvq_attn.cu -- instantiations of the split attention kernel with the
// hardware E4M3 conversion and for fp16 pools, the dispatch to the bitcast
// decoder's instantiations, and the log-sum-exp combine kernel.
#include "kvq_attn_kernel.cuh"

namespace kvq {

cudaError_t launch_attention(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    if (a.batch == 0) return cudaSuccess;
    // The fused step: on the split kernel, instances of their own append inside the launch (the
    // attention-only instances compile without that code).  The tcgen05 kernel, whose registers
    // are at their limit, ran measurably slower with it compiled in, even unused; there a small
    // kernel appends by block table first, and the attention-only instance follows.
    if (a.k_new) {
        if (a.mma_sync || !tc_supported(head_dim, a.rows)) return launch_attention_step(e4m3, head_dim, a, stream);
        const cudaError_t e = launch_append_step(e4m3, head_dim, a, stream);
        if (e != cudaSuccess) return e;
        AttnArgs plain = a;
        plain.k_new = plain.v_new = nullptr;
        return launch_attention_tc(e4m3, plain, stream);
    }
    // many query rows per kv head (MTP verify): the tcgen05 kernel (either E4M3 decoder)
    if (!a.mma_sync && tc_supported(head_dim, a.rows)) return launch_attention_tc(e4m3, a, stream);
    if (e4m3 && a.bitcast_decode) return launch_attention_bitcast(head_dim, a, stream);
    if (a.longest_first) return launch_attention_lpt(e4m3, head_dim, a, stream);
    if (e4m3)
        return head_dim == 128 ? launch_rows<true, 128, false>(a, stream)
                               : launch_rows<true, 64, false>(a, stream);
    return head_dim == 128 ? launch_rows<false, 128, false>(a, stream)
                           : launch_rows<false, 64, false>(a, stream);
}

// ---------------------------------------------------------------------------
// Log-sum-exp combine.  WPR warps per (b, h, i) row (4 rows of one warp each,
// or one row of 4 warps for long split lists): every warp finds the row's
// M = max m_s and W = sum l_s exp(m_s - M) with the lanes reading the splits'
// (m, l) side by side; warp w then sums w_s * o_s over splits w, w + WPR, ...
// (merge_splits), and the warps add their sums in shared memory.
// Log-sum-exp merge of one workspace row's S split partials, by one warp:
// M = max m_s and W = sum l_s exp(m_s - M) over the non-empty splits, then
// this lane's V = D/32 channels of sum w_s o_s, w_s = l_s exp(m_s - M), over
// splits s_first, s_first + stride, ...  Every split's m and l are written
// (-inf and 0 when empty), so they are loaded without a test, together with
// the first kB o vectors of this warp's share: one round trip to memory for
// up to 32 splits.  An empty split's o (unwritten) is loaded but never used:
// its weight is 0 and the sum takes it by a select.  Returns W (0 for a row
// without keys, whose acc stays 0).
template <int D>
__device__ __forceinline__ float merge_splits(const float *o_row, const float *m, const float *l, int S, int lane,
                                              int s_first, int s_stride, float (&acc)[D / 32])
{
    constexpr int V = D / 32;
    constexpr int kB = 8;
    constexpr float kLog2e = 1.4426950408889634f;
    auto ld = [](const float *p) { return *p; };
    auto load_batch = [&](float (&x)[kB][V], int s0) {
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int s = s0 + u * s_stride;
#pragma unroll
            for (int v = 0; v < V; ++v) x[u][v] = 0.f;
            if (s < S) {
                const float *p = o_row + (int64_t)s * D + lane * V;
                if (V == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(p);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                    x[u][2] = t.z;
                    x[u][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2 *>(p);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                }
            }
        }
    };
    float x[kB][V];
    load_batch(x, s_first);
    const float ms = lane < S ? ld(m + lane) : -INFINITY;
    const float ls = lane < S ? ld(l + lane) : 0.f;
    float M = ls > 0.f ? ms : -INFINITY;
    for (int s = lane + 32; s < S; s += 32) {
        const float m2 = ld(m + s), l2 = ld(l + s);
        if (l2 > 0.f) M = fmaxf(M, m2);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    // this lane's weight of split `lane` (of the chunk of 32 splits in use)
    float wc = (ls > 0.f && M != -INFINITY) ? ls * fast_exp2((ms - M) * kLog2e) : 0.f;
    float W = wc;
    for (int s = lane + 32; s < S; s += 32) {
        const float m2 = ld(m + s), l2 = ld(l + s);
        if (l2 > 0.f) W += l2 * fast_exp2((m2 - M) * kLog2e);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(kFull, W, off);
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    if (M == -INFINITY) return 0.f;
    int chunk = 0;
    for (int s0 = s_first; s0 < S; s0 += kB * s_stride) {
        if (s0 != s_first) load_batch(x, s0);
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int s = s0 + u * s_stride;   // the same on every lane
            if (s >= S) break;
            if ((s >> 5) != chunk) {            // weights of the next 32 splits
                chunk = s >> 5;
                const int sl = (chunk << 5) + lane;
                const float m2 = sl < S ? ld(m + sl) : -INFINITY, l2 = sl < S ? ld(l + sl) : 0.f;
                wc = l2 > 0.f ? l2 * fast_exp2((m2 - M) * kLog2e) : 0.f;
            }
            const float w = __shfl_sync(kFull, wc, s & 31);
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] += (w != 0.f) ? w * x[u][v] : 0.f;
        }
    }
    return W;
}

// out[b][i][h][lane*V ..] = acc / W in fp16 (0 for W = 0)
template <int D>
__device__ __forceinline__ void store_merged(__half *out, int b, int i, int h, int q_len, int num_q_heads, int lane,
                                             const float (&acc)[D / 32], float W)
{
    constexpr int V = D / 32;
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __half *dst = out + (((int64_t)b * q_len + i) * num_q_heads + h) * D + lane * V;
    if (V == 4) {
        uint2 o2;
        o2.x = pack_half2(acc[0] * inv, acc[1] * inv);
        o2.y = pack_half2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(dst) = o2;
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_half2(acc[0] * inv, acc[1] * inv);
    }
}

template <int D, int WPR>
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ ws_o,
                                                      const float *__restrict__ ws_m,
                                                      const float *__restrict__ ws_l,
                                                      __half *__restrict__ out, int rows, int q_len,
                                                      int num_q_heads, int S)
{
    constexpr int V = D / 32;   // channels per lane (4 or 2)
    constexpr int kRowsPerCta = 4 / WPR;
    __shared__ float red[WPR > 1 ? WPR - 1 : 1][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerCta + warp / WPR;
    const int wr = warp % WPR;   // this warp's share of the splits
    grid_dependency_wait();   // the partials come from the attention kernel
    launch_dependents();
    const bool live = row < rows;   // the same on a row's WPR whole warps
    float acc[V];
    float W = 0.f;
    if (live) {
        W = merge_splits<D>(ws_o + (int64_t)row * S * D, ws_m + (int64_t)row * S, ws_l + (int64_t)row * S, S,
                            lane, wr, WPR, acc);
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
    }
    if (WPR > 1) {
        if (wr > 0)
#pragma unroll
            for (int v = 0; v < V; ++v) red[wr - 1][lane * V + v] = acc[v];
        __syncthreads();
        if (wr > 0) return;
#pragma unroll
        for (int q = 0; q < WPR - 1; ++q)
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] += red[q][lane * V + v];
    }
    if (!live) return;
    // row = (b * Hq + h) * q_len + i  ->  out[b][i][h][:]
    const int i = row % q_len;
    const int bh = row / q_len;
    store_merged<D>(out, bh / num_q_heads, i, bh % num_q_heads, q_len, num_q_heads, lane, acc, W);
}

cudaError_t launch_combine(const float *ws_o, const float *ws_m, const float *ws_l, void *out,
                           int32_t batch, int32_t q_len, int32_t num_q_heads, int32_t head_dim,
                           int32_t num_splits, cudaStream_t stream)
{
    const int rows = batch * num_q_heads * q_len;
    if (rows == 0) return cudaSuccess;
    __half *o = static_cast<__half *>(out);
    if (num_splits >= 16) {   // one row per CTA, four warps over its splits
        const dim3 grid(rows);
        if (head_dim == 128)
            return launch_pdl(combine_kernel<128, 4>, grid, dim3(128), 0, stream, ws_o, ws_m, ws_l, o,
                              rows, q_len, num_q_heads, num_splits);
        return launch_pdl(combine_kernel<64, 4>, grid, dim3(128), 0, stream, ws_o, ws_m, ws_l, o,
                          rows, q_len, num_q_heads, num_splits);
    }
    const dim3 grid((rows + 3) / 4);
    if (head_dim == 128)
        return launch_pdl(combine_kernel<128, 1>, grid, dim3(128), 0, stream, ws_o, ws_m, ws_l, o,
                          rows, q_len, num_q_heads, num_splits);
    return launch_pdl(combine_kernel<64, 1>, grid, dim3(128), 0, stream, ws_o, ws_m, ws_l, o, rows,
                      q_len, num_q_heads, num_splits);
}

}  // namespace kvq
