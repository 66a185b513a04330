// kvq_attn.cu -- instantiations of the split attention kernel with the
// hardware E4M3 conversion and for fp16 pools, the dispatch to the bitcast
// decoder's instantiations, and the log-sum-exp combine kernel.
#include "kvq_attn_kernel.cuh"

namespace kvq {

bool cluster_merge_applies(bool e4m3, int64_t batch, int num_kv_heads, int rows, int num_splits, bool bitcast,
                           bool longest_first)
{
    const int64_t resident = int64_t(device_sm_count()) * (e4m3 ? 4 : 2);   // the instances' CTAs per SM
    const int64_t ctas = batch * num_kv_heads * num_splits;
    return rows <= 8 && num_splits <= 8 && ctas <= resident && !bitcast && !longest_first;
}

cudaError_t launch_attention(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream, bool *merged)
{
    *merged = false;
    if (a.batch == 0) return cudaSuccess;
    // The full call with up to 8 query rows per kv head and up to 8 splits (hardware decoder, index
    // order), on a grid that is resident in one wave: the splits of each (sequence, kv head) run as
    // one cluster and merge into `out` themselves, with the combine's arithmetic, instead of a
    // combine launch after the whole grid.  A CTA then waits at its end for its cluster's other
    // splits, which costs nothing while every CTA is resident, but on a grid of several waves it
    // would hold an SM slot the next wave needs (the fp16 decode step, 1.7 waves: 48.9 -> 51.2 us).
    if (a.out && cluster_merge_applies(e4m3, a.batch, a.num_kv_heads, a.rows, a.num_splits,
                                       e4m3 && a.bitcast_decode, a.longest_first)) {
        *merged = true;
        return launch_attention_cm(e4m3, head_dim, a, stream);
    }
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
