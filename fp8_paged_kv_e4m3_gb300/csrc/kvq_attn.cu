// kvq_attn.cu -- instantiations of the split attention kernel with the
// hardware E4M3 conversion and for fp16 pools, the dispatch to the bitcast
// decoder's instantiations, and the log-sum-exp combine kernel.
#include "kvq_attn_kernel.cuh"

namespace kvq {

cudaError_t launch_attention(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    if (a.batch == 0) return cudaSuccess;
    if (e4m3 && a.bitcast_decode) return launch_attention_bitcast(head_dim, a, stream);
    // many query rows per kv head (MTP verify): the tcgen05 kernel
    if (!a.mma_sync && tc_supported(head_dim, a.rows)) return launch_attention_tc(e4m3, a, stream);
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
// with independent loads in flight, and the warps add their sums in shared
// memory.
template <int D, int WPR>
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ ws_o,
                                                      const float *__restrict__ ws_m,
                                                      const float *__restrict__ ws_l,
                                                      __half *__restrict__ out, int rows, int q_len,
                                                      int num_q_heads, int S)
{
    constexpr int V = D / 32;   // channels per lane (4 or 2)
    constexpr int kRowsPerCta = 4 / WPR;
    constexpr int kUnroll = 4;
    __shared__ float red[WPR > 1 ? WPR - 1 : 1][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerCta + warp / WPR;
    const int wr = warp % WPR;   // this warp's share of the splits
    grid_dependency_wait();   // the partials come from the attention kernel
    launch_dependents();
    const bool live = row < rows;
    const float *m = ws_m + (int64_t)row * S;
    const float *l = ws_l + (int64_t)row * S;
    // row max over the non-empty splits, lanes striding over s
    float M = -INFINITY;
    if (live)
        for (int s = lane; s < S; s += 32)
            if (l[s] > 0.f) M = fmaxf(M, m[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float W = 0.f;
    if (live && M != -INFINITY)
        for (int s = lane; s < S; s += 32) {
            const float ls = l[s];
            if (ls > 0.f) W += ls * fast_exp2((m[s] - M) * 1.4426950408889634f);
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(kFull, W, off);

    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    if (live && M != -INFINITY) {
        const float *src0 = ws_o + (int64_t)row * S * D + lane * V;
        for (int s0 = wr; s0 < S; s0 += WPR * kUnroll) {
            float w[kUnroll];
            float x[kUnroll][V];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int s = s0 + u * WPR;
                const float ls = s < S ? l[s] : 0.f;
                w[u] = ls > 0.f ? ls * fast_exp2((m[s] - M) * 1.4426950408889634f) : 0.f;
#pragma unroll
                for (int v = 0; v < V; ++v) x[u][v] = 0.f;
                if (w[u] != 0.f) {   // empty splits leave tmp_out unwritten: never read it
                    if (V == 4) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(src0 + (int64_t)s * D);
                        x[u][0] = t4.x;
                        x[u][1] = t4.y;
                        x[u][2] = t4.z;
                        x[u][3] = t4.w;
                    } else {
                        const float2 t2 = *reinterpret_cast<const float2 *>(src0 + (int64_t)s * D);
                        x[u][0] = t2.x;
                        x[u][1] = t2.y;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int v = 0; v < V; ++v) acc[v] += w[u] * x[u][v];
        }
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
    const float inv = W > 0.f ? 1.f / W : 0.f;
    // row = (b * Hq + h) * q_len + i  ->  out[b][i][h][:]
    const int i = row % q_len;
    const int bh = row / q_len;
    const int h = bh % num_q_heads, b = bh / num_q_heads;
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
