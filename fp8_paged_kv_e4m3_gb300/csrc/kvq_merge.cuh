// kvq_merge.cuh -- the log-sum-exp merge of one workspace row's split
// partials, shared by the combine kernel and the split kernel's cluster merge,
// so that both give the same bits.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_device.cuh"

namespace kvq {

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
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
    // this lane's weight of split `lane` (of the chunk of 32 splits in use)
    float wc = (ls > 0.f && M != -INFINITY) ? ls * fast_exp2((ms - M) * kLog2e) : 0.f;
    float W = wc;
    for (int s = lane + 32; s < S; s += 32) {
        const float m2 = ld(m + s), l2 = ld(l + s);
        if (l2 > 0.f) W += l2 * fast_exp2((m2 - M) * kLog2e);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xFFFFFFFFu, W, off);
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
            const float w = __shfl_sync(0xFFFFFFFFu, wc, s & 31);
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

}  // namespace kvq
