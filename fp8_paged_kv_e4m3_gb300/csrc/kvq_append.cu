// kvq_append.cu -- quantise-on-append into page-4 pools, and the amax
// reduction used for calibration.
//
// PR "[Model][SM70][FP8] Integrate calibrated E4M3 QSA KV capacity path",
// section Changes: the main K/V cache is stored in calibrated E4M3 (one scale
// per layer for K, one for V); mixed catch-up/decode batches append prefill
// chunks and decode tokens through the same path; offline calibration gives
// scale = amax / 448.
//
// Layout: one thread owns 8 consecutive channels of one token of one kv head
// for both K and V: two 16-byte fp16 loads, two 8-byte E4M3 stores (or two
// 16-byte stores for the fp16 twin).  Each element is divided by its scale
// in IEEE binary32 (round to nearest even), then converted with the
// hardware satfinite E4M3 conversion, which rounds to nearest even and
// saturates finite overflow to +-448: together, the method's two-step
// rounding.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

// four fp16 -> four E4M3 bytes (element 0 in the lowest byte)
__device__ __forceinline__ uint32_t quantize4(uint2 h, float scale)
{
    const __half2 a = *reinterpret_cast<const __half2 *>(&h.x);
    const __half2 b = *reinterpret_cast<const __half2 *>(&h.y);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    const float2 qa = make_float2(__fdiv_rn(fa.x, scale), __fdiv_rn(fa.y, scale));
    const float2 qb = make_float2(__fdiv_rn(fb.x, scale), __fdiv_rn(fb.y, scale));
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(qa, __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(qb, __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// Grid: x over (token, 8-channel vector) pairs of one kv head, y over the kv
// heads.  With a power-of-two count of vectors per head (D = 64, 128, ...)
// the split of x is a shift (vph_log2 >= 0), else a 32-bit division.
template <bool E4M3>
__global__ void __launch_bounds__(256) append_kernel(const uint4 *__restrict__ k_new,
                                                     const uint4 *__restrict__ v_new,
                                                     const int32_t *__restrict__ slot_mapping,
                                                     int32_t num_tokens, int vph, int vph_log2, int head_dim,
                                                     uint8_t *__restrict__ k_cache,
                                                     uint8_t *__restrict__ v_cache, int64_t num_pages,
                                                     float k_scale, float v_scale, int32_t *err_flag)
{
    grid_dependency_wait();   // new K/V and slots may come from the previous kernel
    launch_dependents();
    const int j = blockIdx.x * blockDim.x + threadIdx.x;   // (token, vector) of kv head g
    const int g = blockIdx.y, num_kv_heads = gridDim.y;
    const int tok = vph_log2 >= 0 ? j >> vph_log2 : j / vph;
    if (tok >= num_tokens) return;
    const int vec = j - tok * vph;
    const int32_t slot = __ldg(slot_mapping + tok);
    if (slot < 0) return;
    const int64_t page = slot >> 2;
    if (page >= num_pages) {
        if (vec == 0 && g == 0) report(err_flag, KVQ_DEV_BAD_SLOT);
        return;
    }
    const int64_t src = ((int64_t)tok * num_kv_heads + g) * vph + vec;
    const int64_t dst = (((page * num_kv_heads + g) * 4) + (slot & 3)) * head_dim + vec * 8;
    const uint4 kv = __ldg(k_new + src);
    const uint4 vv = __ldg(v_new + src);
    if (E4M3) {
        uint2 kq, vq;
        kq.x = quantize4(make_uint2(kv.x, kv.y), k_scale);
        kq.y = quantize4(make_uint2(kv.z, kv.w), k_scale);
        vq.x = quantize4(make_uint2(vv.x, vv.y), v_scale);
        vq.y = quantize4(make_uint2(vv.z, vv.w), v_scale);
        *reinterpret_cast<uint2 *>(k_cache + dst) = kq;
        *reinterpret_cast<uint2 *>(v_cache + dst) = vq;
    } else {
        *reinterpret_cast<uint4 *>(k_cache + 2 * dst) = kv;
        *reinterpret_cast<uint4 *>(v_cache + 2 * dst) = vv;
    }
}

cudaError_t launch_append(bool e4m3, const void *k_new, const void *v_new,
                          const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                          int32_t head_dim, void *k_cache, void *v_cache, int64_t num_pages,
                          float k_scale, float v_scale, int32_t *err_flag, cudaStream_t stream)
{
    const int vph = head_dim / 8;
    const int vph_log2 = (vph & (vph - 1)) == 0 ? __builtin_ctz((unsigned)vph) : -1;
    const int64_t per_head = (int64_t)num_tokens * vph;
    if (per_head == 0 || num_kv_heads == 0) return cudaSuccess;
    if (per_head > 0x7FFFFFFF - 255 || num_kv_heads > 65535) return cudaErrorInvalidConfiguration;
    auto kn = static_cast<const uint4 *>(k_new);
    auto vn = static_cast<const uint4 *>(v_new);
    auto kc = static_cast<uint8_t *>(k_cache);
    auto vc = static_cast<uint8_t *>(v_cache);
    const dim3 grid((unsigned)((per_head + 255) / 256), (unsigned)num_kv_heads);
    if (e4m3)
        return launch_pdl(append_kernel<true>, grid, dim3(256), 0, stream, kn, vn, slot_mapping, num_tokens,
                          vph, vph_log2, head_dim, kc, vc, num_pages, k_scale, v_scale, err_flag);
    return launch_pdl(append_kernel<false>, grid, dim3(256), 0, stream, kn, vn, slot_mapping, num_tokens,
                      vph, vph_log2, head_dim, kc, vc, num_pages, 1.f, 1.f, err_flag);
}

// ---------------------------------------------------------------------------
// The fused step's append where the attention kernel does not append itself
// (the tcgen05 kernel's shapes): token t = b * q_len + i of k_new / v_new
// ([B][q_len][Hkv][D]) goes to position L_b - q_len + i of sequence b, in the
// page its block table names.  A sequence with an invalid length, or a row
// whose page entry is out of range, is skipped; the attention launch that
// follows reports both.  Same arithmetic as append_kernel.
template <bool E4M3>
__global__ void __launch_bounds__(256) append_step_kernel(const uint4 *__restrict__ k_new,
                                                          const uint4 *__restrict__ v_new, AttnArgs a,
                                                          int64_t num_vecs, int vecs_per_token,
                                                          int vecs_per_head, int head_dim)
{
    grid_dependency_wait();   // new K/V may come from the previous kernel
    launch_dependents();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= num_vecs) return;
    const int64_t tok = idx / vecs_per_token;
    const int within = (int)(idx - tok * vecs_per_token);
    const int g = within / vecs_per_head;
    const int d0 = (within - g * vecs_per_head) * 8;
    const int b = (int)(tok / a.q_len), i = (int)(tok % a.q_len);
    const int L = __ldg(a.context_lens + b);
    if (L < a.q_len || L > a.max_pages * 4) return;
    const int pos = L - a.q_len + i;
    const int32_t page = __ldg(a.block_tables + (int64_t)b * a.max_pages + pos / 4);
    if (page < 0 || (int64_t)page >= a.num_pages) return;
    const int64_t dst = (((int64_t)page * a.num_kv_heads + g) * 4 + (pos & 3)) * head_dim + d0;
    auto *kc = static_cast<uint8_t *>(const_cast<void *>(a.k_cache));
    auto *vc = static_cast<uint8_t *>(const_cast<void *>(a.v_cache));
    const uint4 kv = __ldg(k_new + idx);
    const uint4 vv = __ldg(v_new + idx);
    if (E4M3) {
        uint2 kq, vq;
        kq.x = quantize4(make_uint2(kv.x, kv.y), a.k_scale);
        kq.y = quantize4(make_uint2(kv.z, kv.w), a.k_scale);
        vq.x = quantize4(make_uint2(vv.x, vv.y), a.v_scale);
        vq.y = quantize4(make_uint2(vv.z, vv.w), a.v_scale);
        *reinterpret_cast<uint2 *>(kc + dst) = kq;
        *reinterpret_cast<uint2 *>(vc + dst) = vq;
    } else {
        *reinterpret_cast<uint4 *>(kc + 2 * dst) = kv;
        *reinterpret_cast<uint4 *>(vc + 2 * dst) = vv;
    }
}

cudaError_t launch_append_step(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    const int vph = head_dim / 8;
    const int vpt = vph * a.num_kv_heads;
    const int64_t n = (int64_t)a.batch * a.q_len * vpt;
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    auto kn = static_cast<const uint4 *>(a.k_new);
    auto vn = static_cast<const uint4 *>(a.v_new);
    const dim3 grid((unsigned)blocks);
    if (e4m3)
        return launch_pdl(append_step_kernel<true>, grid, dim3(256), 0, stream, kn, vn, a, n, vpt, vph, head_dim);
    return launch_pdl(append_step_kernel<false>, grid, dim3(256), 0, stream, kn, vn, a, n, vpt, vph, head_dim);
}

// ---------------------------------------------------------------------------
// amax = max |x| over an fp16 tensor, one CTA (calibration is off the hot
// loop; a single CTA keeps the result a plain store with no atomics and no
// pre-zeroing).  NaN anywhere gives NaN.
__global__ void __launch_bounds__(1024) amax_kernel(const __half *__restrict__ x, int64_t n,
                                                    float *__restrict__ out)
{
    __shared__ float red[32];
    __shared__ int nan_seen;
    if (threadIdx.x == 0) nan_seen = 0;
    __syncthreads();
    float m = 0.f;
    bool nan = false;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const float v = fabsf(__half2float(x[i]));
        nan |= (v != v);
        m = fmaxf(m, v);
    }
    if (nan) nan_seen = 1;
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (threadIdx.x == 0) *out = nan_seen ? __int_as_float(0x7FC00000) : m;
    }
}

cudaError_t launch_amax(const void *x, int64_t n, float *amax_out, cudaStream_t stream)
{
    amax_kernel<<<1, 1024, 0, stream>>>(static_cast<const __half *>(x), n, amax_out);
    return cudaGetLastError();
}

}  // namespace kvq
