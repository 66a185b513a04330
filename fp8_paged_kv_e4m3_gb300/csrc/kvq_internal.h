// kvq_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

// Arguments of one split-K attention launch (device pointers).
struct AttnArgs {
    const void *q;               // fp16 [B][q_len][Hq][D]
    const void *k_cache;         // pools [P][Hkv][4][D]
    const void *v_cache;
    int64_t num_pages;
    const int32_t *block_tables; // [B][max_pages]
    const int32_t *context_lens; // [B]
    const int32_t *topk_idx;     // [B][Hkv][max_topk] or null
    const int32_t *topk_lens;    // [B] or null
    float *ws_o;                 // [B][Hq][q_len][S][D]
    float *ws_m;                 // [B][Hq][q_len][S]
    float *ws_l;                 // [B][Hq][q_len][S]
    int32_t *err_flag;
    int32_t batch, q_len, num_q_heads, num_kv_heads, group, rows, num_splits;
    int32_t split_pages;   // 0 = equal division of each sequence, else pages per split
    int32_t max_pages, max_topk;
    float qk_scale_log2;         // hoisted: sm_scale * log2(e) [* k_scale for E4M3]
    float out_scale;             // hoisted: v_scale for E4M3, 1 for fp16
    bool bitcast_decode;         // E4M3: the bitcast decoder instead of the hardware conversion
    bool mma_sync;               // keep many-row tiles on the mma.sync kernel
    bool fp8_qk;                 // E4M3 scores on the tcgen05 kernel (query quantised per CTA)
    bool early_pages;            // split kernel, no top-k list: block tables, lengths and pages of
                                 // positions < L - q_len may be read before the dependency wait
    bool longest_first;          // split kernel (hardware decoder): CTAs take the sequences longest first
    // Fused step (no top-k list): this step's new rows, fp16 [B][q_len][Hkv][D], quantised
    // (E4M3: divided by k_scale / v_scale) or copied (fp16) into the pools -- by the split
    // kernel's FUSED instances before they copy the pages that hold them, or by the append
    // kernel that precedes the tcgen05 kernel; null for the attention-only calls.
    const void *k_new = nullptr;
    const void *v_new = nullptr;
    float k_scale = 1.f, v_scale = 1.f;
    // fp16 [B][q_len][Hq][D] output of the full call, or null (partials only); the split
    // kernel's cluster-merge instances write it themselves
    void *out = nullptr;
};

// Arguments of one chunked-prefill attention call (device pointers).
struct PrefillArgs {
    const void *q;               // fp16 [q_start[B]][Hq][128]
    const void *k_cache;         // pools [P][Hkv][4][128]
    const void *v_cache;
    int64_t num_pages;
    const int32_t *block_tables; // [B][max_pages]
    const int32_t *context_lens; // [B]
    const int32_t *q_start;      // [B + 1]
    void *out;                   // fp16 [q_start[B]][Hq][128]
    uint8_t *tiles;              // fp16 K/V tiles [B][Hkv][max_tiles][2][128 x 128]
    uint32_t *tile_mask;         // [B][Hkv][max_tiles][4]: keys with a bad page
    int32_t *err_flag;
    int32_t batch, num_q_heads, num_kv_heads, group, max_pages, max_q_len, max_tiles, total_q;
    float qk_scale_log2;         // sm_scale * log2(e) [* k_scale for E4M3]
    float out_scale;             // v_scale for E4M3, 1 for fp16
};

size_t prefill_tiles_bytes(int32_t batch, int32_t num_kv_heads, int32_t max_tiles);
size_t prefill_mask_offset(int32_t batch, int32_t num_kv_heads, int32_t max_tiles);
int32_t prefill_max_tiles(int32_t max_pages);
cudaError_t launch_prefill(bool e4m3, const PrefillArgs &a, cudaStream_t stream);

struct WorkspaceLayout {
    size_t o_off, m_off, l_off, total;
};

WorkspaceLayout workspace_layout(int64_t rows_total, int32_t num_splits, int32_t head_dim);

// *merged: set when the launch also merged the partials into a.out (the cluster merge), so that
// no combine follows
cudaError_t launch_attention(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream, bool *merged);
// whether a full call takes the cluster merge (the rule launch_attention applies)
bool cluster_merge_applies(bool e4m3, int64_t batch, int num_kv_heads, int rows, int num_splits, bool bitcast,
                           bool longest_first);
// the split kernel's cluster-merge instances (kvq_attn_cm.cu)
cudaError_t launch_attention_cm(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream);
// the split kernel's longest-first instances (kvq_attn_lpt.cu)
cudaError_t launch_attention_lpt(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream);
cudaError_t launch_attention_bitcast(int head_dim, const AttnArgs &a, cudaStream_t stream);
cudaError_t launch_attention_bitcast_lpt(int head_dim, const AttnArgs &a, cudaStream_t stream);
cudaError_t launch_attention_tc(bool e4m3, const AttnArgs &a, cudaStream_t stream);
// the fused step (a.k_new set): the split kernel's instances that append in the launch
// (kvq_attn_step.cu), and the append by block table that precedes the tcgen05 kernel
// (kvq_append.cu)
cudaError_t launch_attention_step(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream);
cudaError_t launch_append_step(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream);
bool tc_supported(int head_dim, int rows);
cudaError_t launch_combine(const float *ws_o, const float *ws_m, const float *ws_l, void *out,
                           int32_t batch, int32_t q_len, int32_t num_q_heads, int32_t head_dim,
                           int32_t num_splits, cudaStream_t stream);
cudaError_t launch_append(bool e4m3, const void *k_new, const void *v_new,
                          const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                          int32_t head_dim, void *k_cache, void *v_cache, int64_t num_pages,
                          float k_scale, float v_scale, int32_t *err_flag, cudaStream_t stream);
cudaError_t launch_amax(const void *x, int64_t n, float *amax_out, cudaStream_t stream);

int device_sm_count();

// Launch `kernel` on `stream` with programmatic stream serialisation, so that
// it may begin while the previous kernel in the stream drains (the kernel
// waits with griddepcontrol.wait before reading its inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace kvq
