// kvq_attn_cm.cu -- the split attention kernel's cluster-merge instances
// (CMERGE: one cluster per (sequence, kv head), whose splits merge their
// partials into the output themselves; up to 8 query rows per kv head,
// hardware E4M3 conversion and fp16 pools, index order; with and without the
// fused step's append), in a translation unit of their own so that they
// compile in parallel with the others.
#include "kvq_attn_kernel.cuh"

namespace kvq {

template <bool E4M3, int D>
static cudaError_t launch_cm(const AttnArgs &a, cudaStream_t stream)
{
    if (a.k_new) return launch_one<E4M3, D, 1, 1, false, false, true, true>(a, stream);
    return launch_one<E4M3, D, 1, 1, false, false, false, true>(a, stream);
}

cudaError_t launch_attention_cm(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    if (e4m3) return head_dim == 128 ? launch_cm<true, 128>(a, stream) : launch_cm<true, 64>(a, stream);
    return head_dim == 128 ? launch_cm<false, 128>(a, stream) : launch_cm<false, 64>(a, stream);
}

}  // namespace kvq
