// kvq_attn_lpt.cu -- the split attention kernel's instances that take the
// sequences longest first (KVQ_ATTN_LONGEST_FIRST), in a translation unit of
// their own so that they compile in parallel with the index-order ones.
#include "kvq_attn_kernel.cuh"

namespace kvq {

cudaError_t launch_attention_lpt(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    if (e4m3)
        return head_dim == 128 ? launch_rows<true, 128, false, true>(a, stream)
                               : launch_rows<true, 64, false, true>(a, stream);
    return head_dim == 128 ? launch_rows<false, 128, false, true>(a, stream)
                           : launch_rows<false, 64, false, true>(a, stream);
}

}  // namespace kvq
