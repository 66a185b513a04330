// kvq_attn_bitcast_lpt.cu -- the bitcast decoder's instances of the split
// attention kernel that take the sequences longest first
// (KVQ_ATTN_LONGEST_FIRST with KVQ_ATTN_BITCAST_DECODE), in a translation unit
// of their own so that they compile in parallel with the others.
#include "kvq_attn_kernel.cuh"

namespace kvq {

cudaError_t launch_attention_bitcast_lpt(int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    return head_dim == 128 ? launch_rows<true, 128, true, true>(a, stream)
                           : launch_rows<true, 64, true, true>(a, stream);
}

}  // namespace kvq
