// kvq_attn_bitcast.cu -- instantiations of the split attention kernel with
// the bitcast E4M3 decoder of the source pages (PR "[Model][SM70][FP8]
// Integrate calibrated E4M3 QSA KV capacity path", section Changes: an exact
// bitcast software decoder replaced the slower one in the hot loop).  A
// translation unit of its own so that the two decoder families compile in
// parallel.
#include "kvq_attn_kernel.cuh"

namespace kvq {

cudaError_t launch_attention_bitcast(int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    if (a.batch == 0) return cudaSuccess;
    if (a.longest_first) return launch_attention_bitcast_lpt(head_dim, a, stream);
    return head_dim == 128 ? launch_rows<true, 128, true>(a, stream)
                           : launch_rows<true, 64, true>(a, stream);
}

}  // namespace kvq
