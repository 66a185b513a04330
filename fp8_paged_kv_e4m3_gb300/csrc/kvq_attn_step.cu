// kvq_attn_step.cu -- the split attention kernel's fused-step instances
// (FUSED: the producers append this step's rows before copying their pages;
// hardware E4M3 conversion and fp16 pools, index order), in a translation
// unit of their own so that they compile in parallel with the others.  The
// append code lives only in these instances: compiled into an instance, even
// unused, it changes that kernel's register allocation and its speed.
#include "kvq_attn_kernel.cuh"

namespace kvq {

cudaError_t launch_attention_step(bool e4m3, int head_dim, const AttnArgs &a, cudaStream_t stream)
{
    if (e4m3)
        return head_dim == 128 ? launch_rows<true, 128, false, false, true>(a, stream)
                               : launch_rows<true, 64, false, false, true>(a, stream);
    return head_dim == 128 ? launch_rows<false, 128, false, false, true>(a, stream)
                           : launch_rows<false, 64, false, false, true>(a, stream);
}

}  // namespace kvq
