// decode_bf16.cu -- instantiates the split-K decode kernel for __nv_bfloat16 K/V pools (q and out:
// __nv_bfloat16), head_dim 64 and 128, 1/2/4/8 query heads per CTA.
#include "decode_split.cuh"

namespace pkv {

cudaError_t launch_split_bf16(const SplitParams& p, int D, int heads_per_cta, cudaStream_t s) {
    return launch_split_dispatch<__nv_bfloat16, __nv_bfloat16>(p, D, heads_per_cta, s);
}

}  // namespace pkv
