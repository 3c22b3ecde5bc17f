// decode_i8.cu -- instantiates the split-K decode kernel for int8_t K/V pools (q and out:
// __nv_bfloat16), head_dim 64 and 128, 1/2/4/8 query heads per CTA.
#include "decode_split.cuh"

namespace pkv {

cudaError_t launch_split_i8(const SplitParams& p, int D, int heads_per_cta, cudaStream_t s) {
    return launch_split_dispatch<int8_t, __nv_bfloat16>(p, D, heads_per_cta, s);
}

}  // namespace pkv
