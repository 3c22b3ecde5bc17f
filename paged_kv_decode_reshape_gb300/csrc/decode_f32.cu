// decode_f32.cu -- instantiates the split-K decode kernel for float K/V pools (q and out:
// float), head_dim 64 and 128, 1/2/4/8 query heads per CTA.
#include "decode_split.cuh"

namespace pkv {

cudaError_t launch_split_f32(const SplitParams& p, int D, int heads_per_cta, cudaStream_t s) {
    return launch_split_dispatch<float, float>(p, D, heads_per_cta, s);
}

}  // namespace pkv
