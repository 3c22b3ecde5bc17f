// decode_mma2.cu -- the tensor-core split kernel with two 8-column n-tiles per CTA (16 query heads,
// or multi-token columns, per kv head read in one pass), in its own translation unit so that the
// library's sources compile in parallel.
#include "decode_mma.cuh"

namespace pkv {

namespace {

template <bool kI8, bool kPacked>
cudaError_t launch_t2(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
    using G = MmaGeom<kI8, 2>;
    auto kern = mma_split_kernel<kI8, kPacked, 2>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.max_splits, p.Hkv * p.head_chunks, p.packed ? p.B : p.B * p.L),
                      dim3(G::THREADS), G::SMEM, s, p, tk, tv);
}

}  // namespace

cudaError_t launch_split_mma_nt2(const SplitParams& p, bool i8, const CUtensorMap& tk,
                                 const CUtensorMap& tv, cudaStream_t s) {
    if (p.packed) return i8 ? launch_t2<true, true>(p, tk, tv, s) : launch_t2<false, true>(p, tk, tv, s);
    return i8 ? launch_t2<true, false>(p, tk, tv, s) : launch_t2<false, false>(p, tk, tv, s);
}

}  // namespace pkv
