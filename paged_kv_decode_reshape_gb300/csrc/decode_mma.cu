// decode_mma.cu -- instantiates the tensor-core split kernel with one n-tile (bf16 and INT8 K/V,
// head_dim 128; decode_mma2.cu has the two-n-tile kernels) and builds the TMA tensor maps that
// describe a K or V pool to the copy engine.
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_mma.cuh"

namespace pkv {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // The driver entry point is looked up once per process (a function pointer, not state of
    // any call).
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

template <bool kI8, bool kPacked>
cudaError_t launch_t(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
    using G = MmaGeom<kI8, 1>;
    auto kern = mma_split_kernel<kI8, kPacked, 1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.max_splits, p.Hkv * p.head_chunks, p.packed ? p.B : p.B * p.L), dim3(G::THREADS), G::SMEM, s,
                      p, tk, tv);
}

}  // namespace

// A pool [NB][Hkv][16][128] as the TMA sees it, 128-byte swizzle. INT8: a 2-D tensor of NB*Hkv*16
// rows of 128 bytes, one box = one (block, kv head) tile [16 rows][128 B]. bf16: a 3-D tensor
// (64 dims, NB*Hkv*16 rows, 2 halves of the 128 dims), one box = one tile as [half][16 rows][128 B]:
// a single copy per tile (a copy's cost on the TMA unit is per box as much as per byte).
bool make_pool_tensor_map(CUtensorMap* map, const void* pool, int num_blocks, int num_kv_heads, bool i8) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t rows = (cuuint64_t)num_blocks * num_kv_heads * kBlockSize;
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r;
    if (i8) {
        const cuuint64_t dims[2] = {(cuuint64_t)kMmaD, rows};
        const cuuint64_t strides[1] = {(cuuint64_t)kMmaD};
        const cuuint32_t box[2] = {128u, (cuuint32_t)kBlockSize};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[3] = {64, rows, 2};
        const cuuint64_t strides[2] = {(cuuint64_t)kMmaD * 2, 128};  // row, half (bytes)
        const cuuint32_t box[3] = {64u, (cuuint32_t)kBlockSize, 2u};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// A bf16 pool as a 4-D tensor (64 dims, 8 rows, 2 halves, NB*Hkv*2 groups of 8 rows): one box is a
// whole (block, kv head) tile laid out as [row group][half][8 rows][128 B], so that in a run of
// tiles every 8 consecutive keys of one 64-dim half sit 2 KB after the previous 8.
bool make_pool_tensor_map_blocks(CUtensorMap* map, const void* pool, int num_blocks, int num_kv_heads) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t groups = (cuuint64_t)num_blocks * num_kv_heads * (kBlockSize / 8);
    const cuuint64_t dims[4] = {64, 8, 2, groups};
    const cuuint64_t strides[3] = {(cuuint64_t)kMmaD * 2, 128, 8 * kMmaD * 2};  // row, half, group
    const cuuint32_t box[4] = {64u, 8u, 2u, 2u};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_split_mma(const SplitParams& p, bool i8, const CUtensorMap& tk, const CUtensorMap& tv,
                             cudaStream_t s) {
    if (p.ntiles == 2) return launch_split_mma_nt2(p, i8, tk, tv, s);
    if (p.packed) return i8 ? launch_t<true, true>(p, tk, tv, s) : launch_t<false, true>(p, tk, tv, s);
    return i8 ? launch_t<true, false>(p, tk, tv, s) : launch_t<false, false>(p, tk, tv, s);
}

}  // namespace pkv
