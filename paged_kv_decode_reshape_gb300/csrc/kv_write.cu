// kv_write.cu -- slot-mapped KV-cache write.
//
// "AMD ATOM inference engine", introduction (the request-lifecycle step of writing into the KV
// cache) and section 5.1 (16-token blocks, one block table per sequence); "LLM Primer VI,
// Chapter 8", section 8.1 (a slot is a position inside a physical block of the flat pool).
// Token i with slot s >= 0 lands in block s / 16, row s % 16, for every kv head, K and V alike.
//
// One thread per 16-byte vector of a row: a warp moves whole 128-512 byte rows with coalesced
// 16-byte loads and stores; the byte copy is exact for every element type. INT8 pools carry one
// fp32 scale per (token, kv head), copied by the thread holding the row's first vector.
#include "pkv_device.cuh"

namespace pkv {

namespace {

__global__ void __launch_bounds__(256) kv_write_kernel(const WriteParams p) {
    grid_dependency_wait();    // the new K/V rows may come from the kernel before this one
    grid_dependents_launch();  // let the attention kernel start its launch meanwhile
    const int vpr = p.row_bytes / 16;
    const long long per_pool = (long long)p.T * p.Hkv * vpr;
    const long long total = 2 * per_pool;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int which = idx >= per_pool;  // 0: K, 1: V
        long long r = idx - which * per_pool;
        const int v = (int)(r % vpr);
        r /= vpr;
        const int h = (int)(r % p.Hkv);
        const long long i = r / p.Hkv;
        const long long s = p.slot_mapping[i];
        if (s < 0) continue;  // padding token
        if (s >= (long long)p.NB * kBlockSize) {
            if (v == 0 && h == 0 && which == 0) flag(p.status, PKV_FLAG_BAD_SLOT);
            continue;
        }
        const long long dst_row = ((s / kBlockSize) * p.Hkv + h) * kBlockSize + s % kBlockSize;
        const long long src_row = i * p.Hkv + h;
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const unsigned char*>(which ? p.v_new : p.k_new) + src_row * p.row_bytes) + v;
        uint4* dst = reinterpret_cast<uint4*>(
            static_cast<unsigned char*>(which ? p.v_pool : p.k_pool) + dst_row * p.row_bytes) + v;
        *dst = *src;
        if (p.k_scales != nullptr && v == 0) {
            if (which) p.v_scales[dst_row] = p.v_new_scales[src_row];
            else p.k_scales[dst_row] = p.k_new_scales[src_row];
        }
    }
}

// Quantising write ("EchoLLMServing inference framework notes", section 3: an INT8 KV cache
// with a per-token scale): each (token, kv head) row of K or V becomes int8 codes plus one fp32
// scale, scale = max|x| / 127 (1 for an all-zero row), code = clamp(rint(x / scale), -127, 127),
// all in IEEE fp32 (correctly rounded divide, round-half-even rint) so the result is bit-exact.
// One warp per row: lane i holds D/32 consecutive values, the row maximum is a warp reduction,
// and the codes go out as one 32- or 16-bit store per lane.
template <typename T, int D>
__global__ void __launch_bounds__(256) kv_write_quant_kernel(const QuantWriteParams p) {
    grid_dependency_wait();
    grid_dependents_launch();
    constexpr int V = D / 32;
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)p.T * p.Hkv;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < 2 * rows; w += nwarps) {
        const int which = w >= rows;  // 0: K, 1: V
        const long long r = w - which * rows;
        const int h = (int)(r % p.Hkv);
        const long long i = r / p.Hkv;
        const long long s = p.slot_mapping[i];
        if (s < 0) continue;
        if (s >= (long long)p.NB * kBlockSize) {
            if (lane == 0 && h == 0 && which == 0) flag(p.status, PKV_FLAG_BAD_SLOT);
            continue;
        }
        const T* src = static_cast<const T*>(which ? p.v_new : p.k_new) + r * D + lane * V;
        float x[V];
#pragma unroll
        for (int e = 0; e < V; ++e) {
            if constexpr (sizeof(T) == 4) x[e] = reinterpret_cast<const float*>(src)[e];
            else x[e] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[e]);
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        float scale = amax / 127.0f;
        if (scale == 0.0f) scale = 1.0f;
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < V; ++e) {
            float q = rintf(x[e] / scale);
            q = fminf(fmaxf(q, -127.0f), 127.0f);
            packed |= (uint32_t)(uint8_t)(int8_t)q << (8 * e);
        }
        const long long dst_row = ((s / kBlockSize) * p.Hkv + h) * kBlockSize + s % kBlockSize;
        int8_t* dst = (which ? p.v_pool : p.k_pool) + dst_row * D + lane * V;
        if constexpr (V == 4) *reinterpret_cast<uint32_t*>(dst) = packed;
        else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
        if (lane == 0) (which ? p.v_scales : p.k_scales)[dst_row] = scale;
    }
}

// Copy-on-write of forked sequences ("LLM Primer VI, Chapter 8", section 8.1: blocks shared by
// reference count): for each (src, dst) pair, block dst of the K pool, the V pool and -- INT8
// pools -- both scale arrays becomes a copy of block src. A block of one array is contiguous
// ([Hkv][16][D] elements, or [Hkv][16] scales), so the copy is a flat run of 16-byte vectors:
// one thread per vector, grid-stride, each pair's ids validated before use.
__global__ void __launch_bounds__(256) kv_copy_blocks_kernel(const CopyBlocksParams p) {
    grid_dependency_wait();    // the pairs, and the pools' last writes, may come from the kernel before
    grid_dependents_launch();  // the write that follows waits for this grid to complete
    long long per_pair = 0;
    for (int a = 0; a < 4; ++a) per_pair += p.vec_per_block[a];
    const long long total = (long long)p.num_pairs * per_pair;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int pair = (int)(idx / per_pair);
        long long v = idx - (long long)pair * per_pair;
        int a = 0;
        while (v >= p.vec_per_block[a]) v -= p.vec_per_block[a++];
        const int src = p.pairs[2 * pair], dst = p.pairs[2 * pair + 1];
        if (src < 0 || src >= p.NB || dst < 0 || dst >= p.NB || src == dst) {
            if (v == 0 && a == 0) flag(p.status, PKV_FLAG_BAD_BLOCK);
            continue;
        }
        uint4* base = static_cast<uint4*>(p.arrays[a]);
        base[(long long)dst * p.vec_per_block[a] + v] = base[(long long)src * p.vec_per_block[a] + v];
    }
}

}  // namespace

cudaError_t launch_kv_write_quant(const QuantWriteParams& p, pkv_dtype src, int D, cudaStream_t s) {
    const long long rows = 2LL * p.T * p.Hkv;
    if (rows == 0) return cudaSuccess;
    long long blocks = (rows + 7) / 8;  // 8 warps (rows) per CTA
    if (blocks > 152 * 8) blocks = 152 * 8;
    const dim3 g((unsigned)blocks), b(256);
    if (src == PKV_F32)
        return D == 128 ? launch_pdl(kv_write_quant_kernel<float, 128>, g, b, 0, s, p)
                        : launch_pdl(kv_write_quant_kernel<float, 64>, g, b, 0, s, p);
    return D == 128 ? launch_pdl(kv_write_quant_kernel<__nv_bfloat16, 128>, g, b, 0, s, p)
                    : launch_pdl(kv_write_quant_kernel<__nv_bfloat16, 64>, g, b, 0, s, p);
}

cudaError_t launch_kv_write(const WriteParams& p, cudaStream_t s) {
    const long long total = 2LL * p.T * p.Hkv * (p.row_bytes / 16);
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;  // grid-stride beyond 32 CTAs per SM
    return launch_pdl(kv_write_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p);
}

}  // namespace pkv

namespace pkv {

cudaError_t launch_kv_copy_blocks(const CopyBlocksParams& p, cudaStream_t s) {
    long long per_pair = 0;
    for (int a = 0; a < 4; ++a) per_pair += p.vec_per_block[a];
    const long long total = (long long)p.num_pairs * per_pair;
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    return launch_pdl(kv_copy_blocks_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p);
}

}  // namespace pkv
