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

}  // namespace

cudaError_t launch_kv_write(const WriteParams& p, cudaStream_t s) {
    const long long total = 2LL * p.T * p.Hkv * (p.row_bytes / 16);
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;  // grid-stride beyond 32 CTAs per SM
    return launch_pdl(kv_write_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p);
}

}  // namespace pkv
