// decode_static_ws.cu -- paged decode attention for callers that cannot allocate device memory.
//
// pkv_paged_decode_attention needs a workspace for the split-K partial states, which its caller
// allocates. Some callers cannot call cudaMalloc: a plugin that runs inside another runtime's
// memory plan (the host framework owns every device allocation and hands out none for scratch),
// or a latency-critical serving loop where an allocation, with the device-wide synchronisation
// it can imply, is not acceptable. This entry point gives them the same attention with the
// workspace taken from a fixed array that lives in the library itself.
//
// The array is a file-scope __device__ array of PKV_STATIC_WORKSPACE_BYTES bytes; every GPU that
// loads this library holds it until the process exits. Its name in host code is only a host-side
// stand-in, so the device address is looked up with cudaGetSymbolAddress, once per device, on
// the first call made while that device is current, and cached.
#include <mutex>

#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {};

// Device address of the static workspace on the current device (set-up on first use).
pkv_status static_workspace(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_device_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr)
            return PKV_ERR_CUDA;
        g_device_ptr[dev] = p;
    }
    *out = g_device_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_static_ws(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    pkv_dtype dtype, int split_chunk_tokens, int32_t* status, void* stream) {
    // bytes of partial states this batch needs; beyond the array's size the call is refused
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                   max_context_len, split_chunk_tokens);
    if (need > (size_t)PKV_STATIC_WORKSPACE_BYTES) return PKV_ERR_WORKSPACE;
    void* ws = nullptr;
    const pkv_status st = static_workspace(&ws);
    if (st != PKV_OK) return st;
    // Nothing in the workspace has to start at zero: the merge kernel reads only partial states
    // that this call's split kernel wrote.
    return pkv_paged_decode_attention(out, q, k_pool, v_pool, block_tables, context_lens, num_seqs,
                                      num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                      max_blocks_per_seq, max_context_len, scale, dtype,
                                      split_chunk_tokens, ws, PKV_STATIC_WORKSPACE_BYTES, status,
                                      stream);
}
