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
// stand-in, so the device address is looked up with cudaGetSymbolAddress on the first call made
// while a device is current, and cached for that device together with the unique id of the
// context it was looked up in. A later call in another context on the same device (after
// cudaDeviceReset, say, when the module may load at another address) looks the address up again.
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {};
unsigned long long g_context_id[kMaxDevices] = {};

// Unique id of the current context (cuCtxGetId, through the runtime's driver entry-point query so
// that the library needs no link against the driver library); false if it cannot be read.
bool current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the static workspace on the current device (looked up on first use there,
// and again whenever the device's context has changed since).
pkv_status static_workspace(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (have_ctx && g_device_ptr[dev] != nullptr && g_context_id[dev] == ctx) {
        *out = g_device_ptr[dev];
        return PKV_OK;
    }
    // set-up: the lookup also makes the device's primary context current on this thread if no
    // context was, so the context id is read after it
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
    if (!current_context_id(&ctx)) return PKV_ERR_CUDA;
    g_device_ptr[dev] = p;
    g_context_id[dev] = ctx;
    *out = p;
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_static_ws(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    pkv_dtype dtype, int split_chunk_tokens, int32_t* status, void* stream) {
    if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    // the exact bytes of partial states this call uses (its own chunk for this dtype); beyond the
    // array's size the call is refused before anything is enqueued
    const size_t need = pkv_decode_workspace_bytes_dtype(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                         max_context_len, split_chunk_tokens, dtype);
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
