// pkv_internal.h -- internal interface between the C ABI (pkv_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"  // include/ is on the compiler include path

namespace pkv {

constexpr int kBlockSize = 16;      // tokens per KV block (the only size built)
constexpr int kMaxSplits = 8192;    // split extent the merge kernel supports
constexpr int kMinAutoChunk = 256;   // auto chunk range (tokens per split before block rounding)
constexpr int kMaxAutoChunk = 4096;
// (sequence, kv head, split) units the auto chunk aims at, per kernel: measured on GB300 (152 SMs)
// over chunks 256..4096 on the Llama-3-8B GQA, 131k-context, INT8 and shared-prefix batches. The
// bf16 tensor-core kernel keeps 3 CTAs per SM and does best with fewer, longer splits (with its
// block loop unrolled by two, 1024 units beat 2048 by ~0.4 % on the Llama-3-8B and 131k batches);
// the INT8 one keeps 5 per SM and, doing more arithmetic per byte, does best with more of them.
constexpr long long kTargetUnitsBf16Mma = 1024;
constexpr long long kTargetUnits = 4096;  // INT8 tensor-core and CUDA-core kernels
#ifndef PKV_LPT_MAX_ROWS
#define PKV_LPT_MAX_ROWS 128
#endif
// the tensor-core split kernel starts the longest units first for batches of up to this many
// sequences (each CTA ranks the sequences' split lengths at entry: work grows with the square)
constexpr int kLptMaxRows = PKV_LPT_MAX_ROWS;
constexpr int kMinChunkI8Mma = 512;       // INT8 tensor-core kernel: auto chunk at least this,
constexpr int kMaxSplitsI8Mma = 32;       // and at most this many splits for the longest sequence

// Split rule ("EchoLLMServing inference framework notes", section 2, FlashDecoding):
// split_num = max(1, n // chunk), capped at max_splits; each split is a whole number of
// blocks, per = ceil(n / split_num) rounded up to the block size; split j covers
// [j * per, min(n, (j + 1) * per)); trailing empty splits are dropped. n <= 0 -> 1 split.
__host__ __device__ __forceinline__ int split_count(int n, int chunk, int max_splits, int* per) {
    if (n <= 0) {
        *per = 0;
        return 1;
    }
    int s0 = n / chunk;
    s0 = s0 < 1 ? 1 : (s0 > max_splits ? max_splits : s0);
    int p = (n + s0 - 1) / s0;
    p = (p + kBlockSize - 1) / kBlockSize * kBlockSize;
    *per = p;
    return (n + p - 1) / p;
}

// Context length seen by query token lq (0 <= lq < L) of a sequence whose stored length is n
// (multi-token decode: the L new tokens are the last L positions and attend causally, so token
// lq sees the first n - (L - 1 - lq)). n is first clamped to [0, ncap]; *bad is set when n was
// outside that range or shorter than L.
__host__ __device__ __forceinline__ int query_context_len(int n, int L, int lq, int ncap, bool* bad) {
    *bad = n < L || n > ncap;
    n = n < 0 ? 0 : (n > ncap ? ncap : n);
    n -= L - 1 - lq;
    return n < 0 ? 0 : n;
}

struct SplitParams {
    void* out;                  // [B][Hq][D], element type of q
    const void* q;              // [B][Hq][D]
    const void* k_pool;         // [NB][Hkv][16][D]
    const void* v_pool;
    const float* k_scales;      // [NB][Hkv][16] (int8 only)
    const float* v_scales;
    const int32_t* block_tables;  // [B][MBPS]
    const int32_t* context_lens;  // [B]
    float* ws_acc;              // [B][Hq][S][D]  unnormalised accumulators
    float* ws_ml;               // [B][Hq][S][2]  (m in log2 units, l)
    int32_t* status;
    int B, Hq, Hkv, G, NB, MBPS;
    int L;                      // query tokens per sequence (1: decode); grid.z = B * L
    int chunk, max_splits;      // S = max_splits
    int head_chunks;            // CTAs per kv head along grid.y (ceil(G / heads per CTA))
    int max_context_len;
    float scale_log2;           // scale * log2(e): scores are kept in base-2 units
    int kv_start;               // tokens [0, kv_start) are handled elsewhere (shared prefix), else 0
    int always_partial;         // write (m, l, acc) even for single-split rows (merged later)
    int ws_stride;              // partial slots per (row, query head) in the workspace (>= max_splits)
    int packed;                 // multi-token: one CTA column per (query token, head) of a sequence
    int ntiles;                 // tensor-core kernel: 8-column MMA n-tiles per CTA (1 or 2)
    int lpt;                    // tensor-core kernel: grid row z = the sequence of rank z, longest
                                // splits first (one row per sequence, B <= its row limit)
};

struct MergeParams {
    void* out;
    const float* ws_acc;
    const float* ws_ml;
    const int32_t* context_lens;
    int B, Hq, MBPS, L, chunk, max_splits;  // B: sequences; rows are (sequence, query token)
    int kv_start;          // the split kernel's kv_start (its splits cover [kv_start, n))
    int extra0, extra;     // extra partial slots [extra0, extra0 + extra) per row (shared prefix)
    int ws_stride;         // partial slots per (row, query head) in the workspace
    int packed;            // the split kernel ran packed: splits follow the sequence's last token
};

struct WriteParams {
    const void* k_new;
    const void* v_new;
    void* k_pool;
    void* v_pool;
    const float* k_new_scales;
    const float* v_new_scales;
    float* k_scales;
    float* v_scales;
    const int64_t* slot_mapping;
    int32_t* status;
    int T, Hkv, row_bytes, NB;
};

// Launch `kern` on `s` with programmatic stream serialization (see grid_dependency_wait()).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

struct CopyBlocksParams {
    void* arrays[4];              // K pool, V pool, K scales, V scales (unused ones: 0 vectors)
    long long vec_per_block[4];   // 16-byte vectors one block occupies in each array
    const int32_t* pairs;         // [num_pairs][2]: source block, destination block
    int32_t* status;
    int num_pairs, NB;
};

struct QuantWriteParams {
    const void* k_new;          // [T][Hkv][D] fp32 or bf16
    const void* v_new;
    int8_t* k_pool;             // [NB][Hkv][16][D]
    int8_t* v_pool;
    float* k_scales;            // [NB][Hkv][16]
    float* v_scales;
    const int64_t* slot_mapping;
    int32_t* status;
    int T, Hkv, NB;
};

struct PrefillParams {
    void* out;                    // [total][Hq][128] bf16
    const void* q;                // [total][Hq][128] bf16
    const int32_t* block_tables;  // [B][MBPS]
    const int32_t* context_lens;  // [B]
    const int32_t* query_start;   // [B + 1]
    int32_t* status;
    int B, Hq, Hkv, G, NB, MBPS;
    float scale_log2;
    // INT8 cache (else null): the pools [NB][Hkv][16][128] int8 and scales [NB][Hkv][16] fp32
    const int8_t* k_i8;
    const int8_t* v_i8;
    const float* k_scales;
    const float* v_scales;
};

// Shared-prefix (cascade) decode, prefix part: every (sequence, query head) row of one kv head
// against the first prefix_tokens tokens of block_tables[0], split into key ranges; each range
// writes a partial state (m, l, acc) into partial slot slot0 + split of the decode workspace.
struct PrefixParams {
    const void* q;                // [B][Hq][128] bf16
    const int32_t* block_tables;  // [B][MBPS]; row 0's first prefix blocks are the shared ones
    float* ws_acc;                // [B][Hq][S][128]
    float* ws_ml;                 // [B][Hq][S][2]
    int32_t* status;
    int B, Hq, Hkv, G, NB, MBPS;
    int S, slot0;                 // partial slots per (row, head); first prefix slot
    int prefix_tokens, split_tokens;  // both multiples of 128
    float scale_log2;
    // INT8 cache (else null): the pools [NB][Hkv][16][128] int8 and scales [NB][Hkv][16] fp32
    const int8_t* k_i8;
    const int8_t* v_i8;
    const float* k_scales;
    const float* v_scales;
};

// Launchers (return the launch's error code).
cudaError_t launch_kv_write(const WriteParams& p, cudaStream_t s);
cudaError_t launch_kv_write_quant(const QuantWriteParams& p, pkv_dtype src, int D, cudaStream_t s);
cudaError_t launch_kv_copy_blocks(const CopyBlocksParams& p, cudaStream_t s);
cudaError_t launch_split_f32(const SplitParams& p, int D, int heads_per_cta, cudaStream_t s);
cudaError_t launch_split_bf16(const SplitParams& p, int D, int heads_per_cta, cudaStream_t s);
cudaError_t launch_split_i8(const SplitParams& p, int D, int heads_per_cta, cudaStream_t s);
cudaError_t launch_merge(const MergeParams& p, pkv_dtype out_dtype, int D, cudaStream_t s);

// Tensor-core split kernel for head_dim 128, bf16 or INT8 pools, 8 query heads per CTA; the K and
// V pools are described by TMA tensor maps built with make_pool_tensor_map (false on failure).
bool make_pool_tensor_map(CUtensorMap* map, const void* pool, int num_blocks, int num_kv_heads, bool i8);
// The tcgen05 prefill / prefix kernels' view of a bf16 pool (one box per block tile).
bool make_pool_tensor_map_blocks(CUtensorMap* map, const void* pool, int num_blocks, int num_kv_heads);
// the kernel with two n-tiles (16 columns per CTA); same arguments as launch_split_mma
cudaError_t launch_split_mma_nt2(const SplitParams& p, bool i8, const CUtensorMap& tk,
                                 const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_prefix(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int splits,
                          cudaStream_t s);
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           int max_query_len, cudaStream_t s);
cudaError_t launch_split_mma(const SplitParams& p, bool i8, const CUtensorMap& tk, const CUtensorMap& tv,
                             cudaStream_t s);

}  // namespace pkv
