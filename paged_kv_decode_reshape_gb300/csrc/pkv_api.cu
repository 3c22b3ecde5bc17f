// pkv_api.cu -- the C ABI of libpkv.so (declared in include/pkv.h).
//
// Validates arguments on the host (nothing is enqueued on failure), chooses the split chunk,
// sizes the grids and launches the kernels on the caller's stream. Allocates nothing, keeps no
// state, never synchronises.
#include <stdint.h>

#include "pkv_internal.h"

namespace {

using namespace pkv;

constexpr float kLog2e = 1.4426950408889634f;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [a, a + na) and [b, b + nb) share a byte
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

size_t elem_bytes(pkv_dtype t) { return t == PKV_F32 ? 4 : t == PKV_BF16 ? 2 : t == PKV_I8 ? 1 : 0; }

// the tensor-core kernel serves head_dim 128 with bf16 or INT8 pools; the CUDA-core kernel the rest
bool uses_mma(int head_dim, pkv_dtype kv_dtype) {
    return head_dim == 128 && (kv_dtype == PKV_BF16 || kv_dtype == PKV_I8);
}

long long target_units(int head_dim, pkv_dtype kv_dtype) {
    return uses_mma(head_dim, kv_dtype) && kv_dtype == PKV_BF16 ? kTargetUnitsBf16Mma : kTargetUnits;
}

// Tokens per split before block rounding: the request, or in auto mode the power of two in
// [kMinAutoChunk, kMaxAutoChunk] nearest below (work units of the batch) / (target units of the
// kernel), so that a batch yields about that many (row, kv head, split) units for the GPU's SMs to
// share. The INT8 tensor-core kernel, whose units each pay a start-up of a few microseconds
// against a slower per-byte rate, also keeps at least kMinChunkI8Mma tokens per split and at most
// kMaxSplitsI8Mma splits for the longest sequence (measured on GB300: a 64-sequence, 512-4096
// token batch runs 16 % faster at chunk 512 than 256, a 131k-context batch 8 % faster at 4096
// than 1024). Doubled further while the split extent exceeds what the merge kernel supports.
int choose_chunk(int num_seqs, int num_kv_heads, int max_context_len, int requested, int head_dim,
                 pkv_dtype kv_dtype) {
    if (requested > 0) return requested;
    const long long target = target_units(head_dim, kv_dtype);
    const long long tokens = (long long)num_seqs * num_kv_heads * max_context_len;
    int c = kMinAutoChunk;
    while (c < kMaxAutoChunk && tokens / (2LL * c) >= target) c *= 2;
    if (uses_mma(head_dim, kv_dtype) && kv_dtype == PKV_I8) {
        if (c < kMinChunkI8Mma) c = kMinChunkI8Mma;
        while (c < kMaxAutoChunk && max_context_len / c > kMaxSplitsI8Mma) c *= 2;
    }
    while (max_context_len / c > kMaxSplits) c *= 2;
    return c;
}

// The smallest auto chunk any K/V dtype gets for this shape (the most splits): what a workspace
// sized without knowing the dtype must cover.
int min_chunk_any_dtype(int num_seqs, int num_kv_heads, int max_context_len, int requested, int head_dim) {
    int c = choose_chunk(num_seqs, num_kv_heads, max_context_len, requested, head_dim, PKV_F32);
    for (pkv_dtype t : {PKV_BF16, PKV_I8}) {
        const int x = choose_chunk(num_seqs, num_kv_heads, max_context_len, requested, head_dim, t);
        c = x < c ? x : c;
    }
    return c;
}

int split_extent(int max_context_len, int chunk) {
    const int s = max_context_len / chunk;
    return s < 1 ? 1 : s;
}

size_t workspace_bytes_for(int B, int Hq, int D, int S) {
    if (S <= 1) return 0;
    return (size_t)B * Hq * S * ((size_t)D + 2) * sizeof(float);
}

// Key splits of a shared prefix (cascade decode): enough (row tile, kv head, split) CTAs for about
// kPrefixTargetCtas, each split a whole number of 128-key tiles. Measured on the 256-sequence,
// 2048-token-prefix batch: 64 CTAs (no key split) beat 148, 296 and 600 -- a CTA's set-up (TMEM,
// Q, pipeline fill) outweighs the parallelism splitting the prefix adds.
#ifndef PKV_PREFIX_TARGET_CTAS
#define PKV_PREFIX_TARGET_CTAS 64
#endif
constexpr long long kPrefixTargetCtas = PKV_PREFIX_TARGET_CTAS;
void prefix_splits(int rows, int g, int Hkv, int prefix, int* splits, int* split_tokens) {
    const long long base = (long long)((rows * (long long)g + 127) / 128) * Hkv;
    const int tiles = (prefix + 127) / 128;
    long long s = (kPrefixTargetCtas + base - 1) / base;
    s = s < 1 ? 1 : (s > tiles ? tiles : s);
    const int per = (int)((tiles + s - 1) / s) * 128;
    *split_tokens = per;
    *splits = (prefix + per - 1) / per;
}

int heads_per_cta(int g) { return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8; }

struct Decode {
    void* out; const void* q; const void* k_pool; const void* v_pool;
    const float* k_scales; const float* v_scales;
    const int32_t* block_tables; const int32_t* context_lens;
    int B, L, Hq, Hkv, D, BS, NB, MBPS, max_ctx;  // L: query tokens per sequence
    float scale;
    pkv_dtype q_dtype, kv_dtype;
    int chunk_req;
    void* ws; size_t ws_bytes;
    int32_t* status;
    cudaStream_t stream;
    int prefix;  // shared-prefix tokens (cascade decode), else 0
};

pkv_status run_decode(const Decode& a) {
    if (a.B < 0 || a.L < 1 || a.Hq <= 0 || a.Hkv <= 0 || a.D <= 0 || a.NB <= 0 || a.MBPS <= 0)
        return PKV_ERR_INVALID_ARG;
    if (a.Hq % a.Hkv != 0) return PKV_ERR_INVALID_ARG;
    if (a.BS != kBlockSize || (a.D != 64 && a.D != 128)) return PKV_ERR_UNSUPPORTED;
    if (a.max_ctx < 0 || (long long)a.max_ctx > (long long)a.MBPS * kBlockSize) return PKV_ERR_INVALID_ARG;
    if (a.chunk_req < 0 || a.chunk_req % kBlockSize != 0) return PKV_ERR_INVALID_ARG;
    if (!(a.scale == a.scale) || a.scale == INFINITY || a.scale == -INFINITY) return PKV_ERR_INVALID_ARG;
    if (a.B == 0) return PKV_OK;
    if (!a.out || !a.q || !a.k_pool || !a.v_pool || !a.block_tables || !a.context_lens)
        return PKV_ERR_INVALID_ARG;
    const bool i8 = a.kv_dtype == PKV_I8;
    if (i8 && (!a.k_scales || !a.v_scales)) return PKV_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)a.out, a.q, a.k_pool, a.v_pool, (const void*)a.k_scales,
                            (const void*)a.v_scales})
        if (ptr && !aligned(ptr, 16)) return PKV_ERR_INVALID_ARG;
    if (!aligned(a.block_tables, 4) || !aligned(a.context_lens, 4)) return PKV_ERR_INVALID_ARG;
    const int rows = a.B * a.L;  // (sequence, query token) rows of q and out
    if ((long long)a.B * a.L > 65535) return PKV_ERR_UNSUPPORTED;  // grid.z
    const int g = a.Hq / a.Hkv;
    // head_dim 128 bf16 / INT8 pools run on the tensor-core kernel (8 heads per CTA); fp32 and
    // head_dim 64 on the CUDA-core kernel
    const bool mma = uses_mma(a.D, a.kv_dtype);
    const int hg = mma ? 8 : heads_per_cta(g);
    // Tensor-core kernel: 8 or 16 MMA columns per CTA (one or two n-tiles), holding the query
    // heads of one (sequence, query token) row, or -- multi-token decode -- the (token, head)
    // pairs of a sequence's kv head. Pick the layout with the fewest passes over each sequence's
    // K/V, the narrower and unpacked one on ties.
    bool packed = false;
    int ntiles = 1, head_chunks = (g + hg - 1) / hg;
    if (mma) {
        long long best = -1;
        for (int nt = 1; nt <= 2; ++nt)
            for (int pk = 0; pk <= (a.L > 1 && a.prefix == 0 ? 1 : 0); ++pk) {
                const int cap = 8 * nt;
                const long long passes = pk ? (long long)(a.L * g + cap - 1) / cap
                                            : (long long)a.L * ((g + cap - 1) / cap);
                if (best < 0 || passes < best) {
                    best = passes;
                    ntiles = nt;
                    packed = pk;
                    head_chunks = pk ? (a.L * g + cap - 1) / cap : (g + cap - 1) / cap;
                }
            }
    }
    if ((long long)a.NB * a.Hkv * kBlockSize > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // TMA row index
    if ((long long)a.Hkv * head_chunks > 65535 || a.Hq > 65535) return PKV_ERR_UNSUPPORTED;

    // shared prefix (cascade): tokens [0, prefix) of every sequence are the same blocks; they go to
    // the tcgen05 prefix kernel as P key splits, the split kernel covers [prefix, n)
    const int prefix = a.prefix;
    if (prefix < 0) return PKV_ERR_INVALID_ARG;
    if (prefix > 0) {
        if ((a.kv_dtype != PKV_BF16 && a.kv_dtype != PKV_I8) || a.D != 128 || a.L != 1) return PKV_ERR_UNSUPPORTED;
        if (prefix % kBlockSize || prefix > a.max_ctx) return PKV_ERR_INVALID_ARG;
    }
    const int suffix_max = a.max_ctx - prefix;
    const int chunk = choose_chunk(rows, a.Hkv, suffix_max, a.chunk_req, a.D, a.kv_dtype);
    const int S = split_extent(suffix_max, chunk);
    if (S > kMaxSplits) return PKV_ERR_UNSUPPORTED;
    int P = 0, split_tokens = 0;
    if (prefix > 0) prefix_splits(rows, g, a.Hkv, prefix, &P, &split_tokens);
    const int Sw = S + P;  // partial slots per (row, query head)
    const size_t need = P > 0 ? (size_t)rows * a.Hq * Sw * ((size_t)a.D + 2) * sizeof(float)
                              : workspace_bytes_for(rows, a.Hq, a.D, S);
    if (need > 0) {
        if (!a.ws || a.ws_bytes < need) return PKV_ERR_WORKSPACE;
        if (!aligned(a.ws, 256)) return PKV_ERR_INVALID_ARG;
    }

    // out must not alias an input or the workspace
    const size_t qe = elem_bytes(a.q_dtype), ke = elem_bytes(a.kv_dtype);
    const size_t out_b = (size_t)rows * a.Hq * a.D * qe;
    const size_t pool_b = (size_t)a.NB * a.Hkv * kBlockSize * a.D * ke;
    const size_t sc_b = i8 ? (size_t)a.NB * a.Hkv * kBlockSize * 4 : 0;
    if (overlap(a.out, out_b, a.q, out_b) || overlap(a.out, out_b, a.k_pool, pool_b) ||
        overlap(a.out, out_b, a.v_pool, pool_b) || overlap(a.out, out_b, a.k_scales, sc_b) ||
        overlap(a.out, out_b, a.v_scales, sc_b) ||
        overlap(a.out, out_b, a.block_tables, (size_t)a.B * a.MBPS * 4) ||
        overlap(a.out, out_b, a.context_lens, (size_t)a.B * 4) ||
        overlap(a.out, out_b, a.ws, need))
        return PKV_ERR_INVALID_ARG;

    SplitParams p{};
    p.out = a.out; p.q = a.q; p.k_pool = a.k_pool; p.v_pool = a.v_pool;
    p.k_scales = a.k_scales; p.v_scales = a.v_scales;
    p.block_tables = a.block_tables; p.context_lens = a.context_lens;
    p.ws_acc = need ? static_cast<float*>(a.ws) : nullptr;
    p.ws_ml = need ? static_cast<float*>(a.ws) + (size_t)rows * a.Hq * Sw * a.D : nullptr;
    p.status = a.status;
    p.B = a.B; p.L = a.L; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = g; p.NB = a.NB; p.MBPS = a.MBPS;
    p.chunk = chunk; p.max_splits = S; p.head_chunks = head_chunks;
    p.max_context_len = a.max_ctx;
    p.scale_log2 = a.scale * kLog2e;
    p.kv_start = prefix;
    p.always_partial = P > 0;
    p.ws_stride = Sw;
    p.packed = packed;
    p.ntiles = ntiles;
    // longest units first: the bf16 kernel (measured on GB300: the Llama-3-8B GQA batch 103.1 ->
    // 98.3 us); not the INT8 one, whose many short CTAs pay more for the ranking than they gain
    // (the INT8 batch 212.8 -> 234.9 us)
    p.lpt = mma && a.kv_dtype == PKV_BF16 && (a.L == 1 || packed) && a.B > 1 && a.B <= kLptMaxRows;

    cudaError_t e;
    if (mma) {
        CUtensorMap tk, tv;
        const bool i8m = a.kv_dtype == PKV_I8;
        if (!make_pool_tensor_map(&tk, a.k_pool, a.NB, a.Hkv, i8m) ||
            !make_pool_tensor_map(&tv, a.v_pool, a.NB, a.Hkv, i8m))
            return PKV_ERR_CUDA;
        if (P > 0) {
            // the prefix kernel's one-box-per-block view of the same pools (bf16; an INT8 cache is
            // copied row by row, no tensor map)
            CUtensorMap pk{}, pv{};
            if (!i8m && (!make_pool_tensor_map_blocks(&pk, a.k_pool, a.NB, a.Hkv) ||
                         !make_pool_tensor_map_blocks(&pv, a.v_pool, a.NB, a.Hkv)))
                return PKV_ERR_CUDA;
            PrefixParams x{};
            if (i8m) {
                x.k_i8 = static_cast<const int8_t*>(a.k_pool); x.v_i8 = static_cast<const int8_t*>(a.v_pool);
                x.k_scales = a.k_scales; x.v_scales = a.v_scales;
            }
            x.q = a.q; x.block_tables = a.block_tables; x.ws_acc = p.ws_acc; x.ws_ml = p.ws_ml;
            x.status = a.status; x.B = a.B; x.Hq = a.Hq; x.Hkv = a.Hkv; x.G = g; x.NB = a.NB;
            x.MBPS = a.MBPS; x.S = Sw; x.slot0 = S; x.prefix_tokens = prefix;
            x.split_tokens = split_tokens; x.scale_log2 = p.scale_log2;
            if (launch_prefix(x, pk, pv, P, a.stream) != cudaSuccess) return PKV_ERR_CUDA;
        }
        e = launch_split_mma(p, i8m, tk, tv, a.stream);
    } else if (a.kv_dtype == PKV_F32) e = launch_split_f32(p, a.D, hg, a.stream);
    else if (a.kv_dtype == PKV_BF16) e = launch_split_bf16(p, a.D, hg, a.stream);
    else e = launch_split_i8(p, a.D, hg, a.stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    if (S > 1 || P > 0) {
        MergeParams m{};
        m.out = a.out; m.ws_acc = p.ws_acc; m.ws_ml = p.ws_ml; m.context_lens = a.context_lens;
        m.B = a.B; m.L = a.L; m.Hq = a.Hq; m.MBPS = a.MBPS; m.chunk = chunk; m.max_splits = S;
        m.kv_start = prefix; m.extra0 = S; m.extra = P; m.ws_stride = Sw; m.packed = packed;
        if (launch_merge(m, a.q_dtype, a.D, a.stream) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace

extern "C" {

const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_WORKSPACE: return "workspace too small";
        case PKV_ERR_CUDA: return "CUDA launch failed";
        case PKV_ERR_NO_BLOCKS: return "not enough free KV blocks";
    }
    return "unknown status";
}

const char* pkv_version(void) { return "pkv 0.1 sm_103a"; }

pkv_status pkv_kv_cache_write(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                              const float* k_new_scales, const float* v_new_scales,
                              float* k_scales, float* v_scales, const int64_t* slot_mapping,
                              int num_tokens, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, pkv_dtype dtype, int32_t* status, void* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F32 && dtype != PKV_BF16 && dtype != PKV_I8) return PKV_ERR_INVALID_ARG;
    if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    const bool i8 = dtype == PKV_I8;
    const bool any_scale = k_new_scales || v_new_scales || k_scales || v_scales;
    const bool all_scale = k_new_scales && v_new_scales && k_scales && v_scales;
    if (i8 ? !all_scale : any_scale) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping) return PKV_ERR_INVALID_ARG;
    for (const void* ptr : {k_new, v_new, (const void*)k_pool, (const void*)v_pool})
        if (!aligned(ptr, 16)) return PKV_ERR_INVALID_ARG;
    if (!aligned(slot_mapping, 8)) return PKV_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)k_new_scales, (const void*)v_new_scales,
                            (const void*)k_scales, (const void*)v_scales})
        if (ptr && !aligned(ptr, 4)) return PKV_ERR_INVALID_ARG;
    const size_t row = (size_t)head_dim * elem_bytes(dtype);
    const size_t new_b = (size_t)num_tokens * num_kv_heads * row;
    const size_t pool_b = (size_t)num_blocks * num_kv_heads * kBlockSize * row;
    if (overlap(k_pool, pool_b, v_pool, pool_b) || overlap(k_pool, pool_b, k_new, new_b) ||
        overlap(k_pool, pool_b, v_new, new_b) || overlap(v_pool, pool_b, k_new, new_b) ||
        overlap(v_pool, pool_b, v_new, new_b))
        return PKV_ERR_INVALID_ARG;
    WriteParams p{};
    p.k_new = k_new; p.v_new = v_new; p.k_pool = k_pool; p.v_pool = v_pool;
    p.k_new_scales = k_new_scales; p.v_new_scales = v_new_scales;
    p.k_scales = k_scales; p.v_scales = v_scales;
    p.slot_mapping = slot_mapping; p.status = status;
    p.T = num_tokens; p.Hkv = num_kv_heads; p.row_bytes = (int)row; p.NB = num_blocks;
    return launch_kv_write(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_kv_cache_write_int8(const void* k_new, const void* v_new, int8_t* k_pool,
                                   int8_t* v_pool, float* k_scales, float* v_scales,
                                   const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                   int head_dim, int block_size, int num_blocks,
                                   pkv_dtype src_dtype, int32_t* status, void* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (src_dtype != PKV_F32 && src_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_pool || !v_pool || !k_scales || !v_scales || !slot_mapping)
        return PKV_ERR_INVALID_ARG;
    for (const void* ptr : {k_new, v_new, (const void*)k_pool, (const void*)v_pool})
        if (!aligned(ptr, 16)) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_scales, 4) || !aligned(v_scales, 4) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    const size_t new_b = (size_t)num_tokens * num_kv_heads * head_dim * elem_bytes(src_dtype);
    const size_t pool_b = (size_t)num_blocks * num_kv_heads * kBlockSize * head_dim;
    const size_t sc_b = (size_t)num_blocks * num_kv_heads * kBlockSize * 4;
    const void* outs[4] = {k_pool, v_pool, k_scales, v_scales};
    const size_t out_b[4] = {pool_b, pool_b, sc_b, sc_b};
    for (int i = 0; i < 4; ++i) {
        if (overlap(outs[i], out_b[i], k_new, new_b) || overlap(outs[i], out_b[i], v_new, new_b))
            return PKV_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (overlap(outs[i], out_b[i], outs[j], out_b[j])) return PKV_ERR_INVALID_ARG;
    }
    QuantWriteParams p{};
    p.k_new = k_new; p.v_new = v_new; p.k_pool = k_pool; p.v_pool = v_pool;
    p.k_scales = k_scales; p.v_scales = v_scales; p.slot_mapping = slot_mapping; p.status = status;
    p.T = num_tokens; p.Hkv = num_kv_heads; p.NB = num_blocks;
    return launch_kv_write_quant(p, src_dtype, head_dim, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_kv_cache_copy_blocks(void* k_pool, void* v_pool, float* k_scales, float* v_scales,
                                    const int32_t* block_pairs, int num_pairs, int num_kv_heads,
                                    int head_dim, int block_size, int num_blocks, pkv_dtype dtype,
                                    int32_t* status, void* stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F32 && dtype != PKV_BF16 && dtype != PKV_I8) return PKV_ERR_INVALID_ARG;
    if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    const bool i8 = dtype == PKV_I8;
    if (i8 ? !(k_scales && v_scales) : (k_scales || v_scales)) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!k_pool || !v_pool || !block_pairs) return PKV_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)k_pool, (const void*)v_pool, (const void*)k_scales,
                            (const void*)v_scales})
        if (ptr && !aligned(ptr, 16)) return PKV_ERR_INVALID_ARG;
    if (!aligned(block_pairs, 4)) return PKV_ERR_INVALID_ARG;
    const size_t blk = (size_t)num_kv_heads * kBlockSize * head_dim * elem_bytes(dtype);
    const size_t sblk = (size_t)num_kv_heads * kBlockSize * 4;
    if (overlap(k_pool, blk * num_blocks, v_pool, blk * num_blocks)) return PKV_ERR_INVALID_ARG;
    CopyBlocksParams p{};
    p.arrays[0] = k_pool; p.arrays[1] = v_pool; p.arrays[2] = k_scales; p.arrays[3] = v_scales;
    p.vec_per_block[0] = p.vec_per_block[1] = (long long)(blk / 16);
    p.vec_per_block[2] = p.vec_per_block[3] = i8 ? (long long)(sblk / 16) : 0;
    p.pairs = block_pairs; p.status = status; p.num_pairs = num_pairs; p.NB = num_blocks;
    return launch_kv_copy_blocks(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_decode_split_chunk(int num_seqs, int num_kv_heads, int head_dim, int max_context_len,
                           int split_chunk_tokens, pkv_dtype kv_dtype) {
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
        split_chunk_tokens < 0 || split_chunk_tokens % kBlockSize ||
        (kv_dtype != PKV_F32 && kv_dtype != PKV_BF16 && kv_dtype != PKV_I8))
        return 0;
    return choose_chunk(num_seqs, num_kv_heads, max_context_len, split_chunk_tokens, head_dim, kv_dtype);
}

size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_context_len, int split_chunk_tokens) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_context_len < 0 || split_chunk_tokens < 0 || split_chunk_tokens % kBlockSize)
        return 0;
    // the smallest chunk (most splits) of any K/V dtype: an upper bound for all
    const int chunk = min_chunk_any_dtype(num_seqs, num_kv_heads, max_context_len, split_chunk_tokens, head_dim);
    return workspace_bytes_for(num_seqs, num_q_heads, head_dim, split_extent(max_context_len, chunk));
}

size_t pkv_decode_workspace_bytes_dtype(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int max_context_len, int split_chunk_tokens,
                                        pkv_dtype kv_dtype) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_context_len < 0 || split_chunk_tokens < 0 || split_chunk_tokens % kBlockSize ||
        (kv_dtype != PKV_F32 && kv_dtype != PKV_BF16 && kv_dtype != PKV_I8))
        return 0;
    // the chunk run_decode picks for this shape and K/V dtype, hence its exact split extent
    const int chunk = choose_chunk(num_seqs, num_kv_heads, max_context_len, split_chunk_tokens, head_dim,
                                   kv_dtype);
    return workspace_bytes_for(num_seqs, num_q_heads, head_dim, split_extent(max_context_len, chunk));
}

pkv_status pkv_paged_decode_attention(void* out, const void* q, const void* k_pool,
                                      const void* v_pool, const int32_t* block_tables,
                                      const int32_t* context_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, int max_blocks_per_seq,
                                      int max_context_len, float scale, pkv_dtype dtype,
                                      int split_chunk_tokens, void* workspace,
                                      size_t workspace_bytes, int32_t* status, void* stream) {
    if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    Decode a{out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens,
             num_seqs, 1, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
             max_blocks_per_seq, max_context_len, scale, dtype, dtype, split_chunk_tokens,
             workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream)};
    return run_decode(a);
}

pkv_status pkv_paged_decode_attention_int8(void* out, const void* q, const int8_t* k_pool,
                                           const int8_t* v_pool, const float* k_scales,
                                           const float* v_scales, const int32_t* block_tables,
                                           const int32_t* context_lens, int num_seqs,
                                           int num_q_heads, int num_kv_heads, int head_dim,
                                           int block_size, int num_blocks,
                                           int max_blocks_per_seq, int max_context_len,
                                           float scale, int split_chunk_tokens, void* workspace,
                                           size_t workspace_bytes, int32_t* status,
                                           void* stream) {
    Decode a{out, q, k_pool, v_pool, k_scales, v_scales, block_tables, context_lens,
             num_seqs, 1, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
             max_blocks_per_seq, max_context_len, scale, PKV_BF16, PKV_I8, split_chunk_tokens,
             workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream)};
    return run_decode(a);
}

}  // extern "C"

namespace {

// Paged prefill over a bf16 cache (k_scales == v_scales == null) or an INT8 cache with its scales.
pkv_status run_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                       const float* k_scales, const float* v_scales, bool i8,
                       const int32_t* block_tables, const int32_t* context_lens,
                       const int32_t* query_start, int num_seqs, int total_query_tokens,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int max_blocks_per_seq, int max_query_len, float scale,
                       int32_t* status, void* stream) {
    if (num_seqs < 0 || total_query_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || max_query_len < 0 ||
        num_q_heads % num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim != 128 || block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PKV_ERR_INVALID_ARG;
    if (i8 && (!k_scales || !v_scales)) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_query_tokens == 0 || max_query_len == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens || !query_start)
        return PKV_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)out, q, k_pool, v_pool, (const void*)k_scales, (const void*)v_scales})
        if (ptr && !aligned(ptr, 16)) return PKV_ERR_INVALID_ARG;
    if (num_seqs > 65535 || num_q_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if ((long long)num_blocks * num_kv_heads * kBlockSize > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    const size_t io_b = (size_t)total_query_tokens * num_q_heads * head_dim * 2;
    const size_t pool_b = (size_t)num_blocks * num_kv_heads * kBlockSize * head_dim * (i8 ? 1 : 2);
    const size_t sc_b = i8 ? (size_t)num_blocks * num_kv_heads * kBlockSize * 4 : 0;
    if (overlap(out, io_b, q, io_b) || overlap(out, io_b, k_pool, pool_b) ||
        overlap(out, io_b, v_pool, pool_b) || overlap(out, io_b, k_scales, sc_b) ||
        overlap(out, io_b, v_scales, sc_b) ||
        overlap(out, io_b, block_tables, (size_t)num_seqs * max_blocks_per_seq * 4) ||
        overlap(out, io_b, context_lens, (size_t)num_seqs * 4) ||
        overlap(out, io_b, query_start, (size_t)(num_seqs + 1) * 4))
        return PKV_ERR_INVALID_ARG;
    CUtensorMap tk{}, tv{};  // INT8: the kernel copies rows with 1-D bulk copies, no tensor map
    if (!i8 && (!make_pool_tensor_map_blocks(&tk, k_pool, num_blocks, num_kv_heads) ||
                !make_pool_tensor_map_blocks(&tv, v_pool, num_blocks, num_kv_heads)))
        return PKV_ERR_CUDA;
    PrefillParams p{};
    p.out = out; p.q = q; p.block_tables = block_tables; p.context_lens = context_lens;
    p.query_start = query_start; p.status = status;
    p.B = num_seqs; p.Hq = num_q_heads; p.Hkv = num_kv_heads; p.G = num_q_heads / num_kv_heads;
    p.NB = num_blocks; p.MBPS = max_blocks_per_seq; p.scale_log2 = scale * kLog2e;
    if (i8) {
        p.k_i8 = static_cast<const int8_t*>(k_pool); p.v_i8 = static_cast<const int8_t*>(v_pool);
        p.k_scales = k_scales; p.v_scales = v_scales;
    }
    return launch_prefill(p, tk, tv, max_query_len, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_prefill_attention(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* query_start,
                                       int num_seqs, int total_query_tokens, int num_q_heads,
                                       int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, int max_blocks_per_seq, int max_query_len,
                                       float scale, int32_t* status, void* stream) {
    return run_prefill(out, q, k_pool, v_pool, nullptr, nullptr, false, block_tables, context_lens,
                       query_start, num_seqs, total_query_tokens, num_q_heads, num_kv_heads, head_dim,
                       block_size, num_blocks, max_blocks_per_seq, max_query_len, scale, status, stream);
}

pkv_status pkv_paged_prefill_attention_int8(void* out, const void* q, const int8_t* k_pool,
                                            const int8_t* v_pool, const float* k_scales,
                                            const float* v_scales, const int32_t* block_tables,
                                            const int32_t* context_lens, const int32_t* query_start,
                                            int num_seqs, int total_query_tokens, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int num_blocks, int max_blocks_per_seq,
                                            int max_query_len, float scale, int32_t* status,
                                            void* stream) {
    return run_prefill(out, q, k_pool, v_pool, k_scales, v_scales, true, block_tables, context_lens,
                       query_start, num_seqs, total_query_tokens, num_q_heads, num_kv_heads, head_dim,
                       block_size, num_blocks, max_blocks_per_seq, max_query_len, scale, status, stream);
}

pkv_status pkv_paged_decode_attention_multi(void* out, const void* q, const void* k_pool,
                                            const void* v_pool, const float* k_scales,
                                            const float* v_scales, const int32_t* block_tables,
                                            const int32_t* context_lens, int num_seqs,
                                            int num_query_tokens, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int num_blocks, int max_blocks_per_seq,
                                            int max_context_len, float scale, pkv_dtype kv_dtype,
                                            int split_chunk_tokens, void* workspace,
                                            size_t workspace_bytes, int32_t* status,
                                            void* stream) {
    if (kv_dtype != PKV_F32 && kv_dtype != PKV_BF16 && kv_dtype != PKV_I8) return PKV_ERR_INVALID_ARG;
    if (kv_dtype != PKV_I8 && (k_scales || v_scales)) return PKV_ERR_INVALID_ARG;
    const pkv_dtype q_dtype = kv_dtype == PKV_I8 ? PKV_BF16 : kv_dtype;
    Decode a{out, q, k_pool, v_pool, k_scales, v_scales, block_tables, context_lens,
             num_seqs, num_query_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
             num_blocks, max_blocks_per_seq, max_context_len, scale, q_dtype, kv_dtype,
             split_chunk_tokens, workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream)};
    return run_decode(a);
}

pkv_status pkv_paged_decode_attention_shared_prefix_int8(
    void* out, const void* q, const int8_t* k_pool, const int8_t* v_pool, const float* k_scales,
    const float* v_scales, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
    int max_blocks_per_seq, int max_context_len, float scale, int shared_prefix_tokens,
    int split_chunk_tokens, void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
    if (shared_prefix_tokens <= 0) return PKV_ERR_INVALID_ARG;
    Decode a{out, q, k_pool, v_pool, k_scales, v_scales, block_tables, context_lens,
             num_seqs, 1, num_q_heads, num_kv_heads, head_dim, block_size,
             num_blocks, max_blocks_per_seq, max_context_len, scale, PKV_BF16, PKV_I8,
             split_chunk_tokens, workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream)};
    a.prefix = shared_prefix_tokens;
    return run_decode(a);
}

size_t pkv_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                                int head_dim, int max_context_len,
                                                int shared_prefix_tokens, int split_chunk_tokens) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        head_dim != 128 || max_context_len < 0 || split_chunk_tokens < 0 ||
        split_chunk_tokens % kBlockSize || shared_prefix_tokens <= 0 ||
        shared_prefix_tokens % kBlockSize || shared_prefix_tokens > max_context_len)
        return 0;
    const int suffix_max = max_context_len - shared_prefix_tokens;
    // the bf16 and the INT8 call: the smaller chunk (more suffix splits) covers both
    const int cb = choose_chunk(num_seqs, num_kv_heads, suffix_max, split_chunk_tokens, head_dim, PKV_BF16);
    const int ci = choose_chunk(num_seqs, num_kv_heads, suffix_max, split_chunk_tokens, head_dim, PKV_I8);
    const int chunk = cb < ci ? cb : ci;
    const int S = split_extent(suffix_max, chunk);
    int P = 0, split_tokens = 0;
    prefix_splits(num_seqs, num_q_heads / num_kv_heads, num_kv_heads, shared_prefix_tokens, &P,
                  &split_tokens);
    return (size_t)num_seqs * num_q_heads * (S + P) * ((size_t)head_dim + 2) * sizeof(float);
}

pkv_status pkv_paged_decode_attention_shared_prefix(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    int shared_prefix_tokens, int split_chunk_tokens, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream) {
    if (shared_prefix_tokens <= 0) return PKV_ERR_INVALID_ARG;
    Decode a{out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens,
             num_seqs, 1, num_q_heads, num_kv_heads, head_dim, block_size,
             num_blocks, max_blocks_per_seq, max_context_len, scale, PKV_BF16, PKV_BF16,
             split_chunk_tokens, workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream)};
    a.prefix = shared_prefix_tokens;
    return run_decode(a);
}

}  // extern "C"
