/*
 * pkv.h -- C ABI of libpkv.so: paged KV-cache decode on one NVIDIA GB300 (sm_103a).
 *
 * The hot path, each operation the GPU form of a step the pages describe:
 *   pkv_kv_cache_write                 -- store the new tokens' K and V into their slots of the
 *                                         paged pool ("AMD ATOM inference engine", introduction:
 *                                         the request-lifecycle step of writing into the KV
 *                                         cache; section 5.1: 16-token blocks, one block table
 *                                         per sequence).
 *   pkv_paged_decode_attention         -- decode attention that gathers K and V through the
 *                                         block tables ("LLM Primer VI, Chapter 8", section 8.1)
 *                                         with split-K online softmax and a second merge kernel
 *                                         ("EchoLLMServing inference framework notes", section 2,
 *                                         PagedAttention V2 and FlashDecoding).
 *   pkv_paged_decode_attention_int8    -- the same over an INT8 K/V cache with per-token scales,
 *                                         dequantised inside the kernel (same notes, section 3).
 * Around it:
 *   pkv_kv_cache_write_int8            -- the INT8 cache's write: quantise each row, keep its scale.
 *   pkv_paged_decode_attention_multi   -- L query tokens per sequence, causal among themselves.
 *   pkv_paged_decode_attention_shared_prefix[_int8] -- decode of a batch sharing a prefix: the prefix once
 *                                         per kv head on the tcgen05 tensor cores, then the suffixes.
 *   pkv_paged_prefill_attention        -- chunked, variable-length prefill (mixed batches) on tcgen05.
 *   pkv_paged_prefill_attention_int8   -- the same over an INT8 cache, dequantised in the kernel.
 *   pkv_paged_decode_attention_static_ws -- decode with a library-held workspace (no allocation).
 *   pkv_bm_*                           -- host block manager: allocation, refcounted prefix sharing.
 *   pkv_xxh64, pkv_block_hash          -- the chained per-block prefix hash it keys shared blocks by.
 *   pkv_kv_cache_copy_blocks             -- copy-on-write of blocks shared by forked sequences.
 *   pkv_decode_split_chunk, pkv_decode_workspace_bytes, pkv_decode_workspace_bytes_dtype,
 *   pkv_decode_shared_prefix_workspace_bytes
 *                                      -- the split rule and workspace sizes the calls use.
 *
 * Layouts (all row-major, element strides implied by the shapes):
 *   q, out       [num_seqs][num_q_heads][head_dim]
 *   k_new, v_new [num_tokens][num_kv_heads][head_dim]
 *   k/v pool     [num_blocks][num_kv_heads][block_size][head_dim]
 *   k/v scales   [num_blocks][num_kv_heads][block_size]      (fp32, INT8 pools only)
 *   block_tables [num_seqs][max_blocks_per_seq] int32; entry j of row b is the physical block
 *                holding logical tokens [16 j, 16 j + 16) of sequence b
 *   context_lens [num_seqs] int32: tokens of each sequence, counting this step's new token
 *   slot_mapping [num_tokens] int64: physical slot block * block_size + offset; < 0 = padding
 * Query head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: every array pointer is DEVICE memory owned by the caller; the library allocates
 * nothing, keeps no state between calls and never synchronises. Work is enqueued on `stream`
 * (a cudaStream_t; NULL = the legacy default stream) and is asynchronous to the host.
 * Pointers to device arrays must be 16-byte aligned; `out` must not alias any input.
 *
 * Errors: argument checks run on the host before any launch; on failure nothing is enqueued
 * and the status says why. PKV_ERR_CUDA means a launch was rejected by the CUDA runtime.
 * Bad VALUES inside device arrays (a block id outside [0, num_blocks), a slot outside the pool,
 * a context_len above max_blocks_per_seq * block_size) are never dereferenced: the kernels
 * skip them and, when `status` is non-NULL, OR a PKV_FLAG_* bit into that device int32.
 * The caller clears it; the library only sets bits.
 *
 * Pool contents: only the first context_lens[b] slots of each table are read into a result. The
 * other slots of a sequence's last block, and blocks no table references, may hold any bits (stale
 * tokens, NaN, never-written memory; INT8: any scales) without changing an output: K scores past
 * the context are masked to -inf and their V rows (bf16 / fp32) or V scales (INT8) are zeroed or
 * not read before a weight of 0 could meet them. Outputs are written in their own rows only.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, misalignment, aliasing */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim not 64/128, block_size not 16,
                                  or a pool / grid past the kernels' index limits */
    PKV_ERR_WORKSPACE = 3,     /* workspace smaller than pkv_decode_workspace_bytes() */
    PKV_ERR_CUDA = 4,          /* the CUDA runtime rejected a launch */
    PKV_ERR_NO_BLOCKS = 5      /* block manager: not enough free blocks (nothing was changed) */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_I8 = 2 } pkv_dtype;

/* bits the kernels OR into *status (device int32) when they meet bad values */
#define PKV_FLAG_BAD_SLOT 0x1         /* slot >= num_blocks * block_size: token not written */
#define PKV_FLAG_BAD_BLOCK 0x2        /* block id outside [0, num_blocks): block skipped */
#define PKV_FLAG_BAD_CONTEXT 0x4      /* context_len < 0 or > max_blocks_per_seq * block_size:
                                         clamped to [0, max_blocks_per_seq * block_size] */
#define PKV_FLAG_LONG_CONTEXT 0x8     /* context_len > max_context_len: still correct, the
                                         sequence's splits were made longer (informational) */
#define PKV_FLAG_TIMEOUT 0x10         /* a wait for a staged copy exceeded 1 s: that unit was
                                         abandoned and its output rows are undefined */
#define PKV_FLAG_BAD_PREFIX 0x20      /* shared-prefix call: a sequence's table does not start with
                                         the shared blocks, or its context is shorter than the
                                         prefix; that sequence's output is undefined */

/* Static text for a status code. Never NULL. */
const char* pkv_status_string(pkv_status s);

/* Library build identification, e.g. "pkv 0.1 sm_103a". */
const char* pkv_version(void);

/*
 * Slot-mapped KV write ("AMD ATOM inference engine", introduction and section 5.1;
 * "LLM Primer VI, Chapter 8", section 8.1). For every token i < num_tokens with
 * s = slot_mapping[i] >= 0, and every kv head h:
 *     k_pool[s / block_size][h][s % block_size][:] = k_new[i][h][:]      (likewise v)
 * as a bit copy. For dtype PKV_I8 the per-token scales move with the rows:
 *     k_scales[s / block_size][h][s % block_size] = k_new_scales[i][h]   (likewise v)
 * (the four scale pointers must be NULL for other dtypes). Slots must be unique within a
 * call; negative slots are skipped; slots >= num_blocks * block_size are skipped and flagged.
 */
pkv_status pkv_kv_cache_write(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                              const float* k_new_scales, const float* v_new_scales,
                              float* k_scales, float* v_scales, const int64_t* slot_mapping,
                              int num_tokens, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, pkv_dtype dtype, int32_t* status, void* stream);

/*
 * Quantising KV write for an INT8 cache ("EchoLLMServing inference framework notes", section 3:
 * INT8 KV cache with a per-token scale, dequantised inside the attention kernel). For every token
 * i with s = slot_mapping[i] >= 0 and kv head h, the row x = k_new[i][h][:] (fp32 or bf16,
 * src_dtype) is stored as
 *     scale = max_d |x_d| / 127            (1 if the row is all zeros)
 *     k_pool[s / 16][h][s % 16][d] = clamp(rint(x_d / scale), -127, 127)   (round half to even)
 *     k_scales[s / 16][h][s % 16]   = scale
 * in IEEE fp32 arithmetic (so it is bit-reproducible), and likewise for V. Codes never use -128.
 * Slot rules, flags and errors as pkv_kv_cache_write. Dequantised values x_d ~ code * scale are
 * within scale / 2 of x_d.
 */
pkv_status pkv_kv_cache_write_int8(const void* k_new, const void* v_new, int8_t* k_pool,
                                   int8_t* v_pool, float* k_scales, float* v_scales,
                                   const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                   int head_dim, int block_size, int num_blocks,
                                   pkv_dtype src_dtype, int32_t* status, void* stream);

/*
 * Paged (chunked, variable-length) prefill attention on tcgen05 tensor cores ("EchoLLMServing
 * inference framework notes", section 2: FlashAttention tiles the prefill queries; section 3:
 * chunked prefill; "LLM Primer VI, Chapter 8", section 8.1: K/V through the block table).
 * Sequence b owns query rows query_start[b] .. query_start[b + 1] - 1 of q and out
 * ([total_query_tokens][num_q_heads][128], bf16): they are the last
 * L_b = query_start[b + 1] - query_start[b] tokens of its context_lens[b] tokens, whose K/V are
 * already in the pool (written with pkv_kv_cache_write). Row i of sequence b attends causally:
 *     out[query_start[b] + i][h][:] = sum_{t < n_b - L_b + 1 + i} softmax_t(scale * <q, K_t>) V_t
 * bf16 pools [num_blocks][num_kv_heads][16][128] only (head_dim 128; PKV_ERR_UNSUPPORTED
 * otherwise). query_start is int32 [num_seqs + 1], non-decreasing, query_start[0] = 0;
 * max_query_len >= every L_b (sizes the grid; a longer sequence's extra rows are not computed).
 * A sequence with context_lens[b] < L_b or beyond the table is flagged (PKV_FLAG_BAD_CONTEXT) and
 * its rows are not written. Needs no workspace. Accumulation fp32 in TMEM; the softmax weights
 * enter the second product as bf16.
 */
pkv_status pkv_paged_prefill_attention(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* query_start,
                                       int num_seqs, int total_query_tokens, int num_q_heads,
                                       int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, int max_blocks_per_seq, int max_query_len,
                                       float scale, int32_t* status, void* stream);

/*
 * Paged prefill over an INT8 cache ("EchoLLMServing inference framework notes", section 3: the
 * per-token dequantisation fused into the attention kernels, FlashAttention prefill as well as
 * FlashDecoding; chunked prefill and mixed prefill + decode batches over the same cache). Same
 * rows, causal rule, arguments and errors as pkv_paged_prefill_attention, with
 *     K_t = k_pool[blk][g][off][:] * k_scales[blk][g][off],  V_t likewise with v_scales
 * (int8 pools [num_blocks][num_kv_heads][16][128], fp32 scales [num_blocks][num_kv_heads][16],
 * all 16-byte aligned; q and out bf16). Inside the kernel the tcgen05 products run on fp16
 * operands (they take both operands in one 16-bit type): the int8 codes exactly (K with an offset
 * of 1152 removed from each score), q scaled by one power of two per 128 rows (exact for bf16
 * values, within fp16's range), each key's K scale applied to its fp32 score and its V scale to
 * its weight before the weight is rounded to fp16; accumulation fp32.
 */
pkv_status pkv_paged_prefill_attention_int8(void* out, const void* q, const int8_t* k_pool,
                                            const int8_t* v_pool, const float* k_scales,
                                            const float* v_scales, const int32_t* block_tables,
                                            const int32_t* context_lens, const int32_t* query_start,
                                            int num_seqs, int total_query_tokens, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int num_blocks, int max_blocks_per_seq,
                                            int max_query_len, float scale, int32_t* status,
                                            void* stream);

/*
 * Multi-token decode: L = num_query_tokens new tokens per sequence, verified in one pass, as MTP
 * speculative decoding does ("AMD ATOM inference engine", section 4: a decode step reserves
 * num_new_tokens = mtp_k + 1 cache slots per sequence). The L new tokens are the last L of
 * context_lens[b] (already written with pkv_kv_cache_write[_int8]); query token l attends
 * causally to the first context_lens[b] - (L - 1 - l) tokens:
 *     out[b][l][h][:] = sum_{t < n_b - L + 1 + l} softmax_t(scale * <q[b][l][h], K_t>) V_t
 * q and out are [num_seqs][L][num_q_heads][head_dim]. kv_dtype PKV_F32 / PKV_BF16: q, out and the
 * pools share it and the scale pointers must be NULL; PKV_I8: int8 pools with fp32 scales
 * (as pkv_paged_decode_attention_int8), q and out bf16. Every (sequence, query token) row is
 * split like a decode row, so the workspace is pkv_decode_workspace_bytes(num_seqs * L, ...).
 * num_query_tokens = 1 is pkv_paged_decode_attention(_int8). A context_lens[b] < L is a caller
 * error: it is flagged (PKV_FLAG_BAD_CONTEXT) and the rows with no visible token are zeros.
 */
pkv_status pkv_paged_decode_attention_multi(void* out, const void* q, const void* k_pool,
                                            const void* v_pool, const float* k_scales,
                                            const float* v_scales, const int32_t* block_tables,
                                            const int32_t* context_lens, int num_seqs,
                                            int num_query_tokens, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int num_blocks, int max_blocks_per_seq,
                                            int max_context_len, float scale, pkv_dtype kv_dtype,
                                            int split_chunk_tokens, void* workspace,
                                            size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Decode attention for a batch whose sequences all begin with the same shared_prefix_tokens
 * tokens stored in the same blocks -- the refcounted prefix sharing of "LLM Primer VI, Chapter 8",
 * section 8.1 (one system prompt, or the samples of one request). The result is that of
 * pkv_paged_decode_attention with the same arguments (the same softmax, summed in another
 * order). The pages run each sequence over the whole context; here the prefix is read once per
 * kv head and multiplied against every sequence's query heads at once on the tensor cores
 * (tcgen05, the prefill kernel's machinery, split into key ranges), each sequence's own suffix
 * [shared_prefix_tokens, context_len) goes through the split-K decode kernel, and the merge
 * kernel combines both sets of (m, l, acc) states ("EchoLLMServing inference framework notes",
 * section 2).
 * bf16 q / out / pools, head_dim 128, one query token per sequence. shared_prefix_tokens is a
 * positive multiple of block_size, <= max_context_len. The shared blocks are read from
 * block_tables row 0; a sequence whose table does not start with them, or whose context_len is
 * below shared_prefix_tokens, is flagged PKV_FLAG_BAD_PREFIX and its output is undefined.
 * workspace: at least pkv_decode_shared_prefix_workspace_bytes(...) bytes, 256-byte aligned,
 * contents on entry irrelevant. Other arguments and errors as pkv_paged_decode_attention.
 */
pkv_status pkv_paged_decode_attention_shared_prefix(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    int shared_prefix_tokens, int split_chunk_tokens, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream);

/*
 * The same over an INT8 cache ("EchoLLMServing inference framework notes", section 3): int8 pools
 * with their fp32 per-token scales [num_blocks][num_kv_heads][16], q and out bf16. The prefix goes
 * through the INT8 prefill kernel's machinery (rows dequantised in shared memory), the suffixes
 * through the INT8 split-K decode kernel; the result is pkv_paged_decode_attention_int8's.
 */
pkv_status pkv_paged_decode_attention_shared_prefix_int8(
    void* out, const void* q, const int8_t* k_pool, const int8_t* v_pool, const float* k_scales,
    const float* v_scales, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
    int max_blocks_per_seq, int max_context_len, float scale, int shared_prefix_tokens,
    int split_chunk_tokens, void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* Workspace bytes pkv_paged_decode_attention_shared_prefix[_int8] needs (0 for invalid arguments):
 * num_seqs * num_q_heads * (suffix splits + prefix key splits) * (head_dim + 2) * 4, with the
 * suffix split count of whichever of the bf16 and INT8 calls splits more (an upper bound for
 * both). Pure host arithmetic. */
size_t pkv_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                                int head_dim, int max_context_len,
                                                int shared_prefix_tokens, int split_chunk_tokens);

/*
 * Bytes of device workspace pkv_paged_decode_attention[_int8] needs for the split-K partial
 * states (m, l, acc) of a batch: the split count per sequence follows "EchoLLMServing
 * inference framework notes", section 2 (split_num = max(1, context_len // chunk)), so the
 * bound uses max_context_len. split_chunk_tokens = 0 selects the library's chunk for this batch
 * shape. The auto chunk depends on the K/V dtype (pkv_decode_split_chunk); this bound takes the
 * smallest chunk any dtype would get, so it covers them all. Returns 0 for invalid arguments.
 * Pure host arithmetic.
 */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_context_len, int split_chunk_tokens);

/*
 * The exact workspace bytes of one call of pkv_paged_decode_attention (kv_dtype PKV_F32 or
 * PKV_BF16) or pkv_paged_decode_attention_int8 (kv_dtype PKV_I8) with this batch shape: the
 * same split rule as pkv_decode_workspace_bytes, at the chunk pkv_decode_split_chunk gives for
 * that K/V dtype, so it is never larger than that dtype-free bound (at most half of it when the
 * bf16 head_dim-128 kernel takes a longer auto chunk). For the multi-token call pass
 * num_seqs * num_query_tokens as num_seqs. 0 when no split is needed or for invalid arguments.
 * Pure host arithmetic.
 */
size_t pkv_decode_workspace_bytes_dtype(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int max_context_len, int split_chunk_tokens,
                                        pkv_dtype kv_dtype);

/* The chunk (tokens per split before block rounding) that pkv_paged_decode_attention[_int8,
 * _multi] use for a request of split_chunk_tokens (0 = auto), this batch shape and K/V dtype
 * (num_seqs counts (sequence, query token) rows for the multi-token call); 0 for invalid
 * arguments. The same notes call the chunk a value calibrated by profiling the GPU; the auto rule
 * here is the power of two in [256, 4096] nearest below num_seqs * num_kv_heads *
 * max_context_len / (2 * U), where U is the number of (sequence, kv head, split) units the kernel
 * that serves the call does best with on a GB300 (152 SMs): 1024 for the bf16 head_dim-128
 * tensor-core kernel, 4096 for the INT8 one and for the CUDA-core kernel (fp32, head_dim 64).
 * The INT8 head_dim-128 kernel then takes at least 512 and doubles the chunk while the longest
 * sequence would get more than 32 splits. The chunk then grows until the split extent
 * max(1, max_context_len / chunk) is at most 8192.
 * Pure host arithmetic. */
int pkv_decode_split_chunk(int num_seqs, int num_kv_heads, int head_dim, int max_context_len,
                           int split_chunk_tokens, pkv_dtype kv_dtype);

/*
 * Paged decode attention ("LLM Primer VI, Chapter 8", section 8.1; "EchoLLMServing inference
 * framework notes", section 2). For every sequence b and query head h, with n = context_lens[b]
 * and kv head g = h / (num_q_heads / num_kv_heads):
 *     K_t = k_pool[block_tables[b][t / bs]][g][t % bs][:],  V_t likewise,  t < n
 *     out[b][h][:] = sum_t softmax_t(scale * <q[b][h], K_t>) V_t          (zeros if n == 0)
 * Sequence b is cut into split_num = max(1, n // chunk) splits of whole blocks (capped at
 * max(1, max_context_len // chunk)); one kernel computes each split's (m, l, acc) for the whole
 * GQA group of a kv head, a second kernel merges them. Sequences with one split skip the merge.
 * dtype is the element type of q, out, k_pool and v_pool: PKV_F32 or PKV_BF16. Accumulation is
 * fp32; out is rounded to dtype (nearest-even). max_context_len >= every context_lens[b]
 * (a larger context is still computed correctly and flagged). split_chunk_tokens: 0 = auto,
 * else a multiple of block_size. workspace: device memory of at least
 * pkv_decode_workspace_bytes(...) bytes, 256-byte aligned; its contents on entry do not matter.
 */
pkv_status pkv_paged_decode_attention(void* out, const void* q, const void* k_pool,
                                      const void* v_pool, const int32_t* block_tables,
                                      const int32_t* context_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, int max_blocks_per_seq,
                                      int max_context_len, float scale, pkv_dtype dtype,
                                      int split_chunk_tokens, void* workspace,
                                      size_t workspace_bytes, int32_t* status, void* stream);

/*
 * INT8-KV paged decode attention ("EchoLLMServing inference framework notes", section 3:
 * per-token dequantisation fused into the attention kernel). Identical to
 * pkv_paged_decode_attention with q and out in bf16 and
 *     K_t = k_pool[blk][g][off][:] * k_scales[blk][g][off]   (int8 times fp32)
 *     V_t = v_pool[blk][g][off][:] * v_scales[blk][g][off]
 * The scales are applied to the scores and to the softmax weights, not to every element.
 */
pkv_status pkv_paged_decode_attention_int8(void* out, const void* q, const int8_t* k_pool,
                                           const int8_t* v_pool, const float* k_scales,
                                           const float* v_scales, const int32_t* block_tables,
                                           const int32_t* context_lens, int num_seqs,
                                           int num_q_heads, int num_kv_heads, int head_dim,
                                           int block_size, int num_blocks,
                                           int max_blocks_per_seq, int max_context_len,
                                           float scale, int split_chunk_tokens, void* workspace,
                                           size_t workspace_bytes, int32_t* status,
                                           void* stream);

/*
 * Paged decode attention that allocates nothing and takes no workspace argument.
 *
 * The pages this library follows have no counterpart of this entry point: it exists for callers
 * that cannot call cudaMalloc -- a plugin running inside another runtime's memory plan, where the
 * host framework owns every device allocation and offers none for scratch, or a latency-critical
 * loop where an allocation and the device-wide synchronisation it can bring are not acceptable.
 *
 * Same arguments, semantics and errors as pkv_paged_decode_attention without `workspace` and
 * `workspace_bytes`: the split-K partial states go to a fixed array of
 * PKV_STATIC_WORKSPACE_BYTES bytes inside the library (a file-scope __device__ array; every GPU
 * that loads the library holds it until the process exits). A batch whose partial states need
 * more than that (pkv_decode_workspace_bytes_dtype(..., dtype) > PKV_STATIC_WORKSPACE_BYTES, the
 * exact size at the chunk this call uses) is refused with PKV_ERR_WORKSPACE before anything is
 * enqueued; a larger split_chunk_tokens needs less.
 * The first call made while a given device is current looks up the array's device address on
 * that device (cudaGetSymbolAddress) and caches it with the id of the current context; a call in
 * another context on that device (after cudaDeviceReset, for one) looks it up again. Make the
 * first call on each device, and the first after a reset, before any stream capture. The current
 * device must be the one `stream` belongs to.
 * All calls share the one array per device and it keeps the last call's contents (nothing in it
 * needs to start at zero): calls whose work overlaps on the GPU -- on different streams, or from
 * different host threads -- race on it and must be serialised by the caller.
 */
#define PKV_STATIC_WORKSPACE_BYTES (32u << 20)

pkv_status pkv_paged_decode_attention_static_ws(void* out, const void* q, const void* k_pool,
                                                const void* v_pool, const int32_t* block_tables,
                                                const int32_t* context_lens, int num_seqs,
                                                int num_q_heads, int num_kv_heads, int head_dim,
                                                int block_size, int num_blocks,
                                                int max_blocks_per_seq, int max_context_len,
                                                float scale, pkv_dtype dtype,
                                                int split_chunk_tokens, int32_t* status,
                                                void* stream);

/*
 * Copy-on-write of forked sequences ("LLM Primer VI, Chapter 8", section 8.1: sequences share
 * blocks by reference count; the block manager reports a copy when one of them writes into a
 * shared, partly filled block). For each pair i of block_pairs ([num_pairs][2] int32, device
 * memory: source block, destination block), block destination of k_pool and v_pool -- all kv
 * heads, all 16 slots, [num_kv_heads][16][head_dim] elements of dtype -- and, for PKV_I8 pools,
 * of k_scales and v_scales ([num_kv_heads][16] fp32) becomes a bit copy of block source. Pairs
 * must name distinct destinations, none of which is a source of another pair. A pair with an id
 * outside [0, num_blocks), or source == destination, is skipped and flagged PKV_FLAG_BAD_BLOCK.
 * Enqueue it before the pkv_kv_cache_write of the step's new tokens, on the same stream.
 * Pools and scale arrays 16-byte aligned; scale pointers NULL unless dtype is PKV_I8.
 */
pkv_status pkv_kv_cache_copy_blocks(void* k_pool, void* v_pool, float* k_scales, float* v_scales,
                                    const int32_t* block_pairs, int num_pairs, int num_kv_heads,
                                    int head_dim, int block_size, int num_blocks, pkv_dtype dtype,
                                    int32_t* status, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Host block manager: the step before the decode path, producing block_tables, context_lens and
 * slot_mapping. "AMD ATOM inference engine", section 5.1 (the KV cache as fixed 16-token blocks, a
 * block table per sequence, a reference count per block) and section 5.2 (prefix caching with
 * xxhash64 chained over blocks); "LLM Primer VI, Chapter 8", section 8.1 (blocks shared by
 * reference count, which makes best-of-n sampling on one prompt nearly free).
 *
 * A pkv_block_manager is host memory owned by the caller (create / destroy); no device memory and
 * no CUDA call is involved, and it is not thread-safe. Sequences are named by caller-chosen int64
 * ids. Free blocks are handed out first-in first-out, initially 0, 1, 2, ...; freed blocks go to
 * the back of the free list, tail block first. With prefix caching on, every full block carries
 * the chained hash of its tokens; a prompt block whose hash (and tokens) match a cached block
 * shares it (ref_count + 1) instead of taking a free block, even when that block sits freed but
 * not yet reused in the free list. The cache never shares partial blocks; a fork shares every
 * block, and copy-on-write (pkv_bm_append_cow) splits a shared partial tail block when one of its
 * sequences writes into it.
 * --------------------------------------------------------------------------------------------- */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager over num_blocks blocks of block_size tokens; NULL on bad arguments / no memory. */
pkv_block_manager* pkv_bm_create(int num_blocks, int block_size, int enable_prefix_cache);
void pkv_bm_destroy(pkv_block_manager* bm);
int pkv_bm_num_free_blocks(const pkv_block_manager* bm);
int pkv_bm_ref_count(const pkv_block_manager* bm, int block_id);  /* -1 for a bad id */

/* xxhash64 (the published XXH64 algorithm) of len bytes. */
uint64_t pkv_xxh64(const void* data, size_t len, uint64_t seed);
/* Chained block hash of section 5.2: XXH64, seed 0, over prefix_hash as 8 little-endian bytes
 * (omitted when prefix_hash == -1) followed by the token ids as int64 little-endian. */
uint64_t pkv_block_hash(const int64_t* token_ids, int num_tokens, int64_t prefix_hash);

/* Prefill: enough free blocks for num_tokens (cache hits not counted)? */
int pkv_bm_can_allocate(const pkv_block_manager* bm, int num_tokens);
/* Prefill: give a new sequence blocks for its prompt, sharing cached full blocks of the same
 * chained prefix; *num_cached_tokens (optional) gets the tokens found in the cache.
 * PKV_ERR_NO_BLOCKS if pkv_bm_can_allocate is false; INVALID_ARG for a known seq_id. */
pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int64_t* token_ids,
                           int num_tokens, int* num_cached_tokens);
/* Decode: room for num_new_tokens more tokens (scheduler's can_append)? */
int pkv_bm_can_append(const pkv_block_manager* bm, int64_t seq_id, int num_new_tokens);
/* Decode (may_append): add the tokens, taking a new block at each block boundary; slot_mapping
 * (optional, [num_new_tokens]) receives each token's slot block_id * block_size + offset, ready
 * for pkv_kv_cache_write. A block that becomes full gets its chained hash. */
pkv_status pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, const int64_t* new_token_ids,
                         int num_new_tokens, int64_t* slot_mapping);
/* Decode with copy-on-write: as pkv_bm_append, for sequences that may share their tail block
 * (after pkv_bm_fork). If the tail block is partly filled and another sequence also references it,
 * the sequence first takes a free block for its own copy and drops its reference to the shared
 * one; copy_src_dst[0..1] receive (shared block, new block) and *num_copies 1 (else 0). The caller
 * copies that block on the device (pkv_kv_cache_copy_blocks) before writing the new tokens into
 * their slots. The last sequence referencing a shared block writes in place. pkv_bm_can_append
 * counts the copy's block. pkv_bm_append returns PKV_ERR_INVALID_ARG, changing nothing, where a
 * copy would be needed. */
pkv_status pkv_bm_append_cow(pkv_block_manager* bm, int64_t seq_id, const int64_t* new_token_ids,
                             int num_new_tokens, int64_t* slot_mapping, int32_t* copy_src_dst,
                             int* num_copies);
/* Parallel sampling (best-of-n): a new sequence child_id with the parent's tokens and block table;
 * every block gains a reference, none is copied. INVALID_ARG for an unknown parent or a known
 * child id. */
pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id);
/* Finish or preempt a sequence: its blocks lose a reference; unreferenced ones become free. */
pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id);
int pkv_bm_context_len(const pkv_block_manager* bm, int64_t seq_id);  /* -1 if unknown */
/* The decode inputs of a batch: block_tables [num_seqs][max_blocks_per_seq] (unused entries -1)
 * and context_lens [num_seqs] in host memory, for upload to the device. */
pkv_status pkv_bm_batch_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int num_seqs,
                               int max_blocks_per_seq, int32_t* block_tables,
                               int32_t* context_lens);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
