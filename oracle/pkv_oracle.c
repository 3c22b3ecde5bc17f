/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, obviously-correct CPU statement of the paged-KV decode path, in fp64.
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg load it.
 * It shares no code, header, table or helper with the CUDA library; the two meet only in
 * the seeded input generators (workloads/), which hold none of the method's arithmetic.
 *
 * What it follows (page title, section):
 *  [PRIMER]  "LLM Primer VI, Chapter 8 -- the next generation of KV memory management",
 *            section 8.1 "PagedAttention is virtual memory for the KV cache": the KV cache is
 *            cut into fixed-size blocks (usually 16 tokens) held in one flat physical pool; a
 *            sequence is a block table mapping logical positions to physical block ids; the
 *            attention kernel takes the block table as an extra input and gathers K and V
 *            through it instead of slicing a contiguous buffer.
 *  [ECHO2]   "EchoLLMServing inference framework notes", section 2 "Core operators",
 *            PagedAttention V2 and FlashDecoding: the context is cut into chunks, each chunk
 *            keeps an online-softmax state (m, l, acc), a second (reduce) kernel merges the
 *            partial states; the split count is max(1, context_len // optimal_chunk_size).
 *  [ECHO3]   same page, section 3, "KV Cache INT8 quantisation": per-token dequantisation
 *            with the accompanying scale, fused into the attention kernel.
 *  [ATOM]    "AMD ATOM inference engine" (itsolotime.com), introduction (the request
 *            lifecycle step "writing into the KV cache") and section 5.1 (blocks of 16
 *            tokens, one block_table per sequence).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - pool layout [num_blocks][num_kv_heads][block_size][head_dim], K and V alike;
 *  - GQA: query head h reads kv head h / (Hq / Hkv);
 *  - a slot is block_id * block_size + offset; a negative slot is a padding token and is
 *    not written;
 *  - context_len == 0 gives an all-zero output row;
 *  - INT8 K/V values are dequantised as (double)value * (double)scale, one fp32 scale per
 *    (block, kv head, token) for K and one for V.
 *
 * Parity pins live in tests/test_oracle_pins.py: closed forms (one token, identical keys,
 * two-key logistic weights, one-hot keys), invariance under block permutation and prefix
 * sharing, agreement with a library attention routine on contiguous layouts, the split /
 * merge identity and the bf16 bit patterns.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element codes (match workloads/ and tests; not shared with the CUDA library) */
#define ORC_F32 0
#define ORC_BF16 1
#define ORC_I8 2

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_BAD_BLOCK 2
#define ORC_BAD_SLOT 3
#define ORC_NO_MEMORY 4

static size_t elem_size(int dtype) {
    return dtype == ORC_F32 ? 4 : dtype == ORC_BF16 ? 2 : dtype == ORC_I8 ? 1 : 0;
}

/* bf16 is the upper half of an IEEE binary32: widen by placing it in the high 16 bits. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, size_t idx, int dtype) {
    switch (dtype) {
        case ORC_F32: return (double)((const float*)base)[idx];
        case ORC_BF16: return bf16_to_double(((const uint16_t*)base)[idx]);
        default: return (double)((const int8_t*)base)[idx];
    }
}

double orc_bf16_to_double(uint16_t b) { return bf16_to_double(b); }

/* ------------------------------------------------------------------------------------------
 * KV write [ATOM intro, PRIMER 8.1]: the new token i goes to slot s = slot_mapping[i];
 * block s / BS, row s % BS; every kv head's row is copied unchanged (a byte copy).
 * Applied in token order. For INT8 pools the token's per-head scales go with it.
 * Returns ORC_BAD_SLOT (after writing every valid token) if a slot is >= NB * BS.
 * ---------------------------------------------------------------------------------------- */
int orc_kv_cache_write(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                       const float* k_new_scales, const float* v_new_scales,
                       float* k_scales, float* v_scales,
                       const int64_t* slot_mapping, int T, int Hkv, int D, int BS, int NB,
                       int dtype) {
    size_t es = elem_size(dtype);
    if (es == 0 || T < 0 || Hkv <= 0 || D <= 0 || BS <= 0 || NB < 0) return ORC_BAD_ARG;
    size_t row = (size_t)D * es;
    int status = ORC_OK;
    for (int i = 0; i < T; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= (int64_t)NB * BS) { status = ORC_BAD_SLOT; continue; }
        int64_t blk = s / BS, off = s % BS;
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = (((size_t)blk * Hkv + h) * BS + (size_t)off);
            size_t src = (size_t)i * Hkv + h;
            memcpy((char*)k_pool + dst * row, (const char*)k_new + src * row, row);
            memcpy((char*)v_pool + dst * row, (const char*)v_new + src * row, row);
            if (dtype == ORC_I8) {
                k_scales[dst] = k_new_scales[src];
                v_scales[dst] = v_new_scales[src];
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------------------------
 * Quantising KV write [ECHO3: INT8 KV cache with a per-token scale]. Each (token, kv head) row x
 * of D values (fp32 or bf16) is stored as int8 codes with one fp32 scale, in fp32 arithmetic:
 *   amax = max_d |x_d|,  scale = amax / 127 (1 if that is 0),
 *   code_d = clamp(rint(x_d / scale), -127, 127)   (rint: round half to even)
 * The scale is symmetric per row, so the largest-magnitude element maps to +-127. Reading where
 * the page is silent: the divisor 127 and half-even rounding follow the int8 recipe of the input
 * generator; codes never use -128. Then the row goes to its slot as in orc_kv_cache_write.
 * ---------------------------------------------------------------------------------------- */
static float load_f32(const void* base, size_t idx, int dtype) {
    if (dtype == ORC_F32) return ((const float*)base)[idx];
    uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

void orc_quantize_row_int8(const void* src, size_t off, int D, int dtype, int8_t* codes,
                           float* scale_out) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(load_f32(src, off + d, dtype));
        if (a > amax) amax = a;
    }
    float scale = amax / 127.0f;
    if (scale == 0.0f) scale = 1.0f;
    for (int d = 0; d < D; ++d) {
        float q = rintf(load_f32(src, off + d, dtype) / scale);
        if (q > 127.0f) q = 127.0f;
        if (q < -127.0f) q = -127.0f;
        codes[d] = (int8_t)q;
    }
    *scale_out = scale;
}

int orc_kv_cache_write_quant(const void* k_new, const void* v_new, int8_t* k_pool, int8_t* v_pool,
                             float* k_scales, float* v_scales, const int64_t* slot_mapping, int T,
                             int Hkv, int D, int BS, int NB, int src_dtype) {
    if ((src_dtype != ORC_F32 && src_dtype != ORC_BF16) || T < 0 || Hkv <= 0 || D <= 0 ||
        BS <= 0 || NB < 0)
        return ORC_BAD_ARG;
    int status = ORC_OK;
    for (int i = 0; i < T; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= (int64_t)NB * BS) { status = ORC_BAD_SLOT; continue; }
        int64_t blk = s / BS, off = s % BS;
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = ((size_t)blk * Hkv + h) * BS + (size_t)off;
            size_t src = ((size_t)i * Hkv + h) * (size_t)D;
            orc_quantize_row_int8(k_new, src, D, src_dtype, k_pool + dst * D, &k_scales[dst]);
            orc_quantize_row_int8(v_new, src, D, src_dtype, v_pool + dst * D, &v_scales[dst]);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------------------------
 * Split rule [ECHO2, FlashDecoding answer]: split_num = max(1, n // chunk), capped at
 * max_splits (the grid's split extent, max(1, max_context_len // chunk)). Each split covers
 * a whole number of blocks: per = ceil(n / split_num) rounded up to BS; split j is
 * [j*per, min(n, (j+1)*per)); trailing splits that would be empty are dropped, so the count
 * returned is ceil(n / per). n <= 0 gives one (empty) split.
 * ---------------------------------------------------------------------------------------- */
int orc_split_count(int n, int chunk, int max_splits, int BS, int* per_out) {
    if (n <= 0 || chunk <= 0) { if (per_out) *per_out = 0; return 1; }
    int s0 = n / chunk;
    if (s0 < 1) s0 = 1;
    if (max_splits >= 1 && s0 > max_splits) s0 = max_splits;
    int per = (n + s0 - 1) / s0;
    per = ((per + BS - 1) / BS) * BS;
    if (per_out) *per_out = per;
    return (n + per - 1) / per;
}

/* Everything one (sequence, query head) pair needs. */
typedef struct {
    const void* q; int q_dtype;
    const void* k_pool; const void* v_pool; int kv_dtype;
    const float* k_scales; const float* v_scales;
    const int32_t* block_tables; const int32_t* context_lens;
    int B, Hq, Hkv, D, BS, NB, MBPS;
    double scale;
} orc_problem;

/* Gather the K or V row of logical token t of sequence b for kv head kvh into `row`
 * (widened to double, INT8 dequantised) [PRIMER 8.1, ECHO3]. */
static int gather_row(const orc_problem* P, int b, int kvh, int t, int which_v, double* row) {
    int32_t blk = P->block_tables[(size_t)b * P->MBPS + t / P->BS];
    if (blk < 0 || blk >= P->NB) return ORC_BAD_BLOCK;
    int off = t % P->BS;
    size_t r = ((size_t)blk * P->Hkv + kvh) * P->BS + off;
    const void* pool = which_v ? P->v_pool : P->k_pool;
    double sc = 1.0;
    if (P->kv_dtype == ORC_I8) sc = (double)(which_v ? P->v_scales : P->k_scales)[r];
    for (int d = 0; d < P->D; ++d) {
        double x = load_elem(pool, r * P->D + d, P->kv_dtype);
        row[d] = P->kv_dtype == ORC_I8 ? x * sc : x;
    }
    return ORC_OK;
}

/* s_t = scale * sum_d q[d] * k_t[d] for t in [lo, hi); qrow is element index of q's first dim. */
static int scores(const orc_problem* P, size_t qrow, int b, int h, int lo, int hi, double* s,
                  double* row) {
    int kvh = h / (P->Hq / P->Hkv);
    for (int t = lo; t < hi; ++t) {
        int rc = gather_row(P, b, kvh, t, 0, row);
        if (rc) return rc;
        double dot = 0.0;
        for (int d = 0; d < P->D; ++d) dot += load_elem(P->q, qrow + d, P->q_dtype) * row[d];
        s[t - lo] = P->scale * dot;
    }
    return ORC_OK;
}

/* Softmax attention of query vector q[qrow ..] (head h, K/V of sequence b's table) over tokens
 * [lo, hi) in the partial form of [ECHO2]: m = max_t s_t, l = sum_t exp(s_t - m),
 * acc = sum_t exp(s_t - m) v_t. Empty range: m = -inf, l = 0, acc = 0. */
static int partial_q(const orc_problem* P, size_t qrow, int b, int h, int lo, int hi,
                     double* m_out, double* l_out, double* acc, double* s, double* row) {
    for (int d = 0; d < P->D; ++d) acc[d] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (hi <= lo) return ORC_OK;
    int rc = scores(P, qrow, b, h, lo, hi, s, row);
    if (rc) return rc;
    double m = s[0];
    for (int t = 1; t < hi - lo; ++t) if (s[t] > m) m = s[t];
    int kvh = h / (P->Hq / P->Hkv);
    double l = 0.0;
    for (int t = lo; t < hi; ++t) {
        double p = exp(s[t - lo] - m);
        l += p;
        rc = gather_row(P, b, kvh, t, 1, row);
        if (rc) return rc;
        for (int d = 0; d < P->D; ++d) acc[d] += p * row[d];
    }
    *m_out = m;
    *l_out = l;
    return ORC_OK;
}

/* The decode case: query row (b, h) of q [B][Hq][D]. */
static int partial(const orc_problem* P, int b, int h, int lo, int hi, double* m_out,
                   double* l_out, double* acc, double* s, double* row) {
    return partial_q(P, ((size_t)b * P->Hq + h) * P->D, b, h, lo, hi, m_out, l_out, acc, s, row);
}

typedef struct {
    const orc_problem* P;
    double* out;
    int first, stride;
    int status;
} orc_job;

/* out[b][h][:] = sum_t softmax(s)_t v_t over the whole context: the plain definition. */
static void* attention_worker(void* arg) {
    orc_job* J = (orc_job*)arg;
    const orc_problem* P = J->P;
    int maxn = 0;
    for (int b = 0; b < P->B; ++b) if (P->context_lens[b] > maxn) maxn = P->context_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)(maxn > 0 ? maxn : 1));
    double* row = (double*)malloc(sizeof(double) * (size_t)P->D);
    double* acc = (double*)malloc(sizeof(double) * (size_t)P->D);
    if (!s || !row || !acc) { J->status = ORC_NO_MEMORY; free(s); free(row); free(acc); return NULL; }
    for (int pair = J->first; pair < P->B * P->Hq; pair += J->stride) {
        int b = pair / P->Hq, h = pair % P->Hq;
        double* o = J->out + (size_t)pair * P->D;
        int n = P->context_lens[b];
        if (n <= 0) { for (int d = 0; d < P->D; ++d) o[d] = 0.0; continue; }
        double m, l;
        int rc = partial(P, b, h, 0, n, &m, &l, acc, s, row);
        if (rc) { J->status = rc; break; }
        for (int d = 0; d < P->D; ++d) o[d] = acc[d] / l;
    }
    free(s); free(row); free(acc);
    return NULL;
}

static int check_problem(const orc_problem* P) {
    if (P->B < 0 || P->Hq <= 0 || P->Hkv <= 0 || P->Hq % P->Hkv || P->D <= 0 || P->BS <= 0 ||
        P->MBPS < 0 || elem_size(P->q_dtype) == 0 || elem_size(P->kv_dtype) == 0 ||
        P->q_dtype == ORC_I8)
        return ORC_BAD_ARG;
    if (P->kv_dtype == ORC_I8 && (!P->k_scales || !P->v_scales)) return ORC_BAD_ARG;
    for (int b = 0; b < P->B; ++b)
        if (P->context_lens[b] > P->MBPS * P->BS) return ORC_BAD_ARG;
    return ORC_OK;
}

/* Paged decode attention [PRIMER 8.1, ECHO2, ECHO3] for every (b, h), in fp64, into
 * out[B][Hq][D] (double). num_threads host threads split the (b, h) pairs round-robin. */
int orc_paged_decode_attention(double* out, const void* q, int q_dtype, const void* k_pool,
                               const void* v_pool, int kv_dtype, const float* k_scales,
                               const float* v_scales, const int32_t* block_tables,
                               const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                               int BS, int NB, int MBPS, double scale, int num_threads) {
    orc_problem P = {q, q_dtype, k_pool, v_pool, kv_dtype, k_scales, v_scales,
                     block_tables, context_lens, B, Hq, Hkv, D, BS, NB, MBPS, scale};
    int rc = check_problem(&P);
    if (rc) return rc;
    if (num_threads < 1) num_threads = 1;
    orc_job* jobs = (orc_job*)calloc((size_t)num_threads, sizeof(orc_job));
    pthread_t* th = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return ORC_NO_MEMORY; }
    for (int i = 0; i < num_threads; ++i) {
        jobs[i] = (orc_job){&P, out, i, num_threads, ORC_OK};
        if (num_threads == 1) attention_worker(&jobs[i]);
        else pthread_create(&th[i], NULL, attention_worker, &jobs[i]);
    }
    if (num_threads > 1)
        for (int i = 0; i < num_threads; ++i) pthread_join(th[i], NULL);
    for (int i = 0; i < num_threads; ++i) if (jobs[i].status) rc = jobs[i].status;
    free(jobs); free(th);
    return rc;
}

/* Multi-token decode ("AMD ATOM inference engine", section 4, decode scheduling: with MTP
 * speculative decoding a decode step reserves num_new_tokens = mtp_k + 1 cache slots per
 * sequence; the target model verifies all of them in one pass). Sequence b's L new tokens are
 * its last L context positions; query token l (0 <= l < L) attends causally to positions
 * t <= n_b - L + l, i.e. to the first n_b - (L - 1 - l) tokens. q and out are [B][L][Hq][D].
 * n_b < L is a bad argument. Computed by the plain definition per (b, l, h). */
int orc_paged_decode_attention_multi(double* out, const void* q, int q_dtype, const void* k_pool,
                                     const void* v_pool, int kv_dtype, const float* k_scales,
                                     const float* v_scales, const int32_t* block_tables,
                                     const int32_t* context_lens, int B, int L, int Hq, int Hkv,
                                     int D, int BS, int NB, int MBPS, double scale) {
    if (L < 1) return ORC_BAD_ARG;
    orc_problem P = {q, q_dtype, k_pool, v_pool, kv_dtype, k_scales, v_scales,
                     block_tables, context_lens, B, Hq, Hkv, D, BS, NB, MBPS, scale};
    int rc = check_problem(&P);
    if (rc) return rc;
    int maxn = 1;
    for (int b = 0; b < B; ++b) {
        if (context_lens[b] < L) return ORC_BAD_ARG;
        if (context_lens[b] > maxn) maxn = context_lens[b];
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)maxn);
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    if (!s || !row || !acc) { free(s); free(row); free(acc); return ORC_NO_MEMORY; }
    /* query token l of sequence b: q row (b * L + l), sequence b's block table */
    for (int b = 0; b < B && rc == ORC_OK; ++b) {
        for (int l = 0; l < L && rc == ORC_OK; ++l) {
            int n_l = context_lens[b] - (L - 1 - l);
            for (int h = 0; h < Hq; ++h) {
                size_t r = (size_t)(b * L + l) * Hq + h;
                double m, lsum;
                rc = partial_q(&P, r * D, b, h, 0, n_l, &m, &lsum, acc, s, row);
                if (rc) break;
                double* o = out + r * D;
                for (int d = 0; d < D; ++d) o[d] = acc[d] / lsum;
            }
        }
    }
    free(s); free(row); free(acc);
    return rc;
}

/* Paged prefill (chunked prefill; "EchoLLMServing inference framework notes", section 2
 * FlashAttention for prefill, section 3 chunked prefill and mixed batches): sequence b has
 * L_b = query_start[b + 1] - query_start[b] query tokens, the last L_b of its context n_b, at
 * rows query_start[b] .. of q / out [total][Hq][D]. Row i of sequence b attends causally to the
 * first n_b - (L_b - 1 - i) tokens -- the multi-token rule with a per-sequence L. */
int orc_paged_prefill_attention(double* out, const void* q, int q_dtype, const void* k_pool,
                                const void* v_pool, int kv_dtype, const float* k_scales,
                                const float* v_scales, const int32_t* block_tables,
                                const int32_t* context_lens, const int32_t* query_start, int B,
                                int Hq, int Hkv, int D, int BS, int NB, int MBPS, double scale) {
    orc_problem P = {q, q_dtype, k_pool, v_pool, kv_dtype, k_scales, v_scales,
                     block_tables, context_lens, B, Hq, Hkv, D, BS, NB, MBPS, scale};
    int rc = check_problem(&P);
    if (rc) return rc;
    int maxn = 1;
    for (int b = 0; b < B; ++b) {
        int L = query_start[b + 1] - query_start[b];
        if (L < 0 || context_lens[b] < L) return ORC_BAD_ARG;
        if (context_lens[b] > maxn) maxn = context_lens[b];
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)maxn);
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    if (!s || !row || !acc) { free(s); free(row); free(acc); return ORC_NO_MEMORY; }
    for (int b = 0; b < B && rc == ORC_OK; ++b) {
        int L = query_start[b + 1] - query_start[b];
        for (int i = 0; i < L && rc == ORC_OK; ++i) {
            int n_i = context_lens[b] - (L - 1 - i);
            for (int h = 0; h < Hq; ++h) {
                size_t r = (size_t)(query_start[b] + i) * Hq + h;
                double m, lsum;
                rc = partial_q(&P, r * D, b, h, 0, n_i, &m, &lsum, acc, s, row);
                if (rc) break;
                double* o = out + r * D;
                for (int d = 0; d < D; ++d) o[d] = acc[d] / lsum;
            }
        }
    }
    free(s); free(row); free(acc);
    return rc;
}

/* Split mode [ECHO2]: per (b, h, split j) the partial state (m_j, l_j, acc_j) of the tokens in
 * split j (orc_split_count's ranges). m/l are [B][Hq][max_splits], acc [B][Hq][max_splits][D];
 * unused split slots are left as m = -inf, l = 0, acc = 0. n_splits[b] receives the count. */
int orc_paged_decode_partials(double* m, double* l, double* acc, int32_t* n_splits,
                              const void* q, int q_dtype, const void* k_pool,
                              const void* v_pool, int kv_dtype, const float* k_scales,
                              const float* v_scales, const int32_t* block_tables,
                              const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                              int BS, int NB, int MBPS, double scale, int chunk,
                              int max_splits) {
    orc_problem P = {q, q_dtype, k_pool, v_pool, kv_dtype, k_scales, v_scales,
                     block_tables, context_lens, B, Hq, Hkv, D, BS, NB, MBPS, scale};
    int rc = check_problem(&P);
    if (rc) return rc;
    if (chunk <= 0 || max_splits < 1) return ORC_BAD_ARG;
    int maxn = 1;
    for (int b = 0; b < B; ++b) if (context_lens[b] > maxn) maxn = context_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)maxn);
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
    if (!s || !row) { free(s); free(row); return ORC_NO_MEMORY; }
    for (int b = 0; b < B && rc == ORC_OK; ++b) {
        int n = context_lens[b], per;
        int ns = orc_split_count(n, chunk, max_splits, BS, &per);
        n_splits[b] = ns;
        for (int h = 0; h < Hq && rc == ORC_OK; ++h) {
            for (int j = 0; j < max_splits; ++j) {
                size_t idx = ((size_t)b * Hq + h) * max_splits + j;
                int lo = j * per, hi = lo + per < n ? lo + per : n;
                if (j >= ns) hi = lo;  /* unused slot: the empty state */
                rc = partial(&P, b, h, lo, hi, &m[idx], &l[idx], acc + idx * D, s, row);
                if (rc) break;
            }
        }
    }
    free(s); free(row);
    return rc;
}

/* Reduce kernel of [ECHO2]: M = max_j m_j, L = sum_j l_j e^(m_j - M),
 * out = sum_j acc_j e^(m_j - M) / L over the first n_splits[b] splits. L == 0 gives zeros. */
int orc_merge_partials(double* out, const double* m, const double* l, const double* acc,
                       const int32_t* n_splits, int B, int Hq, int D, int max_splits) {
    for (int b = 0; b < B; ++b) {
        int ns = n_splits[b];
        if (ns < 1 || ns > max_splits) return ORC_BAD_ARG;
        for (int h = 0; h < Hq; ++h) {
            size_t base = ((size_t)b * Hq + h) * max_splits;
            double M = -INFINITY;
            for (int j = 0; j < ns; ++j) if (m[base + j] > M) M = m[base + j];
            double L = 0.0;
            double* o = out + ((size_t)b * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (M == -INFINITY) continue;
            for (int j = 0; j < ns; ++j) {
                double w = exp(m[base + j] - M);
                L += l[base + j] * w;
                for (int d = 0; d < D; ++d) o[d] += acc[(base + j) * D + d] * w;
            }
            for (int d = 0; d < D; ++d) o[d] /= L;
        }
    }
    return ORC_OK;
}
