// decode_mma.cuh -- split-K paged decode attention, kernel 1 of 2, tensor-core path (head_dim 128,
// bf16 or INT8 K/V, 8 MMA columns per CTA).
//
// Same unit and outputs as the CUDA-core kernel (decode_split.cuh): one CTA per (sequence b,
// kv head, split) for the GQA group of that kv head ("EchoLLMServing inference framework
// notes", section 2: one program per split emitting (m, l, acc); "LLM Primer VI, Chapter 8",
// section 8.1: K/V gathered through the block table). What changes is how a 16-token block is
// consumed: the per-block work is a dense [16 tokens x 128] x [128 x 8 heads] product and its
// transpose, done with warp-level mma.sync m16n8k16 so that one instruction covers what took
// 64 FMAs plus conversions, and the kernel stays far from the issue limit at HBM speed.
//
// The 8 MMA columns are query heads of one (sequence, query token) row, or, in packed multi-token
// decode, the (token, head) pairs of one sequence's kv head, each column masked at its own causal
// limit. With kv_start > 0 (shared-prefix calls) the CTA covers only tokens [kv_start, n) and
// always emits a partial state: the prefix is merged in from the tcgen05 prefix kernel.
//
// Warp roles: every warp is its own producer and consumer. Warp w takes blocks w, w+NC, ... of
// the split (NC warps per CTA) and owns the stages w, w+NC, ... of a STAGES-deep shared-memory
// ring (STAGES = NC * stages per warp). Its lane 0 issues, per block, one TMA tensor copy of each
// of the K and V tiles with 128-byte swizzle (bank-conflict-free ldmatrix), plus 1-D bulk copies of
// the INT8 scale rows, completing on the stage's mbarrier; as soon as the warp has consumed a
// block it refills that stage with its block STAGES further on. No warp waits for another until
// the end, where the NC online-softmax states are merged in shared memory. Block ids come from
// the table 32 at a time (one per lane, validated) a window ahead of use.
//
// Per block and consumer warp (tokens on the MMA M dimension, heads on N):
//   S^T[16 x 8]   = K[16 x 128] . Q^T[128 x 8]      8 MMAs (k = 16 dims each)
//   online softmax on S^T (scores in base-2 units; the running max is only raised when a block
//   exceeds it by more than 2^8, so rescaling the accumulators is rare -- exact in real arithmetic
//   because l and acc always share the reference max)
//   P^T fragments = movmatrix.trans of the score fragments (no shared-memory round trip)
//   O^T[128 x 8] += V^T[128 x 16] . P^T[16 x 8]       8 MMAs (k = 16 tokens)
// bf16: K fragments by ldmatrix, V^T fragments by ldmatrix.trans, P rounded to bf16.
// INT8 ("EchoLLMServing notes", section 3): K fragments by ldmatrix and V^T fragments by
// ldmatrix.trans of the int8 tiles read as 16-bit pairs; each register of 4 int8 becomes two
// fp16x2 operands holding 1152 + x exactly (byte-permute conversion of Kim et al. 2022), and the
// constant 1152 is taken out once per score (1152 * sum q') and once per output (1152 * sum of
// the fp16 weights), not per element. q enters fp16 exactly, scaled by one power of two per CTA;
// the per-token K scale times scale*log2(e) and that power's inverse multiplies the score, and the
// V scale the softmax weight. Dims are consumed in a fixed
// permuted order that q's fragments and the output mapping follow, which leaves the dot
// products unchanged.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pkv_device.cuh"

namespace pkv {

constexpr int kMmaD = 128;          // head_dim of this path
constexpr int kMmaHeads = 8;        // MMA N: query heads per CTA
// warps per CTA and stages per warp, per element type (build-time tunables)
#ifndef PKV_MMA_WARPS_BF16
#define PKV_MMA_WARPS_BF16 4
#endif
#ifndef PKV_MMA_SPW_BF16
#define PKV_MMA_SPW_BF16 2
#endif
#ifndef PKV_MMA_WARPS_I8
#define PKV_MMA_WARPS_I8 4
#endif
#ifndef PKV_MMA_SPW_I8
#define PKV_MMA_SPW_I8 2
#endif
#ifndef PKV_MMA_PROXY_FENCE
#define PKV_MMA_PROXY_FENCE 1
#endif
#ifndef PKV_MMA_MINB_I8  // minimum resident CTAs per SM the INT8 kernel is compiled for (0: no bound)
#define PKV_MMA_MINB_I8 0
#endif
#ifndef PKV_MMA_UNROLL_I8  // INT8 blocks per trip of the block loop
#define PKV_MMA_UNROLL_I8 1
#endif
constexpr int kUnrollI8 = PKV_MMA_UNROLL_I8;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only when the max grows by > 2^8

template <bool kI8, int kNT = 1>
struct MmaGeom {
    static constexpr int NC = kI8 ? PKV_MMA_WARPS_I8 : PKV_MMA_WARPS_BF16;  // warps per CTA
    static constexpr int SPW = kI8 ? PKV_MMA_SPW_I8 : PKV_MMA_SPW_BF16;     // stages per warp
    static constexpr int THREADS = 32 * NC;
    static constexpr int TILE = kBlockSize * kMmaD * (kI8 ? 1 : 2);  // one K (or V) tile
    static constexpr int BOX = kBlockSize * 128;  // [16 rows][128 B]: a bf16 tile's 64-dim half, an INT8 tile
    static constexpr int STAGE = 2 * TILE;                           // K then V
    // Stage s is only ever used by warp s % NC, so each warp waits on a stage's phases strictly
    // in order and a parity wait can never match a phase two behind.
    static constexpr int STAGES = NC * SPW;
    static constexpr int RING = STAGES * STAGE;
    static constexpr int SCALES = kI8 ? STAGES * 2 * kBlockSize * 4 : 0;
    static constexpr int NCOL = kMmaHeads * kNT;                     // MMA columns per CTA
    static constexpr int MERGE = NC * NCOL * (kMmaD + 2) * 4;
    static constexpr int MAIN = RING > MERGE ? RING : MERGE;
    // + 1024 for aligning the ring to the 128-byte-swizzle atom
    static constexpr int SMEM = 1024 + MAIN + SCALES + STAGES * 8;
    static_assert(RING % 1024 == 0 && STAGE % 1024 == 0, "swizzled boxes need 1024-byte alignment");
    static_assert(RING >= 4 * (kLptMaxRows + 1), "longest-first scratch fits in the ring");

};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <bool kI8>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (kI8) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// int8 -> biased fp16, two values per instruction (the byte-permute / magic-number conversion
// of Kim et al. 2022): placing the byte x + 128 (x XOR 0x80) in the low byte of the fp16 1024
// gives exactly 1152 + x. For a word of four int8 [b0 b1 b2 b3], lo -> fp16x2(1152+b0, 1152+b2)
// and hi -> fp16x2(1152+b1, 1152+b3); the sign flip and the exponent byte are one XOR with
// 0x64806480 after masking. The 1152 offset is removed once per score / per output (below),
// never per element.
constexpr float kI8Bias = 1152.0f;
constexpr int kBiasFoldBlocks = 8;  // INT8: blocks between removals of the V offset from O
__device__ __forceinline__ uint32_t i8_lo_h2(uint32_t w) { return (w & 0x00FF00FFu) ^ 0x64806480u; }
__device__ __forceinline__ uint32_t i8_hi_h2(uint32_t w) { return ((w >> 8) & 0x00FF00FFu) ^ 0x64806480u; }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// kPacked: the columns are (query token, head) pairs (packed multi-token decode); a template
// parameter so that the one-token path keeps its exact instruction stream.
// kNT: 8-column MMA n-tiles per CTA. With 2, a warp reads and widens each K/V tile once for 16
// columns (G = 16, or multi-token rows of G = 8).
template <bool kI8, bool kPacked, int kNT>
// bf16: three CTAs per SM (shared memory bounds it there anyway), so up to 170 registers a thread;
// INT8: the compiler's own choice (96, five CTAs per SM), or the tunable minimum
#if PKV_MMA_MINB_I8 > 0
#define PKV_MMA_BOUNDS __launch_bounds__(MmaGeom<kI8, kNT>::THREADS, kI8 ? PKV_MMA_MINB_I8 : 3)
#else
#define PKV_MMA_BOUNDS __launch_bounds__(MmaGeom<kI8, kNT>::THREADS, kI8 ? 0 : 3)
#endif
__global__ void PKV_MMA_BOUNDS mma_split_kernel(const SplitParams p,
                                                               const __grid_constant__ CUtensorMap tmk,
                                                               const __grid_constant__ CUtensorMap tmv) {
    using G = MmaGeom<kI8, kNT>;
    constexpr int STAGES = G::STAGES, STAGE = G::STAGE, TILE = G::TILE, NCOL = G::NCOL;
    constexpr float kNegInf = -INFINITY;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned
    float* scl = reinterpret_cast<float*>(smem + G::MAIN);              // [STAGES][K16 | V16]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::MAIN + G::SCALES);
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.head_chunks;
    const int hc = blockIdx.y - kvh * p.head_chunks;
    // MMA columns: query heads of one (sequence, query token) row, or -- packed multi-token
    // decode -- the (query token, head) pairs of one sequence's kv head, so that the L tokens
    // being verified read each K/V tile once. The splits follow the longest context (the last
    // token's); each column masks the keys past its own context n - (L - 1 - l).
    // Inputs (new K/V rows, tables) may come from the previous kernel: wait for it. In a
    // shared-prefix call the previous kernel is the prefix kernel, which releases this one only
    // after its own wait (so the inputs are complete) and writes nothing this kernel reads; this
    // kernel then runs alongside it and waits for it only at exit, which keeps the merge kernel
    // (waiting for this grid) behind both.
    if (p.kv_start == 0) grid_dependency_wait();

    // Grid row z of the launch is row z of q / out, or with p.lpt (one row per sequence, at most
    // kLptMaxRows of them) the sequence of rank z when the sequences are ordered by the length of
    // their splits, longest first (ties by index). CTAs start in grid order, so the longest
    // (sequence, kv head, split) units start first and the last wave holds the shortest ones.
    int zrow = (int)blockIdx.z;
    if (p.lpt) {
        // scratch at the start of the ring, which no copy has reached yet
        int* lpt_key = reinterpret_cast<int*>(smem);
        int& lpt_row = lpt_key[kLptMaxRows];
        for (int i = tid; i < p.B; i += G::THREADS) {
            bool bd;
            const int ni = query_context_len(p.context_lens[i], p.L, p.L - 1, p.MBPS * kBlockSize, &bd);
            int pi;
            split_count(ni > p.kv_start ? ni - p.kv_start : 0, p.chunk, p.max_splits, &pi);
            lpt_key[i] = pi;
        }
        __syncthreads();
        for (int i = tid; i < p.B; i += G::THREADS) {
            const int ki = lpt_key[i];
            int rank = 0;
            for (int j = 0; j < p.B; ++j) {
                const int kj = lpt_key[j];
                rank += (kj > ki) | ((kj == ki) & (j < i));
            }
            if (rank == zrow) lpt_row = i;
        }
        __syncthreads();
        zrow = lpt_row;
    }
    const int b = kPacked ? zrow : zrow / p.L;
    const int lq = kPacked ? p.L - 1 : zrow - b * p.L;  // the token the splits follow
    const int c0 = hc * NCOL;                                    // first column of this CTA
    const int ncols = kPacked ? p.L * p.G : p.G;
    const int nh = ncols - c0 < NCOL ? ncols - c0 : NCOL;        // columns in use
    auto col_zb = [&](int j) { return kPacked ? b * p.L + (c0 + j) / p.G : zrow; };
    auto col_head = [&](int j) { return kvh * p.G + (kPacked ? (c0 + j) % p.G : c0 + j); };

    const int stored = p.context_lens[b];
    bool bad;
    const int n = query_context_len(stored, p.L, lq, p.MBPS * kBlockSize, &bad);
    const bool reporter = tid == 0 && split == 0 && blockIdx.y == 0 && (kPacked || lq == 0);
    if (bad && reporter) flag(p.status, PKV_FLAG_BAD_CONTEXT);
    else if (stored > p.max_context_len && reporter) flag(p.status, PKV_FLAG_LONG_CONTEXT);
    // tokens [kv_start, n) are this kernel's (kv_start > 0: a shared prefix is handled elsewhere)
    if (p.kv_start > 0 && split == 0 && blockIdx.y == 0 && lq == 0) {
        bool badp = n < p.kv_start;
        const int nb = p.kv_start / kBlockSize;
        for (int j = tid; j < nb && !badp; j += G::THREADS)
            badp = p.block_tables[(size_t)b * p.MBPS + j] != p.block_tables[j];
        if (badp) flag(p.status, PKV_FLAG_BAD_PREFIX);
    }
    int per;
    const int ns = split_count(n > p.kv_start ? n - p.kv_start : 0, p.chunk, p.max_splits, &per);
    if (split >= ns) {
        if (p.kv_start > 0) grid_dependency_wait();
        return;
    }
    const int t0 = p.kv_start + split * per;
    const int t1 = n < t0 + per ? n : t0 + per;
    const int nblk = t1 > t0 ? (t1 - t0 + kBlockSize - 1) / kBlockSize : 0;
    const int blk0 = t0 / kBlockSize;

    const uint32_t ring = smem_addr(smem);
    const uint32_t full0 = smem_addr(full);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(full0 + 8 * s, 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    // per-lane MMA coordinates
    const int r = lane >> 2;  // fragment row group: token (QK) / head (B operand)
    const int c = lane & 3;   // thread in group: head pair 2c, 2c+1 of the C fragments
    // context of columns 2c and 2c + 1 (packed: token (c0 + col) / G sees n - (L - 1 - l) keys)
    auto col_ctx = [&](int j) { return kPacked ? n - (p.L - 1 - (c0 + j) / p.G) : n; };
    int ncol_lim[kNT][2];
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        ncol_lim[t][0] = col_ctx(8 * t + 2 * c);
        ncol_lim[t][1] = col_ctx(8 * t + 2 * c + 1);
    }

    // per n-tile t, for this lane's columns 8t + 2c and 8t + 2c + 1: the reference max m (base-2
    // units; set from the column's first block with a valid key and raised only when a block
    // exceeds it by more than 2^8), the sum l of 2^(s - m), and O^T. A column that never sees a
    // valid key keeps l = 0 and reports its max as -inf.
    float m[kNT][2], l[kNT][2];
    float o[kNT][8][4];
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        m[t][0] = m[t][1] = 0.f;
        l[t][0] = l[t][1] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[t][i][0] = o[t][i][1] = o[t][i][2] = o[t][i][3] = 0.f;
    }

    // ---- this warp's blocks: k-th is split block j = warp + k * NC, in stage warp + (k % SPW) * NC ----
    constexpr int NC = G::NC, SPW = G::SPW;
    const int nmine = nblk > warp ? (nblk - warp + NC - 1) / NC : 0;
    const int32_t* bt_row = p.block_tables + (size_t)b * p.MBPS + blk0;
    auto load_window = [&](int w) {  // lane i: id of this warp's block 32 * w + i (-1: none / bad)
        const int k = 32 * w + lane;
        int id = -1;
        if (k < nmine) {
            id = bt_row[warp + k * NC];
            if (id < 0 || id >= p.NB) {
                flag(p.status, PKV_FLAG_BAD_BLOCK);
                id = -1;
            }
        }
        return id;
    };
    int win = 0;
    int ids_a = load_window(0), ids_b = nmine > 32 ? load_window(1) : -1;
    auto id_of = [&](int k) {  // warp-uniform; k within windows win, win + 1
        const int va = __shfl_sync(0xffffffffu, ids_a, k & 31);
        const int vb = __shfl_sync(0xffffffffu, ids_b, k & 31);
        return (k >> 5) == win ? va : vb;
    };
    auto issue = [&](int k, int bid) {  // lane 0: start this warp's k-th block into its stage
        const int st = warp + (k % SPW) * NC;
        const uint32_t bar = full0 + 8 * st;
        const uint32_t dst = ring + st * STAGE;
        if (bid >= 0) {
            const int row = (bid * p.Hkv + kvh) * kBlockSize;
            mbar_arrive_expect_tx(bar, STAGE + (kI8 ? 2 * kBlockSize * 4 : 0));
            if constexpr (kI8) {  // one [16 rows][128 B] box per tile
                tma_load_2d(dst, &tmk, 0, row, bar);
                tma_load_2d(dst + TILE, &tmv, 0, row, bar);
            } else {  // one box per tile: both 64-dim halves, [half][16 rows][128 B]
                tma_load_3d(dst, &tmk, 0, row, 0, bar);
                tma_load_3d(dst + TILE, &tmv, 0, row, 0, bar);
            }
            if constexpr (kI8) {
                const size_t srow = (size_t)bid * p.Hkv + kvh;
                const uint32_t sd = smem_addr(scl + st * 2 * kBlockSize);
                bulk_g2s(sd, p.k_scales + srow * kBlockSize, kBlockSize * 4, bar);
                bulk_g2s(sd + kBlockSize * 4, p.v_scales + srow * kBlockSize, kBlockSize * 4, bar);
            }
        } else {
            mbar_arrive(bar);  // nothing to load: complete the phase so the wait stays in step
        }
    };
#pragma unroll 1
    for (int k = 0; k < SPW && k < nmine; ++k) {
        const int bid = id_of(k);
        if (lane == 0) issue(k, bid);
    }

    // INT8: q enters the fp16 MMAs as q' = q * 2^e, e one power of two for the CTA's columns, so
    // that the largest |q'| lies in [2^14, 2^15): exact, as a bf16 value scaled by a power of two
    // fits fp16's 11-bit significand, and never past fp16's range whatever q's magnitude. The
    // scores' multiplier (the per-token K scale) then carries scale * log2(e) * 2^-e in fp32.
    float score_mult = p.scale_log2;  // bf16: scale * log2(e); INT8: that times 2^-e
    {
        // q as the B operand of S^T = K Q^T: b0b1 = (dims k0 + 2c, +1; head r), b2b3 = (+8, +9)
        uint32_t qb[kNT][8][2];
        float qsum[kNT];  // INT8: sum of this lane's fp16 q' values of column 8t + r (as the MMA sees them)
        float q_up = 1.f;  // INT8: 2^e
        if constexpr (kI8) {
            // every warp loads all of the CTA's columns, so a warp-wide max covers them all
            float amax = 0.f;
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
                if (8 * t + r < nh) {
                    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                                ((size_t)col_zb(8 * t + r) * p.Hq + col_head(8 * t + r)) * kMmaD;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint2 raw4 = *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c);
                        float f0, f1, f2, f3;
                        bf16x2_to_f32(raw4.x, f0, f1);
                        bf16x2_to_f32(raw4.y, f2, f3);
                        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))));
                    }
                }
            }
#pragma unroll
            for (int off = 1; off <= 16; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            int e = 0;
            if (amax > 0.f) {  // floor(log2(amax)) from the exponent field (-127 for a subnormal amax)
                e = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xffu) - 127);
                e = e < -126 ? -126 : (e > 126 ? 126 : e);  // 2^e and 2^-e stay normal floats
            }
            q_up = __uint_as_float((uint32_t)(127 + e) << 23);
            score_mult = p.scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23);
        }
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            qsum[t] = 0.f;
            const bool hv = 8 * t + r < nh;
            const int col = hv ? 8 * t + r : 0;
            const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                        ((size_t)col_zb(col) * p.Hq + col_head(col)) * kMmaD;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                if constexpr (kI8) {
                    // permuted dims: k-pos 2c,2c+1 <- dims 16ks+4c+0, +2; k-pos 2c+8,2c+9 <- +1, +3
                    // (the order in which i8_lo_h2 / i8_hi_h2 deliver a row's bytes)
                    const uint2 raw4 = *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c);
                    float f0, f1, f2, f3;
                    bf16x2_to_f32(raw4.x, f0, f1);
                    bf16x2_to_f32(raw4.y, f2, f3);
                    qb[t][ks][0] = hv ? pack_h2(f0 * q_up, f2 * q_up) : 0u;
                    qb[t][ks][1] = hv ? pack_h2(f1 * q_up, f3 * q_up) : 0u;
                    const float2 u0 = __half22float2(*reinterpret_cast<const __half2*>(&qb[t][ks][0]));
                    const float2 u1 = __half22float2(*reinterpret_cast<const __half2*>(&qb[t][ks][1]));
                    qsum[t] += (u0.x + u0.y) + (u1.x + u1.y);
                } else {
                    qb[t][ks][0] = hv ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c) : 0u;
                    qb[t][ks][1] = hv ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c + 8) : 0u;
                }
            }
        }
        // INT8: 1152 * sum_d q'_d of columns 2c and 2c+1 is what the biased K adds to each score
        float kcorr[kNT][2], psum[kNT][2];
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            kcorr[t][0] = kcorr[t][1] = 0.f;
            psum[t][0] = psum[t][1] = 0.f;
            if constexpr (kI8) {
                float qs = qsum[t];
                qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                qs += __shfl_xor_sync(0xffffffffu, qs, 2);  // lanes 4r..4r+3: column r's full sum
                kcorr[t][0] = kI8Bias * __shfl_sync(0xffffffffu, qs, 4 * (2 * c));
                kcorr[t][1] = kI8Bias * __shfl_sync(0xffffffffu, qs, 4 * (2 * c + 1));
            }
        }
        bool fresh = true;  // warp-uniform: no block consumed yet, so m is not set
        // bf16: two blocks per trip, so stage indices and parities are compile-time (measured: the
        // Llama-3-8B GQA batch 100.1 -> 98.4 us); INT8 stays at one, where the extra registers
        // would cost a CTA per SM
#pragma unroll(kI8 ? kUnrollI8 : 2)
        for (int k = 0; k < nmine; ++k) {
            const int j = warp + k * NC;
            const int st = warp + (k % SPW) * NC;
            if ((k & 31) == 0 && k > 0) {  // consumption enters the next id window
                ++win;
                ids_a = ids_b;
                ids_b = nmine > 32 * (win + 1) ? load_window(win + 1) : -1;
            }
            const int bid = id_of(k);
            if (!mbar_wait_bounded(full0 + 8 * st, (k / SPW) & 1)) {
                if (lane == 0) {
                    flag(p.status, PKV_FLAG_TIMEOUT);
                    atomicExch(&abort_flag, 1);
                    // let this warp's copies already issued land before giving up
                    for (int q = k; q < k + SPW && q < nmine; ++q)
                        mbar_wait_bounded(full0 + 8 * (warp + (q % SPW) * NC), (q / SPW) & 1);
                }
                break;
            }
            if (bid >= 0) {
                const uint32_t kt = ring + st * STAGE;
                const uint32_t vt = kt + TILE;
                // ---- S^T = K . Q^T (each K fragment serves every n-tile) ----
                // INT8: the accumulators start at -1152 * sum q', which removes the bias of the
                // widened K from every score
                float s[kNT][4];
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
                    s[t][0] = s[t][2] = -kcorr[t][0];
                    s[t][1] = s[t][3] = -kcorr[t][1];
                }
                const int lr = lane & 7, mi = lane >> 3;
                if constexpr (kI8) {
#pragma unroll
                    for (int kp = 0; kp < 4; ++kp) {  // chunks 2kp, 2kp+1 (16 dims each)
                        const int y = (mi & 1) * 8 + lr;
                        const int ch = 2 * kp + (mi >> 1);
                        uint32_t rr[4];
                        ldsm_x4(kt + y * 128 + ((ch ^ (y & 7)) << 4), rr);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t lo = rr[2 * h];      // token r: bytes 4c..4c+3
                            const uint32_t hi = rr[2 * h + 1];  // token r + 8
                            uint32_t a[4];
                            a[0] = i8_lo_h2(lo);
                            a[1] = i8_lo_h2(hi);
                            a[2] = i8_hi_h2(lo);
                            a[3] = i8_hi_h2(hi);
#pragma unroll
                            for (int t = 0; t < kNT; ++t)
                                mma16816<true>(s[t], a, qb[t][2 * kp + h][0], qb[t][2 * kp + h][1]);
                        }
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int y = (mi & 1) * 8 + lr;
                        const int ch = (ks & 3) * 2 + (mi >> 1);
                        uint32_t a[4];
                        ldsm_x4(kt + (ks >> 2) * G::BOX + y * 128 + ((ch ^ (y & 7)) << 4), a);
#pragma unroll
                        for (int t = 0; t < kNT; ++t) mma16816<false>(s[t], a, qb[t][ks][0], qb[t][ks][1]);
                    }
                }
                // s[t][0] = (tok r, col 8t+2c), [1] = (tok r, 8t+2c+1), [2] = (tok r+8, 8t+2c), [3] = (tok r+8, 8t+2c+1)
                const int nvalid = t1 - (t0 + j * kBlockSize);  // >= 1; >= 16 for full blocks
                // score multipliers: the K scale (INT8) or scale * log2(e) (bf16) per token row
                float vs0 = 1.f, vs1 = 1.f, ks0 = score_mult, ks1 = score_mult;
                if constexpr (kI8) {
                    // A block that ends the context: the V scales of its slots past the context
                    // may be any bits (NaN included), and those tokens' weights of 0 times NaN
                    // would poison O, so they are zeroed here (their K scores are masked to -inf
                    // below). The fence orders these writes before the stage's next bulk copy.
                    if (nvalid < kBlockSize) {
                        if (lane < kBlockSize - nvalid) {
                            scl[st * 2 * kBlockSize + kBlockSize + nvalid + lane] = 0.f;
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        }
                        __syncwarp();
                    }
                    const float* sc = scl + st * 2 * kBlockSize;
                    ks0 = sc[r] * score_mult;
                    ks1 = sc[r + 8] * score_mult;
                    vs0 = sc[kBlockSize + r];
                    vs1 = sc[kBlockSize + r + 8];
                }
                // d = score - m (base 2), one FFMA per score; keys past a column's limit get -inf
                float dm[kNT][2];
                bool any_up = false;
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
                    s[t][0] = fmaf(s[t][0], ks0, -m[t][0]);
                    s[t][1] = fmaf(s[t][1], ks0, -m[t][1]);
                    s[t][2] = fmaf(s[t][2], ks1, -m[t][0]);
                    s[t][3] = fmaf(s[t][3], ks1, -m[t][1]);
                    // keys of this block visible to this lane's columns 8t + 2c and 8t + 2c + 1
                    const int lim0 = kPacked ? min(nvalid, ncol_lim[t][0] - (t0 + j * kBlockSize)) : nvalid;
                    const int lim1 = kPacked ? min(nvalid, ncol_lim[t][1] - (t0 + j * kBlockSize)) : nvalid;
                    if (kPacked ? (lim0 < kBlockSize || lim1 < kBlockSize) : nvalid < kBlockSize) {
                        s[t][0] = r < lim0 ? s[t][0] : kNegInf;
                        s[t][1] = r < lim1 ? s[t][1] : kNegInf;
                        s[t][2] = r + 8 < lim0 ? s[t][2] : kNegInf;
                        s[t][3] = r + 8 < lim1 ? s[t][3] : kNegInf;
                    }
                    dm[t][0] = fmaxf(s[t][0], s[t][2]);
                    dm[t][1] = fmaxf(s[t][1], s[t][3]);
                    any_up = any_up || dm[t][0] > kRescaleThreshold || dm[t][1] > kRescaleThreshold;
                }
                // Raising m needs the column's maximum over the 8 lanes that hold its tokens; that
                // reduction runs only on the warp's first block (m is set from it) and when some
                // lane's keys exceed m by more than 2^8, which is rare.
                if (fresh || __any_sync(0xffffffffu, any_up)) {
#pragma unroll
                    for (int t = 0; t < kNT; ++t) {
#pragma unroll
                        for (int off = 4; off <= 16; off <<= 1) {
                            dm[t][0] = fmaxf(dm[t][0], __shfl_xor_sync(0xffffffffu, dm[t][0], off));
                            dm[t][1] = fmaxf(dm[t][1], __shfl_xor_sync(0xffffffffu, dm[t][1], off));
                        }
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const bool up = fresh ? dm[t][e] != kNegInf : dm[t][e] > kRescaleThreshold;
                            const float delta = up ? dm[t][e] : 0.f;
                            // on the first block l and O are still 0: nothing to rescale (and
                            // 2^-delta may overflow for very negative scores)
                            const float a = up && !fresh ? ex2(-delta) : 1.f;
                            m[t][e] += delta;
                            s[t][e] -= delta;
                            s[t][e + 2] -= delta;
                            l[t][e] *= a;
                            psum[t][e] *= a;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                o[t][i][e] *= a;
                                o[t][i][e + 2] *= a;
                            }
                        }
                    }
                    fresh = false;
                }
                // ---- O^T += V^T . P^T ----
                uint32_t pb[kNT][2];
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
                    const float p0 = ex2(s[t][0]), p1 = ex2(s[t][1]);
                    const float p2 = ex2(s[t][2]), p3 = ex2(s[t][3]);
                    l[t][0] += p0 + p2;
                    l[t][1] += p1 + p3;
                    if constexpr (kI8) {
                        const uint32_t h01 = pack_h2(p0 * vs0, p1 * vs0);
                        const uint32_t h23 = pack_h2(p2 * vs1, p3 * vs1);
                        // the weights exactly as the MMA uses them: their sum times 1152 is what
                        // the biased V adds to each output
                        const float2 w01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
                        const float2 w23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
                        psum[t][0] += w01.x + w23.x;
                        psum[t][1] += w01.y + w23.y;
                        pb[t][0] = movm_t(h01);
                        pb[t][1] = movm_t(h23);
                    } else {
                        pb[t][0] = movm_t(pack_bf16(p0, p1));
                        pb[t][1] = movm_t(pack_bf16(p2, p3));
                    }
                }
                const bool partial = nvalid < kBlockSize;
                if constexpr (kI8) {
                    // V^T fragments by ldmatrix.trans of the int8 tile read as 16-bit pairs: for
                    // 16-byte chunk j the lane gets [V(2c,d) V(2c,d+1) V(2c+1,d) V(2c+1,d+1)] with
                    // d = 16j + 2r, i.e. A rows r <- dim d and r + 8 <- dim d + 1 of m-tile j.
                    // Tokens past the context need no masking: their weight is 0 and every biased
                    // int8 value is finite.
                    const int lr2 = lane & 7, mi2 = lane >> 3;
#pragma unroll
                    for (int jp = 0; jp < 4; ++jp) {  // chunks 2jp, 2jp+1
                        const int y = (mi2 & 1) * 8 + lr2;
                        const int ch = 2 * jp + (mi2 >> 1);
                        uint32_t rr[4];
                        ldsm_x4_t(vt + y * 128 + ((ch ^ (y & 7)) << 4), rr);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t t0w = rr[2 * h];      // tokens 2c, 2c+1
                            const uint32_t t8w = rr[2 * h + 1];  // tokens 2c+8, 2c+9
                            uint32_t a[4];
                            a[0] = i8_lo_h2(t0w);
                            a[1] = i8_hi_h2(t0w);
                            a[2] = i8_lo_h2(t8w);
                            a[3] = i8_hi_h2(t8w);
#pragma unroll
                            for (int t = 0; t < kNT; ++t) mma16816<true>(o[t][2 * jp + h], a, pb[t][0], pb[t][1]);
                        }
                    }
                } else {
                    const int lr2 = lane & 7, mi2 = lane >> 3;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int y = (mi2 >> 1) * 8 + lr2;
                        const int ch = (i & 3) * 2 + (mi2 & 1);
                        uint32_t a[4];
                        ldsm_x4_t(vt + (i >> 2) * G::BOX + y * 128 + ((ch ^ (y & 7)) << 4), a);
                        if (partial) {  // zero the token columns past the context
                            const bool k0 = 2 * c < nvalid, k1 = 2 * c + 1 < nvalid;
                            const bool k8 = 2 * c + 8 < nvalid, k9 = 2 * c + 9 < nvalid;
                            const uint32_t mlo = (k0 ? 0xffffu : 0u) | (k1 ? 0xffff0000u : 0u);
                            const uint32_t mhi = (k8 ? 0xffffu : 0u) | (k9 ? 0xffff0000u : 0u);
                            a[0] &= mlo; a[1] &= mlo; a[2] &= mhi; a[3] &= mhi;
                        }
#pragma unroll
                        for (int t = 0; t < kNT; ++t) mma16816<false>(o[t][i], a, pb[t][0], pb[t][1]);
                    }
                }
            }
            if constexpr (kI8) {
                // Every kBiasFoldBlocks blocks, take the 1152 offset of the biased V out of O (the
                // column's weight sum over the warp's 8 token rows), so O never holds more than
                // that many blocks' worth of offset: the subtraction then cancels no more digits
                // of O than a short split would, whatever the split's length.
                if ((k % kBiasFoldBlocks) == kBiasFoldBlocks - 1) {
#pragma unroll
                    for (int t = 0; t < kNT; ++t) {
                        float w0 = psum[t][0], w1 = psum[t][1];
#pragma unroll
                        for (int off = 4; off <= 16; off <<= 1) {
                            w0 += __shfl_xor_sync(0xffffffffu, w0, off);
                            w1 += __shfl_xor_sync(0xffffffffu, w1, off);
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            o[t][i][0] = fmaf(-kI8Bias, w0, o[t][i][0]); o[t][i][2] = fmaf(-kI8Bias, w0, o[t][i][2]);
                            o[t][i][1] = fmaf(-kI8Bias, w1, o[t][i][1]); o[t][i][3] = fmaf(-kI8Bias, w1, o[t][i][3]);
                        }
                        psum[t][0] = psum[t][1] = 0.f;
                    }
                }
            }
            __syncwarp();  // every lane is done reading the stage
            if (k + SPW < nmine) {
                const int nb = id_of(k + SPW);
                if (lane == 0) {
#if PKV_MMA_PROXY_FENCE
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // reads before the async write
#endif
                    issue(k + SPW, nb);
                }
            }
        }
        // finish l (and the INT8 weight sums) over the 8 token rows (lanes with the same c)
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                l[t][0] += __shfl_xor_sync(0xffffffffu, l[t][0], off);
                l[t][1] += __shfl_xor_sync(0xffffffffu, l[t][1], off);
                if constexpr (kI8) {
                    psum[t][0] += __shfl_xor_sync(0xffffffffu, psum[t][0], off);
                    psum[t][1] += __shfl_xor_sync(0xffffffffu, psum[t][1], off);
                }
            }
            if constexpr (kI8) {  // remove the 1152 offset of the biased V from every output
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[t][i][0] -= kI8Bias * psum[t][0]; o[t][i][2] -= kI8Bias * psum[t][0];
                    o[t][i][1] -= kI8Bias * psum[t][1]; o[t][i][3] -= kI8Bias * psum[t][1];
                }
            }
            // a column with no valid key in this warp's blocks has l = 0 (any other has l >= 1:
            // the key that set m contributed 2^0)
            m[t][0] = l[t][0] > 0.f ? m[t][0] : kNegInf;
            m[t][1] = l[t][1] > 0.f ? m[t][1] : kNegInf;
        }
    }

    __syncthreads();  // every warp is done with the ring (its copies all consumed or drained)
    if (abort_flag) {
        if (p.kv_start > 0) grid_dependency_wait();
        return;
    }
    grid_dependents_launch();  // the merge kernel may start launching
    // ---- merge the consumer warps' states (ring memory reused) ----
    float* sm_m = reinterpret_cast<float*>(smem);               // [NC][NCOL]
    float* sm_l = sm_m + G::NC * NCOL;                          // [NC][NCOL]
    float* sm_o = sm_l + G::NC * NCOL;                          // [NC][NCOL][128]
    {
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            const int cl = 8 * t + 2 * c;
            if (r == 0) {
                sm_m[warp * NCOL + cl] = m[t][0];
                sm_m[warp * NCOL + cl + 1] = m[t][1];
                sm_l[warp * NCOL + cl] = l[t][0];
                sm_l[warp * NCOL + cl + 1] = l[t][1];
            }
            float* ow = sm_o + warp * NCOL * kMmaD;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d0 = kI8 ? 16 * i + 2 * r : 16 * i + r;
                const int d1 = kI8 ? d0 + 1 : d0 + 8;
                ow[cl * kMmaD + d0] = o[t][i][0];
                ow[(cl + 1) * kMmaD + d0] = o[t][i][1];
                ow[cl * kMmaD + d1] = o[t][i][2];
                ow[(cl + 1) * kMmaD + d1] = o[t][i][3];
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < NCOL * kMmaD; e += G::THREADS) {
        const int hh = e / kMmaD, d = e % kMmaD;
        if (hh >= nh) continue;
        const int zb = col_zb(hh);
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < G::NC; ++w) M = fmaxf(M, sm_m[w * NCOL + hh]);
        float L = 0.f, A = 0.f;
        if (M != kNegInf) {
#pragma unroll
            for (int w = 0; w < G::NC; ++w) {
                const float wt = ex2(sm_m[w * NCOL + hh] - M);
                L = fmaf(wt, sm_l[w * NCOL + hh], L);
                A = fmaf(wt, sm_o[(w * NCOL + hh) * kMmaD + d], A);
            }
        }
        const size_t qh = (size_t)zb * p.Hq + col_head(hh);
        if (ns == 1 && !p.always_partial) {
            store_out<__nv_bfloat16>(static_cast<__nv_bfloat16*>(p.out) + qh * kMmaD + d, L > 0.f ? A / L : 0.f);
        } else {
            const size_t u = qh * p.ws_stride + split;
            p.ws_acc[u * kMmaD + d] = A;
            if (d == 0) {
                p.ws_ml[2 * u] = M;
                p.ws_ml[2 * u + 1] = L;
            }
        }
    }
    if (p.kv_start > 0) grid_dependency_wait();
}

}  // namespace pkv
