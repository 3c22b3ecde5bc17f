// prefill_tc.cu -- paged (chunked, variable-length) prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM), head_dim 128, bf16.
//
// "EchoLLMServing inference framework notes", section 2: FlashAttention for prefill tiles the
// queries by BLOCK_M and keeps the working set on chip; section 3: chunked prefill and mixed
// batches. "LLM Primer VI, Chapter 8", section 8.1: K and V are gathered through the block table.
// Sequence b's L_b query tokens are the last L_b of its context (written to the cache first);
// query row i attends causally to the first n_b - (L_b - 1 - i) tokens.
//
// The same kernel (kPrefix) also runs the shared-prefix part of a cascade decode: there a CTA's 128
// rows are (sequence, query head) pairs of one kv head, all attending to one key range of the
// prefix every sequence shares, and it writes partial states (m, l, acc) for the merge kernel.
//
// One CTA computes 128 query rows of one query head against 128-key tiles. Both products read
// their A operand from tensor memory: a tcgen05.mma with M = N = 128, K = 16 takes 64 cycles and
// reads its B operand from shared memory at 64 B a cycle; an A operand from shared memory would
// double that, to the whole shared-memory bandwidth, and the TMA copies into the rings would then
// slow the products (measured: Q in shared memory, 4 % slower). TMEM columns:
//   O   0-127     fp32 accumulator, row r in lane r
//   Q   128-191   the CTA's 128 query rows, two bf16 dims per column (written once)
//   P   192-255   bf16 weights of a key tile, two keys per column
//   S   256-383 (buffer 0), 384-511 (buffer 1): S = Q . K^T of a key tile, fp32
// Warp roles (384 threads):
//   warps 0-7  softmax. Warp w owns TMEM lanes 32 (w % 4) .. + 31 (query rows). bf16 cache: the
//              two warps of a lane quadrant take alternate key tiles (warps 0-3 the even ones from
//              S buffer 0, warps 4-7 the odd ones from S buffer 1), one thread per row over all
//              128 keys; a row's reference maximum after each tile is handed to the other warp
//              through shared memory (m_ready). The two warps run out of phase, one loading S or
//              waiting while the other computes (measured: 1300 TFLOP/s against 1210 for a split
//              of every tile between them). INT8 cache (one S buffer): warps 0-3 take keys 0-63 of
//              every tile, warps 4-7 keys 64-127; per tile the two warps of a quadrant vote whether
//              any row may raise its reference maximum, and only then swap maxima.
//   warp 8     lane 0 issues the S products (and their commits); the warp owns the TMEM allocation
//   warp 11    lane 0 issues the PV products. Two issuers, because a thread that has just issued a
//              batch of products takes several hundred cycles to notice its next barrier, and
//              the S and PV streams depend on each other only through the softmax.
//   warps 9-10 producers: block ids from the table, one 4-D TMA copy (4 KB, 128-byte swizzle) per
//              pool block of a key tile, K by warp 9 into one ring, V by warp 10 into another. A
//              K slot is free once S of its tile is done, so K runs well ahead of V. (Measured on
//              GB300: an SM takes in ~53 GB/s of 2 KB TMA boxes but ~82 GB/s of 4 KB ones, so
//              one box per block rather than one per 64-dim half.)
// Per key tile t the S issuer computes S(t) = Q . K(t)^T into S buffer t % 2 as soon as K(t) has
// landed and the softmax has read S(t-2) from that buffer (s_free), so it runs up to two tiles
// ahead of the softmax; the PV issuer computes O += P(t) . V(t) once P(t) is written (p_full).
// The softmax writes P(t) once PV(t-1), the product that last read P, is done (pv_done); PV(t-1)
// was issued when the softmax finished tile t-1, so it has usually completed by then. S has one
// barrier per buffer, so no barrier completes a phase its waiter has not yet seen (a parity wait
// would miss it). The running max is raised lazily (only when a tile exceeds it by more than
// 2^8), so O is rarely rescaled; at the end each row is divided by its sum.
#include <cuda.h>

#include <cuda_fp16.h>

#include "pkv_device.cuh"
#include "tc_common.cuh"

namespace pkv {

namespace {

constexpr int kPfQ = 128;                      // query rows per CTA (MMA M)
constexpr int kPfK = 128;                      // keys per tile (MMA N of S, K of PV)
// A K (or V) tile is the 8 pool blocks of 128 keys, one 4 KB TMA box each, block jj at 4 KB jj as
// [row group (keys 0-7, 8-15)][64-dim half][8 keys][128 B]: in every half, key k's 128-byte row is
// at (k / 8) * 2 KB + (k % 8) * 128 (+ 1 KB for dims 64-127), a uniform stride for both products.
constexpr int kPfBlockBytes = kBlockSize * 256;  // one block's keys, both halves
constexpr int kPfStage = 8 * kPfBlockBytes;     // one K (or V) tile
// Softmax threads per query row (a build-time tunable): each takes 128 / kPfSplit keys of every
// tile and 128 / kPfSplit dims of the row's output. The kPfSplit warps sharing a TMEM lane quadrant
// (w, w + 4, ...) form one barrier group. Measured on GB300 (the 4 x 4096-token prefill): 2 threads
// per row 1138 TFLOP/s, 4 threads per row (640-thread CTAs) 1112.
#ifndef PKV_PF_SPLIT
#define PKV_PF_SPLIT 2
#endif
constexpr int kPfSplit = PKV_PF_SPLIT;
static_assert(kPfSplit == 2 || kPfSplit == 4, "threads per row");
constexpr int kPfKeysPer = kPfK / kPfSplit;         // keys of a tile per thread
constexpr int kPfDimsPer = 128 / kPfSplit;          // output dims per thread
constexpr int kPfSoftWarps = 4 * kPfSplit;
constexpr int kPfSoftThreads = 32 * kPfSoftWarps;
constexpr int kPfGroup = 32 * kPfSplit;             // threads of one barrier group
constexpr int kPfThreads = kPfSoftThreads + 128;
// INT8 cache: the producers copy each block's int8 K (or V) rows (2 KB) into the second half of the
// tile's slot and its 16 scales into a row of the scale area, completing on staged[ring slot]; four
// converter warps (two per ring) widen them in place into fp16 rows of the layout above and then
// complete full[ring slot] for the MMA issuers, as the tensor copies do for a bf16 cache.
constexpr int kPfConvWarp0 = kPfSoftWarps + 4;       // warps 12-13: K ring, 14-15: V ring
constexpr int kPfConvThreads = 64;                   // per ring
constexpr int kPfI8Half = kPfStage / 2;              // int8 rows of a tile start here in the slot
constexpr int kPfThreadsI8 = kPfThreads + 32 * 4;

// Ring depths, buffering and shared-memory layout of the bf16 (kI8 false) and INT8 kernels.
//  - bf16: two S buffers, so the S products run up to two tiles ahead of the softmax, and one P
//    buffer (TMEM has room for one more 128-column buffer, not for both). K 3 slots, V 2: measured
//    on GB300 (the 4 x 4096-token prefill) 1210-1220 TFLOP/s, against 1162 with V 3 slots and
//    1137 with one S and two P buffers (with the alternate-tile softmax: 1315-1320 against 1143;
//    with one S buffer, S(t + 1) starts only after S(t) is read and then queues behind PV(t)).
//  - INT8: a PV waits for its V conversion, so the softmax keeps two P buffers (it need not wait
//    for PV(t-1) before writing P(t)) and S one buffer (two S and one P measured the same); the
//    alternate-tile softmax needs ~160 registers, above the 128 of a 512-thread CTA.
#ifndef PKV_PF_STAGES_K
#define PKV_PF_STAGES_K 3
#endif
#ifndef PKV_PF_STAGES_V
#define PKV_PF_STAGES_V 2
#endif
template <bool kI8>
struct PfGeom {
    static constexpr int SK = kI8 ? 3 : PKV_PF_STAGES_K;  // K ring slots
    static constexpr int SV = kI8 ? 3 : PKV_PF_STAGES_V;  // V ring slots
    static constexpr int R = SK + SV;
    static constexpr int SBufs = kI8 ? 1 : 2;             // S buffers (128 TMEM columns each)
    static constexpr int PBufs = kI8 ? 2 : 1;             // P buffers (64 columns each)
    // bf16: the two softmax warps of a TMEM lane quadrant take alternate key tiles, one thread per
    // row over all 128 keys (needs the two S buffers: warp parity e reads S buffer e)
    static constexpr bool Alt = !kI8 && kPfSplit == 2;
    static constexpr int OffV = SK * kPfStage;
    static constexpr int OffX = R * kPfStage;             // row maxima [2][kPfSplit][128], sums [kPfSplit][128]
    static constexpr int OffBar = OffX + 3 * kPfSplit * kPfQ * 4;
    // barriers: full[ring slots], empty[ring slots] (K slots, then V slots), s_full[2], s_free[2],
    // p_full[2], pv_done[2], o_done, drain[2], (Alt) m_ready[4 quadrants][2 parities]; then the
    // TMEM slot
    static constexpr int NumBars = 2 * R + 11 + (Alt ? 8 : 0);
    static constexpr int OffStaged = OffBar + NumBars * 8 + 16;              // INT8: after the TMEM slot
    static constexpr int OffScl = (OffStaged + R * 8 + 15) / 16 * 16;        // INT8: [ring slot][8 blocks][16] fp32
    static constexpr int Smem = kI8 ? 1024 + OffScl + R * 8 * kBlockSize * 4 : 1024 + OffBar + NumBars * 8 + 16;
    static constexpr int Threads = kI8 ? kPfThreadsI8 : kPfThreads;
    // TMEM columns: O 0-127, Q 128-191, then the P buffers (64 each), then the S buffers (128 each)
    static constexpr uint32_t PCol = 192, SCol = PCol + 64 * PBufs;
    static_assert(SK >= 2 && SV >= 2, "a slot loads while the other is read");
    static_assert(Smem <= 227 * 1024, "shared memory");
    static_assert(OffScl % 16 == 0, "scale rows are bulk-copy targets");
    static_assert(SCol + 128 * SBufs <= 512, "TMEM columns");
};
constexpr int kPfOffK = 0;
constexpr int kPfMmaWarp = kPfSoftWarps, kPfLoadWarpK = kPfSoftWarps + 1, kPfLoadWarpV = kPfSoftWarps + 2,
              kPfMmaWarpPV = kPfSoftWarps + 3;
constexpr uint32_t kPfTmemCols = 512;
// named barriers: 1-4 the softmax warps of a TMEM lane quadrant, 5-6 the INT8 converters of a
// ring, 7 Q written (the softmax warps and the S issuer's warp)
constexpr int kPfQBar = 7;
constexpr uint32_t kOCol = 0, kQCol = 128;
constexpr float kPfRescale = 8.0f;             // log2 units

// What one launch computes, filled by launch_prefill (kPrefix false) or launch_prefix (true).
struct PfWork {
    const void* q;
    const int32_t* block_tables;
    int32_t* status;
    int Hq, Hkv, G, NB, MBPS;
    float scale_log2;
    // prefill: rows are query tokens of sequence blockIdx.z, one query head (blockIdx.y) per CTA
    void* out;
    const int32_t* context_lens;
    const int32_t* query_start;
    // shared prefix: rows are the (sequence, head-in-group) pairs of kv head blockIdx.y; keys are
    // split blockIdx.z of the prefix (block_tables row 0); output is a partial state per row
    float* ws_acc;
    float* ws_ml;
    int B, S, slot0, prefix_tokens, split_tokens;
    // INT8 cache: the pools as [NB][Hkv][16][128] int8 and their scales [NB][Hkv][16]
    const int8_t* k_i8;
    const int8_t* v_i8;
    const float* k_scales;
    const float* v_scales;
};

// INT8 cache: the products run on fp16 operands. Four int8 values (one 32-bit word, bytes b0..b3)
// become two fp16 pairs exactly by the byte-permute / magic-number conversion (Kim et al. 2022):
// the byte x + 128 (x XOR 0x80) in the low byte of the fp16 1024 is exactly 1152 + x, so
// lo = (1152 + b0, 1152 + b2) is one LOP3 and hi = (1152 + b1, 1152 + b3) a shift and a LOP3. A
// row's dims thus come in the order 4j, 4j + 2, 4j + 1, 4j + 3 within every group of four; Q is
// written in the same order (so S is unchanged) and O's columns are put back in order when stored.
constexpr float kPfI8Bias = 1152.0f;
__device__ __forceinline__ uint32_t pf_i8_lo(uint32_t w) { return (w & 0x00FF00FFu) ^ 0x64806480u; }
__device__ __forceinline__ uint32_t pf_i8_hi(uint32_t w) { return ((w >> 8) & 0x00FF00FFu) ^ 0x64806480u; }
// the biased pair minus 1152 in each half: the codes themselves, exact in fp16
__device__ __forceinline__ uint32_t pf_unbias(uint32_t h) {
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2half2(__float2half_rn(kPfI8Bias)));
    return *reinterpret_cast<const uint32_t*>(&r);
}
// O columns 4j .. 4j + 3 hold dims 4j, 4j + 2, 4j + 1, 4j + 3: back in order
__device__ __forceinline__ void pf_unpermute(float (&o)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float t = o[4 * j + 1];
        o[4 * j + 1] = o[4 * j + 2];
        o[4 * j + 2] = t;
    }
}
__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <bool kPrefix, bool kI8>
__global__ void __launch_bounds__(PfGeom<kI8>::Threads, 1) prefill_kernel(const PfWork p,
                                                                const __grid_constant__ CUtensorMap tmk,
                                                                const __grid_constant__ CUtensorMap tmv) {
    grid_dependency_wait();
    // shared prefix: the suffix kernel after this one reads nothing this one writes, so it may
    // start now and run on the SMs this grid leaves free (it waits for this grid before it exits)
    if constexpr (kPrefix) grid_dependents_launch();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int qt, h, kvh, b, L, q0, first_visible, n_tile_max, split;
    const int32_t* bt_row;
    if constexpr (!kPrefix) {
        // heaviest query tiles (most keys under the causal mask) first
        qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
        kvh = h / p.G;
        split = 0;
        q0 = p.query_start[b];
        L = p.query_start[b + 1] - q0;
        if (qt * kPfQ >= L) return;
        const int n = p.context_lens[b];
        if (n < L || n > p.MBPS * kBlockSize) {
            if (tid == 0 && qt == 0 && h == 0) flag(p.status, PKV_FLAG_BAD_CONTEXT);
            return;
        }
        first_visible = n - L + 1;                          // keys visible to query row 0
        const int rows = min(kPfQ, L - qt * kPfQ);
        n_tile_max = first_visible + qt * kPfQ + rows - 1;  // keys visible to the last row
        bt_row = p.block_tables + (size_t)b * p.MBPS;
    } else {
        qt = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
        h = 0, b = 0, q0 = 0, first_visible = 0;
        L = p.B * p.G;                                      // rows of this kv head
        const int key0 = split * p.split_tokens;            // keys [key0, key0 + n_tile_max)
        n_tile_max = min(p.split_tokens, p.prefix_tokens - key0);
        bt_row = p.block_tables + key0 / kBlockSize;
    }
    const int ntiles = (n_tile_max + kPfK - 1) / kPfK;
    // Block ids come in windows of 32 (4 key tiles), lane j holding block 32 w + j (-1: not needed
    // or invalid), the next window loaded while the current one is used.
    auto load_window = [&](int w, bool report) {
        const int j = 32 * w + lane_of();
        int id = -1;
        if (j * kBlockSize < n_tile_max) {
            const int v = bt_row[j];
            if (v >= 0 && v < p.NB) id = v;
            else if (report) flag(p.status, PKV_FLAG_BAD_BLOCK);
        }
        return id;
    };
    auto has_window = [&](int w) { return 32 * w * kBlockSize < n_tile_max; };

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_addr(smem);
    float* xmax = reinterpret_cast<float*>(smem + PfGeom<kI8>::OffX);  // [2 buffers][kPfSplit parts][128 rows]
    float* xsum = xmax + 2 * kPfSplit * kPfQ;                // [kPfSplit parts][128 rows]
    using Gm = PfGeom<kI8>;
    constexpr bool kAlt = Gm::Alt;
    const uint32_t bar0 = sbase + Gm::OffBar;
    // ring g (0: K, 1: V) has nst(g) slots; tile t uses slot t % nst(g), ring slot ridx(g, s)
    auto nst = [](int g) { return g ? Gm::SV : Gm::SK; };
    auto ridx = [](int g, int s) { return g ? Gm::SK + s : s; };
    auto full = [&](int g, int s) { return bar0 + 8 * ridx(g, s); };
    auto empty = [&](int g, int s) { return bar0 + 8 * (Gm::R + ridx(g, s)); };
    auto slot = [&](int g, int t) { return sbase + (g ? Gm::OffV : kPfOffK) + (t % nst(g)) * kPfStage; };
    const uint32_t bar1 = bar0 + 8 * (2 * Gm::R);
    auto s_full = [&](int u) { return bar1 + 8 * u; };
    auto s_free = [&](int u) { return bar1 + 8 * (2 + u); };
    auto p_full = [&](int u) { return bar1 + 8 * (4 + u); };
    auto pv_done = [&](int u) { return bar1 + 8 * (6 + u); };
    const uint32_t o_done = bar1 + 8 * 8;
    auto drain = [&](int x) { return bar1 + 8 * (9 + x); };
    // alternate-tile softmax: the reference max after a tile of lane quadrant q4 by warp parity e
    // is published
    auto m_ready = [&](int q4, int e) { return bar1 + 8 * (11 + 2 * q4 + e); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Gm::OffBar + Gm::NumBars * 8);
    // INT8: the int8 rows of ring g's slot s have landed (the producer's copies)
    auto staged = [&](int g, int s) { return sbase + Gm::OffStaged + 8 * ridx(g, s); };
    auto scl = [&](int g, int s) { return sbase + Gm::OffScl + ridx(g, s) * 8 * kBlockSize * 4; };
    __shared__ int abort_flag;
    __shared__ unsigned q_amax_bits;  // INT8: the CTA's largest |q| (a non-negative float's bits)

    // softmax thread (hf, r): row r, keys kPfKeysPer hf .. of each tile, output dims kPfDimsPer hf ..
    const int hf = (warp >> 2) & (kPfSplit - 1);
    const int r = tid & 127;
    const int i = qt * kPfQ + r;
    const bool row_valid = i < L;
    // the (token, head) row of q / out: prefill query token q0 + i of head h; shared prefix: the
    // (sequence i / G, head kvh * G + i % G) pair
    const size_t qrow = !kPrefix ? (size_t)(q0 + (row_valid ? i : 0)) * p.Hq + h
                                 : (row_valid ? (size_t)(i / p.G) * p.Hq + kvh * p.G + i % p.G : 0);
    const uint32_t tl = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lane quadrant
    // Q row r, dims kPfDimsPer hf .. (zeros past the rows): loaded before the set-up below so that
    // its latency overlaps it
    uint32_t qw[kPfDimsPer / 2];
    if (warp < kPfSoftWarps) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                          qrow * 128 + kPfDimsPer * hf);
#pragma unroll
        for (int c = 0; c < kPfDimsPer / 8; ++c) {
            const uint4 v = row_valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
            qw[4 * c] = v.x; qw[4 * c + 1] = v.y; qw[4 * c + 2] = v.z; qw[4 * c + 3] = v.w;
        }
    }

    // the producers' first two windows of block ids, read before the set-up too (the first copies
    // wait for them)
    int ids_first = -1, ids_second = -1;
    if (warp == kPfLoadWarpK || warp == kPfLoadWarpV) {
        ids_first = load_window(0, warp == kPfLoadWarpK);
        ids_second = has_window(1) ? load_window(1, warp == kPfLoadWarpK) : -1;
    }

    if (tid == 0) {
        for (int g = 0; g < 2; ++g)
            for (int s = 0; s < nst(g); ++s) {
                mbar_init(full(g, s), kI8 ? kPfConvThreads : 1);
                // INT8 K slot: its scale row is read by the softmax warps after S is done
                mbar_init(empty(g, s), kI8 && g == 0 ? 1 + kPfSoftWarps : 1);
                if constexpr (kI8) mbar_init(staged(g, s), 1);
            }
        // alternate tiles: S buffer u and P of tile parity u come from the 4 warps of parity u
        constexpr int kTileThreads = kAlt ? kPfSoftThreads / 2 : kPfSoftThreads;
        for (int u = 0; u < 2; ++u) {
            mbar_init(s_full(u), 1);
            mbar_init(s_free(u), kTileThreads);
            mbar_init(p_full(u), kTileThreads);
            mbar_init(pv_done(u), 1);
        }
        if constexpr (kAlt)
            for (int x = 0; x < 8; ++x) mbar_init(m_ready(x >> 1, x & 1), 32);
        mbar_init(o_done, 1);
        mbar_init(drain(0), 1);
        mbar_init(drain(1), 1);
        abort_flag = 0;
        q_amax_bits = 0u;
        mbar_init_fence();
    }
    if (warp == kPfMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kPfTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Q into TMEM columns 128 + kPfDimsPer / 2 hf .. (two bf16 per column). For a bf16 cache only
    // the S issuer waits for it (named barrier kPfQBar) and the producers start their copies at
    // once (measured: 7 % faster than a CTA-wide barrier). For an INT8 cache the CTA-wide barrier
    // stays: producers and converters started before Q was written made that kernel 7 % slower.
    // INT8: q enters the fp16 products as q' = q * 2^e, e one power of two for the CTA's rows, so
    // that the largest |q'| lies in [2^14, 2^15) (a bf16 value scaled by a power of two is exact in
    // fp16 there, and nothing passes fp16's range); the scores' factor carries 2^-e. kcorr =
    // 1152 * (sum of the row's q' as the product sees them) is what the biased K codes add to each
    // of the row's scores.
    float q_down = 1.f, kcorr = 0.f;
    if constexpr (kI8) {
        if (warp < kPfSoftWarps) {
            float amax = 0.f;
#pragma unroll
            for (int c = 0; c < kPfDimsPer / 2; ++c)
                amax = fmax3(amax, fabsf(__uint_as_float(qw[c] << 16)), fabsf(__uint_as_float(qw[c] & 0xffff0000u)));
            atomicMax(&q_amax_bits, __float_as_uint(amax));
        }
        __syncthreads();
        const float amax = __uint_as_float(q_amax_bits);
        int e = 0;
        if (amax > 0.f) {  // floor(log2(amax)) from the exponent field (-127 for a subnormal amax)
            e = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xffu) - 127);
            e = e < -126 ? -126 : (e > 126 ? 126 : e);  // 2^e and 2^-e stay normal floats
        }
        const float q_up = __uint_as_float((uint32_t)(127 + e) << 23);
        q_down = __uint_as_float((uint32_t)(127 - e) << 23);
        if (warp < kPfSoftWarps) {
            float qsum = 0.f;
#pragma unroll
            for (int j = 0; j < kPfDimsPer / 4; ++j) {  // dims 4j .. 4j + 3 of this thread's part
                const uint32_t w0 = qw[2 * j], w1 = qw[2 * j + 1];
                const uint32_t lo = pack2_f16(__uint_as_float(w0 << 16) * q_up, __uint_as_float(w1 << 16) * q_up);
                const uint32_t hi = pack2_f16(__uint_as_float(w0 & 0xffff0000u) * q_up,
                                              __uint_as_float(w1 & 0xffff0000u) * q_up);
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
                const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                qsum += (a.x + a.y) + (b.x + b.y);
                qw[2 * j] = lo;
                qw[2 * j + 1] = hi;
            }
            xsum[hf * kPfQ + r] = qsum;  // the row's other part is read after the barrier below
            tmem_st_words(tmem + tl + kQCol + kPfDimsPer / 2 * hf, qw);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp < kPfSoftWarps) {
            float qs = 0.f;
#pragma unroll
            for (int q2 = 0; q2 < kPfSplit; ++q2) qs += xsum[q2 * kPfQ + r];
            kcorr = kPfI8Bias * qs;
        }
    } else if (warp < kPfSoftWarps) {
        tmem_st_words(tmem + tl + kQCol + kPfDimsPer / 2 * hf, qw);
        tc_fence_before();
        named_barrier_arrive(kPfQBar, kPfSoftThreads + 32);
    } else if (warp == kPfMmaWarp) {
        named_barrier_sync(kPfQBar, kPfSoftThreads + 32);
        tc_fence_after();
    }

    if (warp == kPfLoadWarpK || warp == kPfLoadWarpV) {
        // ---------------- producers: ring g = K (warp 9) or V (warp 10) ----------------
        const int g = warp - kPfLoadWarpK;
        const CUtensorMap* map = g ? &tmv : &tmk;
        int issued = 0;
        int ids_cur = ids_first, ids_next = ids_second;
        for (int t = 0; t < ntiles; ++t) {
            const int ns = nst(g), st = t % ns;
            if (t > 0 && (t & 3) == 0) {
                ids_cur = ids_next;
                ids_next = has_window((t >> 2) + 1) ? load_window((t >> 2) + 1, true) : -1;
            }
            const bool got = t < ns || mbar_wait_bounded(empty(g, st), ((t / ns) - 1) & 1);
            if (!__all_sync(0xffffffffu, got)) {  // warp-uniform exit
                if (lane == 0) { atomicExch(&abort_flag, 1); flag(p.status, PKV_FLAG_TIMEOUT); }
                break;
            }
            if (__any_sync(0xffffffffu, aborted(&abort_flag))) break;
            // lane jj < 8: the pool block of keys 128 t + 16 jj .. (-1 when not needed or invalid)
            int id = __shfl_sync(0xffffffffu, ids_cur, 8 * (t & 3) + (lane & 7));
            if (lane >= 8) id = -1;
            const unsigned valid = __ballot_sync(0xffffffffu, id >= 0);
            // bf16: the tensor copies complete full(g); INT8: the row copies complete staged(g)
            const uint32_t done = kI8 ? staged(g, st) : full(g, st);
            constexpr int kBytes = kI8 ? kPfBlockBytes / 2 + kBlockSize * 4 : kPfBlockBytes;
            if constexpr (kI8) {
                // V scales of blocks not copied: zero, so that a masked key's weight times its
                // scale is 0 (a stale scale could be a NaN)
                if (g == 1 && lane < 8 && id < 0) {
                    float4* z = reinterpret_cast<float4*>(smem + Gm::OffScl + ridx(1, st) * 8 * kBlockSize * 4) +
                                lane * (kBlockSize / 4);
#pragma unroll
                    for (int c = 0; c < kBlockSize / 4; ++c) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                __syncwarp();
            }
            if (lane == 0) {
                if (valid == 0) mbar_arrive(done);
                else mbar_arrive_expect_tx(done, __popc(valid) * kBytes);
            }
            __syncwarp();
            if (id >= 0) {
                if constexpr (kI8) {  // 2 KB of int8 rows and 64 B of scales per (block, kv head)
                    const size_t tile = (size_t)id * p.Hkv + kvh;
                    bulk_g2s(slot(g, t) + kPfI8Half + lane * (kPfBlockBytes / 2),
                             (g ? p.v_i8 : p.k_i8) + tile * (kPfBlockBytes / 2), kPfBlockBytes / 2, done);
                    bulk_g2s(scl(g, st) + lane * kBlockSize * 4, (g ? p.v_scales : p.k_scales) + tile * kBlockSize,
                             kBlockSize * 4, done);
                } else {
                    const int grp = (id * p.Hkv + kvh) * (kBlockSize / 8);  // the block's first 8-row group
                    tma_load_4d(slot(g, t) + lane * kPfBlockBytes, map, 0, 0, 0, grp, done);
                }
            }
            issued = t + 1;
        }
        if (aborted(&abort_flag) && lane == 0) {
            // let this CTA's own copies land before shared memory goes away
            const int ns = nst(g);
            for (int t = issued - ns < 0 ? 0 : issued - ns; t < issued; ++t)
                mbar_wait_bounded(kI8 ? staged(g, t % ns) : full(g, t % ns), (t / ns) & 1);
        }
    } else if (kI8 && warp >= kPfConvWarp0) {
        // ---------------- INT8: converters of ring g (warps 12-13: K, 14-15: V) ----------------
        // Thread c widens keys c and c + 64 of each tile: the key's 128 int8 values into fp16
        // (K: the codes plus 1152; V: the codes) in the 128-byte-swizzled rows the MMA
        // descriptors read. All of the ring's int8 rows are read into registers before any fp16
        // row is written, since the fp16 tile fills the whole slot, over the int8 rows in its
        // second half.
        const int g = (warp - kPfConvWarp0) >> 1;
        const int c = tid - 32 * (kPfConvWarp0 + 2 * g);
        const int bar_id = 5 + g;  // named barrier of the ring's kPfConvThreads threads
        const int ns = nst(g);
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % ns;
            const bool got = mbar_wait_bounded(staged(g, st), (t / ns) & 1);
            if (!got && lane_of() == 0) { atomicExch(&abort_flag, 1); flag(p.status, PKV_FLAG_TIMEOUT); }
            if (barrier_or(bar_id, kPfConvThreads, !got || aborted(&abort_flag))) break;
            uint4 in[2][8];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int key = c + 64 * kk, blk = key >> 4, kin = key & 15;
                const uint4* row = reinterpret_cast<const uint4*>(smem + (g ? Gm::OffV : kPfOffK) + st * kPfStage +
                                                                   kPfI8Half + blk * (kPfBlockBytes / 2) + kin * 128);
#pragma unroll
                for (int v = 0; v < 8; ++v) in[kk][v] = row[(v + lane) & 7];  // rotated: no bank conflicts
            }
            named_barrier_sync(bar_id, kPfConvThreads);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int key = c + 64 * kk, blk = key >> 4, kin = key & 15;
                // K: the codes plus 1152 (the softmax subtracts kcorr from each score and applies
                // the key's scale); V: the codes themselves (the key's scale goes onto its weight)
                unsigned char* base = smem + (g ? Gm::OffV : kPfOffK) + st * kPfStage + blk * kPfBlockBytes +
                                      (kin >> 3) * 2048 + (kin & 7) * 128;
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const int vv = (v + lane) & 7;  // dims 16 vv .. 16 vv + 15
                    uint32_t o[8];
                    const uint32_t wv[4] = {in[kk][v].x, in[kk][v].y, in[kk][v].z, in[kk][v].w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        o[2 * x] = pf_i8_lo(wv[x]);
                        o[2 * x + 1] = pf_i8_hi(wv[x]);
                        if (g) {
                            o[2 * x] = pf_unbias(o[2 * x]);
                            o[2 * x + 1] = pf_unbias(o[2 * x + 1]);
                        }
                    }
                    const int half = vv >> 2, ch = (2 * vv) & 7;  // 16-byte chunks ch, ch + 1 of the half
                    unsigned char* hb = base + half * 1024;
                    *reinterpret_cast<uint4*>(hb + ((ch ^ (kin & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4*>(hb + (((ch + 1) ^ (kin & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the MMA reads them async
            if (g == 1) {
                // keys past the CTA's last visible key weigh 0, but their V scales may be any bits
                // (NaN included) and 0 * NaN would poison O: zero them (the softmax reads the scale
                // row only after full(1), which this thread completes below)
                float* vsr = reinterpret_cast<float*>(smem + Gm::OffScl) + ridx(1, st) * 8 * kBlockSize;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    if (t * kPfK + c + 64 * kk >= n_tile_max) vsr[c + 64 * kk] = 0.f;
            }
            mbar_arrive(full(g, st));
        }
    } else if (warp == kPfMmaWarp || warp == kPfMmaWarpPV) {
        // ---------------- MMA issuers: S (warp 8) and PV (warp 11) ----------------
        if (lane == 0) {
            const bool is_s = warp == kPfMmaWarp;
            // fp16 operands for an INT8 cache, bf16 otherwise
            constexpr uint32_t kIdescS = kI8 ? idesc_f16(kPfQ, kPfK, false) : idesc_bf16(kPfQ, kPfK, false);
            constexpr uint32_t kIdescO = kI8 ? idesc_f16(kPfQ, 128, true) : idesc_bf16(kPfQ, 128, true);
            auto issue_s = [&](int t) {  // S(t) = Q . K(t)^T into S buffer t % SBufs
                const uint32_t kbase = slot(0, t);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    // K-major: 8-key groups 2 KB apart, dims 16 ks.. in half ks / 4 at 32 B (ks % 4)
                    const uint64_t bd = sdesc(kbase + (ks >> 2) * 1024 + (ks & 3) * 32, 16, 2048);
                    umma_ts(tmem + Gm::SCol + 128 * (t % Gm::SBufs), tmem + kQCol + 8 * ks, bd, kIdescS, ks > 0);
                }
                umma_commit(s_full(t % Gm::SBufs));
                umma_commit(empty(0, t % Gm::SK));  // the K slot is free once S(t) is done
            };
            auto issue_pv = [&](int t) {  // O += P(t) . V(t), P(t) in buffer t % PBufs
                const uint32_t vbase = slot(1, t);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    // MN-major: keys 16 kk.. are block kk; 8-key groups 2 KB apart, dims 64.. 1 KB on
                    const uint64_t bd = sdesc(vbase + kk * kPfBlockBytes, 1024, 2048);
                    umma_ts(tmem + kOCol, tmem + Gm::PCol + 64 * (t % Gm::PBufs) + 8 * kk, bd, kIdescO,
                            (t > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(pv_done(t & 1));
                umma_commit(empty(1, t % Gm::SV));  // the V slot is free once PV(t) is done
            };
            bool ok = true;
            auto wait = [&](uint32_t bar, uint32_t par) {
                if (ok && !mbar_wait_bounded(bar, par)) {
                    ok = false;
                    atomicExch(&abort_flag, 1);
                    flag(p.status, PKV_FLAG_TIMEOUT);
                }
                if (ok && aborted(&abort_flag)) ok = false;
                tc_fence_after();
                return ok;
            };
            if (is_s) {
                // S buffer t % SBufs is free once the softmax has read S(t - SBufs) from it
                for (int t = 0; t < ntiles && ok; ++t) {
                    const int tf = t - Gm::SBufs;
                    if (tf >= 0 && !wait(s_free(tf % Gm::SBufs), (tf / Gm::SBufs) & 1)) break;
                    if (!wait(full(0, t % Gm::SK), (t / Gm::SK) & 1)) break;
                    issue_s(t);
                }
            } else {
                for (int t = 0; t < ntiles && ok; ++t) {
                    if (!wait(p_full(t & 1), (t >> 1) & 1)) break;
                    if (!wait(full(1, t % Gm::SV), (t / Gm::SV) & 1)) break;
                    issue_pv(t);
                }
                umma_commit(o_done);
            }
            // every product this thread issued is done before TMEM may go away
            umma_commit(drain(is_s ? 0 : 1));
            mbar_wait_bounded(drain(is_s ? 0 : 1), 0);
        }
        __syncwarp();
    } else if constexpr (kAlt) {
        // ---------------- softmax, alternate tiles: row r, tiles t = e, e + 2, ..., all 128 keys ----------------
        // The two warps of a lane quadrant hold the same rows and take turns: warp parity e reads
        // S buffer e. The reference max of a row after each tile is handed to the other warp
        // (m_ready), which needs it before its own tile's exponents: O and every P are relative
        // to it. Each warp keeps its own part of the row sum, relative to the reference of its
        // latest tile; the parts are combined at the end.
        const int e = warp >> 2, q4 = warp & 3;
        const uint32_t s_col = tmem + tl + Gm::SCol + 128 * e, o_col = tmem + tl + kOCol;
        const uint32_t p_col = tmem + tl + Gm::PCol;
        const int n_row = !row_valid ? 0 : (kPrefix ? n_tile_max : first_visible + i);
        const int pair_bar = 1 + q4;  // named barrier of the quadrant's two warps
        const bool neg = p.scale_log2 < 0.f;
        const float csc = fmaxf(fabsf(p.scale_log2), 1.17549435e-38f);
        float* mref = xmax;                 // [128 rows]: the reference after the latest tile
        float* xm = xmax + kPfQ;            // [2 parities][128 rows]: each warp's final reference
        float m = -INFINITY, l = 0.f;       // this warp's reference and its part of the row sum
        bool ok = true;
        int win = -1;
        unsigned present = 0;
        for (int t = e; t < ntiles; t += 2) {
            if ((t >> 2) != win) {  // block presence of window t / 4 (the producer's test)
                win = t >> 2;
                present = __ballot_sync(0xffffffffu, load_window(win, false) >= 0);
            }
            const int mask8 = (present >> (8 * (t & 3))) & 0xFF;
            const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(s_full(e), (t >> 1) & 1));
            if (!got) {
                atomicExch(&abort_flag, 1);
                flag(p.status, PKV_FLAG_TIMEOUT);
            }
            tc_fence_after();
            if ((t + 1) * kPfK > n_tile_max || mask8 != 0xFF) {
                // V rows of keys no row may see (past the context or in a missing block) must be
                // finite: their weights are 0, and 0 * NaN would poison O. Thread r zeroes key r
                // of the tile once its V copy has landed (PV(t) waits for this warp's P). The
                // parity wait on the slot's barrier is sound only once the slot's previous tile,
                // t - SV, is known landed: PV(t - SV) done says so (and this warp already knows
                // PV(t - SV - 2) done, so that wait is sound too).
                const int k = r;
                const int tv = t - Gm::SV;
                const bool prev_ok = tv < 0 || mbar_wait_bounded(pv_done(tv & 1), (tv >> 1) & 1);
                if (!prev_ok || !mbar_wait_bounded(full(1, t % Gm::SV), (t / Gm::SV) & 1)) {
                    atomicExch(&abort_flag, 1);
                    flag(p.status, PKV_FLAG_TIMEOUT);
                } else if (t * kPfK + k >= n_tile_max || !((mask8 >> (k >> 4)) & 1)) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint4* z = reinterpret_cast<uint4*>(smem + Gm::OffV + (t % Gm::SV) * kPfStage +
                                                            (k >> 4) * kPfBlockBytes + ((k >> 3) & 1) * 2048 +
                                                            half * 1024 + (k & 7) * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) z[c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
            }
            float s[kPfK];
            tmem_ld128(s_col, s);  // (reading TMEM is harmless even when S(t) never came)
            tc_fence_before();
            mbar_arrive(s_free(e));  // S(t + 2) may now be written into this buffer
            // raw scores here; the scale (with log2 e) is applied inside each exponent below
            const int kbase = t * kPfK;
            if (neg || !(kbase + kPfK <= n_row && mask8 == 0xFF)) {  // not all of them visible
#pragma unroll
                for (int c = 0; c < kPfK; ++c) {
                    const bool vis = kbase + c < n_row && ((mask8 >> (c >> 4)) & 1);
                    s[c] = vis ? (neg ? -s[c] : s[c]) : -INFINITY;
                }
            }
            float mx8[8];  // tree maximum with three-input max: 8 chains of keys c8, c8 + 8, ..., c8 + 120
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                float a = fmax3(s[c8], s[c8 + 8], s[c8 + 16]);
#pragma unroll
                for (int j = 24; j + 8 < kPfK - 8; j += 16) a = fmax3(a, s[c8 + j], s[c8 + j + 8]);  // 24 .. 112
                mx8[c8] = fmaxf(a, s[c8 + kPfK - 8]);
            }
            const float mloc = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) * csc;
            // the reference after tile t - 1 (the other warp's), once it is published
            float mprev = -INFINITY;
            bool got_m = true;
            if (t > 0) {
                got_m = __all_sync(0xffffffffu, mbar_wait_bounded(m_ready(q4, e ^ 1), ((t - 1) >> 1) & 1));
                if (!got_m) {
                    atomicExch(&abort_flag, 1);
                    flag(p.status, PKV_FLAG_TIMEOUT);
                }
                mprev = mref[r];
            }
            if (__any_sync(0xffffffffu, !got || !got_m || aborted(&abort_flag))) { ok = false; break; }
            // raise the reference only when the tile's maximum exceeds it by more than 2^8
            const bool up = mloc > mprev + kPfRescale;
            const float mt = up ? mloc : mprev;
            mref[r] = mt;
            mbar_arrive(m_ready(q4, e));
            if (mt != m) {  // this warp's part of the sum follows the reference (m == -inf: l is 0)
                l = m == -INFINITY ? 0.f : l * ex2(m - mt);
                m = mt;
            }
            const float ms = mt == -INFINITY ? 0.f : mt;
            uint32_t pw[kPfK / 2];
            const uint64_t cs2 = f32x2(csc, csc), nms2 = f32x2(-ms, -ms);
            uint64_t ls2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < kPfK / 2; ++c) {
                float y0, y1;
                f32x2_split(fma_f32x2(f32x2(s[2 * c], s[2 * c + 1]), cs2, nms2), y0, y1);
                const float a0 = ex2(y0), a1 = ex2(y1);
                ls2[c & 1] = add_f32x2(ls2[c & 1], f32x2(a0, a1));
                pw[c] = pack2_bf16(a0, a1);
            }
            {
                float e0, e1, o0, o1;
                f32x2_split(ls2[0], e0, e1);
                f32x2_split(ls2[1], o0, o1);
                l += (e0 + o0) + (e1 + o1);
            }
            // P may be written, and O rescaled, once PV(t - 1) is done (it read the last P and
            // accumulated O relative to mprev). This warp waited for PV(t - 3) in its previous
            // tile, so the parity wait for PV(t - 1), on the same barrier, cannot be answered by
            // the phase of PV(t - 3). (With two P buffers and a wait for PV(t - 2) only, a
            // rescale's wait for PV(t - 1) would lack that: measured as wrong results.)
            static_assert(Gm::PBufs == 1, "the waits below assume one P buffer");
            if (t > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(pv_done((t - 1) & 1), ((t - 1) >> 1) & 1))) {
                    atomicExch(&abort_flag, 1);
                    flag(p.status, PKV_FLAG_TIMEOUT);
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, up)) {  // rescale this thread's O row (rare)
                    const float alpha = up ? ex2(mprev - mt) : 1.f;  // mprev == -inf: 0
#pragma unroll 1
                    for (int c0 = 0; c0 < 128; c0 += 32) {
                        float o[32];
                        tmem_ld32(o_col + c0, o);
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] *= alpha;
                        tmem_st32(o_col + c0, o);
                    }
                }
            }
            tmem_st64u(p_col, pw);
            tc_fence_before();
            mbar_arrive(p_full(t & 1));
        }
        if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(o_done, 0))) {
            atomicExch(&abort_flag, 1);
            flag(p.status, PKV_FLAG_TIMEOUT);
        }
        tc_fence_after();
        // the row's sum: both parts, each relative to its warp's last reference, against the
        // final reference (the larger: a row's reference never falls)
        xm[e * kPfQ + r] = m;
        xsum[e * kPfQ + r] = l;
        const bool fail = barrier_or(pair_bar, kPfGroup, !ok || aborted(&abort_flag));
        const float ma = xm[r], mb = xm[kPfQ + r];
        const float mfin = fmaxf(ma, mb);
        float lt = 0.f;
        if (mfin != -INFINITY) {
            if (ma != -INFINITY) lt += xsum[r] * ex2(ma - mfin);
            if (mb != -INFINITY) lt += xsum[kPfQ + r] * ex2(mb - mfin);
        }
        m = mfin;
        const uint32_t o_half = o_col + kPfDimsPer * e;  // this warp writes dims 64 e ..
        if (!fail && kPrefix) {
            // ---- epilogue: the partial state (m in log2 units, l, acc = O unnormalised) ----
            const size_t u = qrow * p.S + p.slot0 + split;
            float* acc = p.ws_acc + u * 128 + kPfDimsPer * e;
#pragma unroll 1
            for (int c0 = 0; c0 < kPfDimsPer; c0 += 32) {
                float o[32];
                tmem_ld32(o_half + c0, o);
                if (row_valid) {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        reinterpret_cast<float4*>(acc + c0)[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                }
            }
            if (row_valid && e == 0) {
                p.ws_ml[2 * u] = m;
                p.ws_ml[2 * u + 1] = lt;
            }
        } else if (!fail) {
            // ---- epilogue: dims 64 e .. of row r of O / l -> out ----
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + qrow * 128 + kPfDimsPer * e);
#pragma unroll 1
            for (int c0 = 0; c0 < kPfDimsPer; c0 += 32) {
                float o[32];
                tmem_ld32(o_half + c0, o);
                if (row_valid) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c0 / 8 + c] = make_uint4(pack2_bf16(o[8 * c] * inv, o[8 * c + 1] * inv),
                                                     pack2_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                                     pack2_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                                     pack2_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                }
            }
        }
    } else {
        // ---------------- softmax: row r, key half hf ----------------
        // + 128 (t % SBufs), + 64 (t % PBufs)
        const uint32_t s_col = tmem + tl + Gm::SCol + kPfKeysPer * hf, o_col = tmem + tl + kOCol + kPfDimsPer * hf;
        const uint32_t p_col = tmem + tl + Gm::PCol + kPfKeysPer / 2 * hf;
        // keys (relative to the CTA's first key) this row sees
        const int n_row = !row_valid ? 0 : (kPrefix ? n_tile_max : first_visible + i);
        const int pair_bar = 1 + (warp & 3);  // named barrier of warps w, w + 4, ... (kPfGroup threads)
        // scores are scaled inside the exponents by |scale| * log2 e; a negative scale flips their
        // sign. |scale| is at least FLT_MIN so a masked score (-inf) never meets a zero factor: a
        // zero scale still gives weights of exactly 1 (every visible score times FLT_MIN is ~0).
        const bool neg = p.scale_log2 < 0.f;
        // (INT8: times 2^-e, undoing q's prescale)
        const float csc = fmaxf(fabsf(p.scale_log2) * q_down, 1.17549435e-38f);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // bit j of `present`: block 32 w + j of the current window is present (the producer's test)
        unsigned present = __ballot_sync(0xffffffffu, load_window(0, false) >= 0);
        int ids_next = has_window(1) ? load_window(1, false) : -1;
        for (int t = 0; t < ntiles; ++t) {
            if (t > 0 && (t & 3) == 0) {
                present = __ballot_sync(0xffffffffu, ids_next >= 0);
                ids_next = has_window((t >> 2) + 1) ? load_window((t >> 2) + 1, false) : -1;
            }
            const int mask8 = (present >> (8 * (t & 3))) & 0xFF;
            constexpr int kMyBlocks = kPfKeysPer / kBlockSize;           // blocks of this thread's keys
            constexpr int kAllMine = (1 << kMyBlocks) - 1;
            const int mask = (mask8 >> (kMyBlocks * hf)) & kAllMine;
            const int u = t & 1;                                       // row-maxima buffer
            const int su = t % Gm::SBufs, pu = t % Gm::PBufs;          // S and P buffers
            const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(s_full(su), (t / Gm::SBufs) & 1));
            if (!got) {
                atomicExch(&abort_flag, 1);
                flag(p.status, PKV_FLAG_TIMEOUT);
            }
            tc_fence_after();
            if ((t + 1) * kPfK > n_tile_max || mask8 != 0xFF) {
                // V rows of keys no row may see (past the context or in a missing block) must be
                // finite: their weights are 0, and 0 * NaN would poison O. Zero them once the V
                // copy of tile t has landed (PV(t) waits for this thread's P, so it reads them
                // zeroed; the next copy into the slot waits for PV(t)).
                // kPfSoftThreads threads: key k, 64-dim half, and a 128 / kPfSplit * 2-byte piece of it
                constexpr int kPieces = kPfSoftThreads / kPfK;     // per key: 2 halves x pieces
                constexpr int kPieceB = 2 * 128 / kPieces;          // bytes of a piece
                const int k = tid / kPieces, half = (tid % kPieces) / (kPieces / 2);
                const int piece = tid % (kPieces / 2);
                if (!mbar_wait_bounded(full(1, t % Gm::SV), (t / Gm::SV) & 1)) {
                    atomicExch(&abort_flag, 1);
                    flag(p.status, PKV_FLAG_TIMEOUT);
                } else if (t * kPfK + k >= n_tile_max || !((mask8 >> (k >> 4)) & 1)) {
                    uint4* z = reinterpret_cast<uint4*>(smem + Gm::OffV + (t % Gm::SV) * kPfStage +
                                                        (k >> 4) * kPfBlockBytes + ((k >> 3) & 1) * 2048 +
                                                        half * 1024 + (k & 7) * 128 + piece * kPieceB);
#pragma unroll
                    for (int c = 0; c < kPieceB / 16; ++c) z[c] = make_uint4(0u, 0u, 0u, 0u);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
            }
            float s[kPfKeysPer];
            tmem_ld_words(s_col + 128 * su, s);  // (reading TMEM is harmless even when S(t) never came)
            if constexpr (kI8) {
                // S holds q' . (codes + 1152): minus kcorr, times each key's K scale (the staged
                // scale row of the K slot, keys in tile order), then the slot may be refilled
                const float4* ks4 = reinterpret_cast<const float4*>(smem + Gm::OffScl) +
                                    ((t % Gm::SK) * 8 * kBlockSize + kPfKeysPer * hf) / 4;
                const uint64_t nk2 = f32x2(-kcorr, -kcorr);
#pragma unroll
                for (int c = 0; c < kPfKeysPer / 4; ++c) {
                    const float4 k4 = ks4[c];
                    float a, b2;
                    f32x2_split(mul_f32x2(add_f32x2(f32x2(s[4 * c], s[4 * c + 1]), nk2), f32x2(k4.x, k4.y)), a, b2);
                    s[4 * c] = a; s[4 * c + 1] = b2;
                    f32x2_split(mul_f32x2(add_f32x2(f32x2(s[4 * c + 2], s[4 * c + 3]), nk2), f32x2(k4.z, k4.w)), a, b2);
                    s[4 * c + 2] = a; s[4 * c + 3] = b2;
                }
                __syncwarp();
                if (lane_of() == 0) mbar_arrive(empty(0, t % Gm::SK));
            }
            tc_fence_before();
            mbar_arrive(s_free(su));  // S(t + SBufs) may now be written into this buffer
            // raw scores here; the scale (with log2 e) is applied inside each exponent below
            const int kbase = t * kPfK + kPfKeysPer * hf;
            if (neg || !(kbase + kPfKeysPer <= n_row && mask == kAllMine)) {  // not all of them visible
#pragma unroll
                for (int c = 0; c < kPfKeysPer; ++c) {
                    const bool vis = kbase + c < n_row && ((mask >> (c >> 4)) & 1);
                    s[c] = vis ? (neg ? -s[c] : s[c]) : -INFINITY;
                }
            }
            float mx8[8];  // tree maximum with three-input max: 8 independent chains, then 2 levels
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if constexpr (kPfKeysPer == 64) {
                    float a = fmax3(s[e], s[e + 8], s[e + 16]);
                    a = fmax3(a, s[e + 24], s[e + 32]);
                    a = fmax3(a, s[e + 40], s[e + 48]);
                    mx8[e] = fmaxf(a, s[e + 56]);
                } else {
                    mx8[e] = fmaxf(fmax3(s[e], s[e + 8], s[e + 16]), s[e + 24]);
                }
            }
            mx8[0] = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
            // One vote of the pair of warps per tile. The reference m changes only when a row's
            // maximum exceeds it by more than 2^8, so if no thread's own half does (and no thread
            // gives up) every row keeps m and the halves need not swap maxima. Otherwise swap them
            // (the row's maximum over both halves, the same in both threads, log2 units) and
            // decide together whether to stop; both warps take the same branch at every barrier.
            const float mloc = mx8[0] * csc;
            const bool stop = !got || aborted(&abort_flag);
            bool up = false;
            float mx = m;
            if (barrier_or(pair_bar, kPfGroup, stop || mloc > m + kPfRescale)) {
                xmax[(u * kPfSplit + hf) * kPfQ + r] = mx8[0];
                named_barrier_sync(pair_bar, kPfGroup);
                float rm = xmax[u * kPfSplit * kPfQ + r];
#pragma unroll
                for (int q2 = 1; q2 < kPfSplit; ++q2) rm = fmaxf(rm, xmax[(u * kPfSplit + q2) * kPfQ + r]);
                mx = rm * csc;
                up = mx > m + kPfRescale;
                if (barrier_or(pair_bar, kPfGroup, stop)) { ok = false; break; }
            }
            float alpha = 1.f;
            if (up) {
                alpha = ex2(m - mx);  // m == -inf: 0
                m = mx;
                l *= alpha;
            }
            const float ms = m == -INFINITY ? 0.f : m;
            // two keys per instruction on the FMA pipe (packed fp32 pairs): the exponents' arguments
            // and the running sums
            uint32_t pw[kPfKeysPer / 2];
            const uint64_t cs2 = f32x2(csc, csc), nms2 = f32x2(-ms, -ms);
            uint64_t ls2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
            // INT8: the weights enter the fp16 product times their key's V scale (the V slot's
            // staged scale row; waited for on every tile, so the parity wait stays in step)
            const float* vsc = nullptr;
            if constexpr (kI8) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(full(1, t % Gm::SV), (t / Gm::SV) & 1))) {
                    atomicExch(&abort_flag, 1);
                    flag(p.status, PKV_FLAG_TIMEOUT);
                }
                vsc = reinterpret_cast<const float*>(smem + Gm::OffScl) +
                      ridx(1, t % Gm::SV) * 8 * kBlockSize + kPfKeysPer * hf;
            }
#pragma unroll
            for (int c = 0; c < kPfKeysPer / 2; ++c) {
                float y0, y1;
                f32x2_split(fma_f32x2(f32x2(s[2 * c], s[2 * c + 1]), cs2, nms2), y0, y1);
                const float a0 = ex2(y0), a1 = ex2(y1);
                ls2[c & 1] = add_f32x2(ls2[c & 1], f32x2(a0, a1));
                if constexpr (kI8) {
                    const float2 v2 = reinterpret_cast<const float2*>(vsc)[c];
                    pw[c] = pack2_f16(a0 * v2.x, a1 * v2.y);
                } else {
                    pw[c] = pack2_bf16(a0, a1);
                }
            }
            {
                float e0, e1, o0, o1;
                f32x2_split(ls2[0], e0, e1);
                f32x2_split(ls2[1], o0, o1);
                l += (e0 + o0) + (e1 + o1);
            }
            // P buffer pu is free once PV(t - PBufs) is done; O may be rescaled once PV(t - 1) is done
            const bool resc = t > 0 && __any_sync(0xffffffffu, up);
            const int wt = resc ? t - 1 : t - Gm::PBufs;  // the tile whose product must be complete
            if (wt >= 0) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(pv_done(wt & 1), (wt >> 1) & 1))) {
                    atomicExch(&abort_flag, 1);
                    flag(p.status, PKV_FLAG_TIMEOUT);
                }
                tc_fence_after();
            }
            if (resc) {  // rescale this thread's dims of its O row (rare)
#pragma unroll 1
                for (int c0 = 0; c0 < kPfDimsPer; c0 += 32) {
                    float o[32];
                    tmem_ld32(o_col + c0, o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] *= alpha;
                    tmem_st32(o_col + c0, o);
                }
            }
            tmem_st_words(p_col + 64 * pu, pw);
            tc_fence_before();
            mbar_arrive(p_full(u));
        }
        if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(o_done, 0))) {
            atomicExch(&abort_flag, 1);
            flag(p.status, PKV_FLAG_TIMEOUT);
        }
        tc_fence_after();
        // the row's sum over its parts; all threads of the group decide together
        xsum[hf * kPfQ + r] = l;
        const bool fail = barrier_or(pair_bar, kPfGroup, !ok || aborted(&abort_flag));
        float lt = xsum[r];
#pragma unroll
        for (int q2 = 1; q2 < kPfSplit; ++q2) lt += xsum[q2 * kPfQ + r];
        if (!fail && kPrefix) {
            // ---- epilogue: the partial state (m in log2 units, l, acc = O unnormalised) ----
            const size_t u = qrow * p.S + p.slot0 + split;
            float* acc = p.ws_acc + u * 128 + kPfDimsPer * hf;
#pragma unroll 1
            for (int c0 = 0; c0 < kPfDimsPer; c0 += 32) {
                float o[32];
                tmem_ld32(o_col + c0, o);
                if constexpr (kI8) pf_unpermute(o);
                if (row_valid) {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        reinterpret_cast<float4*>(acc + c0)[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                }
            }
            if (row_valid && hf == 0) {
                p.ws_ml[2 * u] = m;
                p.ws_ml[2 * u + 1] = lt;
            }
        } else if (!fail) {
            // ---- epilogue: dims kPfDimsPer hf .. of row r of O / l -> out ----
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + qrow * 128 + kPfDimsPer * hf);
#pragma unroll 1
            for (int c0 = 0; c0 < kPfDimsPer; c0 += 32) {
                float o[32];
                tmem_ld32(o_col + c0, o);
                if constexpr (kI8) pf_unpermute(o);
                if (row_valid) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c0 / 8 + c] = make_uint4(pack2_bf16(o[8 * c] * inv, o[8 * c + 1] * inv),
                                                     pack2_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                                     pack2_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                                     pack2_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPfMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPfTmemCols)
                     : "memory");
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           int max_query_len, cudaStream_t s) {
    PfWork w{};
    w.q = p.q; w.block_tables = p.block_tables; w.status = p.status;
    w.Hq = p.Hq; w.Hkv = p.Hkv; w.G = p.G; w.NB = p.NB; w.MBPS = p.MBPS; w.scale_log2 = p.scale_log2;
    w.out = p.out; w.context_lens = p.context_lens; w.query_start = p.query_start; w.B = p.B;
    w.k_i8 = p.k_i8; w.v_i8 = p.v_i8; w.k_scales = p.k_scales; w.v_scales = p.v_scales;
    const dim3 grid((max_query_len + kPfQ - 1) / kPfQ, p.Hq, p.B);
    if (p.k_i8) {
        auto kern = prefill_kernel<false, true>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PfGeom<true>::Smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, grid, dim3(PfGeom<true>::Threads), PfGeom<true>::Smem, s, w, tk, tv);
    }
    auto kern = prefill_kernel<false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PfGeom<false>::Smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, dim3(PfGeom<false>::Threads), PfGeom<false>::Smem, s, w, tk, tv);
}

cudaError_t launch_prefix(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int splits,
                          cudaStream_t s) {
    PfWork w{};
    w.q = p.q; w.block_tables = p.block_tables; w.status = p.status;
    w.Hq = p.Hq; w.Hkv = p.Hkv; w.G = p.G; w.NB = p.NB; w.MBPS = p.MBPS; w.scale_log2 = p.scale_log2;
    w.ws_acc = p.ws_acc; w.ws_ml = p.ws_ml; w.B = p.B; w.S = p.S; w.slot0 = p.slot0;
    w.prefix_tokens = p.prefix_tokens; w.split_tokens = p.split_tokens;
    w.k_i8 = p.k_i8; w.v_i8 = p.v_i8; w.k_scales = p.k_scales; w.v_scales = p.v_scales;
    const dim3 grid((p.B * p.G + kPfQ - 1) / kPfQ, p.Hkv, splits);
    if (p.k_i8) {
        auto kern = prefill_kernel<true, true>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PfGeom<true>::Smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, grid, dim3(PfGeom<true>::Threads), PfGeom<true>::Smem, s, w, tk, tv);
    }
    auto kern = prefill_kernel<true, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PfGeom<false>::Smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, dim3(PfGeom<false>::Threads), PfGeom<false>::Smem, s, w, tk, tv);
}

}  // namespace pkv
