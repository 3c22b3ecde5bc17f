// decode_split.cuh -- split-K paged decode attention, kernel 1 of 2 (CUDA-core path).
//
// One CTA of 128 threads computes one (sequence b, kv head, split) unit for a group of up to HG
// query heads that share the kv head ("EchoLLMServing inference framework notes", section 2:
// one program handles all KV of one split and emits its partial (m, l, acc); "LLM Primer VI,
// Chapter 8", section 8.1: K and V are gathered through the block table).
//
// Data movement. The split's block ids are read once into shared memory. Thread 0 streams each
// 16-token block's K tile and V tile ([16][D] contiguous in the pool, 2-4 KB each) -- plus the
// two 64-byte INT8 scale rows -- into a STAGES-deep shared-memory ring with 1-D bulk copies
// (cp.async.bulk, TMA engine) completing on one mbarrier per stage, so several KB per CTA stay
// in flight while the CTA computes on an earlier block. Block ids outside [0, num_blocks) are
// never dereferenced: the stage is marked invalid and its tokens are masked.
//
// Compute. Thread t owns an 8-element slice (dims 8*(t % TPT) ..) of token (t / TPT) + TPP*p
// of every block and keeps its own online-softmax state (m, l, acc[HG][8]) over those tokens;
// q is held in registers pre-multiplied by scale*log2(e) so scores are in base-2 units. A QK dot
// product is finished by a transposed butterfly across the TPT lanes of the token (each
// exchange halves the number of live values), so the HG*PPB scores of a thread cost about
// 2*HG*PPB shuffles instead of HG*PPB*log2(TPT). The per-thread states are merged in shared
// memory at the end; a single-split sequence writes `out` directly, otherwise the unit writes
// (m, l, acc) to the workspace for the merge kernel. INT8 scales multiply the score (K) and the
// softmax weight (V), not every element ("EchoLLMServing notes", section 3).
#pragma once

#include <math.h>

#include "pkv_device.cuh"

namespace pkv {

template <typename T>
struct KvElem;
template <>
struct KvElem<float> { static constexpr bool kI8 = false; };
template <>
struct KvElem<__nv_bfloat16> { static constexpr bool kI8 = false; };
template <>
struct KvElem<int8_t> { static constexpr bool kI8 = true; };

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }
constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

template <typename KV, int D, int HG>
struct SplitGeom {
    static constexpr bool kI8 = KvElem<KV>::kI8;
    static constexpr int NT = 128;                       // threads per CTA
    static constexpr int TPT = D / 8;                    // threads per token row
    static constexpr int TPP = NT / TPT;                 // tokens per pass (= token groups)
    static constexpr int PPB = kBlockSize / TPP;         // passes per block
    static constexpr int TILE = kBlockSize * D * (int)sizeof(KV);  // one K (or V) tile
    static constexpr int SCALES = kI8 ? 2 * kBlockSize * 4 : 0;    // K and V scale rows
    static constexpr int STAGE = round_up(2 * TILE + SCALES, 128);
    static constexpr int STAGES = cmax(3, cmin(8, 32768 / STAGE));
    static constexpr int RED = TPP * HG * (D + 2) * 4;   // end-of-CTA merge scratch
    static constexpr int MAIN = round_up(cmax(STAGES * STAGE, RED), 128);
    static constexpr int IDWIN = 128;                    // block ids cached per window
    static constexpr int SMEM = MAIN + IDWIN * 4 + round_up(STAGES * 4, 8) + STAGES * 8;
    static_assert(PPB >= 1 && TPP * PPB == kBlockSize, "thread layout must tile a block");
    static_assert(TILE % 16 == 0, "bulk copies move multiples of 16 bytes");
};

// Sum each of the C values over the TPT consecutive lanes of a group (TPT a power of two <= 32)
// and leave every lane of the group holding all C sums. Phase 1 halves the live values at
// each exchange (lanes with the mask bit set keep the upper half), phase 2 finishes the
// remaining masks on what is left, phase 3 gathers the C sums back from the lanes holding them.
template <int C, int TPT>
__device__ __forceinline__ void group_allreduce(float (&v)[C]) {
    constexpr int K = cmin(ilog2(C), ilog2(TPT));
    constexpr int CF = C >> K;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int mask = TPT >> (k + 1);
        const int half = (C >> k) / 2;
        const bool upper = (lane & mask) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float send = upper ? v[j] : v[j + half];
            const float keep = upper ? v[j + half] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
    }
#pragma unroll
    for (int mask = TPT >> (K + 1); mask >= 1; mask >>= 1) {
#pragma unroll
        for (int j = 0; j < CF; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], mask);
    }
    if constexpr (K > 0) {
        float r[C];
        const int gbase = lane & ~(TPT - 1);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int sel = c / CF;
            int src = gbase;
#pragma unroll
            for (int k = 0; k < K; ++k)
                if ((sel >> (K - 1 - k)) & 1) src += TPT >> (k + 1);
            r[c] = __shfl_sync(0xffffffffu, v[c % CF], src);
        }
#pragma unroll
        for (int c = 0; c < C; ++c) v[c] = r[c];
    }
}

template <typename KV, typename QT, int D, int HG>
__global__ void __launch_bounds__(128) split_kernel(const SplitParams p) {
    using G = SplitGeom<KV, D, HG>;
    constexpr int NT = G::NT, TPT = G::TPT, TPP = G::TPP, PPB = G::PPB;
    constexpr int STAGES = G::STAGES, STAGE = G::STAGE, TILE = G::TILE, IDWIN = G::IDWIN;
    constexpr bool kI8 = G::kI8;
    constexpr float kNegInf = -INFINITY;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stages = smem;
    int32_t* ids = reinterpret_cast<int32_t*>(smem + G::MAIN);
    int32_t* stage_ok = ids + IDWIN;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::MAIN + IDWIN * 4 + round_up(STAGES * 4, 8));

    const int tid = threadIdx.x;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.head_chunks;
    const int hc = blockIdx.y - kvh * p.head_chunks;
    const int zb = blockIdx.z;          // row of q / out: query token lq of sequence b
    const int b = zb / p.L, lq = zb - b * p.L;
    const int h0 = kvh * p.G + hc * HG;          // first query head of this CTA
    const int nh = cmin(HG, p.G - hc * HG);      // query heads this CTA produces

    grid_dependency_wait();  // inputs (new K/V rows, tables) may come from the previous kernel

    // context length of this query token, clamped to what the block table can address
    const int stored = p.context_lens[b];
    bool bad;
    const int n = query_context_len(stored, p.L, lq, p.MBPS * kBlockSize, &bad);
    const bool reporter = tid == 0 && split == 0 && blockIdx.y == 0 && lq == 0;
    if (bad && reporter) flag(p.status, PKV_FLAG_BAD_CONTEXT);
    else if (stored > p.max_context_len && reporter) flag(p.status, PKV_FLAG_LONG_CONTEXT);
    int per;
    const int ns = split_count(n, p.chunk, p.max_splits, &per);
    if (split >= ns) return;
    const int t0 = split * per;
    const int t1 = cmin(n, t0 + per);
    const int nblk = (t1 - t0 + kBlockSize - 1) / kBlockSize;
    const int blk0 = t0 / kBlockSize;

    const int slice = tid % TPT;  // dims [8*slice, 8*slice + 8)
    const int tg = tid / TPT;     // tokens tg + TPP*pp of each block

    // q for the CTA's heads, in base-2 score units
    float qf[HG][8];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
        if (hh < nh) {
            const QT* qp = static_cast<const QT*>(p.q) + ((size_t)zb * p.Hq + h0 + hh) * D + slice * 8;
            gload8_f32<QT>(qp, qf[hh]);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[hh][e] *= p.scale_log2;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[hh][e] = 0.f;
        }
    }

    float m[HG], l[HG], acc[HG][8];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
        m[hh] = kNegInf;
        l[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;
    }

    const uint32_t bar0 = smem_addr(bars);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
    }
    const int32_t* bt_row = p.block_tables + (size_t)b * p.MBPS + blk0;
    auto load_ids = [&](int first) {  // ids of blocks [first, first + IDWIN) of the split
        for (int j = first + tid; j < nblk && j < first + IDWIN; j += NT) {
            int id = bt_row[j];
            if (id < 0 || id >= p.NB) {
                flag(p.status, PKV_FLAG_BAD_BLOCK);
                id = -1;
            }
            ids[j % IDWIN] = id;
        }
    };
    load_ids(0);
    __syncthreads();

    const unsigned char* kpool = static_cast<const unsigned char*>(p.k_pool);
    const unsigned char* vpool = static_cast<const unsigned char*>(p.v_pool);
    auto issue = [&](int j) {  // thread 0 only: start block j of the split into its stage
        const int st = j % STAGES;
        const int id = ids[j % IDWIN];
        const uint32_t bar = bar0 + 8 * st;
        const uint32_t dst = smem_addr(stages + st * STAGE);
        stage_ok[st] = id >= 0;
        if (id >= 0) {
            const size_t row = (size_t)id * p.Hkv + kvh;
            mbar_arrive_expect_tx(bar, 2 * TILE + G::SCALES);
            bulk_g2s(dst, kpool + row * TILE, TILE, bar);
            bulk_g2s(dst + TILE, vpool + row * TILE, TILE, bar);
            if constexpr (kI8) {
                bulk_g2s(dst + 2 * TILE, p.k_scales + row * kBlockSize, kBlockSize * 4, bar);
                bulk_g2s(dst + 2 * TILE + kBlockSize * 4, p.v_scales + row * kBlockSize,
                         kBlockSize * 4, bar);
            }
        } else {
            mbar_arrive(bar);
        }
    };
    if (tid == 0)
        for (int j = 0; j < STAGES && j < nblk; ++j) issue(j);

    for (int i = 0; i < nblk; ++i) {
        const int st = i % STAGES;
        const bool ready = mbar_wait_bounded(bar0 + 8 * st, (i / STAGES) & 1);
        if (ready) {
            const unsigned char* kt = stages + st * STAGE;
            const unsigned char* vt = kt + TILE;
            const bool ok = stage_ok[st] != 0;
            const int tok_base = t0 + i * kBlockSize;

            float s[PPB * HG];
#pragma unroll
            for (int pp = 0; pp < PPB; ++pp) {
                const int tok = tg + TPP * pp;
                float kf[8];
                load8_f32<KV>(kt + (tok * D + slice * 8) * sizeof(KV), kf);
#pragma unroll
                for (int hh = 0; hh < HG; ++hh) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) a = fmaf(qf[hh][e], kf[e], a);
                    s[pp * HG + hh] = a;
                }
            }
            group_allreduce<PPB * HG, TPT>(s);

            bool valid[PPB];
#pragma unroll
            for (int pp = 0; pp < PPB; ++pp) {
                const int tok = tg + TPP * pp;
                valid[pp] = ok && (tok_base + tok < t1);
                float ks = 1.f;
                if constexpr (kI8) ks = reinterpret_cast<const float*>(kt + 2 * TILE)[tok];
#pragma unroll
                for (int hh = 0; hh < HG; ++hh)
                    s[pp * HG + hh] = valid[pp] ? s[pp * HG + hh] * ks : kNegInf;
            }
            // online softmax over this thread's tokens, then the weighted V rows
#pragma unroll
            for (int hh = 0; hh < HG; ++hh) {
                float mx = s[hh];
#pragma unroll
                for (int pp = 1; pp < PPB; ++pp) mx = fmaxf(mx, s[pp * HG + hh]);
                const float mnew = fmaxf(m[hh], mx);
                const float msafe = mnew == kNegInf ? 0.f : mnew;
                const float alpha = ex2(m[hh] - msafe);
                l[hh] *= alpha;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[hh][e] *= alpha;
                m[hh] = mnew;
#pragma unroll
                for (int pp = 0; pp < PPB; ++pp) {
                    const float pr = ex2(s[pp * HG + hh] - msafe);
                    s[pp * HG + hh] = pr;
                    l[hh] += pr;
                }
            }
#pragma unroll
            for (int pp = 0; pp < PPB; ++pp) {
                const int tok = tg + TPP * pp;
                float vf[8];
                load8_f32<KV>(vt + (tok * D + slice * 8) * sizeof(KV), vf);
                float vs = 1.f;
                // (a token past the context weighs 0; its scale may be any bits, NaN included, so
                // it is not read into the product)
                if constexpr (kI8) vs = valid[pp] ? reinterpret_cast<const float*>(kt + 2 * TILE + kBlockSize * 4)[tok] : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) vf[e] = valid[pp] ? vf[e] : 0.f;  // rows past the context
#pragma unroll
                for (int hh = 0; hh < HG; ++hh) {
                    const float w = s[pp * HG + hh] * vs;
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(w, vf[e], acc[hh][e]);
                }
            }
        }
        if (__syncthreads_or(!ready)) {
            // a copy never completed: report, wait (bounded) for this CTA's other copies in
            // flight so none lands after exit, and give up on this unit
            if (tid == 0) {
                flag(p.status, PKV_FLAG_TIMEOUT);
                for (int j = i; j < nblk && j < i + STAGES; ++j)
                    mbar_wait_bounded(bar0 + 8 * (j % STAGES), (j / STAGES) & 1);
            }
            return;
        }
        const int j = i + STAGES;
        if (j < nblk) {
            if (j % IDWIN == 0) {
                load_ids(j);
                __syncthreads();
            }
            if (tid == 0) issue(j);
        }
    }

    grid_dependents_launch();  // the merge kernel may start launching
    // merge the per-thread states of the CTA (the ring is idle: every issued copy was consumed)
    float* red_m = reinterpret_cast<float*>(smem);
    float* red_l = red_m + TPP * HG;
    float* red_acc = red_l + TPP * HG;
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
        if (slice == 0) {
            red_m[tg * HG + hh] = m[hh];
            red_l[tg * HG + hh] = l[hh];
        }
        float* dst = red_acc + (tg * HG + hh) * D + slice * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = acc[hh][e];
    }
    __syncthreads();
    for (int o = tid; o < HG * D; o += NT) {
        const int hh = o / D, d = o - (o / D) * D;
        if (hh >= nh) continue;
        float M = kNegInf;
#pragma unroll
        for (int g = 0; g < TPP; ++g) M = fmaxf(M, red_m[g * HG + hh]);
        float L = 0.f, A = 0.f;
        if (M != kNegInf) {
#pragma unroll
            for (int g = 0; g < TPP; ++g) {
                const float w = ex2(red_m[g * HG + hh] - M);
                L = fmaf(w, red_l[g * HG + hh], L);
                A = fmaf(w, red_acc[(g * HG + hh) * D + d], A);
            }
        }
        const size_t qh = (size_t)zb * p.Hq + h0 + hh;
        if (ns == 1) {
            store_out<QT>(static_cast<QT*>(p.out) + qh * D + d, L > 0.f ? A / L : 0.f);
        } else {
            const size_t u = qh * p.ws_stride + split;
            p.ws_acc[u * D + d] = A;
            if (d == 0) {
                p.ws_ml[2 * u] = M;
                p.ws_ml[2 * u + 1] = L;
            }
        }
    }
}

template <typename KV, typename QT, int D, int HG>
cudaError_t launch_split_t(const SplitParams& p, cudaStream_t s) {
    using G = SplitGeom<KV, D, HG>;
    auto kern = split_kernel<KV, QT, D, HG>;
    if (G::SMEM > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, dim3(p.max_splits, p.Hkv * p.head_chunks, p.B * p.L), dim3(G::NT), G::SMEM, s, p);
}

template <typename KV, typename QT>
cudaError_t launch_split_dispatch(const SplitParams& p, int D, int hg, cudaStream_t s) {
    if (D == 128) {
        switch (hg) {
            case 1: return launch_split_t<KV, QT, 128, 1>(p, s);
            case 2: return launch_split_t<KV, QT, 128, 2>(p, s);
            case 4: return launch_split_t<KV, QT, 128, 4>(p, s);
            case 8: return launch_split_t<KV, QT, 128, 8>(p, s);
        }
    } else if (D == 64) {
        switch (hg) {
            case 1: return launch_split_t<KV, QT, 64, 1>(p, s);
            case 2: return launch_split_t<KV, QT, 64, 2>(p, s);
            case 4: return launch_split_t<KV, QT, 64, 4>(p, s);
            case 8: return launch_split_t<KV, QT, 64, 8>(p, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
