// splitk_merge.cu -- kernel 2 of the split-K decode: merges the per-split partial states.
//
// "EchoLLMServing inference framework notes", section 2 (FlashDecoding): each split emits
// (m, l, acc) and a second reduce kernel combines them. For one (sequence, query head) with
// splits j < ns (scores in base-2 units):
//     M = max_j m_j,   w_j = 2^(m_j - M),   L = sum_j w_j l_j,   out = sum_j w_j acc_j / L
// Sequences with a single split were finished by kernel 1 and are skipped here. In a shared-prefix
// call every row also has extra slots (the prefix partials) and is always merged.
//
// One warp per (sequence, query head), eight per CTA, so the whole batch is one wave of CTAs.
// Lane i owns D/32 consecutive columns. The warp loads its split rows eight at a time as
// independent loads and folds each into a running (m, l, acc) (the online rescaling kernel 1
// uses), so no load waits for the global maximum: two dependent global round trips in all
// (context_lens, then the rows).
#include <math.h>

#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kMergeWarps = 8;
constexpr int kMergeBatch = 8;  // rows in flight per warp

template <int V> struct Vec;
template <> struct Vec<2> { using T = float2; };
template <> struct Vec<4> { using T = float4; };

template <typename OT, int D>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const MergeParams p) {
    constexpr int V = D / 32;  // columns per lane
    using VT = typename Vec<V>::T;

    grid_dependency_wait();  // partial states of the split kernel before this one in the stream

    const int lane = threadIdx.x & 31;
    const int pair = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (pair >= p.B * p.L * p.Hq) return;
    const int zb = pair / p.Hq;  // (sequence, query token) row
    const int b = zb / p.L;
    bool bad;
    // the context the split kernel split: the row's own, or (packed) the sequence's last token's
    const int n = query_context_len(p.context_lens[b], p.L, p.packed ? p.L - 1 : zb - b * p.L,
                                    p.MBPS * kBlockSize, &bad);
    int per;
    const int ns = split_count(n > p.kv_start ? n - p.kv_start : 0, p.chunk, p.max_splits, &per);
    if (ns <= 1 && p.extra == 0) return;
    // slots: the row's ns splits, then the extra (shared-prefix) slots
    const int total = ns + p.extra;
    auto slot = [&](int k) { return k < ns ? k : p.extra0 + (k - ns); };

    const size_t base = (size_t)pair * p.ws_stride;
    const float2* ml = reinterpret_cast<const float2*>(p.ws_ml) + base;
    const VT* acc = reinterpret_cast<const VT*>(p.ws_acc + base * D) + lane;
    float m = -INFINITY, l = 0.f, a[V];
#pragma unroll
    for (int e = 0; e < V; ++e) a[e] = 0.f;
    for (int j0 = 0; j0 < total; j0 += kMergeBatch) {
        float2 st[kMergeBatch];
        VT v[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            if (j0 + u < total) {
                const int sl = slot(j0 + u);
                st[u] = ml[sl];
                v[u] = acc[(size_t)sl * (D / V)];
            }
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            if (j0 + u >= total || st[u].x == -INFINITY) continue;  // empty split: no contribution
            const float mn = fmaxf(m, st[u].x);
            const float s0 = ex2(m - mn), s1 = ex2(st[u].x - mn);  // m == -inf: s0 = 0
            l = l * s0 + st[u].y * s1;
            const float* vv = reinterpret_cast<const float*>(&v[u]);
#pragma unroll
            for (int e = 0; e < V; ++e) a[e] = a[e] * s0 + vv[e] * s1;
            m = mn;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    OT* out = static_cast<OT*>(p.out) + (size_t)pair * D + lane * V;
#pragma unroll
    for (int e = 0; e < V; ++e) store_out<OT>(out + e, a[e] * inv);
}

template <typename OT, int D>
cudaError_t launch_merge_t(const MergeParams& p, cudaStream_t s) {
    const int pairs = p.B * p.L * p.Hq;
    return launch_pdl(merge_kernel<OT, D>, dim3((pairs + kMergeWarps - 1) / kMergeWarps),
                      dim3(32 * kMergeWarps), 0, s, p);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, pkv_dtype out_dtype, int D, cudaStream_t s) {
    if (out_dtype == PKV_F32) {
        if (D == 128) return launch_merge_t<float, 128>(p, s);
        if (D == 64) return launch_merge_t<float, 64>(p, s);
    } else {
        if (D == 128) return launch_merge_t<__nv_bfloat16, 128>(p, s);
        if (D == 64) return launch_merge_t<__nv_bfloat16, 64>(p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
