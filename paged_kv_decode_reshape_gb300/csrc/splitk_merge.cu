// splitk_merge.cu -- kernel 2 of the split-K decode: merges the per-split partial states.
//
// "EchoLLMServing inference framework notes", section 2 (FlashDecoding): each split emits
// (m, l, acc) and a second reduce kernel combines them. For one (sequence, query head) with
// splits j < ns (scores in base-2 units):
//     M = max_j m_j,   w_j = 2^(m_j - M),   L = sum_j w_j l_j,   out = sum_j w_j acc_j / L
// Sequences with a single split were finished by kernel 1 and are skipped here.
//
// One CTA of 256 threads per (query head, sequence): J = 256 / (D/4) groups of D/4 threads, each
// group reading whole accumulator rows as float4. A group folds its rows j = g, g + J, ... into a
// running (m, l, acc) of its own as it loads them (the same online rescaling kernel 1 uses), so
// the row loads do not wait for the global maximum; the J group states are then combined once in
// shared memory. Two dependent global round trips in all: context_lens, then the rows.
#include <math.h>

#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kMergeThreads = 256;

template <typename OT, int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
    constexpr int DQ = D / 4;                   // float4 columns per row
    constexpr int J = kMergeThreads / DQ;       // row groups
    __shared__ float g_m[J], g_l[J];
    __shared__ __align__(16) float g_acc[J][D];

    grid_dependency_wait();  // partial states of the split kernel before this one in the stream

    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    int n = p.context_lens[b];
    const int ncap = p.MBPS * kBlockSize;
    n = n < 0 ? 0 : (n > ncap ? ncap : n);
    int per;
    const int ns = split_count(n, p.chunk, p.max_splits, &per);
    if (ns <= 1) return;

    const size_t base = ((size_t)b * p.Hq + h) * p.max_splits;
    const float* ml = p.ws_ml + 2 * base;
    const int dq = tid % DQ, g = tid / DQ;
    const float4* accp = reinterpret_cast<const float4*>(p.ws_acc + base * D) + dq;

    float m = -INFINITY, l = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int j = g; j < ns; j += J) {
        const float mj = ml[2 * j], lj = ml[2 * j + 1];
        const float4 v = accp[(size_t)j * DQ];
        if (mj == -INFINITY) continue;  // a split with no valid token contributes nothing
        const float mn = fmaxf(m, mj);
        const float s0 = ex2(m - mn), s1 = ex2(mj - mn);  // m == -inf: s0 = 0
        l = l * s0 + lj * s1;
        a.x = a.x * s0 + v.x * s1;
        a.y = a.y * s0 + v.y * s1;
        a.z = a.z * s0 + v.z * s1;
        a.w = a.w * s0 + v.w * s1;
        m = mn;
    }
    if (dq == 0) {
        g_m[g] = m;
        g_l[g] = l;
    }
    reinterpret_cast<float4*>(g_acc[g])[dq] = a;
    __syncthreads();
    OT* out = static_cast<OT*>(p.out) + ((size_t)b * p.Hq + h) * D;
    for (int d = tid; d < D; d += kMergeThreads) {
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < J; ++r) M = fmaxf(M, g_m[r]);
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int r = 0; r < J; ++r) {
                const float w = ex2(g_m[r] - M);
                L = fmaf(w, g_l[r], L);
                A = fmaf(w, g_acc[r][d], A);
            }
        }
        store_out<OT>(out + d, L > 0.f ? A / L : 0.f);
    }
}

template <typename OT, int D>
cudaError_t launch_merge_t(const MergeParams& p, cudaStream_t s) {
    return launch_pdl(merge_kernel<OT, D>, dim3(p.Hq, p.B), dim3(kMergeThreads), 0, s, p);
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
