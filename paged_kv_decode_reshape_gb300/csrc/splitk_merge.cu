// splitk_merge.cu -- kernel 2 of the split-K decode: merges the per-split partial states.
//
// "EchoLLMServing inference framework notes", section 2 (FlashDecoding): each split emits
// (m, l, acc) and a second reduce kernel combines them. For one (sequence, query head) with
// splits j < ns (scores in base-2 units):
//     M = max_j m_j,   w_j = 2^(m_j - M),   L = sum_j w_j l_j,   out = sum_j w_j acc_j / L
// Sequences with a single split were finished by kernel 1 and are skipped here.
//
// One CTA of 256 threads per (query head, sequence). The weights w_j go to shared memory; the
// accumulators are read as float4 by D/4 threads per split row and J = 256 / (D/4) rows at a
// time, so a CTA keeps J*D*4 bytes of independent loads in flight per step.
#include <math.h>

#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kMergeThreads = 256;

__device__ __forceinline__ float block_reduce(float v, float* scratch, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, u) : v + u;
    }
    __syncthreads();  // scratch may still be read from a previous reduction
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = scratch[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) v = is_max ? fmaxf(v, scratch[w]) : v + scratch[w];
    return v;
}

template <typename OT, int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
    constexpr int DQ = D / 4;                   // float4 columns per row
    constexpr int J = kMergeThreads / DQ;       // split rows read per step
    extern __shared__ __align__(16) float msm[];
    float* w = msm;                             // [max_splits]
    float* part = msm + ((p.max_splits + 3) & ~3);  // [J][D], 16-byte aligned
    __shared__ float scratch[kMergeThreads / 32];

    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    int n = p.context_lens[b];
    const int ncap = p.MBPS * kBlockSize;
    n = n < 0 ? 0 : (n > ncap ? ncap : n);
    int per;
    const int ns = split_count(n, p.chunk, p.max_splits, &per);
    if (ns <= 1) return;

    const size_t base = ((size_t)b * p.Hq + h) * p.max_splits;
    const float* ml = p.ws_ml + 2 * base;
    float mx = -INFINITY;
    for (int j = tid; j < ns; j += kMergeThreads) mx = fmaxf(mx, ml[2 * j]);
    const float M = block_reduce(mx, scratch, true);
    float ls = 0.f;
    for (int j = tid; j < ns; j += kMergeThreads) {
        const float wj = M == -INFINITY ? 0.f : ex2(ml[2 * j] - M);
        w[j] = wj;
        ls = fmaf(wj, ml[2 * j + 1], ls);
    }
    const float L = block_reduce(ls, scratch, false);  // its barriers also publish w[]

    const int dq = tid % DQ, jl = tid / DQ;
    const float4* accp = reinterpret_cast<const float4*>(p.ws_acc + base * D) + dq;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int j = jl; j < ns; j += J) {
        const float wj = w[j];
        const float4 v = accp[(size_t)j * DQ];
        a.x = fmaf(wj, v.x, a.x);
        a.y = fmaf(wj, v.y, a.y);
        a.z = fmaf(wj, v.z, a.z);
        a.w = fmaf(wj, v.w, a.w);
    }
    reinterpret_cast<float4*>(part + jl * D)[dq] = a;
    __syncthreads();
    const float inv = L > 0.f ? 1.f / L : 0.f;
    OT* out = static_cast<OT*>(p.out) + ((size_t)b * p.Hq + h) * D;
    for (int d = tid; d < D; d += kMergeThreads) {
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < J; ++r) s += part[r * D + d];
        store_out<OT>(out + d, s * inv);
    }
}

template <typename OT, int D>
cudaError_t launch_merge_t(const MergeParams& p, cudaStream_t s) {
    constexpr int J = kMergeThreads / (D / 4);
    const size_t smem = (size_t)((p.max_splits + 3) & ~3) * 4 + (size_t)J * D * 4;
    auto kern = merge_kernel<OT, D>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<dim3(p.Hq, p.B), kMergeThreads, smem, s>>>(p);
    return cudaGetLastError();
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
