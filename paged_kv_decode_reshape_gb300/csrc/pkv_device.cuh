// pkv_device.cuh -- device-side building blocks shared by the libpkv kernels (sm_103a).
//
// Bulk (1-D TMA) copies global -> shared completed through an mbarrier transaction count, the
// bounded mbarrier wait every pipeline uses, and the element conversions the kernels need.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

// Every wait on an mbarrier gives up after this long (device globaltimer, ns): the kernel then
// flags PKV_FLAG_TIMEOUT, drains its own copies (bounded again) and returns.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy before any copy uses it.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Same test, but the warp may be suspended in hardware for up to `hint_ns` waiting for the phase
// (it resumes as soon as the phase completes), so a waiting warp does not spin on issue slots.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier to complete; false if kWaitLimitNs elapsed first. The
// clock is read once per 64 polls so the loop costs few issue slots. With `backoff_ns` > 0 the
// warp also sleeps between polls (for waits whose latency matters less than the issue slots
// they would take from other warps).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t backoff_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i) {
            if (mbar_try_wait_suspend(bar, parity, 1000000u)) return true;
            if (backoff_ns) __nanosleep(backoff_ns);
        }
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// 1-D bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from global memory
// into this CTA's shared memory; completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 2-D TMA tile load (box of the tensor map at coordinates (x, y)) into shared memory; the inner
// coordinate times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 3-D and 4-D tiled TMA copies (x, the innermost coordinate, is 0 in every caller).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two bf16 in one 32-bit word -> two floats (bf16 is the top half of a binary32).
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
}

// Four int8 in one word -> four floats, exactly. Method: bias each byte to unsigned (x + 128)
// by flipping its sign bit, place it in the low mantissa byte of the float 2^23, and subtract
// 2^23 + 128 (the byte-permute conversion of Kim et al., "Who Says Elephants Can't Run:
// Bringing Large Scale MoE Models into Cloud Scale Production", 2022). Tested against a plain
// conversion over all 256 byte values.
__device__ __forceinline__ void s8x4_to_f32(uint32_t w, float (&f)[4]) {
    const uint32_t u = w ^ 0x80808080u;
    const float bias = 8388736.0f;  // 2^23 + 128
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - bias;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - bias;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - bias;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - bias;
}

// Load 8 consecutive elements (16 B of bf16, 32 B of fp32, 8 B of int8) from shared memory and
// widen them to float.
template <typename T>
__device__ __forceinline__ void load8_f32(const unsigned char* p, float (&f)[8]);

template <>
__device__ __forceinline__ void load8_f32<float>(const unsigned char* p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 16);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <>
__device__ __forceinline__ void load8_f32<__nv_bfloat16>(const unsigned char* p, float (&f)[8]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    bf16x2_to_f32(a.x, f[0], f[1]);
    bf16x2_to_f32(a.y, f[2], f[3]);
    bf16x2_to_f32(a.z, f[4], f[5]);
    bf16x2_to_f32(a.w, f[6], f[7]);
}

template <>
__device__ __forceinline__ void load8_f32<int8_t>(const unsigned char* p, float (&f)[8]) {
    const uint2 a = *reinterpret_cast<const uint2*>(p);
    float lo[4], hi[4];
    s8x4_to_f32(a.x, lo);
    s8x4_to_f32(a.y, hi);
#pragma unroll
    for (int i = 0; i < 4; ++i) { f[i] = lo[i]; f[4 + i] = hi[i]; }
}

// Same, from global memory (q vectors).
template <typename T>
__device__ __forceinline__ void gload8_f32(const void* p, float (&f)[8]) {
    load8_f32<T>(reinterpret_cast<const unsigned char*>(p), f);
}

template <typename T>
__device__ __forceinline__ void store_out(T* p, float v);

template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) { *p = v; }

template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

// Programmatic dependent launch: every kernel of this library is launched so that it may start
// while the kernel before it in the stream is finishing. grid_dependency_wait() blocks until that
// kernel has completed and its memory is visible -- each kernel calls it before its first read of
// anything a previous kernel may have written. grid_dependents_launch() lets the next kernel in
// the stream begin launching once every CTA of this one has called it or exited.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void flag(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace pkv
