// prefill_tc.cu -- paged (chunked, variable-length) prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM), head_dim 128, bf16.
//
// "EchoLLMServing inference framework notes", section 2: FlashAttention for prefill tiles the
// queries by BLOCK_M and keeps the working set on chip; section 3: chunked prefill and mixed
// batches. "LLM Primer VI, Chapter 8", section 8.1: K and V are gathered through the block table.
// Sequence b's L_b query tokens are the last L_b of its context (written to the cache first);
// query row i attends causally to the first n_b - (L_b - 1 - i) tokens.
//
// One CTA (4 warps) computes 128 query rows of one query head. The Q tile sits in shared memory
// (K-major, 128-byte swizzle). K and V of 64-token key tiles -- four 16-token pool blocks -- come
// in by TMA through the block table into a 2-stage ring. Per key tile:
//   S[128 x 64]  = Q[128 x 128] . K^T     one thread issues 8 tcgen05.mma (k = 16), D in TMEM
//   thread r reads row r of S from TMEM (tcgen05.ld), masks it (causal limit, context, missing
//   blocks), keeps its own running max and sum (the max is raised lazily, by more than 2^8 only;
//   O is rescaled in TMEM when it is), and writes its bf16 weights as row r of P in shared memory
//   O[128 x 128] += P[128 x 64] . V      4 tcgen05.mma, V read MN-major from its natural layout
// tcgen05.commit signals each product on an mbarrier; the next tile's copy starts as soon as the
// product that read its stage is done. At the end thread r divides its O row by its sum.
#include <cuda.h>

#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kPfQ = 128;                      // query rows per CTA (MMA M)
constexpr int kPfK = 64;                       // keys per tile
constexpr int kPfQBytes = 2 * kPfQ * 128;      // Q: two 64-dim halves of [128 rows x 128 B]
constexpr int kPfPBytes = kPfQ * 128;          // P: [128 rows x 64 keys] bf16
constexpr int kPfHalf = kPfK * 128;            // one 64-dim half of a K or V tile
constexpr int kPfStage = 4 * kPfHalf;          // K half 0, K half 1, V half 0, V half 1
constexpr int kPfStages = 2;
constexpr int kPfOffP = kPfQBytes;
constexpr int kPfOffKV = kPfQBytes + kPfPBytes;
constexpr int kPfOffBar = kPfOffKV + kPfStages * kPfStage;
constexpr int kPfSmem = 1024 + kPfOffBar + 128;
constexpr uint32_t kPfTmemCols = 256;          // O: columns 0..127, S: 128..191
constexpr uint32_t kOCol = 0, kSCol = 128;
constexpr float kPfRescale = 8.0f;             // log2 units

// Shared-memory matrix descriptor (tcgen05): start address, leading / stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major, B K-major or
// MN-major, N and M.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(128) prefill_kernel(const PrefillParams p,
                                                      const __grid_constant__ CUtensorMap tmk,
                                                      const __grid_constant__ CUtensorMap tmv) {
    grid_dependency_wait();
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int q0 = p.query_start[b];
    const int L = p.query_start[b + 1] - q0;
    if (qt * kPfQ >= L) return;
    const int n = p.context_lens[b];
    if (n < L || n > p.MBPS * kBlockSize) {
        if (tid == 0 && qt == 0 && h == 0) flag(p.status, PKV_FLAG_BAD_CONTEXT);
        return;
    }
    const int first_visible = n - L + 1;                       // keys visible to query row 0
    const int rows = min(kPfQ, L - qt * kPfQ);
    const int n_tile_max = first_visible + qt * kPfQ + rows - 1;  // keys visible to the last row
    const int ntiles = (n_tile_max + kPfK - 1) / kPfK;
    const int kvh = h / p.G;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sq = smem_addr(smem), sp = sq + kPfOffP, skv = sq + kPfOffKV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPfOffBar);  // full[2], s, o
    const uint32_t full0 = smem_addr(bars), bar_s = full0 + 16, bar_o = full0 + 24;
    int32_t* tile_mask = reinterpret_cast<int32_t*>(smem + kPfOffBar + 32);  // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPfOffBar + 48);
    __shared__ int abort_flag;

    if (tid == 0) {
        mbar_init(full0, 1);
        mbar_init(full0 + 8, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kPfTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quadrant

    // ---- Q tile: row tid is query i of the sequence (zeros past its queries) ----
    const int i = qt * kPfQ + tid;
    const bool row_valid = i < L;
    const int n_row = row_valid ? first_visible + i : 0;
    {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                          ((size_t)(q0 + (row_valid ? i : 0)) * p.Hq + h) * 128);
#pragma unroll
        for (int c = 0; c < 16; ++c) {  // 16-byte chunk c = dims 8c .. 8c+7
            const uint4 v = row_valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t off = (c >> 3) * (kPfQ * 128) + tid * 128 + ((((c & 7) ^ (tid & 7))) << 4);
            *reinterpret_cast<uint4*>(smem + off) = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }

    // ---- producer (thread 0): key tile kt -> stage kt % 2 ----
    const int32_t* bt_row = p.block_tables + (size_t)b * p.MBPS;
    auto issue = [&](int kt) {
        const int st = kt & 1;
        const uint32_t bar = full0 + 8 * st;
        const uint32_t dst = skv + st * kPfStage;
        int mask = 0, nvalid = 0, ids[4];
        for (int jj = 0; jj < 4; ++jj) {
            const int j = kt * 4 + jj;
            ids[jj] = -1;
            if (j * kBlockSize < n_tile_max) {
                const int id = bt_row[j];
                if (id >= 0 && id < p.NB) {
                    ids[jj] = id;
                    mask |= 1 << jj;
                    ++nvalid;
                } else {
                    flag(p.status, PKV_FLAG_BAD_BLOCK);
                }
            }
        }
        tile_mask[st] = mask;
        if (nvalid == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, nvalid * 4 * (kBlockSize * 128));
        for (int jj = 0; jj < 4; ++jj) {
            if (ids[jj] < 0) continue;
            const int row = (ids[jj] * p.Hkv + kvh) * kBlockSize;
            const uint32_t o = jj * (kBlockSize * 128);
            tma_load_2d(dst + o, &tmk, 0, row, bar);
            tma_load_2d(dst + kPfHalf + o, &tmk, 64, row, bar);
            tma_load_2d(dst + 2 * kPfHalf + o, &tmv, 0, row, bar);
            tma_load_2d(dst + 3 * kPfHalf + o, &tmv, 64, row, bar);
        }
    };
    if (tid == 0) {
        issue(0);
        if (ntiles > 1) issue(1);
    }

    constexpr uint32_t kIdescS = idesc_bf16(kPfQ, kPfK, false);
    constexpr uint32_t kIdescO = idesc_bf16(kPfQ, 128, true);
    float m = -INFINITY, l = 0.f;
    int issued_s = 0, issued_o = 0;  // products issued (for the drain on abort)
    bool failed = false;

    for (int kt = 0; kt < ntiles; ++kt) {
        const int st = kt & 1;
        const uint32_t kvs = skv + st * kPfStage;
        if (!mbar_wait_bounded(full0 + 8 * st, (kt >> 1) & 1)) failed = true;
        if (__syncthreads_or(failed)) break;
        const int mask = tile_mask[st];
        // V rows of keys no row may see (past the context or in a missing block) must be finite:
        // their weights are 0, and 0 * NaN would poison O. Zero them.
        {
            const int r = tid >> 1, half = tid & 1;
            const int k = kt * kPfK + r;
            if (k >= n_tile_max || !((mask >> (r >> 4)) & 1)) {
                uint4* z = reinterpret_cast<uint4*>(smem + kPfOffKV + st * kPfStage + (2 + half) * kPfHalf + r * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c) z[c] = make_uint4(0u, 0u, 0u, 0u);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {  // S = Q . K^T
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t a = sdesc(sq + (ks >> 2) * (kPfQ * 128) + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc(kvs + (ks >> 2) * kPfHalf + (ks & 3) * 32, 16, 1024);
                umma(tmem + kSCol, a, bd, kIdescS, ks > 0);
            }
            umma_commit(bar_s);
        }
        ++issued_s;
        if (!mbar_wait_bounded(bar_s, kt & 1)) failed = true;
        tc_fence_after();
        float s[64];
        {
            float t0[32], t1[32];
            tmem_ld32(tmem + tlane + kSCol, t0);
            tmem_ld32(tmem + tlane + kSCol + 32, t1);
#pragma unroll
            for (int c = 0; c < 32; ++c) { s[c] = t0[c]; s[32 + c] = t1[c]; }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const int k = kt * kPfK + c;
            const bool ok = k < n_row && ((mask >> (c >> 4)) & 1);
            s[c] = ok ? s[c] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, s[c]);
        }
        const bool up = mx > m + kPfRescale;
        float alpha = 1.f;
        if (up) {
            alpha = ex2(m - mx);  // m == -inf: 0
            m = mx;
            l *= alpha;
        }
        const float ms = m == -INFINITY ? 0.f : m;
        // the previous P . V must be done before P, O or its stage are touched again
        if (kt > 0) {
            if (!mbar_wait_bounded(bar_o, (kt - 1) & 1)) failed = true;
            tc_fence_after();
            if (tid == 0 && kt + 1 < ntiles && !failed) issue(kt + 1);
        }
        uint32_t pw[32];
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const float a0 = ex2(s[2 * c] - ms), a1 = ex2(s[2 * c + 1] - ms);
            lsum += a0 + a1;
            pw[c] = pack2_bf16(a0, a1);
        }
        l += lsum;
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // 16-byte chunk j = keys 8j .. 8j+7 of row tid
            const uint32_t off = kPfOffP + tid * 128 + ((j ^ (tid & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + off) = make_uint4(pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
        }
        if (kt > 0 && __any_sync(0xffffffffu, up)) {  // rescale this warp's O rows (rare)
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                float o[32];
                tmem_ld32(tmem + tlane + kOCol + c0, o);
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] *= alpha;
                tmem_st32(tmem + tlane + kOCol + c0, o);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        if (__syncthreads_or(failed)) break;
        tc_fence_after();
        if (tid == 0) {  // O += P . V
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = sdesc(sp + kk * 32, 16, 1024);
                const uint64_t bd = sdesc(kvs + 2 * kPfHalf + kk * (16 * 128), kPfHalf, 1024);
                umma(tmem + kOCol, a, bd, kIdescO, (kt > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(bar_o);
        }
        ++issued_o;
    }

    if (!failed && issued_o > 0 && !mbar_wait_bounded(bar_o, (issued_o - 1) & 1)) failed = true;
    tc_fence_after();
    if (__syncthreads_or(failed)) {
        if (tid == 0) {
            atomicExch(&abort_flag, 1);
            flag(p.status, PKV_FLAG_TIMEOUT);
            // let in-flight products and copies finish before TMEM and shared memory go away
            if (issued_s > 0) mbar_wait_bounded(bar_s, (issued_s - 1) & 1);
            if (issued_o > 0) mbar_wait_bounded(bar_o, (issued_o - 1) & 1);
            for (int kt = 0; kt < ntiles && kt < 2 + issued_o; ++kt) mbar_wait_bounded(full0 + 8 * (kt & 1), (kt >> 1) & 1);
        }
    } else {
        // ---- epilogue: row tid of O / l -> out ----
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                              ((size_t)(q0 + (row_valid ? i : 0)) * p.Hq + h) * 128);
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
            float o[32];
            tmem_ld32(tmem + tlane + kOCol + c0, o);
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
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPfTmemCols)
                     : "memory");
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           int max_query_len, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((max_query_len + kPfQ - 1) / kPfQ, p.Hq, p.B);
    return launch_pdl(prefill_kernel, grid, dim3(128), kPfSmem, s, p, tk, tv);
}

}  // namespace pkv
