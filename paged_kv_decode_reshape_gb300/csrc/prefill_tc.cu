// prefill_tc.cu -- paged (chunked, variable-length) prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM), head_dim 128, bf16.
//
// "EchoLLMServing inference framework notes", section 2: FlashAttention for prefill tiles the
// queries by BLOCK_M and keeps the working set on chip; section 3: chunked prefill and mixed
// batches. "LLM Primer VI, Chapter 8", section 8.1: K and V are gathered through the block table.
// Sequence b's L_b query tokens are the last L_b of its context (written to the cache first);
// query row i attends causally to the first n_b - (L_b - 1 - i) tokens.
//
// One CTA computes the same 128 query rows for two query heads of one GQA group (tiles A and B):
// both read every K/V tile once and have the same causal extent, so their work stays in step.
// Warp roles (320 threads):
//   warps 0-3  softmax of tile A: thread r owns query row r (TMEM lane r)
//   warps 4-7  softmax of tile B
//   warp 8     lane 0 issues every tcgen05.mma and commit; the warp owns the TMEM allocation
//   warp 9     producer: block ids from the table, 2-D TMA copies of 64-key K/V tiles (four pool
//              blocks) into a STAGES-deep ring
// Per key tile t, the tensor core runs, in this order,
//   PV_A(t-1 -> t): O_A += P_A . V_t ;  S_A(t+1) = Q_A . K_{t+1}^T ;  O_B += P_B . V_t ;
//   S_B(t+1) = Q_B . K_{t+1}^T
// so that while one tile's softmax warps turn S into P, the tensor core works on the other tile.
// TMEM columns: O_A 0-127, O_B 128-255, S_A 256-319, S_B 320-383. A commit after S_X(t+1) also
// covers PV_X(t) (commits track every earlier MMA of the issuing thread), so when softmax X sees
// S_X(t+1) it may overwrite P_X and rescale O_X. The running max is raised lazily (only when a
// tile exceeds it by more than 2^8), so O is rarely rescaled; at the end thread r divides its O
// row by its sum.
#include <cuda.h>

#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kPfQ = 128;                      // query rows per tile (MMA M)
constexpr int kPfK = 64;                       // keys per tile
constexpr int kPfQBytes = 2 * kPfQ * 128;      // Q: two 64-dim halves of [128 rows x 128 B]
constexpr int kPfPBytes = kPfQ * 128;          // P: [128 rows x 64 keys] bf16
constexpr int kPfHalf = kPfK * 128;            // one 64-dim half of a K or V tile
constexpr int kPfStage = 4 * kPfHalf;          // K half 0, K half 1, V half 0, V half 1
#ifndef PKV_PF_STAGES
#define PKV_PF_STAGES 4
#endif
constexpr int kPfStages = PKV_PF_STAGES;
constexpr int kPfOffP = 2 * kPfQBytes;         // Q_A, Q_B, then P_A, P_B
constexpr int kPfOffKV = kPfOffP + 2 * kPfPBytes;
constexpr int kPfOffBar = kPfOffKV + kPfStages * kPfStage;
// barriers: kv_full[S], kv_empty[S], s_full[2 tiles][2 buffers], p_full[2], pv_done[2], o_done,
// drain; then the TMEM slot
constexpr int kPfNumBars = 2 * kPfStages + 10;
constexpr int kPfSmem = 1024 + kPfOffBar + kPfNumBars * 8 + 16;
constexpr int kPfThreads = 320;
constexpr int kPfMmaWarp = 8, kPfLoadWarp = 9;
constexpr uint32_t kPfTmemCols = 512;
constexpr uint32_t kOCol = 0, kSCol = 256;     // O_X at 128 X, S_X buffer u at 256 + 128 X + 64 u
constexpr float kPfRescale = 8.0f;             // log2 units
static_assert(kPfSmem <= 227 * 1024, "shared memory");
static_assert(kPfStages >= 3, "S of tile t + 2 is computed while tile t still holds its stage");

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

__device__ __forceinline__ bool aborted(const volatile int* f) { return *f != 0; }

__device__ __forceinline__ int lane_of() { return threadIdx.x & 31; }

__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const PrefillParams p,
                                                                const __grid_constant__ CUtensorMap tmk,
                                                                const __grid_constant__ CUtensorMap tmv) {
    grid_dependency_wait();
    // heaviest query tiles (most keys under the causal mask) first
    const int qt = gridDim.x - 1 - blockIdx.x, b = blockIdx.z;
    const int HP = (p.G + 1) / 2;                       // head pairs per kv head
    const int kvh = blockIdx.y / HP, hp = blockIdx.y - kvh * HP;
    const bool two = 2 * hp + 1 < p.G;                  // tile B exists
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q0 = p.query_start[b];
    const int L = p.query_start[b + 1] - q0;
    if (qt * kPfQ >= L) return;
    const int n = p.context_lens[b];
    if (n < L || n > p.MBPS * kBlockSize) {
        if (tid == 0 && qt == 0 && blockIdx.y == 0) flag(p.status, PKV_FLAG_BAD_CONTEXT);
        return;
    }
    const int first_visible = n - L + 1;                          // keys visible to query row 0
    const int rows = min(kPfQ, L - qt * kPfQ);
    const int n_tile_max = first_visible + qt * kPfQ + rows - 1;  // keys visible to the last row
    const int ntiles = (n_tile_max + kPfK - 1) / kPfK;
    const int32_t* bt_row = p.block_tables + (size_t)b * p.MBPS;
    // Block ids come in windows of 32 (8 key tiles), lane j holding block 32 w + j (-1: not needed
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
    const uint32_t skv = sbase + kPfOffKV;
    const uint32_t bar0 = sbase + kPfOffBar;
    auto kv_full = [&](int s) { return bar0 + 8 * s; };
    auto kv_empty = [&](int s) { return bar0 + 8 * (kPfStages + s); };
    auto s_full = [&](int x, int u) { return bar0 + 8 * (2 * kPfStages + 2 * x + u); };
    auto p_full = [&](int x) { return bar0 + 8 * (2 * kPfStages + 4 + x); };
    auto pv_done = [&](int x) { return bar0 + 8 * (2 * kPfStages + 6 + x); };
    const uint32_t o_done = bar0 + 8 * (2 * kPfStages + 8);
    const uint32_t drain = bar0 + 8 * (2 * kPfStages + 9);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPfOffBar + kPfNumBars * 8);
    __shared__ int abort_flag;

    if (tid == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x, 0), 1);
            mbar_init(s_full(x, 1), 1);
            mbar_init(p_full(x), kPfQ);
            mbar_init(pv_done(x), 1);
        }
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kPfMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kPfTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // ---- Q tiles: softmax thread r of tile X writes query row r (zeros past the sequence's queries) ----
    const int gx = warp >> 2;              // softmax group (tile) of warps 0-7
    const int r = tid & 127;               // its row / TMEM lane
    const int i = qt * kPfQ + r;
    const bool row_valid = i < L;
    if (warp < 8 && (gx == 0 || two)) {
        const int h = kvh * p.G + 2 * hp + gx;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                          ((size_t)(q0 + (row_valid ? i : 0)) * p.Hq + h) * 128);
        unsigned char* qs = smem + gx * kPfQBytes;
#pragma unroll
        for (int c = 0; c < 16; ++c) {  // 16-byte chunk c = dims 8c .. 8c+7
            const uint4 v = row_valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t off = (c >> 3) * (kPfQ * 128) + r * 128 + ((((c & 7) ^ (r & 7))) << 4);
            *reinterpret_cast<uint4*>(qs + off) = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kPfLoadWarp) {
        // ---------------- producer ----------------
        int issued = 0;
        int ids_cur = load_window(0, true), ids_next = has_window(1) ? load_window(1, true) : -1;
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % kPfStages;
            if (t > 0 && (t & 7) == 0) {
                ids_cur = ids_next;
                ids_next = has_window((t >> 3) + 1) ? load_window((t >> 3) + 1, true) : -1;
            }
            const bool got = t < kPfStages || mbar_wait_bounded(kv_empty(st), ((t / kPfStages) - 1) & 1, 200);
            if (!__all_sync(0xffffffffu, got)) {  // warp-uniform exit
                if (lane == 0) { atomicExch(&abort_flag, 1); flag(p.status, PKV_FLAG_TIMEOUT); }
                break;
            }
            if (__any_sync(0xffffffffu, aborted(&abort_flag))) break;
            // lane jj < 4: the pool block of keys 64t + 16jj .. (-1 when not needed or invalid)
            int id = __shfl_sync(0xffffffffu, ids_cur, 4 * (t & 7) + (lane & 3));
            if (lane >= 4) id = -1;
            const unsigned valid = __ballot_sync(0xffffffffu, id >= 0);
            if (lane == 0) {
                const uint32_t bar = kv_full(st);
                if (valid == 0) {
                    mbar_arrive(bar);
                } else {
                    mbar_arrive_expect_tx(bar, __popc(valid) * 4 * (kBlockSize * 128));
                }
            }
            __syncwarp();
            if (lane < 4 && id >= 0) {
                const uint32_t bar = kv_full(st), dst = skv + st * kPfStage;
                const int row = (id * p.Hkv + kvh) * kBlockSize;
                const uint32_t o = lane * (kBlockSize * 128);
                tma_load_2d(dst + o, &tmk, 0, row, bar);
                tma_load_2d(dst + kPfHalf + o, &tmk, 64, row, bar);
                tma_load_2d(dst + 2 * kPfHalf + o, &tmv, 0, row, bar);
                tma_load_2d(dst + 3 * kPfHalf + o, &tmv, 64, row, bar);
            }
            issued = t + 1;
        }
        if (aborted(&abort_flag) && lane == 0) {
            // let this CTA's own copies land before shared memory goes away
            for (int t = issued - kPfStages < 0 ? 0 : issued - kPfStages; t < issued; ++t)
                mbar_wait_bounded(kv_full(t % kPfStages), (t / kPfStages) & 1);
        }
    } else if (warp == kPfMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(kPfQ, kPfK, false);
            constexpr uint32_t kIdescO = idesc_bf16(kPfQ, 128, true);
            auto issue_s = [&](int x, int t) {  // S_X(t) = Q_X . K_t^T into buffer t % 2
                const uint32_t kvs = skv + (t % kPfStages) * kPfStage;
                const uint32_t qs = sbase + x * kPfQBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = sdesc(qs + (ks >> 2) * (kPfQ * 128) + (ks & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc(kvs + (ks >> 2) * kPfHalf + (ks & 3) * 32, 16, 1024);
                    umma(tmem + kSCol + 128 * x + 64 * (t & 1), a, bd, kIdescS, ks > 0);
                }
                umma_commit(s_full(x, t & 1));
            };
            auto issue_pv = [&](int x, int t) {  // O_X += P_X . V_t
                const uint32_t kvs = skv + (t % kPfStages) * kPfStage;
                const uint32_t ps = sbase + kPfOffP + x * kPfPBytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = sdesc(ps + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc(kvs + 2 * kPfHalf + kk * (16 * 128), kPfHalf, 1024);
                    umma(tmem + kOCol + 128 * x, a, bd, kIdescO, (t > 0 || kk > 0) ? 1u : 0u);
                }
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
            // S of the first two tiles, then per tile t: the products of t once its P is ready, and
            // S of tile t + 2 into the buffer tile t has just released
            for (int t = 0; t < 2 && t < ntiles && ok; ++t) {
                if (!wait(kv_full(t % kPfStages), (t / kPfStages) & 1)) break;
                issue_s(0, t);
                if (two) issue_s(1, t);
            }
            for (int t = 0; t < ntiles && ok; ++t) {
                if (!wait(p_full(0), t & 1)) break;
                issue_pv(0, t);
                umma_commit(pv_done(0));
                if (two) {
                    if (!wait(p_full(1), t & 1)) break;
                    issue_pv(1, t);
                    umma_commit(pv_done(1));
                }
                umma_commit(kv_empty(t % kPfStages));  // every product that reads stage t is issued
                if (t + 2 < ntiles) {  // the S buffers tile t used are free (its P is written)
                    if (!wait(kv_full((t + 2) % kPfStages), ((t + 2) / kPfStages) & 1)) break;
                    issue_s(0, t + 2);
                    if (two) issue_s(1, t + 2);
                }
            }
            umma_commit(o_done);
            umma_commit(drain);
            mbar_wait_bounded(drain, 0);  // every issued product is done before TMEM may go away
        }
        __syncwarp();
    } else if (gx == 0 || two) {
        // ---------------- softmax of tile gx ----------------
        const uint32_t tl = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lane quadrant
        const uint32_t s_col = tmem + tl + kSCol + 128 * gx, o_col = tmem + tl + kOCol + 128 * gx;
        unsigned char* ps = smem + kPfOffP + gx * kPfPBytes;
        const int n_row = row_valid ? first_visible + i : 0;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // bit j of `present`: block 32 w + j of the current window is present (the producer's test)
        unsigned present = __ballot_sync(0xffffffffu, load_window(0, false) >= 0);
        int ids_next = has_window(1) ? load_window(1, false) : -1;
        for (int t = 0; t < ntiles; ++t) {
            if (t > 0 && (t & 7) == 0) {
                present = __ballot_sync(0xffffffffu, ids_next >= 0);
                ids_next = has_window((t >> 3) + 1) ? load_window((t >> 3) + 1, false) : -1;
            }
            const int mask = (present >> (4 * (t & 7))) & 0xF;
            const bool got = mbar_wait_bounded(s_full(gx, t & 1), (t >> 1) & 1);
            if (!__all_sync(0xffffffffu, got)) {  // warp-uniform exit
                atomicExch(&abort_flag, 1);
                flag(p.status, PKV_FLAG_TIMEOUT);
                ok = false;
                break;
            }
            if (__any_sync(0xffffffffu, aborted(&abort_flag))) { ok = false; break; }
            tc_fence_after();
            if (gx == 0) {
                // V rows of keys no row may see (past the context or in a missing block) must be
                // finite: their weights are 0, and 0 * NaN would poison O. Zero them. (The copy of
                // tile t has landed: S_A(t) was issued after it.)
                const int kr = r >> 1, half = r & 1;
                const int k = t * kPfK + kr;
                if (k >= n_tile_max || !((mask >> (kr >> 4)) & 1)) {
                    uint4* z = reinterpret_cast<uint4*>(smem + kPfOffKV + (t % kPfStages) * kPfStage +
                                                        (2 + half) * kPfHalf + kr * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) z[c] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            float s[64];
            {
                float t0[32], t1[32];
                tmem_ld32(s_col + 64 * (t & 1), t0);
                tmem_ld32(s_col + 64 * (t & 1) + 32, t1);
#pragma unroll
                for (int c = 0; c < 32; ++c) { s[c] = t0[c]; s[32 + c] = t1[c]; }
            }
            const int kbase = t * kPfK;
            if (kbase + kPfK <= n_row && mask == 0xF) {  // whole tile visible to this row
#pragma unroll
                for (int c = 0; c < 64; ++c) s[c] *= p.scale_log2;
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const bool vis = kbase + c < n_row && ((mask >> (c >> 4)) & 1);
                    s[c] = vis ? s[c] * p.scale_log2 : -INFINITY;
                }
            }
            float mx8[8];  // tree maximum: 8 independent chains, then 3 levels
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = s[e];
#pragma unroll
            for (int c = 8; c < 64; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
#pragma unroll
            for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                for (int e = 0; e < w; ++e) mx8[e] = fmaxf(mx8[e], mx8[e + w]);
            const float mx = mx8[0];
            const bool up = mx > m + kPfRescale;
            float alpha = 1.f;
            if (up) {
                alpha = ex2(m - mx);  // m == -inf: 0
                m = mx;
                l *= alpha;
            }
            const float ms = m == -INFINITY ? 0.f : m;
            // P_X and O_X may be touched once the previous tile's product is done
            bool pv_ready = t == 0;
            auto wait_pv = [&]() {
                if (!pv_ready) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(pv_done(gx), (t - 1) & 1))) {
                        atomicExch(&abort_flag, 1);
                        flag(p.status, PKV_FLAG_TIMEOUT);
                        ok = false;
                    }
                    tc_fence_after();
                    pv_ready = true;
                }
            };
            if (t > 0 && __any_sync(0xffffffffu, up)) {  // rescale this warp's O rows (rare)
                wait_pv();
                if (!ok) break;
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    float o[32];
                    tmem_ld32(o_col + c0, o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] *= alpha;
                    tmem_st32(o_col + c0, o);
                }
            }
            uint32_t pw[32];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float a0 = ex2(s[2 * c] - ms), a1 = ex2(s[2 * c + 1] - ms);
                ls[c & 3] += a0 + a1;
                pw[c] = pack2_bf16(a0, a1);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            wait_pv();
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 16-byte chunk j = keys 8j .. 8j+7 of row r
                const uint32_t off = r * 128 + ((j ^ (r & 7)) << 4);
                *reinterpret_cast<uint4*>(ps + off) = make_uint4(pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            mbar_arrive(p_full(gx));
        }
        if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(o_done, 0))) {
            atomicExch(&abort_flag, 1);
            flag(p.status, PKV_FLAG_TIMEOUT);
            ok = false;
        }
        tc_fence_after();
        if (ok && !__any_sync(0xffffffffu, aborted(&abort_flag))) {
            // ---- epilogue: row r of O / l -> out ----
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int h = kvh * p.G + 2 * hp + gx;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                  ((size_t)(q0 + (row_valid ? i : 0)) * p.Hq + h) * 128);
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                float o[32];
                tmem_ld32(o_col + c0, o);
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
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((max_query_len + kPfQ - 1) / kPfQ, p.Hkv * ((p.G + 1) / 2), p.B);
    return launch_pdl(prefill_kernel, grid, dim3(kPfThreads), kPfSmem, s, p, tk, tv);
}

}  // namespace pkv
