// gdn_ut.cu -- chunk-prep kernels of the forward pass: for every chunk of
// C = 64 tokens of every (sequence, head), with g_r = sum_{i<=r} log_alpha_i
// inside the chunk,
//
//   A_rs = beta_r exp(g_r - g_s) (k_r . k_s)   for s < r, else 0
//   T_u  = (I + A)^{-1} diag(beta),   T_w = (I + A)^{-1} diag(beta gamma)
//
// ("Gated DeltaNet GPU并行实现", section 3.2: everything inside a chunk is
// parallel; the serial state pass needs only the chunk's WY factors
// U = T_u V and W = T_w K.)  Two kernels, one per output form:
//   - k_gdn_ut: T_u and T_w as bf16 in a per-chunk layout [H][chunk_slots]
//     [T_u | T_w][64][64] (dense: slot n * max_chunks + c; packed:
//     floor(cu[n] / 64) + n + c), one bulk-copy box each, for the fused kernel
//     (gdn_fused.cu), which forms W and U on its own tensor cores;
//   - k_gdn_utw, the forward's default: T_u as [rows][64] and W = T_w K as
//     [rows][d_k], bf16, rows indexed like the token rows of the inputs, for
//     the chain kernel (gdn_tc.cu).  W comes from a second tcgen05 product on
//     the staged K tile.
// Rows and columns of tokens past a sequence's end are zero, because beta and
// log_alpha are zero there.
//
// Per unit (chunk, head): the K tile arrives by bulk tensor copy (128-byte
// swizzle), one thread issues the Gram K K^T as tcgen05 MMAs into tensor
// memory (M = 128: rows 64-127 of the operand are whatever follows the tile and
// are never read), four warps read its rows, form A and invert I + A
// (gdn_inv.cuh).  k_gdn_utw then stages T_w (bf16, swizzled) and issues
// W^T = K^T T_w^T (M = d_k lanes, N = 64 tokens) into the unit's Gram
// columns, reads it back, transposes it through shared memory and stores W
// rows.  Both are persistent: each CTA walks units b, b + grid, ... with two K
// buffers and two accumulators in flight.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "gdn_inv.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

// Optional per-CTA timing for profiling builds (-DGDN_TRACE_TIMELINE):
// start and end clock64(), SM and units of every CTA, read back with
// gdn_ut_trace_read().  Compiled out otherwise.
#ifdef GDN_TRACE_TIMELINE
__device__ long long g_ut_cta[2048][4];
__device__ long long g_ut_phase[16][8];   // CTA 0: per local unit, phase stamps
extern "C" int gdn_ut_trace_read(long long *out) {
    return (int)cudaMemcpyFromSymbol(out, g_ut_cta, sizeof(g_ut_cta));
}
extern "C" int gdn_ut_phase_read(long long *out) {
    return (int)cudaMemcpyFromSymbol(out, g_ut_phase, sizeof(g_ut_phase));
}
#define UTRACE(i, ev)                                                       \
    do {                                                                    \
        if (blockIdx.x == 0 && tid == 0 && (i) < 16) g_ut_phase[i][ev] = clock64(); \
    } while (0)
#else
#define UTRACE(i, ev) \
    do {              \
    } while (0)
extern "C" int gdn_ut_debug_ctas();
#endif

namespace gdn {
namespace {

using namespace ptx;
using namespace tcx;
using inv::LDA;

constexpr int kU = 64;
constexpr int kThreadsU = 160;   // warps 0-3 compute, warp 4 copies and issues the Gram

enum {
    U_FULL = 0,        // + buffer: K tile landed, raw gates staged (TMA tx + 32 lanes)
    U_EMPTY = 2,       // + buffer: the tile's MMAs are done (commits) and the gates
                       //   were copied
    U_GDONE = 4,       // + buffer: Gram in tensor memory (commit)
    U_GFREE = 6,       // + buffer: its tensor-memory columns read (A formed)
    U_DRAIN = 8,
    U_COUNT
};

template <int DK>
struct ULay {
    static constexpr int KB = DK / 64;
    static constexpr int SZ_K = KB * 8192;
    static constexpr int OFF_K = 0;                       // + b * SZ_K
    // the Gram's 128-row operand of the last tile's last block reads the 8 KB
    // after the tiles (A's buffer) as its unused rows
    static constexpr int OFF_A = 2 * SZ_K;                // fp32 [64][LDA]
    static constexpr int OFF_T = OFF_A + kU * LDA * 4;    // fp32 [64][LDA]
    static constexpr int OFF_RG = OFF_T + kU * LDA * 4;   // + b * 512: raw log_alpha[64], beta[64]
    static constexpr int OFF_GS = OFF_RG + 2 * 512;       // g, beta, gamma, 1/gamma [64]
    static constexpr int OFF_BAR = OFF_GS + 1024;
    static constexpr int OFF_MISC = OFF_BAR + U_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 16;
    static constexpr int ALLOC = TOTAL + 1024;
    static_assert(kU * LDA * 4 >= 8192, "the last tile's unused operand rows stay in bounds");
    static_assert(OFF_A % 1024 == 0 && OFF_RG % 16 == 0, "align");
};

struct UtParams {
    SeqMap sm;
    const float *log_alpha, *beta;
    const int2 *table;        // packed batches: (sequence, chunk) of every chunk slot
    // per-chunk blocks [H][chunk_slots][2][64][64] of T_u, T_w (k_gdn_ut); or
    // T_u as [rows][64] indexed like the token rows of the inputs (k_gdn_utw)
    __nv_bfloat16 *Tu;
    __nv_bfloat16 *W;         // k_gdn_utw: W = T_w K as [rows][d_k]
    int *err;
    int max_chunks;
    int chunk_slots;
    long long units;          // H * chunk_slots
    uint32_t wait_limit;
};

// Where unit u lives: its output block, the copy coordinates of its first
// token row, its first row in the [rows] gate arrays and its token count
// (0: a slot with no chunk; its output block is never read).
struct Unit {
    long long out_row;   // first row of the unit's [2][64][64] block
    long long row0;
    int y, z, len;
};

__device__ __forceinline__ Unit decode(const UtParams &p, long long u) {
    Unit r{0, 0, 0, 0, 0};
    const int slot = (int)(u % p.chunk_slots), h = (int)(u / p.chunk_slots);
    int n, c;
    if (p.table) {
        const int2 e = p.table[slot];
        n = e.x;
        c = e.y;
        if (n < 0) return r;
    } else {
        n = slot / p.max_chunks;
        c = slot % p.max_chunks;
    }
    if (p.sm.cu) {
        const int a = __ldg(p.sm.cu + n), b = __ldg(p.sm.cu + n + 1);
        if (!(a >= 0 && a <= b && b <= p.sm.T_total)) return r;   // reported by the table kernel
        const int t0 = c * kU;
        if (t0 >= b - a) return r;
        r.len = min(kU, b - a - t0);
        // storage slot of (n, c): floor(cu[n] / 64) + n + c, unique per sequence chunk
        r.out_row = ((long long)h * p.chunk_slots + a / kU + n + c) * 2 * kU;
        r.row0 = (long long)h * p.sm.T_total + a + t0;
        r.y = a + t0;
        r.z = h;
    } else {
        const int t0 = c * kU;
        if (t0 >= p.sm.T) return r;
        r.len = min(kU, p.sm.T - t0);
        r.out_row = u * 2 * kU;
        r.row0 = ((long long)n * p.sm.H + h) * (long long)p.sm.T + t0;
        r.y = t0;
        r.z = n * p.sm.H + h;
    }
    return r;
}

template <int DK>
__global__ void __launch_bounds__(kThreadsU, 3)
k_gdn_ut(const __grid_constant__ CUtensorMap tm_k, UtParams p) {
    using L = ULay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *Ab = reinterpret_cast<float *>(sm + L::OFF_A);
    float *Tb = reinterpret_cast<float *>(sm + L::OFF_T);
    float *gs = reinterpret_cast<float *>(sm + L::OFF_GS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef GDN_TRACE_TIMELINE
    if (tid == 0 && blockIdx.x < 2048) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_ut_cta[blockIdx.x][0] = clock64();
        g_ut_cta[blockIdx.x][2] = smid;
    }
#endif
    const long long nunits =
        blockIdx.x < p.units ? (p.units - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (warp == 4) {
        tmem_alloc(misc, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < U_COUNT; ++i) mbar_init(bar + i, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar + U_FULL + b, 33);
            mbar_init(bar + U_EMPTY + b, 2);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};
    // token rows of the inputs (element counts for the bounds-check build)
    const long long nrows =
        p.sm.cu ? (long long)p.sm.H * p.sm.T_total : (long long)p.sm.N * p.sm.H * p.sm.T;
    (void)nrows;

    if (warp == 4) {
        // ================================ copies (all lanes) and Gram (lane 0)
        if (lane == 0) prefetch_tmap(&tm_k);
        constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);
        const uint32_t sb = smem_u32(sm);
        auto load = [&](long long i) -> bool {
            const int b = (int)(i & 1);
            const bool ok = i < 2 || ctl.wait(U_EMPTY + b, (uint32_t)(((i >> 1) - 1) & 1));
            if (!__all_sync(0xffffffffu, ok)) return false;
            const Unit un = decode(p, blockIdx.x + i * gridDim.x);
            if (lane == 0) {
                mbar_arrive_expect_tx(bar + U_FULL + b, (uint32_t)L::SZ_K);
#pragma unroll
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_3d(sm + L::OFF_K + b * L::SZ_K + kb * 8192, &tm_k, bar + U_FULL + b,
                                kb * 64, un.y, un.z);
            }
            float *rg = reinterpret_cast<float *>(sm + L::OFF_RG + b * 512);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = lane + 32 * h;
                const bool in = r < un.len && GDN_IDX_OK(un.row0 + r, 1, nrows);
                rg[r] = in ? __ldg(p.log_alpha + un.row0 + r) : 0.f;
                rg[64 + r] = in ? __ldg(p.beta + un.row0 + r) : 0.f;
            }
            mbar_arrive(bar + U_FULL + b);
            return true;
        };
        auto gram = [&](long long i) -> bool {
            const int b = (int)(i & 1);
            bool ok = ctl.wait(U_FULL + b, (uint32_t)((i >> 1) & 1));
            if (ok && i >= 2) ok = ctl.wait(U_GFREE + b, (uint32_t)(((i >> 1) - 1) & 1));
            if (!ok) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const uint32_t off = L::OFF_K + b * L::SZ_K + (kk >> 2) * 8192 + (kk & 3) * 32;
                const uint64_t d = make_sdesc(sb + off, 16, 1024, kSwizzle128B);
                mma_bf16(tmem + 64 * b, d, d, idG, kk > 0);
            }
            mma_commit(bar + U_GDONE + b);
            mma_commit(bar + U_EMPTY + b);
            return true;
        };
        long long loaded = 0;
        bool ok = true;
        for (long long i = 0; ok && i < nunits && i < 2; ++i) ok = load(i), loaded = i + 1;
        for (long long i = 0; ok && i < nunits; ++i) {
            int okg = 1;
            if (lane == 0) okg = gram(i);
            ok = __shfl_sync(0xffffffffu, okg, 0) != 0;
            if (ok && i + 2 < nunits) ok = load(i + 2), loaded = i + 3;
        }
        if (lane == 0) {
            // every issued MMA and copy has finished before the CTA leaves
            mma_commit(bar + U_DRAIN);
            mbar_wait(bar + U_DRAIN, 0, ctl.limit);
            if (*abort_flag)
                for (long long i = loaded > 2 ? loaded - 2 : 0; i < loaded; ++i)
                    mbar_wait(bar + U_FULL + (i & 1), (uint32_t)((i >> 1) & 1), ctl.limit);
        }
    } else {
        // ============================================= compute (warps 0-3)
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        auto bar128 = [] { named_bar(1, 128); };
        for (long long i = 0; i < nunits; ++i) {
            const int b = (int)(i & 1);
            const Unit un = decode(p, blockIdx.x + i * gridDim.x);
            // ---- gates: g = in-chunk cumsum of log_alpha, beta (zero past the end)
            if (!named_bar_and(1, 128, ctl.wait(U_FULL + b, (uint32_t)((i >> 1) & 1)))) break;
            UTRACE(i, 0);
            if (warp == 0) {
                const float *rg = reinterpret_cast<const float *>(sm + L::OFF_RG + b * 512);
                float x0 = rg[lane], x1 = rg[32 + lane];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y0 = __shfl_up_sync(0xffffffffu, x0, off);
                    const float y1 = __shfl_up_sync(0xffffffffu, x1, off);
                    if (lane >= off) {
                        x0 += y0;
                        x1 += y1;
                    }
                }
                x1 += __shfl_sync(0xffffffffu, x0, 31);
                gs[lane] = x0;
                gs[32 + lane] = x1;
                gs[64 + lane] = rg[64 + lane];
                gs[96 + lane] = rg[96 + lane];
                gs[128 + lane] = __expf(x0);
                gs[160 + lane] = __expf(x1);
                // used only when the chunk's decay span is moderate (g_C > -80)
                gs[192 + lane] = __expf(-x0);
                gs[224 + lane] = __expf(-x1);
            }
            // ---- A from the Gram rows (lanes 0-63): warps 0-1; warps 2-3 clear
            //      T's upper diagonal blocks.  Every thread finished reading the
            //      previous unit's T before this barrier.
            const bool okg = ctl.wait(U_GDONE + b, (uint32_t)((i >> 1) & 1));
            if (!named_bar_and(1, 128, okg)) break;
            UTRACE(i, 1);
            if (tid == 0) mbar_arrive(bar + U_EMPTY + b);   // gates copied
            __syncwarp();
            tc_fence_after();
            if (warp < 2) {
                const int r = tid;
                uint32_t g0[32], g1[32];
                tmem_ld32(tmem + lane_base + 64 * b, g0);
                tmem_ld32(tmem + lane_base + 64 * b + 32, g1);
                const float gr = gs[r], br = gs[64 + r];
                tmem_wait32(g0);
                tmem_wait32(g1);
                // A_rs = beta_r exp(g_r - g_s) G_rs for s < r: as
                // (beta_r gamma_r) exp(-g_s) G_rs when the chunk's decay span
                // is moderate, else one exponential per entry (never above 1).
                // Entries outside the 16x16 diagonal blocks are rounded to tf32
                // for the merges.
                // (a uniform branch: the common case computes no exponential)
                const bool span_ok = gs[63] > -80.f;
                const float bgr = br * gs[128 + r];
                auto form = [&](auto factor) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = 4 * q + e;
                            const float gv = f32(s < 32 ? g0[s] : g1[s - 32]);
                            const float x = s < r ? factor(s) * gv : 0.f;
                            v[e] = (r >> 4) != (s >> 4) ? inv::tf32(x) : x;
                        }
                        if (GDN_SMEM_OK(smem_u32(Ab + r * LDA + 4 * q), 16))
                            *reinterpret_cast<float4 *>(Ab + r * LDA + 4 * q) =
                                make_float4(v[0], v[1], v[2], v[3]);
                    }
                };
                if (span_ok)
                    form([&](int s) { return bgr * gs[192 + s]; });
                else
                    form([&](int s) { return br * __expf(s < r ? gr - gs[s] : 0.f); });
            } else {
                inv::clear_upper16(Tb, tid - 64, 64);
            }
            tc_fence_before();
            bar128();
            if (tid == 0) mbar_arrive(bar + U_GFREE + b);
            __syncwarp();
            UTRACE(i, 2);
            // ---- T = (I + A)^{-1}
            inv::invert64(Ab, Tb, tid, bar128);
            UTRACE(i, 3);
            // ---- T_u = T diag(beta) and T_w = T diag(beta gamma), bf16 rows:
            //      thread t takes row t/2, columns 32 (t & 1) .. + 31 of both
            if (un.len > 0 && GDN_IDX_OK((un.out_row + (tid >> 1)) * kU, kU * kU + kU,
                                         p.units * 2 * kU * kU)) {
                const int r = tid >> 1, c0 = 32 * (tid & 1);
                uint4 *du = reinterpret_cast<uint4 *>(p.Tu + (un.out_row + r) * kU + c0);
                uint4 *dw = reinterpret_cast<uint4 *>(p.Tu + (un.out_row + kU + r) * kU + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t wu[4], ww[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s = c0 + 8 * q + 2 * e;
                        const float t0 = inv::t_at(Tb, r, s) * gs[64 + s];
                        const float t1 = inv::t_at(Tb, r, s + 1) * gs[64 + s + 1];
                        wu[e] = pack_bf16(t0, t1);
                        ww[e] = pack_bf16(t0 * gs[128 + s], t1 * gs[128 + s + 1]);
                    }
                    du[q] = make_uint4(wu[0], wu[1], wu[2], wu[3]);
                    dw[q] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
                }
            }
            UTRACE(i, 4);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, 128);
    // the fused kernel that follows may launch once every CTA is here (it
    // waits for this grid before it reads T_u): triggered at the start, its
    // CTAs were placed on SMs as this grid's left them, which measured slower
    griddep_launch_dependents();
#ifdef GDN_TRACE_TIMELINE
    if (tid == 0 && blockIdx.x < 2048) {
        g_ut_cta[blockIdx.x][1] = clock64();
        g_ut_cta[blockIdx.x][3] = nunits;
    }
#endif
}

// ---------------------------------------------------------------------------
// k_gdn_utw: the chunk prep with W out, one warpgroup per CTA, four CTAs per
// SM.
//
// Gram, A and the inverse as in k_gdn_ut, arranged for more units in flight
// than its split into copy and compute warps allows: 128 threads do
// everything.  Thread 64 issues the bulk copies and the Grams, the next
// unit's while warps 0-1 form A or run the inverse's first stage (warps 2-3
// are idle in both), so the Gram is done long before it is read;
// thread 0 issues the W^T product; warp 0 prefetches the next unit's gates
// into registers.  The inverse runs in place (A and T share one
// fp32 tile), T_w is staged in that tile once every thread holds its T
// values, and the W transpose reuses it again.  Per CTA: two K buffers, the
// A/T tile and 128 tensor-memory columns (a Gram / W^T accumulator per
// buffer): about 53 KB of shared memory, so four CTAs fit an SM.

enum { V_FULL = 0, V_GDONE = 2, V_WDONE = 4, V_DRAIN = 6, V_DRAIN2, V_COUNT };

template <int DK>
struct VLay {
    static constexpr int KB = DK / 64;
    static constexpr int SZ_K = KB * 8192;
    static constexpr int OFF_K = 0;                         // + b * SZ_K
    // fp32 [64][LDA]: A, then T in place; then T_w (first 8 KB); then W staging.
    // The Gram's unused operand rows of the last tile read its start.
    static constexpr int OFF_AT = 2 * SZ_K;
    static constexpr int OFF_GS = OFF_AT + (kU * LDA * 4 + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_GS + 1024;           // g, beta, gamma, exp(-g)
    static constexpr int OFF_MISC = OFF_BAR + V_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 16;
    static constexpr int ALLOC = TOTAL + 1024;
    static_assert(OFF_AT % 1024 == 0, "the T_w tile is a 128-byte-swizzled operand");
    static_assert(kU * DK * 2 <= kU * LDA * 4, "the W staging fits the A/T tile");
    static_assert(kU * LDA * 4 >= 8192, "the last tile's unused operand rows stay in bounds");
};

template <int DK>
__global__ void __launch_bounds__(128, 4)
k_gdn_utw(const __grid_constant__ CUtensorMap tm_k, UtParams p) {
    using L = VLay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *AT = reinterpret_cast<float *>(sm + L::OFF_AT);
    float *gs = reinterpret_cast<float *>(sm + L::OFF_GS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef GDN_TRACE_TIMELINE
    if (tid == 0 && blockIdx.x < 2048) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_ut_cta[blockIdx.x][0] = clock64();
        g_ut_cta[blockIdx.x][2] = smid;
    }
#endif
    const long long nunits =
        blockIdx.x < p.units ? (p.units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    // token rows of the inputs (element counts for the bounds-check build)
    const long long nrows =
        p.sm.cu ? (long long)p.sm.H * p.sm.T_total : (long long)p.sm.N * p.sm.H * p.sm.T;
    (void)nrows;

    if (warp == 0) {
        tmem_alloc(misc, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < V_COUNT; ++i) mbar_init(bar + i, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};
    const uint32_t sb = smem_u32(sm);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    auto bar128 = [] { named_bar(1, 128); };
    constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);
    constexpr uint32_t idW = make_idesc_bf16(128, 64, true, false);

    // ---- thread 64: the bulk copy of unit i's K tile into buffer i & 1
    constexpr int kIssuer = 64;
    long long loaded = 0, grammed = 0;
    auto load = [&](long long i) {
        const int b = (int)(i & 1);
        const Unit un = decode(p, blockIdx.x + i * gridDim.x);
        mbar_arrive_expect_tx(bar + V_FULL + b, (uint32_t)L::SZ_K);
#pragma unroll
        for (int kb = 0; kb < L::KB; ++kb)
            tma_load_3d(sm + L::OFF_K + b * L::SZ_K + kb * 8192, &tm_k, bar + V_FULL + b,
                        kb * 64, un.y, un.z);
        loaded = i + 1;
    };
    // ---- thread 64: the Gram of unit i into tensor-memory columns 64 (i & 1)
    auto gram = [&](long long i) -> bool {
        const int b = (int)(i & 1);
        if (!ctl.wait(V_FULL + b, (uint32_t)((i >> 1) & 1))) return false;
        grammed = i + 1;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t off = L::OFF_K + b * L::SZ_K + (kk >> 2) * 8192 + (kk & 3) * 32;
            const uint64_t d = make_sdesc(sb + off, 16, 1024, kSwizzle128B);
            mma_bf16(tmem + 64 * b, d, d, idG, kk > 0);
        }
        mma_commit(bar + V_GDONE + b);
        return true;
    };
    // ---- warp 0: unit i's gates (zero past its end) into registers
    float la0 = 0.f, la1 = 0.f, be0 = 0.f, be1 = 0.f;
    auto fetch_gates = [&](long long i) {
        const Unit un = decode(p, blockIdx.x + i * gridDim.x);
        const bool in0 = lane < un.len && GDN_IDX_OK(un.row0 + lane, 1, nrows);
        const bool in1 = lane + 32 < un.len && GDN_IDX_OK(un.row0 + lane + 32, 1, nrows);
        la0 = in0 ? __ldg(p.log_alpha + un.row0 + lane) : 0.f;
        la1 = in1 ? __ldg(p.log_alpha + un.row0 + lane + 32) : 0.f;
        be0 = in0 ? __ldg(p.beta + un.row0 + lane) : 0.f;
        be1 = in1 ? __ldg(p.beta + un.row0 + lane + 32) : 0.f;
    };
    if (warp == 0 && nunits > 0) fetch_gates(0);
    if (tid == kIssuer && nunits > 0) {
        prefetch_tmap(&tm_k);
        load(0);
        if (nunits > 1) load(1);
        gram(0);   // a failed wait sets the abort flag, seen at every thread's next wait
    }

    for (long long i = 0; i < nunits; ++i) {
        const int b = (int)(i & 1);
        const Unit un = decode(p, blockIdx.x + i * gridDim.x);
        UTRACE(i, 0);
        // ---- gates: g = in-chunk cumsum of log_alpha, beta; the next unit's
        //      are fetched meanwhile
        if (warp == 0) {
            float x0 = la0, x1 = la1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, x0, off);
                const float y1 = __shfl_up_sync(0xffffffffu, x1, off);
                if (lane >= off) {
                    x0 += y0;
                    x1 += y1;
                }
            }
            x1 += __shfl_sync(0xffffffffu, x0, 31);
            gs[lane] = x0;
            gs[32 + lane] = x1;
            gs[64 + lane] = be0;
            gs[96 + lane] = be1;
            gs[128 + lane] = __expf(x0);
            gs[160 + lane] = __expf(x1);
            gs[192 + lane] = __expf(-x0);   // used only when the decay span is < 80
            gs[224 + lane] = __expf(-x1);
            if (i + 1 < nunits) fetch_gates(i + 1);
        }
        // ---- A from the Gram rows (warps 0-1), every row written in full
        if (!named_bar_and(1, 128, ctl.wait(V_GDONE + b, (uint32_t)((i >> 1) & 1)))) break;
        UTRACE(i, 1);
        tc_fence_after();
        if (warp < 2) {
            const int r = tid;
            uint32_t g0[32], g1[32];
            tmem_ld32(tmem + lane_base + 64 * b, g0);
            tmem_ld32(tmem + lane_base + 64 * b + 32, g1);
            const float gr = gs[r], br = gs[64 + r];
            tmem_wait32(g0);
            tmem_wait32(g1);
            const bool span_ok = gs[63] > -80.f;
            const float bgr = br * gs[128 + r];
            auto form = [&](auto factor) {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s2 = 4 * q + e;
                        const float gv = f32(s2 < 32 ? g0[s2] : g1[s2 - 32]);
                        const float x = s2 < r ? factor(s2) * gv : 0.f;
                        v[e] = (r >> 4) != (s2 >> 4) ? inv::tf32(x) : x;
                    }
                    if (GDN_SMEM_OK(smem_u32(AT + r * LDA + 4 * q), 16))
                        *reinterpret_cast<float4 *>(AT + r * LDA + 4 * q) =
                            make_float4(v[0], v[1], v[2], v[3]);
                }
            };
            if (span_ok)
                form([&](int s2) { return bgr * gs[192 + s2]; });
            else
                form([&](int s2) { return br * __expf(s2 < r ? gr - gs[s2] : 0.f); });
        }
        // ---- the next unit's Gram into the other buffer's columns (its W^T
        //      was read in the previous unit): now, while warps 0-1 form A, if
        //      its K tile has landed, else while they run the inverse's first
        //      stage
        bool gram_issued = false;
        if (tid == kIssuer && i + 1 < nunits &&
            mbar_test_wait(bar + V_FULL + (b ^ 1), (uint32_t)(((i + 1) >> 1) & 1))) {
            gram(i + 1);
            gram_issued = true;
        }
        tc_fence_before();
        bar128();
        UTRACE(i, 2);
        if (tid == kIssuer && i + 1 < nunits && !gram_issued) gram(i + 1);
        // ---- T = (I + A)^{-1} in place
        inv::invert64_inplace(AT, tid, bar128);
        UTRACE(i, 3);
        // ---- T_u = T diag(beta) rows out; T_w = T diag(beta gamma) staged
        //      (bf16, 128-byte swizzled) over the tile's first 8 KB once every
        //      thread holds its T values.  Item (row r, 8-column chunk ch):
        //      eight consecutive threads read one row of T.
        {
            float tv[4][8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int item = tid + 128 * k, r = item >> 3, c = 8 * (item & 7);
                const float4 ta = *reinterpret_cast<const float4 *>(AT + r * LDA + c);
                const float4 tb = *reinterpret_cast<const float4 *>(AT + r * LDA + c + 4);
                tv[k][0] = ta.x; tv[k][1] = ta.y; tv[k][2] = ta.z; tv[k][3] = ta.w;
                tv[k][4] = tb.x; tv[k][5] = tb.y; tv[k][6] = tb.z; tv[k][7] = tb.w;
            }
            bar128();
            uint8_t *Tw = reinterpret_cast<uint8_t *>(AT);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int item = tid + 128 * k, r = item >> 3, ch = item & 7, c = 8 * ch;
                uint32_t wu[4], ww[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s2 = c + 2 * e;
                    // zero above the diagonal and in the scratch block
                    const bool z0 = s2 > r || (r < 32 && s2 >= 32);
                    const bool z1 = s2 + 1 > r || (r < 32 && s2 + 1 >= 32);
                    const float t0 = z0 ? 0.f : tv[k][2 * e] * gs[64 + s2];
                    const float t1 = z1 ? 0.f : tv[k][2 * e + 1] * gs[64 + s2 + 1];
                    wu[e] = pack_bf16(t0, t1);
                    ww[e] = pack_bf16(t0 * gs[128 + s2], t1 * gs[128 + s2 + 1]);
                }
                if (r < un.len && GDN_IDX_OK((un.row0 + r) * kU + c, 8, nrows * kU))
                    *reinterpret_cast<uint4 *>(p.Tu + (un.row0 + r) * kU + c) =
                        make_uint4(wu[0], wu[1], wu[2], wu[3]);
                st16(Tw + sw128_offset(r, ch), ww[0], ww[1], ww[2], ww[3]);
            }
        }
        fence_proxy_async_smem();
        bar128();
        // ---- thread 0: W^T = K^T T_w^T (M = d_k lanes, N = 64 tokens) into
        //      this unit's columns (the Gram there has been read)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kU / 16; ++kk) {
                const uint64_t da = make_sdesc(sb + L::OFF_K + b * L::SZ_K + kk * 2048, 8192, 1024,
                                               kSwizzle128B);
                const uint64_t dbw = make_sdesc(sb + L::OFF_AT + kk * 32, 16, 1024, kSwizzle128B);
                mma_bf16(tmem + 64 * b, da, dbw, idW, kk > 0);
            }
            mma_commit(bar + V_WDONE + b);
        }
        // ---- W rows: W^T from tensor memory (lane = d_k index) through a
        //      [64][d_k] bf16 tile over the A/T tile, out as rows.  Odd rows
        //      have their 32-bit words XOR 16: the even lanes' row 2m and the
        //      odd lanes' row 2m + 1 then fill different banks, and a 16-byte
        //      vector (four words) stays whole.
        constexpr int WPR = DK / 2;   // 32-bit words per W row
        uint32_t *Ws = reinterpret_cast<uint32_t *>(AT);
        if (!named_bar_and(1, 128, ctl.wait(V_WDONE + b, (uint32_t)((i >> 1) & 1)))) break;
        tc_fence_after();
        if (tid < DK) {
            uint32_t w0[32], w1[32];
            tmem_ld32(tmem + lane_base + 64 * b, w0);
            tmem_ld32(tmem + lane_base + 64 * b + 32, w1);
            tmem_wait32(w0);
            tmem_wait32(w1);
            // lanes t and t ^ 1 hold columns t and t ^ 1 of every row: the
            // even lane writes the pair for rows 2m, the odd lane for 2m + 1
            const bool odd = tid & 1;
            const int cpair = tid & ~1;
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                const int r0 = 2 * m;
                const float a0 = f32(r0 < 32 ? w0[r0] : w1[r0 - 32]);
                const float a1 = f32(r0 + 1 < 32 ? w0[r0 + 1] : w1[r0 - 31]);
                const float give = odd ? a0 : a1;
                const float got = __shfl_xor_sync(0xffffffffu, give, 1);
                const int row = odd ? r0 + 1 : r0;
                const uint32_t word = odd ? pack_bf16(got, a1) : pack_bf16(a0, got);
                uint32_t *dst = Ws + row * WPR + ((cpair >> 1) ^ (odd ? 16 : 0));
                if (GDN_SMEM_OK(smem_u32(dst), 4)) *dst = word;
            }
        }
        tc_fence_before();
        bar128();
        // K buffer b is free (this unit's Gram and W^T are done)
        if (tid == kIssuer && i + 2 < nunits) load(i + 2);
        constexpr int VPR = DK / 8;   // 16-byte vectors per W row
#pragma unroll
        for (int j = 0; j < kU * VPR / 128; ++j) {
            const int idx = tid + 128 * j, r = idx / VPR, q = idx % VPR;
            const uint32_t *src = Ws + r * WPR + ((4 * q) ^ (r & 1 ? 16 : 0));
            if (r < un.len && GDN_IDX_OK((un.row0 + r) * DK + 8 * q, 8, nrows * DK) &&
                GDN_SMEM_OK(smem_u32(src), 16))
                *reinterpret_cast<uint4 *>(p.W + (un.row0 + r) * DK + 8 * q) =
                    *reinterpret_cast<const uint4 *>(src);
        }
        UTRACE(i, 4);
        // (the next unit's first barrier orders these reads before the tile
        // is written again)
    }
    // every issued MMA has finished, and every issued copy landed, before
    // the CTA leaves (each issuing thread drains its own MMAs)
    if (tid == 0) {
        mma_commit(bar + V_DRAIN);
        mbar_wait(bar + V_DRAIN, 0, ctl.limit);
    }
    if (tid == kIssuer) {
        mma_commit(bar + V_DRAIN2);
        mbar_wait(bar + V_DRAIN2, 0, ctl.limit);
        for (long long u = grammed; u < loaded; ++u)
            mbar_wait(bar + V_FULL + (u & 1), (uint32_t)((u >> 1) & 1), ctl.limit);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
    // the chain kernel that follows may launch once every CTA is here (it
    // waits for this grid before it reads T_u and W).  Triggered at the start,
    // its CTAs were placed on SMs as this grid's left them: 0.215 against
    // 0.200 ms per call at B4 H16 T4096 d128
    griddep_launch_dependents();
#ifdef GDN_TRACE_TIMELINE
    if (tid == 0 && blockIdx.x < 2048) {
        g_ut_cta[blockIdx.x][1] = clock64();
        g_ut_cta[blockIdx.x][3] = nunits;
    }
#endif
}

#ifdef GDN_TRACE_TIMELINE
int g_ut_ctas_seen = 0;
#endif

// CTAs the device holds at once, per device: what shared memory holds per SM
// (1 KB reserved per CTA), at most `cap` (the launch bounds' register budget;
// 128 of the 512 tensor-memory columns each), times the SMs.
int resident_ctas(std::atomic<int> (&memo)[kMaxDeviceMemo], int alloc, int cap) {
    return per_device(
        memo,
        [alloc, cap](int dev) {
            int smem_sm = 0, nsm = 0;
            if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                       dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return -1;
            const int fit = smem_sm / (alloc + 1024);
            return max(1, min(fit, cap)) * max(1, nsm);
        },
        0);
}

// The K tensor map and the parameters of a prep launch over every
// (chunk slot, head) unit.
bool ut_setup(const FwdArgs &a, int dk, const int2 *table, __nv_bfloat16 *Tu,
              __nv_bfloat16 *W, CUtensorMap *mk, UtParams *p) {
    const long long ydim = a.sm.cu ? a.sm.T_total : a.sm.T;
    const long long zdim = a.sm.cu ? a.sm.H : (long long)a.sm.N * a.sm.H;
    if (!make_map(mk, a.k, dk, ydim, zdim)) return false;
    p->sm = a.sm;
    p->log_alpha = a.log_alpha;
    p->beta = a.beta;
    p->table = table;
    p->Tu = Tu;
    p->W = W;
    p->err = device_error_word();
    p->max_chunks = a.max_chunks;
    p->chunk_slots = a.chunk_slots;
    p->units = (long long)a.chunk_slots * a.sm.H;
    const long long lim = option(GDN_OPT_WAIT_LIMIT);
    p->wait_limit = lim > 0 ? (uint32_t)(lim > 0x7fffffffLL ? 0x7fffffffLL : lim) : (1u << 22);
    return true;
}

template <int DK>
gdn_status launch_ut(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu) {
    using L = ULay<DK>;
    if (cudaFuncSetAttribute(k_gdn_ut<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(k_gdn_ut<DK>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             100) != cudaSuccess)
        return GDN_ERR_CUDA;
    static std::atomic<int> memo[kMaxDeviceMemo];
    const int ctas = resident_ctas(memo, L::ALLOC, 3);
    if (ctas <= 0) return GDN_ERR_CUDA;
#ifdef GDN_TRACE_TIMELINE
    g_ut_ctas_seen = ctas;
#endif
    if ((long long)a.chunk_slots * a.sm.H <= 0) return GDN_OK;
    CUtensorMap mk;
    UtParams p;
    if (!ut_setup(a, DK, table, Tu, nullptr, &mk, &p)) return GDN_ERR_CUDA;
    const int grid = (int)(p.units < ctas ? p.units : (long long)ctas);
    k_gdn_ut<DK><<<grid, kThreadsU, L::ALLOC, a.stream>>>(mk, p);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <int DK>
gdn_status launch_utw(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu, __nv_bfloat16 *W) {
    using L = VLay<DK>;
    if (cudaFuncSetAttribute(k_gdn_utw<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(k_gdn_utw<DK>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             100) != cudaSuccess)
        return GDN_ERR_CUDA;
    static std::atomic<int> memo[kMaxDeviceMemo];
    const int ctas = resident_ctas(memo, L::ALLOC, 4);
    if (ctas <= 0) return GDN_ERR_CUDA;
#ifdef GDN_TRACE_TIMELINE
    g_ut_ctas_seen = ctas;
#endif
    if ((long long)a.chunk_slots * a.sm.H <= 0) return GDN_OK;
    CUtensorMap mk;
    UtParams p;
    if (!ut_setup(a, DK, table, Tu, W, &mk, &p)) return GDN_ERR_CUDA;
    const int grid = (int)(p.units < ctas ? p.units : (long long)ctas);
    k_gdn_utw<DK><<<grid, 128, L::ALLOC, a.stream>>>(mk, p);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

#ifdef GDN_TRACE_TIMELINE
extern "C" int gdn_ut_debug_ctas() { return g_ut_ctas_seen; }
#endif

gdn_status enqueue_ut(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu) {
    if (a.no_erase || a.vector_gate || a.dt != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (a.dk == 128) return launch_ut<128>(a, table, Tu);
    if (a.dk == 64) return launch_ut<64>(a, table, Tu);
    return GDN_ERR_UNSUPPORTED;
}

gdn_status enqueue_ut_w(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                        __nv_bfloat16 *W) {
    if (a.no_erase || a.vector_gate || a.dt != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (a.dk == 128) return launch_utw<128>(a, table, Tu, W);
    if (a.dk == 64) return launch_utw<64>(a, table, Tu, W);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
