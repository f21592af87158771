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
//     the staged K tile.  Its unit loop (gdn_utw.cuh) also runs inside the
//     chain kernel's overlapped launch, on the SMs the chain leaves free.
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

#include "gdn_utw.cuh"   // UtParams, the unit map and k_gdn_utw's pipeline

namespace gdn {
namespace {

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
// k_gdn_utw: the chunk prep with W out (gdn_utw.cuh), one 128-thread
// pipeline per CTA, four CTAs per SM (shared memory, registers and tensor
// memory all stop at four).  Persistent: each CTA walks the launch's units
// b, b + grid, ...
template <int DK>
__global__ void __launch_bounds__(128, 4)
k_gdn_utw(const __grid_constant__ CUtensorMap tm_k, UtParams p) {
    using L = VLay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5;
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
    // the ready flags of the units that the next launch prepares beside the
    // chain (it sets them)
    if (p.done_zero)
        for (long long i = (long long)blockIdx.x * 128 + tid; i < p.n_done;
             i += (long long)gridDim.x * 128)
            p.done_zero[i] = 0u;
    if (warp == 0) {
        tmem_alloc(misc, 128);
        tmem_relinquish();
    }
    utw_init<DK>(sm, tid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    utw_run<DK>(sm, tmem, tid, 1, &tm_k, p, blockIdx.x, gridDim.x, nunits);
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
gdn_status launch_utw(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu, __nv_bfloat16 *W,
                      int lead = 0, uint32_t *done_zero = nullptr, long long n_done = 0) {
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
    if (lead > 0) {
        // chunks 0 .. lead - 1 of every (sequence, head); the rest are
        // prepared beside the chain, whose ready flags this launch clears
        p.c0 = 0;
        p.nc = lead;
        p.units = (long long)a.sm.N * a.sm.H * lead;
        p.done_zero = done_zero;
        p.n_done = n_done;
    }
    const long long want = p.units > 0 ? p.units : 1;
    const int grid = (int)(want < ctas ? want : (long long)ctas);
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

gdn_status enqueue_ut_w_lead(const FwdArgs &a, __nv_bfloat16 *Tu, __nv_bfloat16 *W, int lead,
                             uint32_t *done, long long n_done) {
    if (a.no_erase || a.vector_gate || a.dt != GDN_BF16 || a.sm.cu || lead < 1 ||
        lead > a.max_chunks)
        return GDN_ERR_UNSUPPORTED;
    if (a.dk == 128) return launch_utw<128>(a, nullptr, Tu, W, lead, done, n_done);
    if (a.dk == 64) return launch_utw<64>(a, nullptr, Tu, W, lead, done, n_done);
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
