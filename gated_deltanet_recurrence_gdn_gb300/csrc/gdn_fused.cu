// gdn_fused.cu -- chunked gated delta rule forward on sm_103a tensor cores:
// the WY factors, the serial state pass and the output of one
// (sequence, head, 64-wide d_v tile) in one CTA, chunks of C = 64 tokens in
// order ("Gated DeltaNet GPU并行实现", section 3.2: products inside a chunk on
// the tensor cores, a serial state pass across chunks).
//
// Inputs per chunk: K, Q (C x d_k), the V tile (C x 64), log_alpha, and
// T_u = (I + A)^{-1} diag(beta), T_w = (I + A)^{-1} diag(beta gamma) from the
// chunk-prep kernel (gdn_ut.cu).  With
// g_r the in-chunk cumulative log gate, gamma_r = exp(g_r), e_r =
// exp(g_C - g_r) and H = S^T (d_k x 64, fp32, in registers of the chain
// warpgroup):
//
//   U  = T_u V                         W = T_w K
//   G  = Q K^T                         P'_rs = exp(-g_s) G_rs  (s <= r)
//   [V' - U; O1] = [-W; Q] H                         (chain MMA 1, M = 128)
//   V' = U + (V' - U)
//   dH = K^T diag(e) V'                              (chain MMA 2)
//   O  = diag(gamma) (O1 + P' V')
//   H <- gamma_C H + dH
//
// When a chunk's total log decay g_C is below -80, exp(-g_s) could overflow:
// that chunk scales Q by gamma in place after the Gram, forms
// P_rs = exp(g_r - g_s) G_rs directly and stores its output rows unscaled.
//
// Two threads issue the MMAs (a tensor-core instruction blocks its issuer while
// the pipe is busy, and each wait between groups costs its issuer time): one
// issues only the two chain MMAs, the moment their operands are ready; the
// other issues the next chunk's W and Gram once chain MMA 1 of chunk j is done
// (they run while the chain forms V') and the next chunk's U and j's output
// product once chain MMA 2 is done (they run while the chain updates H).
// Only the two chain MMAs and the two register passes between them are on the
// state's dependency chain; three input slots keep the copies and the
// per-chunk factors ahead of it.
//
// Warp roles (352 threads):
//   warps 0-3  chain: H (thread t = row t = d_k index t) and V' (threads 0-63 =
//              rows of the chunk) between the chain MMAs.
//   warps 4-5  -W from tensor memory (rows 0-63) into the operand slot;
//              gamma Q in place for wide-span chunks.
//   warps 6-7  P' from the Gram (tensor-memory rows 64-127); output rows.
//   warp 8     bulk tensor copies (one lane); the chunk's gate arrays from
//              log_alpha (all lanes).
//   warp 9     issues W, Gram, U and the output product (one lane); owns
//              tensor memory.
//   warp 10    issues the chain MMAs (one lane).
// Every wait is bounded; a wait that gives up sets the device error word and
// every role leaves its loop; in-flight MMAs are drained before tensor memory
// is freed.
//
// Tokens past the end of a sequence carry beta = log_alpha = 0, so their rows
// and columns of T_u are zero; whatever the copies bring in those rows (the
// next packed sequence, or zero fill) then never reaches a real row.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

// Optional per-role timeline of CTA (0,0,0) for profiling builds
// (-DGDN_TRACE_TIMELINE): clock64() stamps by role, chunk and event, read back
// with gdn_fused_trace_read().  Compiled out otherwise.
#ifdef GDN_TRACE_TIMELINE
__device__ long long g_fused_trace[5][128][8];
__device__ long long g_fused_cta[4096][4];   // per CTA: start, end, SM, chunks
extern "C" int gdn_fused_trace_read(long long *out, long long *cta) {
    int e = (int)cudaMemcpyFromSymbol(out, g_fused_trace, sizeof(g_fused_trace));
    return e ? e : (int)cudaMemcpyFromSymbol(cta, g_fused_cta, sizeof(g_fused_cta));
}
#define FTRACE(role, jj, ev)                                                           \
    do {                                                                               \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (jj) < 128)       \
            g_fused_trace[role][jj][ev] = clock64();                                   \
    } while (0)
#else
#define FTRACE(role, jj, ev) \
    do {                     \
    } while (0)
#endif

namespace gdn {
namespace {

using namespace ptx;
using namespace tcx;

constexpr int kC = 64;
constexpr int kNV = 64;
constexpr int kSlots = 3;
constexpr int kThreadsF = 352;

// mbarriers.  Per-chunk barriers are waited with parity j & 1; "[2]" barriers
// are indexed by j & 1 with parity (j >> 1) & 1; "[3]" by j % 3 with parity
// (j / 3) & 1.  Each barrier's arrivals for chunk j + 2 (resp. j + 3, j + 6)
// depend on its waiters for chunk j having passed, so no waiter can miss a
// phase.
enum {
    F_KQ = 0,              // [3] K and Q landed, gate arrays written (TMA tx + 32 lanes)
    F_TU = F_KQ + 3,       // [2] T_u landed
    F_TW = F_TU + 2,       // T_w landed
    F_V,                   // V tile landed
    E_KQ,                  // [3] slot read by every MMA (commits of both issuers) and
                           //     its gate arrays by the P' warps
    E_TU = E_KQ + 3,       // [2] T_u read by U (commit)
    E_V = E_TU + 2,        // V read by U (commit)
    E_TW,                  // T_w read by W (commit)
    B_WQ,                  // [3] [-W; Q] operand complete
    B_GDONE = B_WQ + 3,    // Gram in tensor memory (commit)
    B_GFREE,               // P' formed from it
    B_UDONE,               // [2] U in tensor memory (commit)
    B_UFREE = B_UDONE + 2, // [2] chain read U
    B_WDONE = B_UFREE + 2, // W in tensor memory (commit)
    B_WFREE,               // -W read out of it
    B_PREADY,              // [2] P' operand written
    B_HREADY = B_PREADY + 2,   // H operand written (chain)
    B_M1,                  // chain MMA 1 done (commit)
    B_VT,                  // decayed V' operand written (chain)
    B_M2,                  // chain MMA 2 done (commit)
    B_VN,                  // [2] V' operand written
    B_OUT = B_VN + 2,      // [2] P' V' done: output rows complete (commit)
    B_DFREE = B_OUT + 2,   // [2] output rows read
    B_DRAIN = B_DFREE + 2, // factor issuer drained
    B_DRAIN2,              // chain issuer drained
    B_COUNT
};

template <int DK>
struct FLay {
    static constexpr int KB = DK / 64;              // 64-column blocks of K, Q, W
    static constexpr int SZ_K = KB * 8192;
    static constexpr int SZ_WQ = KB * 16384;        // per block [-W (64 rows) | Q (64 rows)]
    static constexpr int OFF_K = 0;                 // + s * SZ_K
    static constexpr int OFF_WQ = OFF_K + kSlots * SZ_K;      // + s * SZ_WQ
    // [T_u0 | T_u1 | T_w | P1]: each T tile heads a 128-row operand whose other
    // rows are unused, and [T_w; P1] is the operand whose rows 64-127 are P1
    static constexpr int OFF_TU = OFF_WQ + kSlots * SZ_WQ;    // + b * 8192
    static constexpr int OFF_TW = OFF_TU + 2 * 8192;
    static constexpr int OFF_P1 = OFF_TW + 8192;
    static constexpr int OFF_V = OFF_P1 + 8192;
    // H (DK rows x 64 bf16); the decayed V' of the chunk reuses its first 8 KB
    static constexpr int OFF_H = OFF_V + 8192;
    static constexpr int OFF_VN = OFF_H + DK * 128;           // [V' | P0]
    static constexpr int OFF_P0 = OFF_VN + 8192;
    static constexpr int OFF_GA = OFF_P0 + 8192;              // [3][g | gamma | e | 1/gamma][64]
    static constexpr int OFF_BAR = OFF_GA + kSlots * 1024;
    static constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 16;
    static constexpr int ALLOC = TOTAL + 1024;
    static_assert(ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(OFF_WQ % 1024 == 0 && OFF_TU % 1024 == 0 && OFF_H % 1024 == 0 &&
                      OFF_VN % 1024 == 0 && OFF_V % 1024 == 0,
                  "operand tiles 1024-byte aligned");
};

// Tensor-memory columns (512 allocated; lanes = rows).
constexpr uint32_t TM_G = 0;     // Q K^T in lanes 64-127
constexpr uint32_t TM_U = 64;    // + 64 b: U in lanes 0-63
constexpr uint32_t TM_D = 192;   // + 64 b: [V' - U; O]
constexpr uint32_t TM_DH = 320;  // dH, lanes 0..d_k-1
constexpr uint32_t TM_W = 384;   // W in lanes 0-63, d_k columns

struct FParams {
    SeqMap sm;
    const float *log_alpha, *h0;
    __nv_bfloat16 *o;
    float *hT;
    int *err;
    int dv;
    uint32_t wait_limit;
    long long chunk_slots;   // per head, in the T_u layout [H][chunk_slots][64][64]
    int max_chunks;
};

// Multiplies the 8 bf16 values of a 16-byte piece by f[0..7].
__device__ __forceinline__ uint4 scale8(uint4 v, const float *f) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        w[e] = pack_bf16(x.x * f[2 * e], x.y * f[2 * e + 1]);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Stores 64 fp32 values as bf16 into global memory (128 bytes, 16-byte pieces).
__device__ __forceinline__ void store_row64(__nv_bfloat16 *dst, const uint32_t (&a)[32],
                                            const uint32_t (&b)[32], float sc) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        d[q] = make_uint4(pack_bf16(f32(a[8 * q]) * sc, f32(a[8 * q + 1]) * sc),
                          pack_bf16(f32(a[8 * q + 2]) * sc, f32(a[8 * q + 3]) * sc),
                          pack_bf16(f32(a[8 * q + 4]) * sc, f32(a[8 * q + 5]) * sc),
                          pack_bf16(f32(a[8 * q + 6]) * sc, f32(a[8 * q + 7]) * sc));
#pragma unroll
    for (int q = 0; q < 4; ++q)
        d[4 + q] = make_uint4(pack_bf16(f32(b[8 * q]) * sc, f32(b[8 * q + 1]) * sc),
                              pack_bf16(f32(b[8 * q + 2]) * sc, f32(b[8 * q + 3]) * sc),
                              pack_bf16(f32(b[8 * q + 4]) * sc, f32(b[8 * q + 5]) * sc),
                              pack_bf16(f32(b[8 * q + 6]) * sc, f32(b[8 * q + 7]) * sc));
}

template <int DK>
__global__ void __launch_bounds__(kThreadsF, 1)
k_gdn_fused(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_tu,
            FParams p) {
    using L = FLay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    // chunks whose Gram warps 6-7 have seen complete: a count, so that the
    // wide-span branch of warps 4-5, which waits for the Gram only in some
    // chunks, cannot mistake an older phase of its mbarrier for this one
    uint32_t *g_seen = misc + 2;
    auto GA = [&](int s) { return reinterpret_cast<float *>(sm + L::OFF_GA + s * 1024); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef GDN_TRACE_TIMELINE
    const long long cta_id =
        ((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    if (tid == 0 && cta_id < 4096) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_fused_cta[cta_id][0] = clock64();
        g_fused_cta[cta_id][2] = smid;
    }
#endif
    const int dv0 = (int)blockIdx.x * kNV;
    const int h = blockIdx.y, n = blockIdx.z;

    // ---- sequence bounds (validated; an invalid packed range is an error)
    long long row0 = 0;
    int len = 0, ytok0 = 0, zc = 0;
    if (p.sm.cu) {
        const int a = __ldg(p.sm.cu + n), b = __ldg(p.sm.cu + n + 1);
        if (!(a >= 0 && a <= b && b <= p.sm.T_total)) {
            if (tid == 0) atomicCAS(p.err, 0, kErrBadIndex);
            return;   // before any barrier or tensor-memory use
        }
        row0 = (long long)h * p.sm.T_total + a;
        len = b - a;
        ytok0 = a;
        zc = h;
    } else {
        row0 = ((long long)n * p.sm.H + h) * (long long)p.sm.T;
        len = p.sm.T;
        zc = n * p.sm.H + h;
    }
    const int nch = (len + kC - 1) / kC;
    const long long srow = ((long long)n * p.sm.H + h) * p.dv;   // state rows of (n, h)
    const long long slot0 =
        p.sm.cu ? (long long)(ytok0 / kC) + n : (long long)n * p.max_chunks;
    // rows of chunk 0's [T_u | T_w] block in the chunk-prep kernel's output
    const long long turow0 = ((long long)h * p.chunk_slots + slot0) * 2 * kC;

    if (warp == 9) {
        tmem_alloc(misc, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar + i, 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar + F_KQ + s, 33);
            mbar_init(bar + E_KQ + s, 3);
        }
        *abort_flag = 0;
        *g_seen = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};

    if (warp < 4) {
        // ===================================================== chain warpgroup
        const int t = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float hreg[kNV];
#pragma unroll
        for (int c = 0; c < kNV; ++c)
            hreg[c] = (t < DK && p.h0) ? __ldg(p.h0 + (srow + dv0 + c) * DK + t) : 0.f;
        uint8_t *Hs = sm + L::OFF_H;
        uint8_t *VNs = sm + L::OFF_VN;
        float gC = 1.f;   // gamma_C of the previous chunk
        bool alive = true;
        auto update_h = [&]() {
            if (t < DK) {
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    float d[16];
                    tmem_ld16f(tmem + lane_base + TM_DH + 16 * qq, d);
#pragma unroll
                    for (int i = 0; i < 16; ++i) hreg[16 * qq + i] = fmaf(gC, hreg[16 * qq + i], d[i]);
                }
            }
        };
        for (int j = 0; j < nch; ++j) {
            const int s = j % kSlots, b = j & 1;
            // ---- (A) H <- gamma_C H + dH, published as the bf16 operand of MMA 1
            if (j > 0) {
                if (!named_bar_and(1, 128, ctl.wait(B_M2, (j - 1) & 1))) {
                    alive = false;
                    break;
                }
                if (t == 0) FTRACE(0, j, 0);
                tc_fence_after();
                update_h();
            }
            if (t < DK) put_row64(Hs, t, hreg);
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 128);
            if (t == 0) {
                mbar_arrive(bar + B_HREADY);
                FTRACE(0, j, 1);
            }
            __syncwarp();
            // ---- (B) V' = U + (V' - U): the decayed copy for MMA 2 first, then
            //      the plain copy for P' V'
            if (!named_bar_and(1, 128, ctl.wait(B_M1, j & 1) &&
                                           ctl.wait(B_UDONE + b, (uint32_t)((j >> 1) & 1)))) {
                alive = false;
                break;
            }
            if (t == 0) FTRACE(0, j, 2);
            tc_fence_after();
            const float *ga = GA(s);
            const float gCj = ga[64 + 63];
            if (t < 64) {
                const float er = ga[128 + t];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    float u[16], w[16], x[16];
                    tmem_ld16f(tmem + lane_base + TM_U + 64 * b + 16 * qq, u);
                    tmem_ld16f(tmem + lane_base + TM_D + 64 * b + 16 * qq, w);
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] = (u[i] + w[i]) * er;
                    put8(Hs, t, 2 * qq, x);
                    put8(Hs, t, 2 * qq + 1, x + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 128);
            if (t == 0) {
                mbar_arrive(bar + B_VT);
                FTRACE(0, j, 3);
            }
            __syncwarp();
            // the V' tile is free once the previous chunk's output product is done
            if (j >= 1 && !named_bar_and(1, 128, ctl.wait(B_OUT + ((j - 1) & 1),
                                                          (uint32_t)(((j - 1) >> 1) & 1)))) {
                alive = false;
                break;
            }
            if (t < 64) {
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    float u[16], w[16], x[16];
                    tmem_ld16f(tmem + lane_base + TM_U + 64 * b + 16 * qq, u);
                    tmem_ld16f(tmem + lane_base + TM_D + 64 * b + 16 * qq, w);
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] = u[i] + w[i];
                    put8(VNs, t, 2 * qq, x);
                    put8(VNs, t, 2 * qq + 1, x + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 128);
            if (t == 0) {
                mbar_arrive(bar + B_UFREE + b);
                mbar_arrive(bar + B_VN + b);
                FTRACE(0, j, 4);
            }
            __syncwarp();
            gC = gCj;
        }
        // ---- final state
        if (alive && nch > 0) {
            if (named_bar_and(1, 128, ctl.wait(B_M2, (nch - 1) & 1))) {
                tc_fence_after();
                update_h();
            } else {
                alive = false;
            }
        }
        if (alive && p.hT && t < DK) {
#pragma unroll
            for (int c = 0; c < kNV; ++c) p.hT[(srow + dv0 + c) * DK + t] = hreg[c];
        }
    } else if (warp < 6) {
        // ================================ -W (rows 0-63), gamma Q for wide spans
        const int r = tid - 128;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        for (int j = 0; j < nch; ++j) {
            const int s = j % kSlots;
            const float *ga = GA(s);
            if (!named_bar_and(2, 64, ctl.wait(F_KQ + s, (uint32_t)((j / kSlots) & 1)))) break;
            if (r == 0) FTRACE(1, j, 0);
            // ---- a chunk whose decay span is too wide for exp(-g_s) takes gamma Q
            //      in place once the Gram has read Q; otherwise the output rows
            //      take gamma_r when stored
            if (ga[63] <= -80.f) {
                if (!named_bar_and(2, 64, ctl.flag(g_seen, (uint32_t)j + 1))) break;
                const float gr = ga[64 + r];
                const float f[8] = {gr, gr, gr, gr, gr, gr, gr, gr};
#pragma unroll
                for (int kb = 0; kb < L::KB; ++kb) {
                    uint8_t *qt = sm + L::OFF_WQ + s * L::SZ_WQ + kb * 16384 + 8192;
                    uint4 v[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = *reinterpret_cast<const uint4 *>(qt + sw128_offset(r, c));
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(qt + sw128_offset(r, c)) = scale8(v[c], f);
                }
            }
            // ---- -W into the operand slot
            if (!named_bar_and(2, 64, ctl.wait(B_WDONE, j & 1))) break;
            if (r == 0) FTRACE(1, j, 3);
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < L::KB; ++kb) {
                uint32_t w0[32], w1[32];
                tmem_ld32(tmem + lane_base + TM_W + 64 * kb, w0);
                tmem_ld32(tmem + lane_base + TM_W + 64 * kb + 32, w1);
                tmem_wait32(w0);
                tmem_wait32(w1);
                float x[64];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    x[i] = -f32(w0[i]);
                    x[32 + i] = -f32(w1[i]);
                }
                put_row64(sm + L::OFF_WQ + s * L::SZ_WQ + kb * 16384, r, x);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar(2, 64);
            if (r == 0) {
                mbar_arrive(bar + B_WFREE);
                mbar_arrive(bar + B_WQ + s);
                FTRACE(1, j, 4);
            }
            __syncwarp();
        }
    } else if (warp < 8) {
        // ===================================== P' and output rows (rows 64-127)
        const int r = tid - 192;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        auto epilogue = [&](int jj, float sc) -> bool {
            const int bb = jj & 1;
            if (!named_bar_and(3, 64, ctl.wait(B_OUT + bb, (uint32_t)((jj >> 1) & 1))))
                return false;
            if (r == 0) FTRACE(2, jj, 2);
            tc_fence_after();
            {
                uint32_t o0[32], o1[32];
                tmem_ld32(tmem + lane_base + TM_D + 64 * bb, o0);
                tmem_ld32(tmem + lane_base + TM_D + 64 * bb + 32, o1);
                tmem_wait32(o0);
                tmem_wait32(o1);
                if (r < min(kC, len - jj * kC))
                    store_row64(p.o + (row0 + (long long)jj * kC + r) * p.dv + dv0, o0, o1, sc);
            }
            tc_fence_before();
            named_bar(3, 64);
            if (r == 0) {
                mbar_arrive(bar + B_DFREE + bb);
                FTRACE(2, jj, 3);
            }
            __syncwarp();
            return true;
        };
        bool alive = true;
        float osc = 1.f, osc_prev = 1.f;   // output scales of this and the previous chunk
        for (int j = 0; j < nch; ++j) {
            const int s = j % kSlots, b = j & 1;
            const bool ok = ctl.wait(F_KQ + s, (uint32_t)((j / kSlots) & 1)) &&
                            ctl.wait(B_GDONE, j & 1);
            if (!named_bar_and(3, 64, ok)) {
                alive = false;
                break;
            }
            if (r == 0) st_release_cta(g_seen, (uint32_t)j + 1);
            if (r == 0) FTRACE(2, j, 0);
            tc_fence_after();
            {
                const float *ga = GA(s);
                uint32_t g0[32], g1[32];
                tmem_ld32(tmem + lane_base + TM_G, g0);
                tmem_ld32(tmem + lane_base + TM_G + 32, g1);
                tmem_wait32(g0);
                tmem_wait32(g1);
                // P' = P / gamma_r = exp(-g_s) (Q K^T)_rs for s <= r (the output row
                // takes gamma_r when stored); a chunk whose span is too wide for
                // exp(-g_s) forms P itself (its Q was scaled by gamma in place).
                // P(j) replaces P(j - 2), whose P' V' the epilogue of j - 2 saw done.
                float x[64];
                if (ga[63] > -80.f) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const float gv = f32(i < 32 ? g0[i] : g1[i - 32]);
                        x[i] = (i <= r ? ga[192 + i] : 0.f) * gv;
                    }
                    osc = ga[64 + r];
                } else {
                    const float gr = ga[r];
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const float gv = f32(i < 32 ? g0[i] : g1[i - 32]);
                        x[i] = __expf(i <= r ? gr - ga[i] : -INFINITY) * gv;
                    }
                    osc = 1.f;
                }
                put_row64(sm + (b ? L::OFF_P1 : L::OFF_P0), r, x);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar(3, 64);
            if (r == 0) {
                mbar_arrive(bar + B_GFREE);
                mbar_arrive(bar + B_PREADY + b);
                mbar_arrive(bar + E_KQ + s);   // done with the slot's gate arrays
                FTRACE(2, j, 1);
            }
            __syncwarp();
            if (j >= 1 && !epilogue(j - 1, osc_prev)) {
                alive = false;
                break;
            }
            osc_prev = osc;
        }
        if (alive && nch > 0) epilogue(nch - 1, osc_prev);
    } else if (warp == 8) {
        // ========================================================= copies
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_tu);
        }
        int issued = 0;
        for (int j = 0; j < nch; ++j) {
            const int s = j % kSlots, b = j & 1;
            const int y = ytok0 + j * kC;
            bool ok = j < kSlots || ctl.wait(E_KQ + s, (uint32_t)(((j / kSlots) - 1) & 1));
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                FTRACE(4, j, 0);
                mbar_arrive_expect_tx(bar + F_KQ + s, (uint32_t)(2 * L::SZ_K));
#pragma unroll
                for (int kb = 0; kb < L::KB; ++kb) {
                    tma_load_3d(sm + L::OFF_K + s * L::SZ_K + kb * 8192, &tm_k, bar + F_KQ + s,
                                kb * 64, y, zc);
                    tma_load_3d(sm + L::OFF_WQ + s * L::SZ_WQ + kb * 16384 + 8192, &tm_q,
                                bar + F_KQ + s, kb * 64, y, zc);
                }
            }
            {
                // the chunk's gate arrays: g = in-chunk cumsum of log_alpha (zero
                // past the sequence), gamma = exp(g), e = exp(g_C - g), and
                // exp(-g), used only when the decay span is moderate (g_C > -80)
                const int Lj = min(kC, len - j * kC);
                const long long r0 = row0 + (long long)j * kC;
                float x0 = lane < Lj ? __ldg(p.log_alpha + r0 + lane) : 0.f;
                float x1 = lane + 32 < Lj ? __ldg(p.log_alpha + r0 + lane + 32) : 0.f;
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
                const float gCv = __shfl_sync(0xffffffffu, x1, 31);
                float *ga = GA(s);
                ga[lane] = x0;
                ga[32 + lane] = x1;
                ga[64 + lane] = __expf(x0);
                ga[96 + lane] = __expf(x1);
                ga[128 + lane] = __expf(gCv - x0);
                ga[160 + lane] = __expf(gCv - x1);
                ga[192 + lane] = __expf(-x0);
                ga[224 + lane] = __expf(-x1);
                mbar_arrive(bar + F_KQ + s);
            }
            ok = j < 2 || ctl.wait(E_TU + b, (uint32_t)(((j >> 1) - 1) & 1));
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                // T_u is the chunk-prep kernel's output: wait for that grid
                if (j == 0) griddep_wait();
                FTRACE(4, j, 1);
                mbar_arrive_expect_tx(bar + F_TU + b, 8192u);
                tma_load_3d(sm + L::OFF_TU + b * 8192, &tm_tu, bar + F_TU + b, 0,
                            (int)(turow0 + (long long)j * 2 * kC), 0);
            }
            ok = j < 1 || ctl.wait(E_TW, (uint32_t)((j - 1) & 1));
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar + F_TW, 8192u);
                tma_load_3d(sm + L::OFF_TW, &tm_tu, bar + F_TW, 0,
                            (int)(turow0 + (long long)j * 2 * kC + kC), 0);
            }
            ok = j < 1 || ctl.wait(E_V, (uint32_t)((j - 1) & 1));
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                FTRACE(4, j, 2);
                mbar_arrive_expect_tx(bar + F_V, 8192u);
                tma_load_3d(sm + L::OFF_V, &tm_v, bar + F_V, dv0, y, zc);
            }
            issued = j + 1;
        }
        // on abort, let copies still in flight land before the CTA exits
        if (lane == 0 && *abort_flag) {
            for (int j = max(0, issued - 2); j < issued; ++j) {
                mbar_wait(bar + F_KQ + j % kSlots, (uint32_t)((j / kSlots) & 1), ctl.limit);
                mbar_wait(bar + F_TU + (j & 1), (uint32_t)((j >> 1) & 1), ctl.limit);
            }
            if (issued > 0) {
                mbar_wait(bar + F_TW, (uint32_t)((issued - 1) & 1), ctl.limit);
                mbar_wait(bar + F_V, (uint32_t)((issued - 1) & 1), ctl.limit);
            }
        }
    } else {
        // ===================== warp 9: W, Gram, U, output; warp 10: chain MMAs
        if (lane == 0 && nch > 0) {
            const uint32_t sb = smem_u32(sm);
            auto sdesc = [&](uint32_t off, uint32_t lbo) {
                return make_sdesc(sb + off, lbo, 1024, kSwizzle128B);
            };
            constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);
            constexpr uint32_t idU = make_idesc_bf16(128, kNV, false, true);
            constexpr uint32_t idW = make_idesc_bf16(128, DK, false, true);
            constexpr uint32_t idM1 = make_idesc_bf16(128, kNV, false, true);
            constexpr uint32_t idM2 = make_idesc_bf16(128, kNV, true, true);
            constexpr uint32_t idO = make_idesc_bf16(128, kNV, false, true);
            if (warp == 10) {
                for (int j = 0; j < nch; ++j) {
                    const int s = j % kSlots, b = j & 1;
                    bool ok = ctl.wait(B_HREADY, j & 1) &&
                              ctl.wait(B_WQ + s, (uint32_t)((j / kSlots) & 1));
                    if (ok && j >= 2) ok = ctl.wait(B_DFREE + b, (uint32_t)(((j >> 1) - 1) & 1));
                    if (!ok) break;
                    FTRACE(3, j, 5);
                    tc_fence_after();
                    // chain MMA 1: D = [-W; Q] H
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk) {
                        const uint32_t a = L::OFF_WQ + s * L::SZ_WQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_bf16(tmem + TM_D + 64 * b, sdesc(a, 16),
                                 sdesc(L::OFF_H + kk * 2048, 16), idM1, kk > 0);
                    }
                    mma_commit(bar + B_M1);
                    if (!ctl.wait(B_VT, j & 1)) break;
                    FTRACE(3, j, 4);
                    tc_fence_after();
                    // chain MMA 2: dH = K^T diag(e) V'
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_bf16(tmem + TM_DH, sdesc(L::OFF_K + s * L::SZ_K + kk * 2048, 8192),
                                 sdesc(L::OFF_H + kk * 2048, 16), idM2, kk > 0);
                    mma_commit(bar + B_M2);
                    mma_commit(bar + E_KQ + s);
                }
                // every issued MMA has finished before tensor memory is released
                mma_commit(bar + B_DRAIN2);
                mbar_wait(bar + B_DRAIN2, 0, ctl.limit);
            } else {
                auto mma_w = [&](int jj) -> bool {
                    const int s = jj % kSlots;
                    bool ok = ctl.wait(F_TW, jj & 1) &&
                              ctl.wait(F_KQ + s, (uint32_t)((jj / kSlots) & 1));
                    if (ok && jj >= 1) ok = ctl.wait(B_WFREE, (jj - 1) & 1);
                    if (!ok) return false;
                    FTRACE(3, jj, 2);
                    tc_fence_after();
                    // W = [T_w; x] K, rows 0-63 used
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_bf16(tmem + TM_W, sdesc(L::OFF_TW + kk * 32, 16),
                                 sdesc(L::OFF_K + s * L::SZ_K + kk * 2048, 8192), idW, kk > 0);
                    mma_commit(bar + B_WDONE);
                    mma_commit(bar + E_TW);
                    return true;
                };
                auto mma_g = [&](int jj) -> bool {
                    const int s = jj % kSlots;
                    bool ok = ctl.wait(F_KQ + s, (uint32_t)((jj / kSlots) & 1));
                    if (ok && jj >= 1) ok = ctl.wait(B_GFREE, (jj - 1) & 1);
                    if (!ok) return false;
                    FTRACE(3, jj, 0);
                    tc_fence_after();
                    // Gram: [-W(stale); Q] K^T, rows 64-127 used
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk) {
                        const uint32_t a = L::OFF_WQ + s * L::SZ_WQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint32_t k = L::OFF_K + s * L::SZ_K + (kk >> 2) * 8192 + (kk & 3) * 32;
                        mma_bf16(tmem + TM_G, sdesc(a, 16), sdesc(k, 16), idG, kk > 0);
                    }
                    mma_commit(bar + B_GDONE);
                    mma_commit(bar + E_KQ + s);   // W and Gram are this issuer's readers of the slot
                    return true;
                };
                auto mma_u = [&](int jj) -> bool {
                    const int b = jj & 1;
                    bool ok = ctl.wait(F_TU + b, (uint32_t)((jj >> 1) & 1)) && ctl.wait(F_V, jj & 1);
                    if (ok && jj >= 2) ok = ctl.wait(B_UFREE + b, (uint32_t)(((jj >> 1) - 1) & 1));
                    if (!ok) return false;
                    FTRACE(3, jj, 1);
                    tc_fence_after();
                    // U = [T_u; x] V, rows 0-63 used
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_bf16(tmem + TM_U + 64 * b, sdesc(L::OFF_TU + b * 8192 + kk * 32, 16),
                                 sdesc(L::OFF_V + kk * 2048, 16), idU, kk > 0);
                    mma_commit(bar + B_UDONE + b);
                    mma_commit(bar + E_V);
                    mma_commit(bar + E_TU + b);
                    return true;
                };
                auto mma_o = [&](int jj) -> bool {
                    const int b = jj & 1;
                    const bool ok = ctl.wait(B_VN + b, (uint32_t)((jj >> 1) & 1)) &&
                                    ctl.wait(B_PREADY + b, (uint32_t)((jj >> 1) & 1));
                    if (!ok) return false;
                    FTRACE(3, jj, 3);
                    tc_fence_after();
                    // output: O += [x; P'] V', rows 64-127 used
                    const uint32_t pa = b ? (uint32_t)L::OFF_TW : (uint32_t)L::OFF_VN;
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_bf16(tmem + TM_D + 64 * b, sdesc(pa + kk * 32, 16),
                                 sdesc(L::OFF_VN + kk * 2048, 16), idO, 1u);
                    mma_commit(bar + B_OUT + b);
                    return true;
                };
                // W and Gram of chunk j + 1 go into the pipe behind chain MMA 1
                // of j (while the chain forms V'), U of j + 1 and j's output
                // product behind chain MMA 2 (while the chain updates H)
                bool ok = mma_w(0) && mma_g(0) && mma_u(0);
                for (int j = 0; ok && j < nch; ++j) {
                    ok = ctl.wait(B_M1, j & 1);
                    if (ok && j + 1 < nch) ok = mma_w(j + 1) && mma_g(j + 1);
                    if (ok) ok = ctl.wait(B_M2, j & 1);
                    if (ok && j + 1 < nch) ok = mma_u(j + 1);
                    if (ok) ok = mma_o(j);
                }
                mma_commit(bar + B_DRAIN);
                mbar_wait(bar + B_DRAIN, 0, ctl.limit);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
#ifdef GDN_TRACE_TIMELINE
    if (tid == 0 && cta_id < 4096) {
        g_fused_cta[cta_id][1] = clock64();
        g_fused_cta[cta_id][3] = nch;
    }
#endif
}

#ifdef GDN_TRACE_TIMELINE
int g_fused_launch_err = 0;
#endif

template <int DK>
gdn_status launch_fused(const FwdArgs &a, const __nv_bfloat16 *Tu) {
    using L = FLay<DK>;
    const long long ydim = a.sm.cu ? a.sm.T_total : a.sm.T;
    const long long zdim = a.sm.cu ? a.sm.H : (long long)a.sm.N * a.sm.H;
    CUtensorMap mq, mk, mv, mt;
    if (!make_map(&mq, a.q, DK, ydim, zdim) || !make_map(&mk, a.k, DK, ydim, zdim) ||
        !make_map(&mv, a.v, a.dv, ydim, zdim) ||
        !make_map(&mt, Tu, 64, (long long)a.sm.H * a.chunk_slots * 2 * kC, 1))
        return GDN_ERR_CUDA;
    // the attribute is a per-device property of the function: set on every call
    if (cudaFuncSetAttribute(k_gdn_fused<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC) != cudaSuccess)
        return GDN_ERR_CUDA;
    FParams p;
    p.sm = a.sm;
    p.log_alpha = a.log_alpha;
    p.h0 = a.h0;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.hT = a.hT;
    p.err = device_error_word();
    p.dv = a.dv;
    const long long lim = option(GDN_OPT_WAIT_LIMIT);
    p.wait_limit = lim > 0 ? (uint32_t)(lim > 0x7fffffffLL ? 0x7fffffffLL : lim) : (1u << 22);
    p.chunk_slots = a.chunk_slots;
    p.max_chunks = a.max_chunks;
    dim3 grid(a.dv / kNV, a.sm.H, a.sm.N);
    const int slot = timer_begin(a.stream, "k_gdn_fused");
    // a programmatic dependent of the chunk-prep kernel: its prologue and first
    // copies of K, Q and V overlap that kernel's tail; T_u is read only after
    // griddepcontrol.wait
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsF);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, k_gdn_fused<DK>, mq, mk, mv, mt, p);
#ifdef GDN_TRACE_TIMELINE
    g_fused_launch_err = (int)le;
#endif
    timer_end(slot, a.stream);
    if (le != cudaSuccess) return GDN_ERR_CUDA;
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

#ifdef GDN_TRACE_TIMELINE
extern "C" int gdn_fused_debug_err() { return g_fused_launch_err; }
#endif

bool fused_supported(const FwdArgs &a) {
    return !a.no_erase && !a.vector_gate && a.dt == GDN_BF16 && (a.dk == 64 || a.dk == 128) &&
           a.dv % kNV == 0 && a.dv <= 256 && a.sm.N <= 65535 && a.sm.H <= 65535 &&
           a.rows > 0 && a.sm.H * a.chunk_slots * (long long)(2 * kC) < 0x7fffffffLL;
}

gdn_status fused_forward(const FwdArgs &a) {
    cudaStream_t st = a.stream;
    __nv_bfloat16 *Tu = nullptr;
    int2 *table = nullptr;
    const size_t tu_bytes = (size_t)a.sm.H * a.chunk_slots * 2 * kC * kC * sizeof(__nv_bfloat16);
    if (scratch_alloc((void **)&Tu, tu_bytes, st) != cudaSuccess) return GDN_ERR_CUDA;
    gdn_status rc = GDN_OK;
    if (a.sm.cu) {
        if (scratch_alloc((void **)&table, sizeof(int2) * (size_t)a.chunk_slots, st) !=
            cudaSuccess)
            rc = GDN_ERR_CUDA;
        else
            rc = enqueue_chunk_table(a, table);
    }
    if (rc == GDN_OK) rc = enqueue_ut(a, table, Tu);
    if (rc == GDN_OK) rc = a.dk == 128 ? launch_fused<128>(a, Tu) : launch_fused<64>(a, Tu);
    scratch_free(Tu, st);
    if (table) scratch_free(table, st);
    return rc;
}

}  // namespace gdn
