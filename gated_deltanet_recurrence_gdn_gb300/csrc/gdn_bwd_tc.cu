// gdn_bwd_tc.cu -- the backward pass's state adjoint on sm_103a tensor cores
// (bf16 I/O).
//
// The adjoint of the chunked forward ("Gated DeltaNet GPU并行实现", section
// 3.2) carries dS, the gradient with respect to a chunk's end state, from the
// last chunk to the first.  One CTA owns one (sequence, head, 64-wide d_v
// tile) and keeps dH = dS^T (d_k x 64, fp32) in registers of its chain
// warpgroup.  Per chunk, with g the in-chunk gate cumsum, gamma_r = exp(g_r),
// e_r = exp(g_C - g_r) and P_rs = exp(g_r - g_s) q_r . k_s (s <= r):
//
//   G    = [K; Q] K^T                 (tcgen05, M = 128; rows 64-127 = Q K^T)
//   D    = diag(gamma) dO             (in place, as the tile lands)
//   P'   = P / gamma_r, from G        (P'_rs = exp(-g_s) (Q K^T)_rs, s <= r; bf16)
//   X    = P'^T D                     (tcgen05; = P^T dO)
//   Y    = Q^T D                      (tcgen05; = (diag(gamma) Q)^T dO)
//   Z    = [K; Q] dH                  (tcgen05, the chain; rows 0-63 used)
//   dV'  = X + diag(e) Z              (stored fp32 for the per-chunk kernel)
//   Y   += W^T (-dV')                 (tcgen05, the chain)
//   dH  <- exp(g_C) dH + Y
//
// When a chunk's total log decay g_C is below -80, exp(-g_s) could overflow:
// that chunk leaves dO unscaled, forms P itself (exp(g_r - g_s) per pair)
// and scales Q by gamma in place after the Gram instead, so X = P^T dO and
// Y = (diag(gamma) Q)^T dO.
//
// This is dV' = P^T dO + diag(e) K dS^T and
// dS <- exp(g_C) dS + dO^T diag(gamma) Q - dV'^T W.  Before stepping dH back
// the CTA stores it: the adjoint of the chunk's end state, which the
// per-chunk gradient kernel (gdn_bwd.cu) reads.
//
// Products take bf16 operands (dH, dV', W, P and gamma Q rounded to bf16;
// K, Q, dO are bf16 inputs) with fp32 accumulation in TMEM; the state
// adjoint itself stays fp32.
//
// Warp roles (352 threads), as in the forward's fused kernel (gdn_tc.cu):
//   warps 0-3  chain warpgroup: owns dH (thread t = d_k index t), forms dV',
//              steps dH back, stores dH and dV'.
//   warps 4-5  gates of the chunk, gamma dO in place, clearing of packed-
//              batch tails.
//   warps 6-7  P' (or P and gamma Q in place) from the Gram in TMEM.
//   warp 8     bulk tensor copies (one lane) of K, Q, W and dO tiles, and
//              the chunk's gate cumsum (all lanes, one chunk ahead).
//   warp 9     chain MMA issuer (one lane): Z and the W^T (-dV') update;
//              TMEM owner.
//   warp 10    prep MMA issuer (one lane): G, X and Y.
// Every wait is bounded; a wait that gives up sets the device error word and
// makes every role leave its loop, after which in-flight MMAs are drained and
// TMEM is freed.  Rows past the end of a sequence are zero (bulk-copy fill,
// or cleared when they belong to the next packed sequence) and their gate
// cumsum repeats the last real row's, which leaves every real row unchanged.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gdn_bwd_tc.h"
#include "gdn_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

// Optional per-phase timeline of CTA (0,0,0) for profiling builds
// (-DGDN_TRACE_TIMELINE): clock64() stamps by role, chunk and event, read back
// with gdn_bwd_trace_read().  Compiled out otherwise.
#ifdef GDN_TRACE_TIMELINE
__device__ long long g_bwd_trace[5][128][8];
extern "C" int gdn_bwd_trace_read(long long *out) {
    return (int)cudaMemcpyFromSymbol(out, g_bwd_trace, sizeof(g_bwd_trace));
}
#define BTRACE(role, jj, ev, cond)                                                         \
    do {                                                                                   \
        if ((cond) && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (jj) < 128) \
            g_bwd_trace[role][jj][ev] = clock64();                                         \
    } while (0)
#else
#define BTRACE(role, jj, ev, cond) \
    do {                           \
    } while (0)
#endif

namespace gdn {
namespace {

using namespace ptx;
using namespace tcx;

constexpr int kC = 64;          // chunk length
constexpr int kNV = 64;         // d_v columns per CTA
constexpr int kNS = 2;          // input stages
constexpr int kThreadsB = 352;

// mbarrier slots
enum {
    B_FULL = 0,                 // + stage: bulk copies and gate lanes landed
    B_READY = B_FULL + kNS,     // + stage: gates derived, tails cleared
    B_FREE = B_READY + kNS,     // + stage: every product reading it is done
    B_PREADY = B_FREE + kNS,    // + (j & 1): P written, Q scaled
    B_PFREE = B_PREADY + 2,     // + (j & 1): X has read the P buffer
    B_X = B_PFREE + 2,          // + (j & 1): X done
    B_Y = B_X + 2,              // + (j & 1): Y done
    B_G = B_Y + 2,              // Gram done
    B_GFREE,                    // P warps have read the Gram
    B_Z,                        // Z done
    B_U,                        // Y - W^T dV' done
    B_DRAIN,                    // chain MMA issuer drained
    B_DRAIN2,                   // prep MMA issuer drained
    B_COUNT
};

template <int DK>
struct BLay {
    static constexpr int KB = DK / 64;                 // 64-column blocks of K / Q / W
    // One input stage (tiles of 64 rows x 128 B, 128-byte swizzled): per
    // block [K | Q] (so [K; Q] is one 128-row operand and Q^T one MN-major
    // operand with a 16 KiB block stride), then the W blocks (W^T: 8 KiB
    // stride), then the dO tile.
    static constexpr int OFF_W = KB * 16384;
    static constexpr int OFF_DO = OFF_W + KB * 8192;
    static constexpr int STAGE = OFF_DO + 8192;
    static constexpr int OFF_P = kNS * STAGE;           // two P buffers
    static constexpr int OFF_VN = OFF_P + 2 * 8192;     // -dV' (bf16)
    static constexpr int OFF_H = OFF_VN + 8192;         // dH (bf16), DK rows
    // fp32 staging of the stored dH (DK rows) and dV' (64 rows) for bulk
    // tensor stores: two 32-column halves of 128-byte rows each
    static constexpr int OFF_SH = OFF_H + DK * 128;
    static constexpr int OFF_SV = OFF_SH + DK * 256;
    static constexpr int GSZ = 4 * 64;                  // g, gamma, e, 1 / gamma
    static constexpr int OFF_G = OFF_SV + 64 * 256;     // 2 x GSZ floats
    static constexpr int OFF_GS = OFF_G + 2 * GSZ * 4;  // per stage: raw gate cumsum
    static constexpr int OFF_BAR = OFF_GS + kNS * 64 * 4;
    static constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 64;
    static constexpr int ALLOC = TOTAL + 1024;
    static_assert(STAGE % 1024 == 0 && OFF_P % 1024 == 0 && OFF_VN % 1024 == 0 &&
                      OFF_H % 1024 == 0 && OFF_SH % 1024 == 0 && OFF_SV % 1024 == 0 &&
                      OFF_BAR % 8 == 0,
                  "align");
    // the second 64-row half of an M = 128 operand read past its tile stays
    // inside the allocation: [P^T; x] ends at OFF_VN + 8 KiB, (gamma Q)^T and
    // W^T of a d_k = 64 stage end inside the stage
    static_assert(OFF_VN + 8192 <= TOTAL, "operand halves");
    static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

// Eight bf16 values times `f`, rounded back to bf16.
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float f) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        w[e] = pack_bf16(f2.x * f, f2.y * f);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// TMEM column map (512 allocated): Gram (lanes 64-127 hold Q K^T), X and Y
// double-buffered by chunk parity, Z.
constexpr uint32_t TM_G = 0, TM_X = 64, TM_Z = 192, TM_Y = 256;

struct BwdTcParams {
    SeqMap sm;
    const float *G;        // in-chunk gate cumsum [rows]
    const float *dhT;      // [seq][H][d_v][d_k] or null (zero)
    float *dh0;            // [seq][H][d_v][d_k] or null (not written)
    float *dVn;            // [rows][d_v]
    float *dHc;            // [H][chunk_slots][d_k][d_v]
    int *err;
    int dv;
    int max_chunks;        // dense batches: chunk slot n * max_chunks + c
    long long chunk_slots;
    uint32_t wait_limit;
};

template <int DK>
__global__ void __launch_bounds__(kThreadsB, 1)
k_bwd_dstate_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dh, const __grid_constant__ CUtensorMap tm_dv,
                BwdTcParams p) {
    using L = BLay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    // chunk index + 1 of the last dH / -dV' the chain published
    uint32_t *h_flag = misc + 2, *vn_flag = misc + 3;
    float *gb = reinterpret_cast<float *>(sm + L::OFF_G);   // [2][GSZ]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dv0 = blockIdx.x * kNV, h = blockIdx.y, n = blockIdx.z;

    // ---- sequence bounds (validated; an invalid packed range is an error)
    long long row0 = 0, slot0 = 0;
    int len = 0, ytok0 = 0, zcoord = 0;
    bool ok_seq = true;
    if (p.sm.cu) {
        const int a = __ldg(p.sm.cu + n), b = __ldg(p.sm.cu + n + 1);
        ok_seq = a >= 0 && a <= b && b <= p.sm.T_total;
        if (ok_seq) {
            row0 = (long long)h * p.sm.T_total + a;
            len = b - a;
            slot0 = (long long)(a / kC) + n;
        }
        ytok0 = a;
        zcoord = h;
    } else {
        row0 = ((long long)n * p.sm.H + h) * (long long)p.sm.T;
        len = p.sm.T;
        zcoord = n * p.sm.H + h;
        slot0 = (long long)n * p.max_chunks;
    }
    if (!ok_seq) {
        if (tid == 0) atomicCAS(p.err, 0, kErrBadIndex);
        return;  // before any barrier or TMEM use
    }
    const int nch = (len + kC - 1) / kC;
    const long long srow = ((long long)n * p.sm.H + h) * p.dv;   // state row of (n, h)
    const uint32_t sbase = smem_u32(sm);

    if (warp == 9) {
        tmem_alloc(misc, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar + i, 1);
        for (int s = 0; s < kNS; ++s) mbar_init(bar + B_FREE + s, 2);    // both MMA issuers
        for (int s = 0; s < kNS; ++s) mbar_init(bar + B_FULL + s, 33);   // copies + 32 gate lanes
        *abort_flag = 0;
        *h_flag = 0;
        *vn_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};

    if (warp < 4) {
        // ================================================= chain warpgroup
        const int t = tid;   // d_k index of the dH row / token row of dV'
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float hreg[kNV];
#pragma unroll
        for (int c = 0; c < kNV; ++c)
            hreg[c] = (t < DK && p.dhT) ? __ldg(p.dhT + (srow + dv0 + c) * DK + t) : 0.f;
        uint8_t *Hs = sm + L::OFF_H, *VNs = sm + L::OFF_VN;
        uint8_t *SH = sm + L::OFF_SH, *SV = sm + L::OFF_SV;
        bool alive = true;
        for (int j = 0; j < nch; ++j) {
            const int c = nch - 1 - j, s = j % kNS, bsel = j & 1;
            const int Lc = min(kC, len - c * kC);
            const long long r0 = row0 + (long long)c * kC;
            BTRACE(0, j, 0, t == 0);
            // (i) publish dH as the bf16 B operand of Z, then store it: the
            // adjoint of chunk c's end state
            if (t < DK) put_row64(Hs, t, hreg);
            fence_proxy_async_smem();
            tc_fence_before();
            if (t == 0) bulk_wait_read();   // the staging tiles' last stores have read them
            named_bar(1, 128);
            if (t == 0) st_release_cta(h_flag, (uint32_t)j + 1);
            BTRACE(0, j, 1, t == 0);
            // out through the staging tile and two bulk tensor stores (a
            // thread's own 256-byte row scattered across the warp's stores
            // would touch 32 rows per instruction)
            if (t < DK) put_row64_f32(SH, DK, t, hreg);
            fence_proxy_async_smem();
            named_bar(1, 128);
            if (t == 0) {
                const int y = (int)((h * p.chunk_slots + slot0 + c) * DK);
                tma_store_2d(&tm_dh, SH, dv0, y);
                tma_store_2d(&tm_dh, SH + DK * 128, dv0 + 32, y);
                bulk_commit();
            }
            // (ii) dV' = X + diag(e) Z; -dV' is the bf16 B operand of the update
            {
                bool ok = ctl.wait(B_READY + s, (j / kNS) & 1);
                ok = ok && ctl.wait(B_X + bsel, (j >> 1) & 1) && ctl.wait(B_Z, j & 1);
                if (!named_bar_and(1, 128, ok)) {
                    alive = false;
                    break;
                }
            }
            BTRACE(0, j, 2, t == 0);
            tc_fence_after();
            const float *gj = gb + bsel * L::GSZ;
            // kept in a register: the gate buffer is refilled once this chunk's
            // update MMA has been issued
            const float decayC = gj[64 + 63];
            // dV' rows by bulk tensor store where the box holds this sequence's
            // rows only (dense batches: rows past T are clipped; a packed
            // batch's partial chunk is followed by the next sequence's rows)
            const bool bulk_dv = !p.sm.cu || Lc == kC;
            if (t < kC) {
                const float ev = gj[128 + t];
                float *dvp = (!bulk_dv && t < Lc) ? p.dVn + (r0 + t) * p.dv + dv0 : nullptr;
                const uint32_t ax = tmem + lane_base + TM_X + bsel * 64;
                const uint32_t az = tmem + lane_base + TM_Z;
#pragma unroll
                for (int qt = 0; qt < 4; ++qt) {
                    float xv[16], zv[16];
                    tmem_ld16f(ax + 16 * qt, xv);
                    tmem_ld16f(az + 16 * qt, zv);
#pragma unroll
                    for (int i = 0; i < 16; ++i) xv[i] = fmaf(ev, zv[i], xv[i]);
                    if (bulk_dv) {
                        uint8_t *sv = SV + (qt >> 1) * 8192;
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            *reinterpret_cast<float4 *>(sv + sw128_offset(t, (qt & 1) * 4 + u)) =
                                make_float4(xv[4 * u], xv[4 * u + 1], xv[4 * u + 2],
                                            xv[4 * u + 3]);
                    } else if (dvp) {
                        float4 *d4 = reinterpret_cast<float4 *>(dvp + 16 * qt);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_float4(xv[4 * q], xv[4 * q + 1], xv[4 * q + 2],
                                                xv[4 * q + 3]);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) xv[i] = -xv[i];
                    put8(VNs, t, 2 * qt, xv);
                    put8(VNs, t, 2 * qt + 1, xv + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 128);
            if (t == 0) {
                st_release_cta(vn_flag, (uint32_t)j + 1);
                if (bulk_dv) {
                    const int y = ytok0 + c * kC;
                    tma_store_3d(&tm_dv, SV, dv0, y, zcoord);
                    tma_store_3d(&tm_dv, SV + 8192, dv0 + 32, y, zcoord);
                    bulk_commit();
                }
            }
            BTRACE(0, j, 3, t == 0);
            // (iii) dH <- exp(g_C) dH + (Y - W^T dV')
            if (!named_bar_and(1, 128, ctl.wait(B_U, j & 1))) {
                alive = false;
                break;
            }
            BTRACE(0, j, 4, t == 0);
            tc_fence_after();
            if (t < DK) {
                uint32_t y0[32], y1[32];
                const uint32_t ay = tmem + lane_base + TM_Y + bsel * 64;
                tmem_ld32(ay, y0);
                tmem_ld32(ay + 32, y1);
                tmem_wait32(y0);
                tmem_wait32(y1);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    hreg[i] = fmaf(decayC, hreg[i], f32(y0[i]));
                    hreg[32 + i] = fmaf(decayC, hreg[32 + i], f32(y1[i]));
                }
            }
        }
        if (alive && p.dh0 && t < DK) {
#pragma unroll
            for (int c = 0; c < kNV; ++c) p.dh0[(srow + dv0 + c) * DK + t] = hreg[c];
        }
        if (t == 0) bulk_wait_all();   // every store done before the CTA leaves
    } else if (warp < 6) {
        // ======================================================= gate warps
        const int t = tid - 128;   // row of the chunk
        for (int j = 0; j < nch; ++j) {
            const int c = nch - 1 - j, s = j % kNS;
            const int Lc = min(kC, len - c * kC);
            uint8_t *stg = sm + s * L::STAGE;
            float *gj = gb + (j & 1) * L::GSZ;
            if (!named_bar_and(4, 64, ctl.wait(B_FULL + s, (j / kNS) & 1))) break;
            BTRACE(1, j, 3, t == 0);
            {
                const float *gs = reinterpret_cast<const float *>(sm + L::OFF_GS) + s * 64;
                const float gt = gs[t], gC = gs[63];
                const float gam = __expf(gt);
                gj[t] = gt;
                gj[64 + t] = gam;
                gj[128 + t] = __expf(gC - gt);
                gj[192 + t] = __expf(-gt);   // used only when the span is < 80
                if (gC > -80.f) {
                    // D = diag(gamma) dO: row t of the dO tile in place
                    uint8_t *ds = stg + L::OFF_DO;
                    uint4 v[8];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        v[ch] = *reinterpret_cast<const uint4 *>(ds + sw128_offset(t, ch));
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        v[ch] = scale_bf16x8(v[ch], gam);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        *reinterpret_cast<uint4 *>(ds + sw128_offset(t, ch)) = v[ch];
                }
            }
            if (p.sm.cu && Lc < kC) {
                // rows past this sequence belong to the next one: clear them
                constexpr int per_row = 3 * DK / 8 + 8;   // 16-byte pieces: K, Q, W, dO
                for (int i = t; i < (kC - Lc) * per_row; i += 64) {
                    const int r = Lc + i / per_row, q = i % per_row;
                    uint8_t *base;
                    if (q < DK / 8)   // K
                        base = stg + (q >> 3) * 16384;
                    else if (q < 2 * DK / 8)   // Q
                        base = stg + ((q - DK / 8) >> 3) * 16384 + 8192;
                    else if (q < 3 * DK / 8)   // W
                        base = stg + L::OFF_W + ((q - 2 * DK / 8) >> 3) * 8192;
                    else   // dO
                        base = stg + L::OFF_DO;
                    st16(base + sw128_offset(r, q & 7), 0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            named_bar(4, 64);
            if (t == 0) mbar_arrive(bar + B_READY + s);
            BTRACE(1, j, 4, t == 0);
        }
    } else if (warp < 8) {
        // ========================================================== P warps
        const int r = tid - 192;   // row of the chunk = TMEM lane 64 + r of the Gram
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        for (int j = 0; j < nch; ++j) {
            const int s = j % kNS, bsel = j & 1;
            uint8_t *stg = sm + s * L::STAGE;
            const float *gj = gb + bsel * L::GSZ;
            bool ok = ctl.wait(B_READY + s, (j / kNS) & 1) && ctl.wait(B_G, j & 1);
            if (j >= 2) ok = ok && ctl.wait(B_PFREE + bsel, ((j - 2) >> 1) & 1);
            if (!named_bar_and(3, 64, ok)) break;
            BTRACE(1, j, 1, r == 0);
            tc_fence_after();
            uint32_t g0[32], g1[32];
            tmem_ld32(tmem + lane_base + TM_G, g0);
            tmem_ld32(tmem + lane_base + TM_G + 32, g1);
            const float gr = gj[r], gam = gj[64 + r];
            const bool span_ok = gj[63] > -80.f;
            uint8_t *Pt = sm + L::OFF_P + bsel * 8192;
            tmem_wait32(g0);
            tmem_wait32(g1);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int sidx = 32 * half + i;
                    const bool keep = sidx <= r;
                    const float gv = f32(half == 0 ? g0[i] : g1[i]);
                    // span_ok: P' = exp(-g_s) (q_r . k_s), to pair with gamma dO;
                    // else P itself
                    const float f = span_ok ? gj[192 + sidx]
                                            : __expf(keep ? gr - gj[sidx] : 0.f);
                    x[i] = keep ? f * gv : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) put8(Pt, r, 4 * half + q, x + 8 * q);
            }
            if (!span_ok) {
                // gamma_r Q in place (the Gram has read Q): row r of every
                // block, all loads first, then all stores
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    uint8_t *qs = stg + blk * 16384 + 8192;
                    uint4 v[8];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        v[ch] = *reinterpret_cast<const uint4 *>(qs + sw128_offset(r, ch));
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) v[ch] = scale_bf16x8(v[ch], gam);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        *reinterpret_cast<uint4 *>(qs + sw128_offset(r, ch)) = v[ch];
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(3, 64);
            if (r == 0) {
                mbar_arrive(bar + B_PREADY + bsel);
                mbar_arrive(bar + B_GFREE);
            }
            BTRACE(1, j, 2, r == 0);
        }
    } else if (warp == 8) {
        // ================================================= TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_do);
        }
        int issued = 0;
        // the next chunk's gate cumsum, loaded one chunk ahead; rows past the
        // sequence repeat its last row
        float pg0 = 0.f, pg1 = 0.f;
        auto load_gates = [&](int jj) {
            const int c = nch - 1 - jj;
            const long long r0 = row0 + (long long)c * kC;
            const int Lc = min(kC, len - c * kC);
            pg0 = __ldg(p.G + r0 + min(lane, Lc - 1));
            pg1 = __ldg(p.G + r0 + min(lane + 32, Lc - 1));
        };
        if (nch > 0) load_gates(0);
        for (int j = 0; j < nch; ++j) {
            const int c = nch - 1 - j, s = j % kNS;
            const bool ok = j < kNS || ctl.wait(B_FREE + s, ((j / kNS) - 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            BTRACE(4, j, 0, lane == 0);
            uint8_t *stg = sm + s * L::STAGE;
            uint64_t *fb = bar + B_FULL + s;
            const int y = ytok0 + c * kC;
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, (uint32_t)L::STAGE);
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    tma_load_3d(stg + blk * 16384, &tm_k, fb, blk * 64, y, zcoord);
                    tma_load_3d(stg + blk * 16384 + 8192, &tm_q, fb, blk * 64, y, zcoord);
                    tma_load_3d(stg + L::OFF_W + blk * 8192, &tm_w, fb, blk * 64, y, zcoord);
                }
                tma_load_3d(stg + L::OFF_DO, &tm_do, fb, dv0, y, zcoord);
            }
            float *gs = reinterpret_cast<float *>(sm + L::OFF_GS) + s * 64;
            gs[lane] = pg0;
            gs[32 + lane] = pg1;
            mbar_arrive(fb);
            if (j + 1 < nch) load_gates(j + 1);
            issued = j + 1;
        }
        // on abort, let copies still in flight land before the CTA exits
        if (lane == 0 && *abort_flag) {
            for (int j = max(0, issued - kNS); j < issued; ++j)
                mbar_wait(bar + B_FULL + j % kNS, (j / kNS) & 1, ctl.limit);
        }
    } else if (warp == 9) {
        // ===================================== chain MMA issuer (and TMEM owner)
        if (lane == 0 && nch > 0) {
            constexpr uint32_t idZ = make_idesc_bf16(128, kNV, false, true);   // [K; Q] dH
            constexpr uint32_t idU = make_idesc_bf16(128, kNV, true, true);    // W^T (-dV')
            // descriptor bases; an operand at base + off is base_desc + (off >> 4)
            const uint64_t dS = make_sdesc(sbase, 16, 1024, kSwizzle128B);
            const uint64_t dH = make_sdesc(sbase + L::OFF_H, 16, 1024, kSwizzle128B);
            const uint64_t dWT = make_sdesc(sbase + L::OFF_W, 8192, 1024, kSwizzle128B);
            const uint64_t dVN = make_sdesc(sbase + L::OFF_VN, 16, 1024, kSwizzle128B);
            for (int j = 0; j < nch; ++j) {
                const int s = j % kNS, bsel = j & 1;
                const uint32_t soff = s * L::STAGE;
                if (!ctl.wait(B_READY + s, (j / kNS) & 1) || !ctl.flag(h_flag, (uint32_t)j + 1))
                    break;
                BTRACE(2, j, 0, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = soff + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_Z, dS + (off >> 4), dH + (kk * 2048 >> 4), idZ, kk > 0);
                }
                mma_commit(bar + B_Z);
                BTRACE(2, j, 1, true);
                // Y of this chunk is complete before the update accumulates onto it
                if (!ctl.wait(B_Y + bsel, (j >> 1) & 1) || !ctl.flag(vn_flag, (uint32_t)j + 1))
                    break;
                BTRACE(2, j, 2, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_bf16(tmem + TM_Y + bsel * 64, dWT + ((soff + kk * 2048) >> 4),
                             dVN + (kk * 2048 >> 4), idU, 1u);
                mma_commit(bar + B_U);
                mma_commit(bar + B_FREE + s);
                BTRACE(2, j, 3, true);
            }
            // every issued MMA has finished before TMEM is released
            mma_commit(bar + B_DRAIN);
            mbar_wait(bar + B_DRAIN, 0, ctl.limit);
        }
    } else {
        // ============================================== prep MMA issuer
        if (lane == 0 && nch > 0) {
            constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);   // [K; Q] K^T
            constexpr uint32_t idXY = make_idesc_bf16(128, 64, true, true);    // P^T dO, (gQ)^T dO
            const uint64_t dS = make_sdesc(sbase, 16, 1024, kSwizzle128B);
            const uint64_t dP = make_sdesc(sbase + L::OFF_P, 8192, 1024, kSwizzle128B);
            const uint64_t dQT = make_sdesc(sbase + 8192, 16384, 1024, kSwizzle128B);
            for (int j = 0; j < nch; ++j) {
                const int s = j % kNS, bsel = j & 1;
                const uint32_t soff = s * L::STAGE;
                if (!ctl.wait(B_READY + s, (j / kNS) & 1)) break;
                if (j > 0 && !ctl.wait(B_GFREE, (j - 1) & 1)) break;   // Gram of j-1 read
                BTRACE(3, j, 0, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    // A = [K; Q] and B = K start at the same block
                    const uint32_t off = soff + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_G, dS + (off >> 4), dS + (off >> 4), idG, kk > 0);
                }
                mma_commit(bar + B_G);
                BTRACE(3, j, 1, true);
                if (!ctl.wait(B_PREADY + bsel, (j >> 1) & 1)) break;   // P written, Q scaled
                // X's accumulator was read by the chain two chunks ago
                if (j >= 2 && !ctl.flag(vn_flag, (uint32_t)j - 1)) break;
                BTRACE(3, j, 2, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_bf16(tmem + TM_X + bsel * 64, dP + ((bsel * 8192 + kk * 2048) >> 4),
                             dS + ((soff + L::OFF_DO + kk * 2048) >> 4), idXY, kk > 0);
                mma_commit(bar + B_X + bsel);
                mma_commit(bar + B_PFREE + bsel);
                BTRACE(3, j, 3, true);
                // Y's accumulator: the chain stepped dH with it two chunks ago
                if (j >= 2 && !ctl.flag(h_flag, (uint32_t)j)) break;
                BTRACE(3, j, 4, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_bf16(tmem + TM_Y + bsel * 64, dQT + ((soff + kk * 2048) >> 4),
                             dS + ((soff + L::OFF_DO + kk * 2048) >> 4), idXY, kk > 0);
                mma_commit(bar + B_Y + bsel);
                mma_commit(bar + B_FREE + s);
                BTRACE(3, j, 5, true);
            }
            mma_commit(bar + B_DRAIN2);
            mbar_wait(bar + B_DRAIN2, 0, ctl.limit);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

template <int DK>
gdn_status launch_bwd_tc(const FwdArgs &a, const BwdArgs &b, const __nv_bfloat16 *Wb,
                         const float *G, float *dVn, float *dHc) {
    using L = BLay<DK>;
    const long long ydim = a.sm.cu ? a.sm.T_total : a.sm.T;
    const long long zdim = a.sm.cu ? a.sm.H : (long long)a.sm.N * a.sm.H;
    CUtensorMap mq, mk, mw, mdo, mdh, mdv;
    if (!make_map(&mq, a.q, DK, ydim, zdim) || !make_map(&mk, a.k, DK, ydim, zdim) ||
        !make_map(&mw, Wb, DK, ydim, zdim) || !make_map(&mdo, b.dout, a.dv, ydim, zdim) ||
        !make_map_f32(&mdh, dHc, a.dv, (long long)a.sm.H * a.chunk_slots * DK, DK) ||
        !make_map_f32_3d(&mdv, dVn, a.dv, ydim, zdim))
        return GDN_ERR_CUDA;
    // a per-function attribute of the current device: cheap, set on every launch
    if (cudaFuncSetAttribute(k_bwd_dstate_tc<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC) != cudaSuccess)
        return GDN_ERR_CUDA;
    BwdTcParams p;
    p.sm = a.sm;
    p.G = G;
    p.dhT = b.dhT;
    p.dh0 = b.dh0;
    p.dVn = dVn;
    p.dHc = dHc;
    p.err = device_error_word();
    p.dv = a.dv;
    p.max_chunks = a.max_chunks;
    p.chunk_slots = a.chunk_slots;
    const long long lim = option(GDN_OPT_WAIT_LIMIT);
    p.wait_limit = lim > 0 ? (uint32_t)(lim > 0x7fffffffLL ? 0x7fffffffLL : lim) : (1u << 22);
    const dim3 grid(a.dv / kNV, a.sm.H, a.sm.N);
    k_bwd_dstate_tc<DK><<<grid, kThreadsB, L::ALLOC, a.stream>>>(mq, mk, mw, mdo, mdh, mdv, p);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

bool tc_bwd_supported(const FwdArgs &a) {
    if (a.dt != GDN_BF16 || a.vector_gate) return false;
    if (a.dk != 64 && a.dk != 128) return false;
    if (a.dv % kNV != 0) return false;
    if (a.sm.N > 65535 || a.sm.H > 65535 || a.rows <= 0) return false;
    static std::atomic<int> memo[kMaxDeviceMemo];
    return per_device(
               memo, [](int) { return (device_is_sm10x() && encode_fn() != nullptr) ? 1 : 0; },
               0) == 1;
}

gdn_status tc_bwd_dstate(const FwdArgs &a, const BwdArgs &b, const __nv_bfloat16 *Wb,
                         const float *G, float *dVn, float *dHc) {
    if (!tc_bwd_supported(a)) return GDN_ERR_UNSUPPORTED;
    if (a.sm.N <= 0 || a.sm.H <= 0) return GDN_OK;
    return a.dk == 128 ? launch_bwd_tc<128>(a, b, Wb, G, dVn, dHc)
                       : launch_bwd_tc<64>(a, b, Wb, G, dVn, dHc);
}

}  // namespace gdn
