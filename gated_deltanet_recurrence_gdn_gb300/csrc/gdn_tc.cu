// gdn_tc.cu -- fused chunked gated delta rule forward on sm_103a tensor cores.
//
// One CTA owns one (sequence, head, 64-wide d_v tile) and walks its chunks of
// C = 64 tokens in order ("Gated DeltaNet GPU并行实现", section 3.2: matrix
// products inside a chunk, a serial state pass across chunks).  The chunk-prep
// kernel (gdn_prep.cu) has already written, per chunk, T_u = T diag(beta) and
// W = T diag(beta gamma) K with T = (I + A)^{-1}.  With H = S^T (d_k x 64 tile
// of the state, fp32, kept in registers of the chain warpgroup), g_r the
// in-chunk cumulative log gate and gamma_r = exp(g_r):
//
//   G     = [W; Q] K^T                         (tcgen05, M = 128; rows 64-127 used)
//   P'_rs = exp(-g_s) (Q K^T)_rs,  s <= r      (= P_rs / gamma_r)
//   U     = T_u V                              (tcgen05)
//   [W H; Q H] = [W; Q] H                      (tcgen05, the chain MMA)
//   V'    = U - W H
//   dH    = K^T diag(exp(g_C - g_r)) V'        (tcgen05)
//   O     = diag(gamma) (Q H + P' V')          (tcgen05 accumulate; gamma on store)
//   H    <- exp(g_C) H + dH
//
// When a chunk's total log decay g_C is below -80, exp(-g_s) could overflow:
// that chunk instead scales Q by gamma in place after the Gram, forms
// P_rs = exp(g_r - g_s) (Q K^T)_rs directly and stores O unscaled.
//
// Warp roles (352 threads):
//   warps 0-3  chain warpgroup: owns H (thread t = row t = d_k index t), forms
//              V', updates H, stores O a chunk late from a second TMEM
//              accumulator, off the state's critical path.
//   warps 4-5  gates of the chunk, clearing of packed-batch tails.
//   warps 6-7  P' from the Gram in TMEM, as the bf16 operand of P' V'.
//   warp 8     bulk tensor copies (one lane) of K, W, Q, V and T_u tiles, and
//              the next chunk's gates (all lanes, prefetched in registers).
//   warp 9     chain MMA issuer (one lane): [W; Q] H, K^T V~, P' V'; TMEM owner.
//   warp 10    prep MMA issuer (one lane): [W; Q] K^T, T_u V.
// Every wait is bounded; a wait that gives up sets the device error word and
// makes every role leave its loop, after which in-flight MMAs are drained and
// TMEM is freed.
//
// Rows past the end of a sequence are zero (bulk-copy fill, or cleared by
// warps 4-5 when they belong to the next packed sequence) with
// beta = log_alpha = 0, which leaves every real row unchanged.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>

#include "gdn_bwd_tc.h"
#include "gdn_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

// Optional per-phase timeline of CTA (0,0,0) for profiling builds
// (-DGDN_TRACE_TIMELINE): clock64() stamps by role, chunk and event, read back
// with gdn_trace_read(), and every CTA's start and end, read back with
// gdn_cta_trace_read().  Compiled out otherwise.
#ifdef GDN_TRACE_TIMELINE
__device__ long long g_gdn_trace[4][128][16];
extern "C" int gdn_trace_read(long long *out) {
    return (int)cudaMemcpyFromSymbol(out, g_gdn_trace, sizeof(g_gdn_trace));
}
#define TRACE(role, jj, ev, cond)                                                          \
    do {                                                                                   \
        if ((cond) && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (jj) < 128) \
            g_gdn_trace[role][jj][ev] = clock64();                                         \
    } while (0)
// per CTA (linear index < 4096): global-timer start and end (ns), SM id
__device__ long long g_gdn_cta[4096][3];
extern "C" int gdn_cta_trace_read(long long *out) {
    return (int)cudaMemcpyFromSymbol(out, g_gdn_cta, sizeof(g_gdn_cta));
}
__device__ __forceinline__ long long gtimer() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int smid() {
    int r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}
#define CTA_SPAN(slot)                                                                     \
    do {                                                                                   \
        const long long lin_ = ((long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + \
                               blockIdx.x;                                                 \
        if (threadIdx.x == 0 && lin_ < 4096) {                                             \
            g_gdn_cta[lin_][slot] = gtimer();                                              \
            g_gdn_cta[lin_][2] = smid();                                                   \
        }                                                                                  \
    } while (0)
#else
#define TRACE(role, jj, ev, cond) \
    do {                          \
    } while (0)
#define CTA_SPAN(slot) \
    do {               \
    } while (0)
#endif

#include "gdn_utw.cuh"   // the chunk prep's pipeline, run beside the chain by k_gdn_tc_ov

namespace gdn {
namespace {

using namespace ptx;
using namespace tcx;

constexpr int kC = 64;         // chunk length
constexpr int kNV = 64;        // d_v columns per CTA
constexpr int kNS = 2;         // input stages
constexpr int kThreadsTC = 352;

// mbarrier slots
enum {
    B_FULL = 0,                 // + stage: TMA bytes landed
    B_READY = B_FULL + kNS,     // + stage: pad rows cleared, stage usable by MMA
    B_FREE = B_READY + kNS,     // + stage: consumers done (chain MMA commit + prep)
    B_PFREE = B_FREE + kNS,     // + (chunk & 1): P buffer read by the output MMA
    B_PREADY = B_PFREE + 2,     // + (chunk & 1): P buffer written
    B_G = B_PREADY + 2,         // Gram MMA done (G in TMEM)
    B_GFREE,                    // prep has read G
    B_UW,                       // U and W in TMEM
    B_WQ,                       // [W; Q] (or [W; gamma Q]) in smem for the chain MMA
    B_M2,                       // chain MMA done
    B_VN,                       // V' (bf16) in smem, U consumed
    B_M34,                      // dH and O done
    B_DRAIN,                    // chain MMA issuer drained
    B_DRAIN2,                   // prep MMA issuer drained
    B_M34I,                     // K^T V~ and the output MMA of the chunk issued
    B_HPUB,                     // bf16 H of the chunk in smem (chain -> chain MMA issuer)
    B_COUNT
};

template <int DK>
struct Lay {
    static constexpr int KB = DK / 64;                 // 64-column blocks of K / Q / W
    // One input stage (all tiles 64 rows x 128 B, 128-byte swizzled):
    //   K blocks, then V (so [K | V] would be one operand with 8 KiB block
    //   stride and K^T is one MN-major operand), per block [W | Q] (so
    //   [W; Q] is one 128-row operand), then T_u.
    static constexpr int OFF_V = KB * 8192;
    static constexpr int OFF_WQ = OFF_V + 8192;
    static constexpr int OFF_TU = OFF_WQ + KB * 16384;
    static constexpr int STAGE = OFF_TU + 8192;
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_H = OFF_STAGE + kNS * STAGE;   // DK rows x 128 B
    static constexpr int OFF_R0 = OFF_H + DK * 128;    // [V~ | P0]
    static constexpr int OFF_R1 = OFF_R0 + 16384;      // [V' | P1]
    static constexpr int GSZ = 5 * 64;                 // g, beta, gamma, 1/gamma, beta*gamma
    static constexpr int OFF_G = OFF_R1 + 16384;       // 2 x GSZ floats
    static constexpr int OFF_GS = OFF_G + 2 * GSZ * 4;  // per stage raw gates: log_alpha, beta
    static constexpr int OFF_BAR = OFF_GS + kNS * 128 * 4;
    static constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 64;
    static constexpr int ALLOC = TOTAL + 1024;
    // the backward's state pass only: an fp32 staging tile for bulk tensor
    // stores of each chunk's starting state (DK rows) and then of its V'
    // rows (64), two 32-column halves of 128-byte rows
    static constexpr int OFF_STG = (TOTAL + 1023) / 1024 * 1024;
    static constexpr int ALLOC_S = OFF_STG + DK * 256 + 1024;
    static_assert(ALLOC_S <= 227 * 1024, "shared memory budget (state pass)");
    static_assert(OFF_WQ % 1024 == 0 && OFF_TU % 1024 == 0 && STAGE % 1024 == 0, "align");
    static_assert(OFF_H % 1024 == 0 && OFF_R0 % 1024 == 0 && OFF_G % 16 == 0, "align");
    static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

// TMEM column map (512 allocated): [W; Q] K^T (its lanes 64-127 hold Q K^T),
// two chain / output accumulators, dH, and U = T_u V (lanes 0-63).
constexpr uint32_t TM_G = 0, TM_M2 = 64, TM_H = 192, TM_U = 256;

struct TcParams {
    SeqMap sm;
    const float *log_alpha, *beta, *h0;
    __nv_bfloat16 *o;
    float *hT;
    int *err;
    int dv;
    uint32_t wait_limit;
    // Segment scan (dense batches): sequence n = b * segs + segment; segment 0
    // covers tokens [0, seglen0), segment s > 0 [seglen0 + (s - 1) seglen, +
    // seglen), clipped to T; segs = 0: off.  The wide loop's launch covers
    // segments seg_lo .. segs - 1 of every sequence, segment-major.
    int segs, seglen, seglen0, seg_lo;
    int no_output;   // 1: skip o (state-only pass)
    // Wide loop, first pass of a segment scan: segment 0 runs as the final
    // pass would (from h0x, row b of [N][H][d_v][d_k], with outputs; its
    // final state into hT like the other segments' affine parts) and has no
    // linear-part tile.
    int seg0_full;
    const float *h0x;
    // Wide loop, packed batch: the CTAs of rank r take sequence seq_order[r]
    // (null: sequence r).
    const int *seq_order;
    // CTAs with blockIdx.x >= xsplit run the map's linear part instead: v = 0,
    // h0 = identity (d_k x d_k state), final state into hT2 with width dv2.
    int xsplit, dv2;
    float *hT2;
    int lin_tiles;   // the wide chunk loop's launch of its own: linear-part tiles per (n, h)
    // State pass for the backward (no segments): every chunk's starting state
    // H = S^T as [H][chunk_slots][d_k][d_v] and the rows of V' as [rows][d_v],
    // fp32; null: not stored.  Chunk slot: dense n * max_chunks + c, packed
    // floor(cu[n] / 64) + n + c.
    float *Hst, *Vst;
    long long chunk_slots;
    int max_chunks;
    // Chunk prep beside the chain (k_gdn_tc_ov; dense batches, no segments):
    // chunk j >= prep_c0 of (n, h) waits for its ready flag
    // done[h * chunk_slots + n * max_chunks + j] before its W and T_u tiles
    // are copied.  Null: no wait.
    const uint32_t *done;
    int prep_c0;
};

// Tokens [t0, t0 + len) of segment sg of a segment scan.
__device__ __forceinline__ void seg_range(const TcParams &p, int sg, int &t0, int &len) {
    t0 = sg == 0 ? 0 : p.seglen0 + (sg - 1) * p.seglen;
    len = max(0, min(sg == 0 ? p.seglen0 : p.seglen, p.sm.T - t0));
}

// The kernel body.  STATES: the backward's state pass (stores Hst / Vst),
// a separate kernel (k_gdn_tc_states), so the forward's k_gdn_tc carries
// none of it.  The tensor maps are the kernels' __grid_constant__ parameters.
template <int DK, bool STATES>
__device__ __forceinline__ void gdn_tc_body(const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                                            const CUtensorMap *tm_v, const CUtensorMap *tm_t,
                                            const CUtensorMap *tm_w, const CUtensorMap *tm_hst,
                                            const CUtensorMap *tm_vst, const TcParams &p,
                                            const int bx, const int h, const int n,
                                            const int nseq) {
    using L = Lay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    // chunks whose Gram warps 6-7 have read (P formed): a count, so that the
    // wide-span branch of warps 4-5, which waits for the Gram only in some
    // chunks, cannot mistake an older phase of its mbarrier for this one
    uint32_t *g_seen = misc + 2;
    float *gb = reinterpret_cast<float *>(sm + L::OFF_G);   // [2][GSZ]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA: d_v tile bx (or linear-part tile bx - xsplit) of (sequence n, head h)
    const int dv0 = (bx >= p.xsplit ? bx - p.xsplit : bx) * kNV;

    // ---- sequence bounds (validated; an invalid packed range is an error)
    long long row0 = 0;
    int len = 0;
    bool ok_seq = true;
    int ytok0 = 0, zcoord = 0;   // bulk-copy coordinates of chunk 0
    if (p.sm.cu) {
        const int a = __ldg(p.sm.cu + n), b = __ldg(p.sm.cu + n + 1);
        ok_seq = a >= 0 && a <= b && b <= p.sm.T_total;
        if (ok_seq) {
            row0 = (long long)h * p.sm.T_total + a;
            len = b - a;
        }
        ytok0 = a;
        zcoord = h;
    } else if (p.segs > 0) {
        const int b = n / p.segs, sg = n - b * p.segs;
        int t0;
        seg_range(p, sg, t0, len);
        row0 = ((long long)b * p.sm.H + h) * (long long)p.sm.T + t0;
        ytok0 = t0;
        zcoord = b * p.sm.H + h;
    } else {
        row0 = ((long long)n * p.sm.H + h) * (long long)p.sm.T;
        len = p.sm.T;
        zcoord = n * p.sm.H + h;
    }
    if (!ok_seq) {
        if (tid == 0) atomicCAS(p.err, 0, kErrBadIndex);
        return;  // before any barrier or TMEM use
    }
    const int nch = (len + kC - 1) / kC;
    const bool lin = bx >= p.xsplit;                     // linear-part CTA (v = 0, h0 = I)
    const int dvs = lin ? p.dv2 : p.dv;                  // width of this CTA's state
    float *hTp = lin ? p.hT2 : p.hT;
    const long long srow = ((long long)n * p.sm.H + h) * dvs;   // state row of (n, h)
    const long long slot0 = p.sm.cu ? (long long)(ytok0 / kC) + n : (long long)n * p.max_chunks;

    if (warp == 9) {
        tmem_alloc(misc, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar + i, 1);
        for (int s = 0; s < kNS; ++s) mbar_init(bar + B_FREE + s, 3);   // chain MMA + 2 prep groups
        for (int s = 0; s < kNS; ++s) mbar_init(bar + B_FULL + s, 33);   // TMA tx + 32 gate lanes
        *abort_flag = 0;
        *g_seen = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // everything above touched only this CTA's shared memory and TMEM; global
    // data written by the previous kernel in the stream (T_u / W, segment
    // initial states) is read only from here on
    griddep_wait();
    if (!STATES) CTA_SPAN(0);
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};
    // element counts of the global arrays, for the bounds-check build: token
    // rows of the inputs, and the states of this launch's grid
    const long long nrows =
        p.sm.cu ? (long long)p.sm.H * p.sm.T_total : (long long)p.sm.N * p.sm.H * p.sm.T;
    const long long nstate = (long long)nseq * p.sm.H * dvs * DK;
    (void)nrows;
    (void)nstate;

    if (warp < 4) {
        // ================================================= chain warpgroup
        const int t = tid;   // TMEM lane = H row (d_k index) / output row - 64
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float hreg[kNV];
#pragma unroll
        for (int c = 0; c < kNV; ++c)
            hreg[c] = lin ? ((t < DK && dv0 + c == t) ? 1.f : 0.f)
                          : ((t < DK && p.h0 && GDN_IDX_OK((srow + dv0 + c) * DK + t, 1, nstate))
                                 ? __ldg(p.h0 + (srow + dv0 + c) * DK + t)
                                 : 0.f);
        uint8_t *Hs = sm + L::OFF_H;
        uint8_t *VT = sm + L::OFF_R0, *VN = sm + L::OFF_R1;
        // Output rows of chunk jj (lanes 64-127 of its accumulator) to global,
        // times osc: gamma_r when the chunk's accumulator holds
        // Q H + (P / gamma_r) V' (Q left unscaled), else 1.
        float osc = 1.f;
        auto store_o = [&](int jj) {
            const int r = t - 64;
            const int Lj = min(kC, len - jj * kC);
            uint32_t o0[32], o1[32];
            const uint32_t acc = tmem + lane_base + TM_M2 + (jj & 1) * 64;
            tmem_ld32(acc, o0);
            tmem_ld32(acc + 32, o1);
            tmem_wait32(o0);
            tmem_wait32(o1);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                o0[i] = __float_as_uint(f32(o0[i]) * osc);
                o1[i] = __float_as_uint(f32(o1[i]) * osc);
            }
            if (r < Lj && GDN_IDX_OK((row0 + (long long)jj * kC + r) * p.dv + dv0, kNV,
                                     nrows * p.dv)) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + (row0 + (long long)jj * kC + r) *
                                                                 p.dv + dv0);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(pack_bf16(f32(o0[8 * q]), f32(o0[8 * q + 1])),
                                        pack_bf16(f32(o0[8 * q + 2]), f32(o0[8 * q + 3])),
                                        pack_bf16(f32(o0[8 * q + 4]), f32(o0[8 * q + 5])),
                                        pack_bf16(f32(o0[8 * q + 6]), f32(o0[8 * q + 7])));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[4 + q] = make_uint4(pack_bf16(f32(o1[8 * q]), f32(o1[8 * q + 1])),
                                            pack_bf16(f32(o1[8 * q + 2]), f32(o1[8 * q + 3])),
                                            pack_bf16(f32(o1[8 * q + 4]), f32(o1[8 * q + 5])),
                                            pack_bf16(f32(o1[8 * q + 6]), f32(o1[8 * q + 7])));
            }
        };
        bool alive = true;
        for (int j = 0; j < nch; ++j) {
            TRACE(0, j, 0, t == 0);
            // (i) publish H as the bf16 B operand of the chain MMA
            if (t < DK) put_row64(Hs, t, hreg);
            fence_proxy_async_smem();
            tc_fence_before();
            if (STATES && t == 0) bulk_wait_read();   // the staging tile is free
            named_bar(1, 128);
            if (t == 0) mbar_arrive(bar + B_HPUB);
            TRACE(0, j, 1, t == 0);
            if (STATES) {   // the chunk's starting state, for the backward
                if (t < DK) put_row64_f32(sm + L::OFF_STG, DK, t, hreg);
                fence_proxy_async_smem();
                named_bar(1, 128);
                if (t == 0) {
                    const int y = (int)((h * p.chunk_slots + slot0 + j) * DK);
                    tma_store_2d(tm_hst, sm + L::OFF_STG, dv0, y);
                    tma_store_2d(tm_hst, sm + L::OFF_STG + DK * 128, dv0 + 32, y);
                    bulk_commit();
                }
            }
            // (i') previous chunk's output rows, off the state's critical path
            if (j > 0 && t >= 64 && !p.no_output && !lin) store_o(j - 1);
            TRACE(0, j, 2, t == 64);
            // (ii) V' = U - W H, and its decayed copy for the state update
            {
                // READY orders this chunk's gates; UW and M2 bring U and W H
                if (STATES && t == 0) bulk_wait_read();   // staging free for V'
                bool ok = ctl.wait(B_READY + (j % kNS), (j / kNS) & 1);
                ok = ok && ctl.wait(B_UW, j & 1) && ctl.wait(B_M2, j & 1);
                if (!named_bar_and(1, 128, ok)) {
                    alive = false;
                    break;
                }
            }
            TRACE(0, j, 3, t == 0);
            tc_fence_after();
            const float *gj = gb + (j & 1) * L::GSZ;
            const float gC = gj[63];
            const float decayC = __expf(gC);
            // this chunk's output scale, kept in a register: its gate buffer
            // may be refilled before the rows are stored during chunk j + 1
            const float osc_j = (t >= 64 && gC > -80.f) ? gj[128 + t - 64] : 1.f;
            // V' rows by bulk tensor store where the box holds this sequence's
            // rows only (dense: rows past T are clipped)
            const bool bulk_v = !p.sm.cu || len - j * kC >= kC;
            if (t < 64) {
                const float ev = __expf(gC - gj[t]);
                const uint32_t acc = tmem + lane_base + TM_M2 + (j & 1) * 64;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t wh[32], u[32];
                    tmem_ld32(acc + 32 * half, wh);
                    tmem_ld32(tmem + lane_base + TM_U + 32 * half, u);
                    tmem_wait32(wh);
                    tmem_wait32(u);
                    float vn[32], vt[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        vn[i] = f32(u[i]) - f32(wh[i]);
                        vt[i] = vn[i] * ev;
                    }
                    if (STATES && bulk_v) {   // staged for two bulk tensor stores
                        uint8_t *sv = sm + L::OFF_STG + half * 8192;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            if (GDN_SMEM_OK(smem_u32(sv + sw128_offset(t, q)), 16))
                                *reinterpret_cast<float4 *>(sv + sw128_offset(t, q)) =
                                    make_float4(vn[4 * q], vn[4 * q + 1], vn[4 * q + 2],
                                                vn[4 * q + 3]);
                    } else if (STATES && t < min(kC, len - j * kC) &&
                               GDN_IDX_OK((row0 + (long long)j * kC + t) * p.dv + dv0 + 32 * half,
                                          32, nrows * p.dv)) {
                        float4 *dst = reinterpret_cast<float4 *>(
                            p.Vst + (row0 + (long long)j * kC + t) * p.dv + dv0 + 32 * half);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(vn[4 * q], vn[4 * q + 1], vn[4 * q + 2],
                                                 vn[4 * q + 3]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        put8(VN, t, 4 * half + q, vn + 8 * q);
                        put8(VT, t, 4 * half + q, vt + 8 * q);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 128);
            if (t == 0) {
                mbar_arrive(bar + B_VN);
                if (STATES && bulk_v) {
                    const int y = ytok0 + j * kC;
                    tma_store_3d(tm_vst, sm + L::OFF_STG, dv0, y, zcoord);
                    tma_store_3d(tm_vst, sm + L::OFF_STG + 8192, dv0 + 32, y, zcoord);
                    bulk_commit();
                }
            }
            TRACE(0, j, 4, t == 0);
            // (iii) H <- exp(g_C) H + dH
            if (!named_bar_and(1, 128, ctl.wait(B_M34, j & 1))) {
                alive = false;
                break;
            }
            TRACE(0, j, 5, t == 0);
            tc_fence_after();
            osc = osc_j;
            if (t < DK) {
                uint32_t d0[32], d1[32];
                tmem_ld32(tmem + lane_base + TM_H, d0);
                tmem_ld32(tmem + lane_base + TM_H + 32, d1);
                tmem_wait32(d0);
                tmem_wait32(d1);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    hreg[i] = fmaf(decayC, hreg[i], f32(d0[i]));
                    hreg[32 + i] = fmaf(decayC, hreg[32 + i], f32(d1[i]));
                }
            }
        }
        if (alive && nch > 0 && t >= 64 && !p.no_output && !lin) store_o(nch - 1);
        if (alive && hTp && t < DK) {
#pragma unroll
            for (int c = 0; c < kNV; ++c)
                if (GDN_IDX_OK((srow + dv0 + c) * DK + t, 1, nstate))
                    hTp[(srow + dv0 + c) * DK + t] = hreg[c];
        }
        if (STATES && t == 0) bulk_wait_all();   // every store done before the CTA leaves
    } else if (warp < 8) {
        // ================================================== prep warpgroups
        // Two independent 64-thread pipelines over the chunks:
        //   warps 4-5: gates, clearing of packed-batch tails, and -- only when
        //              the chunk's decay span is too wide for exp(-g_s) -- gamma * Q
        //              in place after the Gram; publishing [W; Q] (or [W; gamma Q])
        //   warps 6-7: P = causal decayed (Q K^T) from TMEM lanes 64-127
        const int t = tid - 128;
        const int w = warp - 4;
        const uint32_t lane_base = (uint32_t)(w * 32) << 16;
        if (t < 64) {
            if (lin) {
                // v = 0: the V tiles are never loaded, so clear them once
                for (int i = t; i < kNS * 512; i += 64)
                    st16(sm + L::OFF_STAGE + (i >> 9) * L::STAGE + L::OFF_V + (i & 511) * 16, 0u,
                         0u, 0u, 0u);
                fence_proxy_async_smem();
            }
            for (int j = 0; j < nch; ++j) {
                const int s = j % kNS;
                uint8_t *stg = sm + L::OFF_STAGE + s * L::STAGE;
                const int L_ = min(kC, len - j * kC);
                float *gj = gb + (j & 1) * L::GSZ;
                TRACE(1, j, 0, t == 0);
                if (!named_bar_and(4, 64, ctl.wait(B_FULL + s, (j / kNS) & 1))) break;
                TRACE(1, j, 1, t == 0);
                if (w == 0) {
                    const float *gs = reinterpret_cast<const float *>(sm + L::OFF_GS) + s * 128;
                    float la0 = gs[lane], la1 = gs[32 + lane];
                    const float b0 = gs[64 + lane], b1 = gs[96 + lane];
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float y0 = __shfl_up_sync(0xffffffffu, la0, off);
                        const float y1 = __shfl_up_sync(0xffffffffu, la1, off);
                        if (lane >= off) {
                            la0 += y0;
                            la1 += y1;
                        }
                    }
                    la1 += __shfl_sync(0xffffffffu, la0, 31);
                    const float e0 = __expf(la0), e1 = __expf(la1);
                    gj[lane] = la0;
                    gj[lane + 32] = la1;
                    gj[64 + lane] = b0;
                    gj[64 + lane + 32] = b1;
                    gj[128 + lane] = e0;
                    gj[128 + lane + 32] = e1;
                    gj[192 + lane] = __expf(-la0);   // used only when the span is < 80
                    gj[192 + lane + 32] = __expf(-la1);
                    gj[256 + lane] = b0 * e0;
                    gj[256 + lane + 32] = b1 * e1;
                }
                if (p.sm.cu && L_ < kC) {
                    // rows past this sequence belong to the next one: clear them
                    constexpr int per_row = 3 * DK / 8 + 16;   // 16-byte pieces: K, W, Q, V, T_u
                    for (int i = t; i < (kC - L_) * per_row; i += 64) {
                        const int r = L_ + i / per_row, q = i % per_row;
                        uint8_t *base;
                        if (q < DK / 8)  // K
                            base = stg + (q >> 3) * 8192;
                        else if (q < 3 * DK / 8)  // W, Q blocks
                            base = stg + L::OFF_WQ + ((q - DK / 8) >> 3) * 8192;
                        else if (q < 3 * DK / 8 + 8)  // V
                            base = stg + L::OFF_V;
                        else  // T_u
                            base = stg + L::OFF_TU;
                        st16(base + sw128_offset(r, q & 7), 0u, 0u, 0u, 0u);
                    }
                }
                named_bar(4, 64);
                TRACE(1, j, 5, t == 0);
                const bool span_ok = gj[63] > -80.f;
                auto scale_q = [&]() {
                    // row t of every Q block: all loads first, then all stores (a
                    // store may alias a later load, so interleaving them would
                    // serialise every round trip)
                    const float gam = gj[128 + t];
#pragma unroll
                    for (int blk = 0; blk < L::KB; ++blk) {
                        uint8_t *qs = stg + L::OFF_WQ + blk * 16384 + 8192;
                        uint4 v[8];
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)
                            v[ch] = *reinterpret_cast<const uint4 *>(qs + sw128_offset(t, ch));
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            uint32_t wv[4] = {v[ch].x, v[ch].y, v[ch].z, v[ch].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&wv[e]);
                                float2 f2 = __bfloat1622float2(b2);
                                wv[e] = pack_bf16(f2.x * gam, f2.y * gam);
                            }
                            v[ch] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        }
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)
                            *reinterpret_cast<uint4 *>(qs + sw128_offset(t, ch)) = v[ch];
                    }
                };
                // span_ok: Q stays unscaled (the output rows take gamma_r at the
                // end, and P is formed divided by gamma_r)
                TRACE(1, j, 6, t == 0);
                fence_proxy_async_smem();
                named_bar(4, 64);
                if (t == 0) mbar_arrive(bar + B_READY + s);
                TRACE(1, j, 7, t == 0);
                if (!span_ok) {
                    // the Gram must read the unscaled Q first
                    if (!named_bar_and(4, 64, ctl.flag(g_seen, (uint32_t)j + 1))) break;
                    scale_q();
                    fence_proxy_async_smem();
                    named_bar(4, 64);
                }
                // publish [W; Q] only once the previous chunk's chain MMA has
                // read its own copy: the barrier then never runs two phases ahead
                // of the chain MMA issuer waiting on it
                if (!named_bar_and(4, 64, j == 0 || ctl.wait(B_M2, (j - 1) & 1))) break;
                if (t == 0) mbar_arrive(bar + B_WQ);
                if (t == 0) mbar_arrive(bar + B_FREE + s);
                TRACE(1, j, 2, t == 0);
            }
        } else {
            for (int j = 0; j < nch; ++j) {
                const int s = j % kNS;
                float *gj = gb + (j & 1) * L::GSZ;
                bool okg = ctl.wait(B_READY + s, (j / kNS) & 1);   // orders this chunk's gates
                okg = okg && ctl.wait(B_G, j & 1);
                if (j >= 2) okg = okg && ctl.wait(B_PFREE + (j & 1), ((j - 2) >> 1) & 1);
                if (!named_bar_and(3, 64, okg)) break;
                TRACE(1, j, 3, t == 64);
                tc_fence_after();
                const int r = t - 64;
                uint32_t g0[32], g1[32];
                tmem_ld32(tmem + lane_base + TM_G, g0);
                tmem_ld32(tmem + lane_base + TM_G + 32, g1);
                const bool span_ok = gj[63] > -80.f;
                const float gr = gj[r];
                uint8_t *Pt = sm + ((j & 1) ? L::OFF_R1 : L::OFF_R0) + 8192;
                tmem_wait32(g0);
                tmem_wait32(g1);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float x[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int sidx = 32 * half + i;
                        const float gv = f32(half == 0 ? g0[i] : g1[i]);
                        const bool keep = sidx <= r;
                        // span_ok: P / gamma_r = exp(-g_s) (q_r . k_s), to pair with the
                        // unscaled Q of the chain MMA; else P itself
                        const float f = span_ok ? gj[192 + sidx]
                                                : __expf(keep ? gr - gj[sidx] : 0.f);
                        x[i] = keep ? f * gv : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) put8(Pt, r, 4 * half + q, x + 8 * q);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(3, 64);
                if (t == 64) {
                    mbar_arrive(bar + B_PREADY + (j & 1));
                    mbar_arrive(bar + B_GFREE);
                    mbar_arrive(bar + B_FREE + s);
                    st_release_cta(g_seen, (uint32_t)j + 1);   // off the P path
                }
                TRACE(1, j, 4, t == 64);
            }
        }
    } else if (warp == 8) {
        // ================================================= TMA producer
        // lane 0 issues the bulk tensor copies; all lanes stage the chunk's
        // gates (log_alpha, beta; zero past the sequence) next to them
        if (lane == 0) {
            prefetch_tmap(tm_q);
            prefetch_tmap(tm_k);
            prefetch_tmap(tm_v);
            prefetch_tmap(tm_t);
            prefetch_tmap(tm_w);
        }
        int issued = 0;
        // gates of the next chunk, loaded one chunk ahead so their latency hides
        // behind the wait for a free stage
        float pla0 = 0.f, pla1 = 0.f, pb0 = 0.f, pb1 = 0.f;
        auto load_gates = [&](int jj) {
            const long long r0 = row0 + (long long)jj * kC;
            const int Lj = min(kC, len - jj * kC);
            const bool in0 = lane < Lj && GDN_IDX_OK(r0 + lane, 1, nrows);
            const bool in1 = lane + 32 < Lj && GDN_IDX_OK(r0 + lane + 32, 1, nrows);
            pla0 = in0 ? __ldg(p.log_alpha + r0 + lane) : 0.f;
            pla1 = in1 ? __ldg(p.log_alpha + r0 + lane + 32) : 0.f;
            pb0 = in0 ? __ldg(p.beta + r0 + lane) : 0.f;
            pb1 = in1 ? __ldg(p.beta + r0 + lane + 32) : 0.f;
        };
        if (nch > 0) load_gates(0);
        for (int j = 0; j < nch; ++j) {
            const int s = j % kNS;
            if (p.done && j >= p.prep_c0) {
                // this chunk's T_u and W rows come from the prep CTAs of the
                // same launch: their ready flag (usually set long before;
                // polled ahead of the wait for a free stage)
                const bool okp =
                    ctl.gflag(p.done + (long long)h * p.chunk_slots + slot0 + j, 1u);
                if (!__all_sync(0xffffffffu, okp)) break;
                fence_proxy_async_global();
            }
            const bool ok = j < kNS || ctl.wait(B_FREE + s, ((j / kNS) - 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            uint8_t *stg = sm + L::OFF_STAGE + s * L::STAGE;
            uint64_t *fb = bar + B_FULL + s;
            const int y = ytok0 + j * kC;
            if (lane == 0) {
                // K, W, Q, V and T_u tiles
                mbar_arrive_expect_tx(fb, (uint32_t)(L::STAGE - (lin ? 8192 : 0)));
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    tma_load_3d(stg + blk * 8192, tm_k, fb, blk * 64, y, zcoord);
                    tma_load_3d(stg + L::OFF_WQ + blk * 16384, tm_w, fb, blk * 64, y, zcoord);
                    tma_load_3d(stg + L::OFF_WQ + blk * 16384 + 8192, tm_q, fb, blk * 64, y,
                                zcoord);
                }
                if (!lin) tma_load_3d(stg + L::OFF_V, tm_v, fb, dv0, y, zcoord);
                tma_load_3d(stg + L::OFF_TU, tm_t, fb, 0, y, zcoord);
            }
            {
                float *gs = reinterpret_cast<float *>(sm + L::OFF_GS) + s * 128;
                gs[lane] = pla0;
                gs[32 + lane] = pla1;
                gs[64 + lane] = pb0;
                gs[96 + lane] = pb1;
                mbar_arrive(fb);
                if (j + 1 < nch) load_gates(j + 1);
            }
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
            constexpr uint32_t idM2 = make_idesc_bf16(128, kNV, false, true);  // [W;Q] H
            constexpr uint32_t idM3 = make_idesc_bf16(128, kNV, true, true);   // K^T V~
            constexpr uint32_t idM4 = make_idesc_bf16(128, kNV, false, true);  // [x;P] V'
            const uint32_t sbase = smem_u32(sm);
            // descriptor bases; an operand at base + off is base_desc + (off >> 4)
            const uint64_t dWQ = make_sdesc(sbase + L::OFF_STAGE + L::OFF_WQ, 16, 1024,
                                            kSwizzle128B);
            const uint64_t dH = make_sdesc(sbase + L::OFF_H, 16, 1024, kSwizzle128B);
            const uint64_t dVT = make_sdesc(sbase + L::OFF_R0, 16, 1024, kSwizzle128B);
            const uint64_t dVN = make_sdesc(sbase + L::OFF_R1, 16, 1024, kSwizzle128B);
            const uint64_t dKT = make_sdesc(sbase + L::OFF_STAGE, 8192, 1024, kSwizzle128B);
            for (int j = 0; j < nch; ++j) {
                const uint32_t soff = (j % kNS) * L::STAGE;
                const uint32_t acc = tmem + TM_M2 + (j & 1) * 64;
                if (!ctl.wait(B_WQ, j & 1) || !ctl.wait(B_HPUB, j & 1)) break;
                TRACE(2, j, 0, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = soff + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(acc, dWQ + (off >> 4), dH + (kk * 2048 >> 4), idM2, kk > 0);
                }
                mma_commit(bar + B_M2);
                TRACE(2, j, 1, true);
                if (!ctl.wait(B_PREADY + (j & 1), (j >> 1) & 1)) break;   // P of this chunk
                if (!ctl.wait(B_VN, j & 1)) break;   // V' of this chunk
                TRACE(2, j, 2, true);
                tc_fence_after();
                const uint64_t dP = (j & 1) ? dVN : dVT;   // [x; P] starts at the region base
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    mma_bf16(tmem + TM_H, dKT + ((soff + kk * 2048) >> 4), dVT + (kk * 2048 >> 4),
                             idM3, kk > 0);
                    mma_bf16(acc, dP + (kk * 32 >> 4), dVN + (kk * 2048 >> 4), idM4, 1u);
                }
                mma_commit(bar + B_M34);
                mma_commit(bar + B_PFREE + (j & 1));
                mma_commit(bar + B_FREE + (j % kNS));
                mbar_arrive(bar + B_M34I);
                TRACE(2, j, 3, true);
            }
            // every issued MMA has finished before TMEM is released
            mma_commit(bar + B_DRAIN);
            mbar_wait(bar + B_DRAIN, 0, ctl.limit);
        }
    } else if (warp == 10) {
        // ============================================== prep MMA issuer
        if (lane == 0 && nch > 0) {
            constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);   // [W;Q] K^T
            constexpr uint32_t idU = make_idesc_bf16(128, 64, false, true);    // [T_u;x] V
            const uint32_t sbase = smem_u32(sm);
            const uint64_t dS = make_sdesc(sbase + L::OFF_STAGE, 16, 1024, kSwizzle128B);
            for (int j = 0; j < nch; ++j) {
                const int s = j % kNS;
                const uint32_t soff = s * L::STAGE;
                if (!ctl.wait(B_READY + s, (j / kNS) & 1)) break;
                if (j > 0 && !ctl.wait(B_GFREE, (j - 1) & 1)) break;   // G of j-1 consumed
                // the tensor pipe runs MMAs in issue order: this chunk's Gram
                // and U go behind the previous chunk's state and output MMAs
                // (K^T V~, P' V'), which the chain waits for, not ahead of them
                if (j > 0 && !ctl.wait(B_M34I, (j - 1) & 1)) break;
                TRACE(3, j, 0, true);
                tc_fence_after();
                // the Gram first: P is the longer path to the output MMA
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t kof = soff + (kk >> 2) * 8192 + (kk & 3) * 32;
                    const uint32_t aof = soff + L::OFF_WQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_G, dS + (aof >> 4), dS + (kof >> 4), idG, kk > 0);
                }
                mma_commit(bar + B_G);
                TRACE(3, j, 1, true);
                if (j > 0 && !ctl.wait(B_VN, (j - 1) & 1)) break;   // U of j-1 consumed
                TRACE(3, j, 2, true);
                tc_fence_after();
                // U = T_u V; rows 64-127 of the A operand are whatever follows T_u
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_bf16(tmem + TM_U, dS + ((soff + L::OFF_TU + kk * 32) >> 4),
                             dS + ((soff + L::OFF_V + kk * 2048) >> 4), idU, kk > 0);
                mma_commit(bar + B_UW);
                TRACE(3, j, 3, true);
            }
            mma_commit(bar + B_DRAIN2);
            mbar_wait(bar + B_DRAIN2, 0, ctl.limit);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!STATES) CTA_SPAN(1);
    if (warp == 9) tmem_dealloc(tmem, 512);
}

template <int DK>
__global__ void __launch_bounds__(kThreadsTC, 1)
k_gdn_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_t,
         const __grid_constant__ CUtensorMap tm_w, TcParams p) {
    gdn_tc_body<DK, false>(&tm_q, &tm_k, &tm_v, &tm_t, &tm_w, nullptr, nullptr, p, blockIdx.x,
                           blockIdx.y, blockIdx.z, gridDim.z);
}

template <int DK>
__global__ void __launch_bounds__(kThreadsTC, 1)
k_gdn_tc_states(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_t,
                const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_hst,
                const __grid_constant__ CUtensorMap tm_vst, TcParams p) {
    gdn_tc_body<DK, true>(&tm_q, &tm_k, &tm_v, &tm_t, &tm_w, &tm_hst, &tm_vst, p, blockIdx.x,
                          blockIdx.y, blockIdx.z, gridDim.z);
}

// The chain with the chunk prep beside it, one cooperative launch of one CTA
// per SM.  CTAs 0 .. nchain - 1 run the chain of (sequence, head, d_v tile)
// (tile fastest, then head); from chunk prep_c0 on, each chunk's W and T_u
// tiles wait for the chunk's ready flag.  Every other CTA runs kPrepPipes
// prep pipelines (gdn_utw.cuh) over the units of chunks prep_c0 ..
// max_chunks - 1, chunk by chunk, and sets those flags; the prep launch
// before this one has prepared the earlier chunks and cleared the flags.
// The chain CTAs, latency-bound on their serial chunk pass, leave the other
// SMs idle otherwise.  A cooperative launch has every CTA resident at once,
// so a chain CTA's wait on a prep CTA always ends.
constexpr int kPrepPipes = 3;
constexpr int kThreadsOV = 128 * kPrepPipes > kThreadsTC ? 128 * kPrepPipes : kThreadsTC;

template <int DK>
struct OvLay {
    static constexpr int PIPE = (VLay<DK>::TOTAL + 1023) / 1024 * 1024;   // per pipeline
    static constexpr int OFF_MISC = kPrepPipes * PIPE;                       // TMEM address
    static constexpr int ALLOC_PREP = OFF_MISC + 16 + 1024;
    static constexpr int ALLOC = ALLOC_PREP > Lay<DK>::ALLOC ? ALLOC_PREP : Lay<DK>::ALLOC;
    static_assert(ALLOC <= 227 * 1024, "shared memory budget (overlapped launch)");
};

// The role of this CTA in an overlapped launch.  With one CTA per SM
// (by_sm) and SM ids 0 .. SMs - 1, the CTA on SM s takes role s, so the chain
// CTAs sit on the lowest-numbered SMs, as a plain launch of the chain alone
// places them (measured: 139 µs for the chain at B4 H16 T4096 d128 there,
// against 152 µs when the roles follow the launch's own placement, which
// spreads the chain CTAs over every GPC).  Otherwise the role is the CTA
// index.
__device__ __forceinline__ int ov_role(int by_sm) {
    uint32_t sm_id, n_smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_id));
    asm volatile("mov.u32 %0, %%nsmid;" : "=r"(n_smid));
    return by_sm && n_smid == gridDim.x ? (int)sm_id : (int)blockIdx.x;
}

// A prep CTA of an overlapped launch (role nchain .. grid - 1): kPrepPipes
// pipelines of 128 threads (threads past them only join the barriers) over
// the launch's prep units, round robin over all prep CTAs' pipelines so the
// chunks finish roughly in order.
template <int DK>
__device__ __forceinline__ void ov_prep_role(const CUtensorMap *tm_k, const UtParams &up,
                                             int role, int nchain) {
    using O = OvLay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + O::OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, pipe = tid >> 7, ptid = tid & 127;
    const bool in_pipe = pipe < kPrepPipes;
    CTA_SPAN(0);
    uint8_t *psm = sm + pipe * O::PIPE;
    if (warp == 0) {
        tmem_alloc(misc, 512);
        tmem_relinquish();
    }
    if (in_pipe) utw_init<DK>(psm, ptid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // the prep launch before this one cleared the ready flags
    griddep_wait();
    const long long stride = (long long)kPrepPipes * (gridDim.x - nchain);
    const long long first = (long long)(role - nchain) * kPrepPipes + pipe;
    const long long nun = first < up.units ? (up.units - 1 - first) / stride + 1 : 0;
    if (in_pipe && nun > 0)
        utw_run<DK>(psm, tmem + 128 * pipe, ptid, 1 + pipe, tm_k, up, first, stride, nun);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    CTA_SPAN(1);
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int DK>
__global__ void __launch_bounds__(kThreadsOV, 1)
k_gdn_tc_ov(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_t,
            const __grid_constant__ CUtensorMap tm_w, TcParams p, UtParams up, int nchain,
            int by_sm) {
    const int role = ov_role(by_sm);
    if (role < nchain) {
        const int ci = role, tiles = p.xsplit, hn = ci / tiles;
        gdn_tc_body<DK, false>(&tm_q, &tm_k, &tm_v, &tm_t, &tm_w, nullptr, nullptr, p,
                               ci - hn * tiles, hn % p.sm.H, hn / p.sm.H, p.sm.N);
        return;
    }
    ov_prep_role<DK>(&tm_k, up, role, nchain);
}

#include "gdn_tcw.cuh"   // the chunk loop with both d_v halves in one CTA (k_gdn_tcw_ov)
static_assert(kThreadsW == kThreadsOV, "both overlapped launches share the prep role");

// -------------------------------------------------------------------- host

// One launch of the fused kernel.  `seq` says how the grid's z axis maps to
// token ranges (plain batch, or b * segs + segment); `lin_tiles` > 0 adds CTAs
// that compute the segments' linear parts (v = 0, h0 = I) into hT2.
struct LaunchCfg {
    int nseq;             // grid.z
    int segs, seglen;     // segment scan view (segs = 0: off)
    int no_output;
    const float *h0;
    float *hT;
    int lin_tiles;
    float *hT2;
    bool timed;
    float *Hst = nullptr, *Vst = nullptr;   // the backward's state pass
    int seglen0 = 0;                        // segment 0's tokens (0: seglen)
    int seg_lo = 0;                         // first segment launched (wide loop)
    const float *h0x = nullptr;             // wide loop: segment 0 from h0x with outputs
    bool seg0_full = false;
    const int *seq_order = nullptr;         // wide loop, packed batch: sequences by rank
};

// The bulk-copy maps of a chain launch: q, k, v, T_u, W (T_u's rows, then W's,
// at Tin).
bool tc_maps(const FwdArgs &a, int dk, const __nv_bfloat16 *Tin, CUtensorMap (&m)[5]) {
    const long long ydim = a.sm.cu ? a.sm.T_total : a.sm.T;
    const long long zdim = a.sm.cu ? a.sm.H : (long long)a.sm.N * a.sm.H;
    const __nv_bfloat16 *Win = Tin + (size_t)a.rows * 64;
    return make_map(&m[0], a.q, dk, ydim, zdim) && make_map(&m[1], a.k, dk, ydim, zdim) &&
           make_map(&m[2], a.v, a.dv, ydim, zdim) && make_map(&m[3], Tin, 64, ydim, zdim) &&
           make_map(&m[4], Win, dk, ydim, zdim);
}

TcParams tc_params(const FwdArgs &a, int dk, const LaunchCfg &c) {
    TcParams p{};
    p.sm = a.sm;
    p.log_alpha = a.log_alpha;
    p.beta = a.beta;
    p.h0 = c.h0;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.hT = c.hT;
    p.err = device_error_word();
    p.dv = a.dv;
    const long long lim = option(GDN_OPT_WAIT_LIMIT);
    p.wait_limit = lim > 0 ? (uint32_t)(lim > 0x7fffffffLL ? 0x7fffffffLL : lim) : (1u << 22);
    p.segs = c.segs;
    p.seglen = c.seglen;
    p.seglen0 = c.seglen0 > 0 ? c.seglen0 : c.seglen;
    p.seg_lo = c.seg_lo;
    p.seg0_full = c.seg0_full ? 1 : 0;
    p.h0x = c.h0x;
    p.seq_order = c.seq_order;
    p.no_output = c.no_output;
    p.xsplit = a.dv / kNV;
    p.dv2 = dk;
    p.hT2 = c.hT2;
    p.lin_tiles = c.lin_tiles;
    p.Hst = c.Hst;
    p.Vst = c.Vst;
    p.chunk_slots = a.chunk_slots;
    p.max_chunks = a.max_chunks;
    p.done = nullptr;
    p.prep_c0 = 0;
    return p;
}

template <int DK>
gdn_status launch_tc(const FwdArgs &a, const __nv_bfloat16 *Tin, const LaunchCfg &c) {
    using L = Lay<DK>;
    const long long ydim = a.sm.cu ? a.sm.T_total : a.sm.T;
    const long long zdim = a.sm.cu ? a.sm.H : (long long)a.sm.N * a.sm.H;
    CUtensorMap m[5];
    if (!tc_maps(a, DK, Tin, m)) return GDN_ERR_CUDA;
    // per-function attributes of the current device: cheap, set on every launch
    if (cudaFuncSetAttribute(k_gdn_tc<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(k_gdn_tc_states<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC_S) != cudaSuccess)
        return GDN_ERR_CUDA;
    // the state pass's outputs (the forward's instantiation never reads these)
    CUtensorMap mh = m[0], mvs = m[0];
    if (c.Hst && (!make_map_f32(&mh, c.Hst, a.dv, (long long)a.sm.H * a.chunk_slots * DK, DK) ||
                  !make_map_f32_3d(&mvs, c.Vst, a.dv, ydim, zdim)))
        return GDN_ERR_CUDA;
    const TcParams p = tc_params(a, DK, c);
    dim3 grid(a.dv / kNV + c.lin_tiles, a.sm.H, c.nseq);
    const int slot = c.timed ? timer_begin(a.stream, "k_gdn_tc") : -1;
    // launched as a programmatic dependent of the previous kernel, which
    // releases it as its CTAs finish (the chunk-prep kernels do so at their
    // end): the prologue (barriers, TMEM) may overlap that kernel's tail
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsTC);
    cfg.dynamicSmemBytes = c.Hst ? L::ALLOC_S : L::ALLOC;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le =
        c.Hst ? cudaLaunchKernelEx(&cfg, k_gdn_tc_states<DK>, m[0], m[1], m[2], m[3], m[4], mh,
                                   mvs, p)
              : cudaLaunchKernelEx(&cfg, k_gdn_tc<DK>, m[0], m[1], m[2], m[3], m[4], p);
    timer_end(slot, a.stream);
    if (le != cudaSuccess) return GDN_ERR_CUDA;
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// The overlapped launch (k_gdn_tc_ov, or k_gdn_tcw_ov with WIDE): nchain
// chain CTAs and nprep prep CTAs over a dense batch whose chunks
// 0 .. lead - 1 are prepared.  GDN_ERR_UNSUPPORTED when the device cannot
// hold the grid at once (the launch did not start; the caller runs the plain
// path).
template <int DK, bool WIDE>
gdn_status launch_tc_ov(const FwdArgs &a, __nv_bfloat16 *Tbuf, uint32_t *done, int lead,
                        int nchain, int nprep) {
    using O = OvLay<DK>;
    constexpr int alloc = WIDE ? (LayW<DK>::ALLOC > O::ALLOC_PREP ? LayW<DK>::ALLOC
                                                                   : O::ALLOC_PREP)
                               : O::ALLOC;
    const auto kern = WIDE ? k_gdn_tcw_ov<DK> : k_gdn_tc_ov<DK>;
    CUtensorMap m[5];
    if (!tc_maps(a, DK, Tbuf, m)) return GDN_ERR_CUDA;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, alloc) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreadsOV, alloc) !=
            cudaSuccess ||
        per_sm < 1)
        return GDN_ERR_UNSUPPORTED;
    // the grid is one CTA per SM (nchain + nprep SMs): with at most one per SM
    // every SM holds exactly one, and the roles may follow SM ids
    const int by_sm = per_sm == 1 ? 1 : 0;
    const LaunchCfg c{a.sm.N, 0, 0, 0, a.h0, a.hT, 0, nullptr, true};
    TcParams p = tc_params(a, DK, c);
    if (WIDE) p.xsplit = a.dv / 128;   // tiles of the wide loop
    p.done = done;
    p.prep_c0 = lead;
    UtParams up;
    ut_params(a, nullptr, Tbuf, Tbuf + (size_t)a.rows * 64, &up);
    up.c0 = lead;
    up.nc = a.max_chunks - lead;
    up.units = (long long)a.sm.N * a.sm.H * up.nc;
    up.done = done;
    // cooperative (every CTA resident at once), and a programmatic dependent
    // of the prep launch where the runtime takes both
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nchain + nprep);
    cfg.blockDim = dim3(kThreadsOV);
    cfg.dynamicSmemBytes = alloc;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const int slot = timer_begin(a.stream, WIDE ? "k_gdn_tcw_ov" : "k_gdn_tc_ov");
    cudaError_t le =
        cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], m[3], m[4], p, up, nchain, by_sm);
    if (le != cudaSuccess) {
        (void)cudaGetLastError();
        cfg.numAttrs = 1;
        le = cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], m[3], m[4], p, up, nchain, by_sm);
    }
    if (le != cudaSuccess) {
        (void)cudaGetLastError();   // a launch that did not start leaves no sticky error
        timer_cancel(slot);
        return GDN_ERR_UNSUPPORTED;
    }
    timer_end(slot, a.stream);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// The wide chunk loop as a launch of its own (k_gdn_tcw), after the prep
// launch over every chunk: one CTA per (sequence, head, 128-column d_v tile),
// plus c.lin_tiles linear-part tiles per (sequence, head) in a segment scan's
// first pass.
template <int DK>
gdn_status launch_tcw(const FwdArgs &a, const __nv_bfloat16 *Tin, const LaunchCfg &c) {
    using L = LayW<DK>;
    CUtensorMap m[5];
    if (!tc_maps(a, DK, Tin, m)) return GDN_ERR_CUDA;
    if (cudaFuncSetAttribute(k_gdn_tcw<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC) != cudaSuccess)
        return GDN_ERR_CUDA;
    TcParams p = tc_params(a, DK, c);
    p.xsplit = a.dv / 128;   // tiles of this loop
    // a programmatic dependent of the previous launch, as the 64-column loop
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)(p.xsplit + c.lin_tiles) * a.sm.H * c.nseq));
    cfg.blockDim = dim3(kThreadsW);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int slot = c.timed ? timer_begin(a.stream, "k_gdn_tcw") : -1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, k_gdn_tcw<DK>, m[0], m[1], m[2], m[3], m[4], p);
    timer_end(slot, a.stream);
    if (le != cudaSuccess) return GDN_ERR_CUDA;
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Exclusive fold of the segment maps ("Gated DeltaNet GPU并行实现", sections
// 2.3 and 3.3): with S -> S A_i + B_i the map of segment i (earlier map
// first), the state entering segment i+1 is S_in[i] A_i + B_i, S_in[0] = h0.
// One CTA per (batch, head, 16 state rows), fp32; each map A_i is copied into
// shared memory (d_k^2 floats, two buffers: the next map's copy runs during
// this one's product).  first_full: segment 0 ran from h0 itself, so B_0 is
// already the state entering segment 1 (and there is no A_0).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(256)
k_seg_fold(const float *__restrict__ h0, const float *__restrict__ Aseg,
           const float *__restrict__ Bseg, float *__restrict__ Sin, int B, int H, int segs,
           int dv, int dk, int first_full) {
    extern __shared__ float Sr[];   // [16][dk], then two A_m buffers [dk][dk]
    const int tid = threadIdx.x;
    const int bh = blockIdx.x, b = bh / H, h = bh - b * H, r0 = blockIdx.y * 16;
    const int tot = 16 * dk, s0 = first_full ? 1 : 0;
    // A_sg into buffer (sg - s0) & 1, 16-byte pieces (the 16-row blocks of one
    // (batch, head) all read it)
    auto fetch = [&](int sg) {
        const long long m = (long long)b * (segs - 1) + sg;
        const float *Am = Aseg + (m * H + h) * (long long)dk * dk;
        float *dst = Sr + 16 * dk + ((sg - s0) & 1) * dk * dk;
        for (int i = tid; i < dk * dk / 4; i += 256) cp_async16(dst + 4 * i, Am + 4 * i);
        cp_async_commit();
    };
    if (s0 < segs - 1) fetch(s0);
    // the state entering the first folded segment: rows r0.. of B_0 or h0
    const float *src = first_full ? Bseg + ((long long)b * (segs - 1) * H + h) * dv * dk
                       : h0       ? h0 + (long long)bh * dv * dk
                                  : nullptr;
    for (int i = tid; i < tot; i += 256) {
        const int r = i / dk, cc = i - r * dk;
        Sr[i] = src ? src[(long long)(r0 + r) * dk + cc] : 0.f;
    }
    __syncthreads();
    for (int sg = s0; sg < segs; ++sg) {
        const long long n = (long long)b * segs + sg;
        for (int i = tid; i < tot; i += 256) {
            const int r = i / dk, cc = i - r * dk;
            Sin[((n * H + h) * dv + r0 + r) * dk + cc] = Sr[i];
        }
        if (sg == segs - 1) break;
        const long long m = (long long)b * (segs - 1) + sg;
        const float *Bm = Bseg + ((m * H + h) * dv + r0) * (long long)dk;
        // entry i = tid + 256 e of the 16 x dk block is row tid / dk + e (256 / dk),
        // column tid % dk (dk divides 256): a thread's entries share their
        // column, so one read of A per kk feeds all of them, and their eight
        // sums run side by side (each in the order kk = 0 .. dk - 1)
        const int cc = tid % dk, rb = tid / dk, rs = 256 / dk, ne = tot / 256;
        float acc[8];   // 16 * dk / 256 <= 8 entries per thread
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[e] = e < ne ? Bm[(long long)(rb + rs * e) * dk + cc] : 0.f;
        // the next map's copy goes out before this one is awaited (its buffer
        // was last read by the product two steps back, before a barrier)
        if (sg + 1 < segs - 1) {
            fetch(sg + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float *As = Sr + 16 * dk + ((sg - s0) & 1) * dk * dk;
#pragma unroll 4
        for (int kk = 0; kk < dk; ++kk) {
            const float a = As[kk * dk + cc];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < ne) acc[e] = fmaf(Sr[(rb + rs * e) * dk + kk], a, acc[e]);
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = tid + 256 * e;
            if (i < tot) Sr[i] = acc[e];
        }
        __syncthreads();
    }
}

// Longest sequences first: order[r] = the packed batch's sequence of rank r
// by length (descending, ties by index: a permutation of 0 .. N - 1).  The
// wide loop's CTAs run sequence-major, so in this order the longest chains
// start in the first wave and the last wave holds the shortest.
constexpr int kMaxOrderSeqs = 4096;   // N^2 comparisons, one thread per sequence
__global__ void __launch_bounds__(256)
k_seq_order(const int32_t *__restrict__ cu, int N, int *__restrict__ order) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    const int ln = __ldg(cu + n + 1) - __ldg(cu + n);
    int r = 0;
    for (int m = 0; m < N; ++m) {
        const int lm = __ldg(cu + m + 1) - __ldg(cu + m);
        r += (lm > ln || (lm == ln && m < n)) ? 1 : 0;
    }
    order[r] = n;
}

int sm_count() {
    static std::atomic<int> memo[kMaxDeviceMemo];
    return per_device(
        memo,
        [](int dev) {
            int n = 0;
            if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                n <= 0)
                n = 148;
            return n;
        },
        148);
}

// Number of sequence segments for the segment scan (1 = none).  Automatic:
// dense batches whose (batch, head, d_v tile) count leaves most SMs idle and
// that have enough chunks per sequence.
int choose_segments(const FwdArgs &a) {
    if (a.sm.cu) return 1;
    const int nch = a.max_chunks;
    const long long opt = option(GDN_OPT_SEGMENTS);
    int S;
    if (opt >= 1) {
        S = (int)opt;
    } else {
        const long long base = (long long)a.sm.N * a.sm.H * (a.dv / kNV);
        if (base * 3 > sm_count() || nch < 64) return 1;
        const long long per = (long long)a.sm.N * a.sm.H * (a.dv / kNV + a.dk / kNV);
        S = 1 + (int)(sm_count() / per);
    }
    S = max(1, min(S, nch));
    return S;
}

bool coop_supported() {
    static std::atomic<int> memo[kMaxDeviceMemo];
    return per_device(
               memo,
               [](int dev) {
                   int v = 0;
                   return cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev) ==
                                      cudaSuccess &&
                                  v
                              ? 1
                              : 0;
               },
               0) == 1;
}

// Whether the forward runs the wide chunk loop (two 64-column halves of d_v
// in one CTA): bf16 batches with scalar gates and erase, d_k 64 or 128, d_v a
// multiple of 128.
// Automatic: where the 64-column loop needs more CTAs than the device has SMs
// (more than one wave): measured at B8 H16 T4096 d128 (256 CTAs against 128),
// 0.290 ms against 0.388 ms per call; with one wave the 64-column loop is
// faster (its chunk period is ≈ 4.0 k cycles against ≈ 5.3 k).
bool wide_applies(const FwdArgs &a, int nchain) {
    if (a.dt != GDN_BF16 || a.no_erase || a.vector_gate) return false;
    if (a.dv % 128 != 0 || (a.dk != 64 && a.dk != 128)) return false;
    const long long opt = option(GDN_OPT_WIDE_CHAIN);
    if (opt < 0) return false;
    return opt > 0 || nchain > sm_count();
}

// Whether a segment scan runs the wide chunk loop: dense bf16 batches with
// scalar gates and erase, d_v a multiple of 128 and d_k = 128 (the linear
// part is one 128-column tile).  Automatic when the segment count is: per
// pass, a CTA per (sequence, head) and per map instead of two, so about
// twice the segments fit one wave (B1 H16 T131072 d128: 5 segments against
// 3); GDN_OPT_WIDE_CHAIN = 1 also with a forced segment count, -1 never.
bool seg_wide_applies(const FwdArgs &a) {
    if (a.sm.cu || a.dt != GDN_BF16 || a.no_erase || a.vector_gate) return false;
    if (a.dv % 128 != 0 || a.dk != 128) return false;
    const long long opt = option(GDN_OPT_WIDE_CHAIN);
    if (opt < 0) return false;
    return opt > 0 || option(GDN_OPT_SEGMENTS) < 1;
}

// The wide segment scan's plan, in chunks.  With head, its first launch runs
// segment 0 in full (from h0, with outputs) on B H d_v / 128 SMs while the
// other SMs form the maps of segments 1 .. S - 2 (B H (d_v / 128 + 1) CTAs
// per segment, w1 waves), and its last launch runs segments 1 .. S - 1 (w3
// waves).  The maps' pass forms no output, its chunk period r = kMapPeriod /
// 1000 of the full one (measured at B1 H16 T131072 d128: 2.04 against 2.81
// us); segment 0 takes as many chunks as the map CTAs' waves take time,
// L0 = r w1 L, the others L = ceil(M / (r w1 + S - 1)).  Cost, in full chunk
// periods: max(L0, r w1 L) + w3 L + kFoldPeriods per fold step.  Without
// head (equal segments, maps of segments 0 .. S - 2, then all S in full):
// (r w1 + w3) ceil(M / S) + the fold; the cheaper of the two is taken.
constexpr long long kMapPeriod = 730;
constexpr long long kFoldPeriods = 4;
struct SegPlan {
    int S = 1, L0 = 0, L = 0;   // segments; chunks of segment 0 and of the others
    bool head = false;
    double cost = 0.0;
};
SegPlan plan_wide(const FwdArgs &a, int S) {
    SegPlan pl;
    const long long M = a.max_chunks, nsm = sm_count();
    const long long bh = (long long)a.sm.N * a.sm.H, v = a.dv / 128, nh = bh * v;
    if (S < 2 || M < 2) return pl;
    const double r = kMapPeriod / 1000.0;
    // equal segments
    {
        const long long L = (M + S - 1) / S, Sr = (M + L - 1) / L;
        const long long w1 = (bh * (v + 1) * (Sr - 1) + nsm - 1) / nsm;
        const long long w3 = (nh * Sr + nsm - 1) / nsm;
        pl.S = (int)Sr;
        pl.L0 = pl.L = (int)L;
        pl.cost = (r * (double)w1 + (double)w3) * (double)L + (double)(kFoldPeriods * (Sr - 1));
    }
    if (nh >= nsm || S < 3) return pl;
    const long long n1 = bh * (v + 1) * (S - 2);
    const long long w1 = (n1 + (nsm - nh) - 1) / (nsm - nh);
    long long L = (long long)std::ceil((double)M / (r * (double)w1 + (double)(S - 1)));
    L = L < 1 ? 1 : L;
    long long L0 = M - (S - 1) * L;
    if (L0 < 1) L0 = std::min<long long>(M - 1, std::max<long long>(1, (long long)(r * w1 * L)));
    const long long Sr = 1 + (M - L0 + L - 1) / L;   // no empty segments
    const long long w3 = (nh * (Sr - 1) + nsm - 1) / nsm;
    const double cost = std::max((double)L0, r * (double)w1 * (double)L) +
                        (double)(w3 * L) + (double)(kFoldPeriods * (Sr - 1));
    if (Sr >= 2 && cost < pl.cost) {
        pl.S = (int)Sr;
        pl.L0 = (int)L0;
        pl.L = (int)L;
        pl.head = true;
        pl.cost = cost;
    }
    return pl;
}

// Segments for the wide segment scan: the count whose plan costs least.
int choose_segments_wide(const FwdArgs &a) {
    const int smax = a.max_chunks < 64 ? a.max_chunks : 64;
    int best = 1;
    double best_cost = -1.0;
    for (int S = 2; S <= smax; ++S) {
        const SegPlan pl = plan_wide(a, S);
        if (pl.S < 2) continue;
        if (best_cost < 0.0 || pl.cost < best_cost) {
            best_cost = pl.cost;
            best = S;
        }
    }
    return best;
}

// Chunks per sequence that the prep launch covers before the overlapped
// launch prepares the rest beside the chain, or -1: no overlap.  Automatic:
// the prep CTAs finish a chunk of every (sequence, head) in
// S = N H u / (prep CTAs x kPrepPipes) cycles and the chain takes tau cycles
// per chunk, so chunk lead + j is ready in time when (j + 1) S <= (lead + j)
// tau; the lead is the smallest that keeps this for every j, plus one.  With
// the 64-column loop and a lead past half the chunks the prep SMs take too
// small a share to pay for the overlapped launch (measured at B4 H16 T4096
// d128: 24 prep SMs, best lead 48 of 64, no faster than the plain path), so
// the overlap is off; the wide loop's alternative is the same loop after a
// prep launch over every chunk, so it overlaps whenever lead < chunks.
// Cycle counts measured on GB300 inside the overlapped launch: tau 4.5 k /
// 3.9 k (d_k 128 / 64) for the 64-column loop, 5.7 k at d_k 128 for the wide
// one (fitted to its best lead at B8 H16 T4096 d128, 53 of 64; 5.0 k at
// d_k 64 is an estimate), u 19.5 k / 18 k per unit and pipeline (three
// pipelines on an SM, beside the chain's memory traffic).
int choose_prep_lead(const FwdArgs &a, int nchain, bool wide) {
    if (a.sm.cu || a.dt != GDN_BF16 || a.no_erase || a.vector_gate) return -1;
    if (a.dk != 64 && a.dk != 128) return -1;
    const long long opt = option(GDN_OPT_PREP_LEAD);
    const int M = a.max_chunks;
    const int nprep = sm_count() - nchain;
    if (opt < 0 || M < 2 || nprep < 1 || !coop_supported()) return -1;
    if (opt > 0) return opt < M ? (int)opt : -1;
    const double tau = wide ? (a.dk == 128 ? 5700.0 : 5000.0) : (a.dk == 128 ? 4500.0 : 3900.0);
    const double u = a.dk == 128 ? 19500.0 : 18000.0;
    const double S = (double)a.sm.N * a.sm.H * u / ((double)nprep * kPrepPipes);
    const double need = S <= tau ? S / tau : M - (M - 1) * tau / S;
    const int lead = max(1, (int)ceil(need) + 1);
    if (wide) return lead < M ? lead : -1;   // the alternative is the wide loop alone
    return 2 * lead > M ? -1 : lead;
}

// The forward with the chunk prep overlapped: the prep launch over chunks
// 0 .. lead - 1 (it also clears the ready flags), then k_gdn_tc_ov.
// GDN_ERR_UNSUPPORTED when the overlapped launch could not start.
gdn_status tc_overlapped(const FwdArgs &a, __nv_bfloat16 *Tbuf, int lead, int nchain,
                         bool wide) {
    const long long nd = (long long)a.sm.H * a.chunk_slots;
    uint32_t *done = nullptr;
    if (scratch_alloc((void **)&done, sizeof(uint32_t) * (size_t)nd, a.stream) != cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_status rc = enqueue_ut_w_lead(a, Tbuf, Tbuf + (size_t)a.rows * 64, lead, done, nd);
    if (rc == GDN_OK) {
        const int nprep = sm_count() - nchain;
        if (wide)
            rc = a.dk == 128 ? launch_tc_ov<128, true>(a, Tbuf, done, lead, nchain, nprep)
                             : launch_tc_ov<64, true>(a, Tbuf, done, lead, nchain, nprep);
        else
            rc = a.dk == 128 ? launch_tc_ov<128, false>(a, Tbuf, done, lead, nchain, nprep)
                             : launch_tc_ov<64, false>(a, Tbuf, done, lead, nchain, nprep);
    }
    scratch_free(done, a.stream);
    return rc;
}

// The segment scan with the 64-column chunk loop, or with the wide one
// (both d_v halves of a 128-column tile, and the d_k = 128 linear part, in
// one CTA each).
gdn_status tc_segmented(const FwdArgs &a, const __nv_bfloat16 *Tbuf, int S, bool wide) {
    cudaStream_t st = a.stream;
    const int nch = a.max_chunks;
    int seglen = ((nch + S - 1) / S) * kC, seglen0 = seglen;
    S = (a.sm.T + seglen - 1) / seglen;   // no empty segments
    // the wide loop may run segment 0 in full beside the other segments' maps
    const SegPlan pl = wide ? plan_wide(a, S) : SegPlan{};
    const bool head = pl.head;
    if (head) {
        S = pl.S;
        seglen = pl.L * kC;
        seglen0 = pl.L0 * kC;
    }
    const int B = a.sm.N, H = a.sm.H, dv = a.dv, dk = a.dk;
    auto pass = [&](const LaunchCfg &c) {
        if (wide) return dk == 128 ? launch_tcw<128>(a, Tbuf, c) : launch_tcw<64>(a, Tbuf, c);
        return dk == 128 ? launch_tc<128>(a, Tbuf, c) : launch_tc<64>(a, Tbuf, c);
    };
    const int lin_tiles = wide ? dk / 128 : dk / kNV;   // the linear part's tiles
    if (S < 2 || (long long)B * S > 65535) {
        LaunchCfg c{B, 0, 0, 0, a.h0, a.hT, 0, nullptr, true};
        return pass(c);
    }
    const size_t st_dv = (size_t)H * dv * dk, st_dk = (size_t)H * dk * dk;
    float *Aseg = nullptr, *Bseg = nullptr, *Sin = nullptr, *Hout = nullptr;
    gdn_status rc = GDN_OK;
    if (scratch_alloc((void **)&Aseg, sizeof(float) * st_dk * B * (S - 1), st) != cudaSuccess ||
        scratch_alloc((void **)&Bseg, sizeof(float) * st_dv * B * (S - 1), st) != cudaSuccess ||
        scratch_alloc((void **)&Sin, sizeof(float) * st_dv * B * S, st) != cudaSuccess ||
        (a.hT && scratch_alloc((void **)&Hout, sizeof(float) * st_dv * B * S, st) != cudaSuccess))
        rc = GDN_ERR_CUDA;
    if (rc == GDN_OK) {
        // pass 1: per segment but the last, the map's affine part (final state
        // from zero) and linear part (final state from the identity, v = 0);
        // with head, segment 0 instead runs in full, its final state the
        // true one entering segment 1
        LaunchCfg c1{B * (S - 1), S - 1, seglen, 1, nullptr, Bseg, lin_tiles, Aseg, true};
        c1.seglen0 = seglen0;
        c1.seg0_full = head;
        c1.h0x = a.h0;
        rc = pass(c1);
    }
    if (rc == GDN_OK) {
        // pass 2: fold the maps into every segment's initial state
        dim3 grid(B * H, dv / 16);
        const int fsm = (16 * dk + 2 * dk * dk) * (int)sizeof(float);   // 136 KB at d_k = 128
        if (cudaFuncSetAttribute(k_seg_fold, cudaFuncAttributeMaxDynamicSharedMemorySize, fsm) !=
            cudaSuccess) {
            rc = GDN_ERR_CUDA;
        } else {
            k_seg_fold<<<grid, 256, fsm, st>>>(a.h0, Aseg, Bseg, Sin, B, H, S, dv, dk,
                                               head ? 1 : 0);
            count_launch();
            if (cudaGetLastError() != cudaSuccess) rc = GDN_ERR_CUDA;
        }
    }
    if (rc == GDN_OK) {
        // pass 3: every segment from its true initial state, with outputs
        // (from segment 1 on with head)
        LaunchCfg c3{B * (S - (head ? 1 : 0)), S, seglen, 0, Sin, Hout, 0, nullptr, true};
        c3.seglen0 = seglen0;
        c3.seg_lo = head ? 1 : 0;
        rc = pass(c3);
    }
    if (rc == GDN_OK && a.hT) {
        for (int b = 0; b < B && rc == GDN_OK; ++b)
            if (cudaMemcpyAsync(a.hT + (size_t)b * st_dv, Hout + ((size_t)b * S + S - 1) * st_dv,
                                sizeof(float) * st_dv, cudaMemcpyDeviceToDevice,
                                st) != cudaSuccess)
                rc = GDN_ERR_CUDA;
    }
    if (Aseg) scratch_free(Aseg, st);
    if (Bseg) scratch_free(Bseg, st);
    if (Sin) scratch_free(Sin, st);
    if (Hout) scratch_free(Hout, st);
    return rc;
}

}  // namespace

bool tc_supported(const FwdArgs &a) {
    if (a.dt != GDN_BF16 || a.vector_gate) return false;
    if (a.dk != 64 && a.dk != 128) return false;
    if (a.dv % kNV != 0 || a.dv > 256) return false;
    if (a.sm.N > 65535 || a.sm.H > 65535) return false;
    if (a.rows <= 0) return false;   // nothing but h0 -> hT: the plain path covers it
    static std::atomic<int> memo[kMaxDeviceMemo];
    return per_device(
               memo, [](int) { return (device_is_sm10x() && encode_fn() != nullptr) ? 1 : 0; },
               0) == 1;
}

gdn_status tc_forward(const FwdArgs &a) {
    // Scratch: T_u (bf16, rows x 64) and W (bf16, rows x d_k) and, for packed batches, the
    // (sequence, chunk) table; stream-ordered, released after the launches.
    cudaStream_t st = a.stream;
    __nv_bfloat16 *Tbuf = nullptr;
    int2 *table = nullptr;
    if (scratch_alloc((void **)&Tbuf, (size_t)a.rows * (64 + a.dk) * sizeof(__nv_bfloat16),
                        st) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_status rc = GDN_OK;
    if (a.sm.cu) {
        if (scratch_alloc((void **)&table, sizeof(int2) * (size_t)a.chunk_slots, st) !=
            cudaSuccess)
            rc = GDN_ERR_CUDA;
        else
            rc = enqueue_chunk_table(a, table);
    }
    int S = choose_segments(a);
    // the segment scan with the wide chunk loop: automatic where the scan is
    // (more segments in one wave of CTAs), or with GDN_OPT_WIDE_CHAIN = 1
    bool wide_seg = false;
    if (S > 1 && seg_wide_applies(a)) {
        wide_seg = true;
        if (option(GDN_OPT_SEGMENTS) < 1) S = choose_segments_wide(a);
    }
    const int nchain = (a.dv / kNV) * a.sm.H * a.sm.N;
    // the overlapped launch: with the wide chunk loop (one CTA per
    // (sequence, head) at d_v = 128) where it is chosen, else the plain one
    int lead = -1;
    bool wide = false;
    const int nchain_w = a.sm.N * a.sm.H * (a.dv / 128);   // wide CTAs
    if (rc == GDN_OK && S <= 1 && wide_applies(a, nchain)) {
        wide = true;
        if (nchain_w < sm_count()) lead = choose_prep_lead(a, nchain_w, true);
    } else if (rc == GDN_OK && S <= 1) {
        lead = choose_prep_lead(a, nchain, false);
    }
    bool done = false;
    if (lead > 0) {
        rc = tc_overlapped(a, Tbuf, lead, wide ? nchain_w : nchain, wide);
        done = rc == GDN_OK;
        if (rc == GDN_ERR_UNSUPPORTED) rc = GDN_OK;   // the plain path below
    }
    // a packed batch on the wide loop: its sequences longest first (launched
    // before the prep, which the chain launch follows programmatically)
    int *order = nullptr;
    if (rc == GDN_OK && !done && wide && a.sm.cu && a.sm.N <= kMaxOrderSeqs) {
        if (scratch_alloc((void **)&order, sizeof(int) * (size_t)a.sm.N, st) != cudaSuccess) {
            rc = GDN_ERR_CUDA;
        } else {
            k_seq_order<<<(a.sm.N + 255) / 256, 256, 0, st>>>(a.sm.cu, a.sm.N, order);
            count_launch();
            if (cudaGetLastError() != cudaSuccess) rc = GDN_ERR_CUDA;
        }
    }
    if (rc == GDN_OK && !done) {
        // the tcgen05 chunk prep (gdn_ut.cu) where it applies, else gdn_prep.cu's
        __nv_bfloat16 *Wbuf = Tbuf + (size_t)a.rows * 64;
        rc = enqueue_ut_w(a, table, Tbuf, Wbuf);
        if (rc == GDN_ERR_UNSUPPORTED) rc = enqueue_tc_prep(a, table, Tbuf, Wbuf);
    }
    if (rc == GDN_OK && !done && wide) {
        LaunchCfg c{a.sm.N, 0, 0, 0, a.h0, a.hT, 0, nullptr, true};
        c.seq_order = order;
        rc = a.dk == 128 ? launch_tcw<128>(a, Tbuf, c) : launch_tcw<64>(a, Tbuf, c);
    } else if (rc == GDN_OK && !done && S > 1) {
        rc = tc_segmented(a, Tbuf, S, wide_seg);
    } else if (rc == GDN_OK && !done) {
        LaunchCfg c{a.sm.N, 0, 0, 0, a.h0, a.hT, 0, nullptr, true};
        rc = a.dk == 128 ? launch_tc<128>(a, Tbuf, c) : launch_tc<64>(a, Tbuf, c);
    }
    scratch_free(Tbuf, st);
    if (table) scratch_free(table, st);
    if (order) scratch_free(order, st);
    return rc;
}

gdn_status tc_state_pass(const FwdArgs &a, const __nv_bfloat16 *Tbuf, float *Hst, float *Vst) {
    if (!tc_supported(a)) return GDN_ERR_UNSUPPORTED;
    LaunchCfg c{a.sm.N, 0, 0, 1, a.h0, nullptr, 0, nullptr, false, Hst, Vst};
    return a.dk == 128 ? launch_tc<128>(a, Tbuf, c) : launch_tc<64>(a, Tbuf, c);
}

}  // namespace gdn
