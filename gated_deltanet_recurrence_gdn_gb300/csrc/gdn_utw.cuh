// gdn_utw.cuh -- the forward's chunk prep with W out (k_gdn_utw's unit
// loop), as a device function that one 128-thread pipeline runs: the prep
// kernel (gdn_ut.cu) runs one per CTA, four CTAs per SM; the chain kernel's
// overlapped launch (gdn_tc.cu) runs three per CTA on the SMs its chain CTAs
// leave free.
//
// Per unit (chunk, head), with g_r the in-chunk cumulative log decay
// ("Gated DeltaNet GPU并行实现", section 3.2):
//   A_rs = beta_r exp(g_r - g_s) (k_r . k_s) for s < r,
//   T_u = (I + A)^{-1} diag(beta),  W = (I + A)^{-1} diag(beta gamma) K,
// T_u as [rows][64] and W as [rows][d_k], bf16, rows indexed like the token
// rows of the inputs.  Thread 64 brings the K tile by bulk tensor copy
// (128-byte swizzle, two buffers in flight) and issues the Gram K K^T as
// tcgen05 MMAs into tensor memory (M = 128: rows 64-127 of the operand are
// whatever follows the tile and are never read), the next unit's while warps
// 0-1 form A or run the inverse's first stage (warps 2-3 are idle in both),
// so the Gram is done long before it is read; warp 0 prefetches the next
// unit's gates into registers.  All four warps invert I + A in place
// (gdn_inv.cuh: A and T share one fp32 tile), write T_u rows and stage T_w
// (bf16, swizzled) in that tile once every thread holds its T values; thread
// 0 issues W^T = K^T T_w^T (M = d_k lanes, N = 64 tokens) into the unit's
// Gram columns; the warps read it back, transpose it through the tile again
// and store W rows.  Per pipeline: two K buffers, the A/T tile and 128
// tensor-memory columns (a Gram / W^T accumulator per buffer), about 51 KB
// of shared memory at d_k = 128.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "gdn_inv.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

#ifndef UTRACE
#define UTRACE(i, ev) \
    do {              \
    } while (0)
#endif

namespace gdn {
namespace {

using namespace ptx;
using namespace tcx;
using inv::LDA;

constexpr int kU = 64;

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
    long long units;          // units of the launch: H * chunk_slots, or N * H * nc
    uint32_t wait_limit;
    // Chunk-major window (dense batches): the launch's units are the
    // (sequence, head) pairs of chunks c0 .. c0 + nc - 1, chunk by chunk;
    // nc = 0: every (head, chunk slot) unit in that order.
    int c0, nc;
    // Ready flags, one per unit (index h * chunk_slots + slot): set to 1 with
    // release semantics at gpu scope once the unit's T_u and W rows are stored
    // (null: not published).  done_zero: n_done flags this launch clears
    // before anything else (null: none).
    uint32_t *done;
    uint32_t *done_zero;
    long long n_done;
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
    // units, one per 64 token rows of a head, number far fewer than 2^31
    const uint32_t uu = (uint32_t)u, cs = (uint32_t)p.chunk_slots;
    const int h = (int)(uu / cs), slot = (int)(uu - (uint32_t)h * cs);
    int n, c;
    if (p.table) {
        const int2 e = p.table[slot];
        n = e.x;
        c = e.y;
        if (n < 0) return r;
    } else {
        n = slot / p.max_chunks;
        c = slot - n * p.max_chunks;
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

// Unit v of a launch as its natural index h * chunk_slots + slot.
// (A window's units, one per 64 token rows of a dense batch, number far
// fewer than 2^31, so the divisions stay in 32 bits.)
__device__ __forceinline__ long long unit_id(const UtParams &p, long long v) {
    if (p.nc <= 0) return v;
    const uint32_t nh = (uint32_t)p.sm.N * (uint32_t)p.sm.H, w = (uint32_t)v;
    const uint32_t c = w / nh, r = w - c * nh;
    const uint32_t n = r / (uint32_t)p.sm.H, h = r - n * (uint32_t)p.sm.H;
    return (long long)h * p.chunk_slots + (long long)n * p.max_chunks + p.c0 + (int)c;
}

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
    static constexpr int OFF_BAR = OFF_GS + 2048;           // 2 x g, beta, gamma, exp(-g)
    static constexpr int OFF_MISC = OFF_BAR + V_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 16;
    static constexpr int ALLOC = TOTAL + 1024;
    static_assert(OFF_AT % 1024 == 0, "the T_w tile is a 128-byte-swizzled operand");
    static_assert(kU * DK * 2 <= kU * LDA * 4, "the W staging fits the A/T tile");
    static_assert(kU * LDA * 4 >= 8192, "the last tile's unused operand rows stay in bounds");
};

// Before the CTA's first barrier: the pipeline's mbarriers and abort flag.
template <int DK>
__device__ __forceinline__ void utw_init(uint8_t *sm, int tid) {
    using L = VLay<DK>;
    if (tid == 0) {
        uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
        for (int i = 0; i < V_COUNT; ++i) mbar_init(bar + i, 1);
        *reinterpret_cast<volatile int *>(sm + L::OFF_MISC + 4) = 0;
        fence_mbar_init();
    }
}

// One pipeline's unit loop over the launch's units first + i * stride,
// i < nunits, in the shared memory at `sm` (1024-byte aligned, VLay<DK>),
// the tensor-memory columns tmem .. tmem + 127 and named barrier bar_id of
// its 128 threads (tid 0..127).  Every MMA it issued has finished and every
// copy it issued has landed when it returns.
template <int DK>
__device__ __forceinline__ void utw_run(uint8_t *sm, uint32_t tmem, int tid, uint32_t bar_id,
                                        const CUtensorMap *tm_k_, const UtParams &p,
                                        long long first, long long stride, long long nunits) {
    using L = VLay<DK>;
    const CUtensorMap &tm_k = *tm_k_;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *AT = reinterpret_cast<float *>(sm + L::OFF_AT);
    float *gsb = reinterpret_cast<float *>(sm + L::OFF_GS);   // unit i's gates at 256 (i & 1)
    const int warp = tid >> 5, lane = tid & 31;
    // token rows of the inputs (element counts for the bounds-check build)
    const long long nrows =
        p.sm.cu ? (long long)p.sm.H * p.sm.T_total : (long long)p.sm.N * p.sm.H * p.sm.T;
    (void)nrows;
    auto uid = [&](long long i) { return unit_id(p, first + i * stride); };
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};
    const uint32_t sb = smem_u32(sm);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    auto bar128 = [bar_id] { named_bar(bar_id, 128); };
    constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);
    constexpr uint32_t idW = make_idesc_bf16(128, 64, true, false);

    // ---- thread 64: the bulk copy of unit i's K tile into buffer i & 1
    constexpr int kIssuer = 64;
    long long loaded = 0, grammed = 0;
    auto load = [&](long long i) {
        const int b = (int)(i & 1);
        const Unit un = decode(p, uid(i));
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
        const Unit un = decode(p, uid(i));
        const bool in0 = lane < un.len && GDN_IDX_OK(un.row0 + lane, 1, nrows);
        const bool in1 = lane + 32 < un.len && GDN_IDX_OK(un.row0 + lane + 32, 1, nrows);
        la0 = in0 ? __ldg(p.log_alpha + un.row0 + lane) : 0.f;
        la1 = in1 ? __ldg(p.log_alpha + un.row0 + lane + 32) : 0.f;
        be0 = in0 ? __ldg(p.beta + un.row0 + lane) : 0.f;
        be1 = in1 ? __ldg(p.beta + un.row0 + lane + 32) : 0.f;
    };
    // ---- warp 3: a unit's g = in-chunk cumsum of log_alpha, gamma = e^g,
    //      e^{-g} and beta into its gate buffer, from the registers
    auto scan_gates = [&](float *gs) {
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
    };
    // unit 0's gates now; later units' one unit ahead, while warps 0-1 form A
    // (warp 3 is idle there), so no unit waits for its gate scan
    if (warp == 3 && nunits > 0) {
        fetch_gates(0);
        scan_gates(gsb);
        if (nunits > 1) fetch_gates(1);
    }
    if (tid == kIssuer && nunits > 0) {
        prefetch_tmap(&tm_k);
        load(0);
        if (nunits > 1) load(1);
        gram(0);   // a failed wait sets the abort flag, seen at every thread's next wait
    }

    long long i = 0;
    for (; i < nunits; ++i) {
        const int b = (int)(i & 1);
        const Unit un = decode(p, uid(i));
        const float *gs = gsb + 256 * b;   // written by warp 3 before an earlier barrier
        UTRACE(i, 0);
        // ---- A from the Gram rows (warps 0-1), every row written in full
        if (!named_bar_and(bar_id, 128, ctl.wait(V_GDONE + b, (uint32_t)((i >> 1) & 1)))) break;
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
        } else if (warp == 3 && i + 1 < nunits) {
            // the next unit's gates into the other buffer (unit i - 1, its last
            // reader, finished before this unit's first barrier)
            scan_gates(gsb + 256 * (b ^ 1));
            if (i + 2 < nunits) fetch_gates(i + 2);
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
            // the previous unit's T_u and W rows, stored a whole unit ago, are
            // published to other CTAs' bulk tensor copies (async proxy) at gpu
            // scope: each thread orders its stores with the async proxy, the
            // barrier gathers them, thread 0 releases the flag.  Here, before
            // this unit stores anything, the fence has nothing left to wait for.
            const bool publish = p.done && i > 0;
            if (publish) fence_proxy_async_global();
            bar128();
            if (publish && tid == 0) st_release_gpu(p.done + uid(i - 1), 1u);
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
        if (!named_bar_and(bar_id, 128, ctl.wait(V_WDONE + b, (uint32_t)((i >> 1) & 1)))) break;
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
    // the last unit's rows (a loop that stopped early publishes nothing more:
    // its error is already recorded, and the chain's waits end on their limit)
    if (p.done && nunits > 0 && i == nunits) {
        fence_proxy_async_global();
        bar128();
        if (tid == 0) st_release_gpu(p.done + uid(nunits - 1), 1u);
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
}

// ---------------------------------------------------------------- host

// The parameters of a prep launch over every (chunk slot, head) unit.
inline void ut_params(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu, __nv_bfloat16 *W,
                      UtParams *p) {
    *p = UtParams{};
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
}

// The same, with the K tensor map.
inline bool ut_setup(const FwdArgs &a, int dk, const int2 *table, __nv_bfloat16 *Tu,
                     __nv_bfloat16 *W, CUtensorMap *mk, UtParams *p) {
    const long long ydim = a.sm.cu ? a.sm.T_total : a.sm.T;
    const long long zdim = a.sm.cu ? a.sm.H : (long long)a.sm.N * a.sm.H;
    if (!make_map(mk, a.k, dk, ydim, zdim)) return false;
    ut_params(a, table, Tu, W, p);
    return true;
}

}  // namespace
}  // namespace gdn
