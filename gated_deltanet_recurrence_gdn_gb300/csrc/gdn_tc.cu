// gdn_tc.cu -- fused chunked gated delta rule forward on sm_103a tensor cores.
//
// One CTA owns one (sequence, head, 64-wide d_v tile) and walks its chunks of
// C = 64 tokens in order ("Gated DeltaNet GPU并行实现", section 3.2: matrix
// products inside a chunk, a serial state pass across chunks).  With
// H = S^T (d_k x 64 tile of the state, fp32, kept in registers of the chain
// warpgroup) and g_r the in-chunk cumulative log gate (gamma_r = exp(g_r)):
//
//   G     = [K; Q] K^T                                  (tcgen05, M = 128)
//   A_rs  = beta_r exp(g_r - g_s) (K K^T)_rs,  s < r     (masked before exp)
//   P_rs  = exp(g_r - g_s) (Q K^T)_rs,         s <= r
//   T     = (I + A)^{-1}                                (16x16 diagonal blocks by
//                                                         forward substitution, merged
//                                                         with tf32 mma.sync)
//   U     = T diag(beta) V,  W = T diag(beta gamma) K   (tcgen05, [T_u; T_w] stacked)
//   [W H; gammaQ H]  = [W; diag(gamma) Q] H             (tcgen05, the chain MMA)
//   V'    = U - W H
//   dH    = K^T diag(exp(g_C - g_r)) V'                 (tcgen05)
//   O     = diag(gamma) Q H + P V'                      (tcgen05, accumulates)
//   H    <- exp(g_C) H + dH
//
// Warp roles (320 threads):
//   warps 0-3  chain warpgroup: owns H (thread t = row t = d_k index t), forms
//              V', updates H, stores O.
//   warps 4-7  prep warpgroup: gates, G epilogue (A, P), the inverse, the WY
//              factors as bf16 operands, gamma-scaled Q.  Runs one chunk ahead
//              of the chain.
//   warp 8     TMA producer (one lane): K, Q, V tiles, 128-byte swizzled.
//   warp 9     MMA issuer (one lane) and TMEM owner.
// Every mbarrier wait is bounded; a wait that gives up sets the device error
// word and makes every role leave its loop, after which in-flight MMAs are
// drained and TMEM is freed.
//
// Rows past the end of a sequence are zero (bulk-copy fill, or cleared by the
// prep warpgroup when they belong to the next packed sequence) with
// beta = log_alpha = 0, which leaves every real row unchanged.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kC = 64;         // chunk length
constexpr int kNV = 64;        // d_v columns per CTA
constexpr int kNS = 2;         // input stages
constexpr int kThreadsTC = 320;

// mbarrier slots
enum {
    B_FULL = 0,                 // + stage: TMA bytes landed
    B_READY = B_FULL + kNS,     // + stage: pad rows cleared, stage usable by MMA
    B_FREE = B_READY + kNS,     // + stage: consumers done (MMA commit + prep)
    B_G = B_FREE + kNS,         // M1 done (G in TMEM)
    B_GFREE,                    // prep has read G
    B_T,                        // T_u / T_w in smem
    B_UW,                       // U and W in TMEM
    B_WQ,                       // W and gamma*Q in smem
    B_M2,                       // chain MMA done
    B_H,                        // H (bf16) in smem, TMEM results consumed
    B_VN,                       // V' (bf16) in smem
    B_M34,                      // dH and O done
    B_DRAIN,
    B_COUNT
};

template <int DK>
struct Lay {
    static constexpr int KB = DK / 64;                 // 64-column blocks of K / Q / W
    static constexpr int STAGE = KB * 16384 + 8192;    // per block [K | Q], then V
    static constexpr int OFF_V = KB * 16384;
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_WQ = kNS * STAGE;         // per block [W | gamma Q]
    static constexpr int OFF_H = OFF_WQ + KB * 16384;  // DK rows x 128 B
    static constexpr int OFF_R0 = OFF_H + DK * 128;    // [V~ | P0]
    static constexpr int OFF_R1 = OFF_R0 + 16384;      // [V' | P1]
    static constexpr int OFF_TT = OFF_R1 + 16384;      // [T_u ; T_w], 128 rows x 128 B
    static constexpr int LDA = 68;                     // fp32 row stride of A / T
    static constexpr int OFF_A = OFF_TT + 16384;
    static constexpr int OFF_T = OFF_A + 64 * LDA * 4;
    static constexpr int LDX = 36;
    static constexpr int OFF_X = OFF_T + 64 * LDA * 4; // fp32 [32][36]
    static constexpr int OFF_G = OFF_X + 32 * LDX * 4; // 2 x {g, beta, gamma, 1/gamma}
    static constexpr int OFF_BAR = OFF_G + 2 * 4 * 64 * 4;
    static constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 64;
    static constexpr int ALLOC = TOTAL + 1024;
    static_assert(OFF_WQ % 1024 == 0 && OFF_H % 1024 == 0 && OFF_R0 % 1024 == 0, "align");
    static_assert(OFF_TT % 1024 == 0 && OFF_A % 16 == 0, "align");
    static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

// TMEM column map (512 allocated)
constexpr uint32_t TM_G = 0, TM_U = 64, TM_M2 = 128, TM_H = 192, TM_W = 256;

struct TcParams {
    SeqMap sm;
    const float *log_alpha, *beta, *h0;
    __nv_bfloat16 *o;
    float *hT;
    int *err;
    int dv;
    uint32_t wait_limit;
};

struct Ctl {
    uint64_t *bar;
    volatile int *abort;
    int *err;
    uint32_t limit;
    // Bounded wait; false when this CTA is aborting (now or because of this wait).
    __device__ __forceinline__ bool wait(int b, uint32_t parity) const {
        if (*abort) return false;
        if (mbar_wait(bar + b, parity, limit)) return true;
        *abort = 1;
        atomicCAS(err, 0, kErrTimeout);
        return false;
    }
};

__device__ __forceinline__ float tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// D += A(16x8, row) * B(8x8, col), tf32 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const float (&a)[4], const float (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(__float_as_uint(a[0])), "r"(__float_as_uint(a[1])), "r"(__float_as_uint(a[2])),
          "r"(__float_as_uint(a[3])), "r"(__float_as_uint(b[0])), "r"(__float_as_uint(b[1])));
}

// One 16x8 output tile of  Y = Am * Bm  over k = 0..K-1, operands fp32 in smem
// (row-major with strides lda / ldb).  Returns the C fragment.
template <int K>
__device__ __forceinline__ void tile_mma(float (&c)[4], const float *Am, int lda, const float *Bm,
                                         int ldb, int lane) {
    const int g = lane >> 2, t = lane & 3;
    c[0] = c[1] = c[2] = c[3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        float a[4], b[2];
        a[0] = tf32(Am[g * lda + k0 + t]);
        a[1] = tf32(Am[(g + 8) * lda + k0 + t]);
        a[2] = tf32(Am[g * lda + k0 + t + 4]);
        a[3] = tf32(Am[(g + 8) * lda + k0 + t + 4]);
        b[0] = tf32(Bm[(k0 + t) * ldb + g]);
        b[1] = tf32(Bm[(k0 + t + 4) * ldb + g]);
        mma_tf32(c, a, b);
    }
}

__device__ __forceinline__ void store_tile(float *D, int ldd, const float (&c)[4], int lane,
                                           float scale) {
    const int g = lane >> 2, t = lane & 3;
    D[g * ldd + 2 * t] = scale * c[0];
    D[g * ldd + 2 * t + 1] = scale * c[1];
    D[(g + 8) * ldd + 2 * t] = scale * c[2];
    D[(g + 8) * ldd + 2 * t + 1] = scale * c[3];
}

__device__ __forceinline__ void st16(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// Writes 16 fp32 values (x[0..15], columns c0..c0+15 of a 64-wide row) as bf16
// into a 128-byte-swizzled row.
__device__ __forceinline__ void put_row16(uint8_t *tile, int row, int c0, const float (&x)[16]) {
    const int ch = c0 >> 3;
    st16(tile + sw128_offset(row, ch), pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
         pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
    st16(tile + sw128_offset(row, ch + 1), pack_bf16(x[8], x[9]), pack_bf16(x[10], x[11]),
         pack_bf16(x[12], x[13]), pack_bf16(x[14], x[15]));
}

template <int DK>
__global__ void __launch_bounds__(kThreadsTC, 1)
k_gdn_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
         const __grid_constant__ CUtensorMap tm_v, TcParams p) {
    using L = Lay<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *gb = reinterpret_cast<float *>(sm + L::OFF_G);   // [2][4][64]
    float *Ab = reinterpret_cast<float *>(sm + L::OFF_A);
    float *Tb = reinterpret_cast<float *>(sm + L::OFF_T);
    float *Xb = reinterpret_cast<float *>(sm + L::OFF_X);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dv0 = blockIdx.x * kNV, h = blockIdx.y, n = blockIdx.z;

    // ---- sequence bounds (validated; an invalid packed range is an error)
    long long row0 = 0;
    int len = 0;
    bool ok_seq = true;
    if (p.sm.cu) {
        const int a = __ldg(p.sm.cu + n), b = __ldg(p.sm.cu + n + 1);
        ok_seq = a >= 0 && a <= b && b <= p.sm.T_total;
        if (ok_seq) {
            row0 = (long long)h * p.sm.T_total + a;
            len = b - a;
        }
    } else {
        row0 = ((long long)n * p.sm.H + h) * (long long)p.sm.T;
        len = p.sm.T;
    }
    if (!ok_seq) {
        if (tid == 0) atomicCAS(p.err, 0, kErrSeqlens);
        return;  // before any barrier or TMEM use
    }
    const int ytok0 = p.sm.cu ? __ldg(p.sm.cu + n) : 0;   // token coordinate of chunk 0
    const int zcoord = p.sm.cu ? h : n * p.sm.H + h;
    const int nch = (len + kC - 1) / kC;
    const long long srow = ((long long)n * p.sm.H + h) * p.dv;   // state row of (n, h)

    if (warp == 9) {
        tmem_alloc(misc, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar + i, 1);
        for (int s = 0; s < kNS; ++s) mbar_init(bar + B_FREE + s, 2);
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};

    if (warp < 4) {
        // ================================================= chain warpgroup
        const int t = tid;   // TMEM lane = H row (d_k index) / output row - 64
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float hreg[kNV];
#pragma unroll
        for (int c = 0; c < kNV; ++c)
            hreg[c] = (t < DK && p.h0) ? __ldg(p.h0 + (srow + dv0 + c) * DK + t) : 0.f;
        uint8_t *Hs = sm + L::OFF_H;
        for (int j = 0; j < nch; ++j) {
            // (i) publish H as the bf16 B operand of the chain MMA
            if (t < DK) {
#pragma unroll
                for (int c0 = 0; c0 < kNV; c0 += 16) {
                    float x[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] = hreg[c0 + i];
                    put_row16(Hs, t, c0, x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 128);
            if (t == 0) mbar_arrive(bar + B_H);
            // (ii) V' = U - W H, and its decayed copy for the state update
            {
                bool ok = ctl.wait(B_WQ, j & 1);   // orders this chunk's gates too
                ok = ok && ctl.wait(B_M2, j & 1);
                if (!named_bar_and(1, 128, ok)) break;
            }
            tc_fence_after();
            const float *gj = gb + (j & 1) * 256;
            const float gC = gj[63];
            const float decayC = __expf(gC);
            if (t < 64) {
                const float ev = __expf(gC - gj[t]);
                uint8_t *VT = sm + L::OFF_R0, *VN = sm + L::OFF_R1;
#pragma unroll
                for (int c0 = 0; c0 < kNV; c0 += 16) {
                    float wh[16], u[16], vt[16];
                    tmem_ld16f(tmem + lane_base + TM_M2 + c0, wh);
                    tmem_ld16f(tmem + lane_base + TM_U + c0, u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        u[i] -= wh[i];
                        vt[i] = u[i] * ev;
                    }
                    put_row16(VN, t, c0, u);
                    put_row16(VT, t, c0, vt);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 128);
            if (t == 0) mbar_arrive(bar + B_VN);
            // (iii) H <- exp(g_C) H + dH;  O rows out
            if (!named_bar_and(1, 128, ctl.wait(B_M34, j & 1))) break;
            tc_fence_after();
            if (t < DK) {
#pragma unroll
                for (int c0 = 0; c0 < kNV; c0 += 16) {
                    float dh[16];
                    tmem_ld16f(tmem + lane_base + TM_H + c0, dh);
#pragma unroll
                    for (int i = 0; i < 16; ++i) hreg[c0 + i] = fmaf(decayC, hreg[c0 + i], dh[i]);
                }
            }
            if (t >= 64) {
                const int r = t - 64;
                const int L_ = min(kC, len - j * kC);
                __nv_bfloat16 *orow = p.o + (row0 + (long long)j * kC + r) * p.dv + dv0;
#pragma unroll
                for (int c0 = 0; c0 < kNV; c0 += 16) {
                    float ov[16];
                    tmem_ld16f(tmem + lane_base + TM_M2 + c0, ov);
                    if (r < L_) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
                        dst[0] = make_uint4(pack_bf16(ov[0], ov[1]), pack_bf16(ov[2], ov[3]),
                                            pack_bf16(ov[4], ov[5]), pack_bf16(ov[6], ov[7]));
                        dst[1] = make_uint4(pack_bf16(ov[8], ov[9]), pack_bf16(ov[10], ov[11]),
                                            pack_bf16(ov[12], ov[13]),
                                            pack_bf16(ov[14], ov[15]));
                    }
                }
            }
        }
        if (!*abort_flag && p.hT && t < DK) {
#pragma unroll
            for (int c = 0; c < kNV; ++c) p.hT[(srow + dv0 + c) * DK + t] = hreg[c];
        }
    } else if (warp < 8) {
        // ================================================== prep warpgroup
        const int t = tid - 128;
        const int w = warp - 4;
        const uint32_t lane_base = (uint32_t)(w * 32) << 16;
        for (int j = 0; j < nch; ++j) {
            const int s = j % kNS;
            uint8_t *stg = sm + L::OFF_STAGE + s * L::STAGE;
            const int L_ = min(kC, len - j * kC);
            float *gj = gb + (j & 1) * 256;   // g, beta, gamma, 1/gamma
            // (a) gates and their in-chunk cumulative sum
            if (w == 0) {
                const long long r0 = row0 + (long long)j * kC;
                float la0 = lane < L_ ? __ldg(p.log_alpha + r0 + lane) : 0.f;
                float la1 = lane + 32 < L_ ? __ldg(p.log_alpha + r0 + lane + 32) : 0.f;
                const float b0 = lane < L_ ? __ldg(p.beta + r0 + lane) : 0.f;
                const float b1 = lane + 32 < L_ ? __ldg(p.beta + r0 + lane + 32) : 0.f;
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
                gj[lane] = la0;
                gj[lane + 32] = la1;
                gj[64 + lane] = b0;
                gj[64 + lane + 32] = b1;
                gj[128 + lane] = __expf(la0);
                gj[128 + lane + 32] = __expf(la1);
                gj[192 + lane] = __expf(-la0);   // used only when the chunk's span is < 80
                gj[192 + lane + 32] = __expf(-la1);
            }
            if (!named_bar_and(2, 128, ctl.wait(B_FULL + s, (j / kNS) & 1))) break;
            if (p.sm.cu && L_ < kC) {
                // rows past this sequence belong to the next one: clear them
                const int per_row = 2 * DK / 8 + kNV / 8;   // 16-byte pieces per row
                for (int i = t; i < (kC - L_) * per_row; i += 128) {
                    const int r = L_ + i / per_row, q = i % per_row;
                    uint8_t *base;
                    int chn;
                    if (q < 2 * DK / 8) {
                        const int blk = q / 16, which = (q / 8) & 1;   // per block: K, then Q
                        base = stg + blk * 16384 + which * 8192;
                        chn = q & 7;
                    } else {
                        base = stg + L::OFF_V;
                        chn = q - 2 * DK / 8;
                    }
                    st16(base + sw128_offset(r, chn), 0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            named_bar(2, 128);
            if (t == 0) mbar_arrive(bar + B_READY + s);
            // (b) G epilogue: A (fp32, for the inverse) and P (bf16 operand)
            if (!named_bar_and(2, 128, ctl.wait(B_G, j & 1))) break;
            tc_fence_after();
            {
                const float gC = gj[63];
                const bool span_ok = gC > -80.f;
                const int r = t & 63;
                const float gr = gj[r];
                float fr = span_ok ? gj[128 + r] : 0.f;
                if (t < 64) fr *= gj[64 + r];   // beta_r folded into A
                uint8_t *Pt = sm + ((j & 1) ? L::OFF_R1 : L::OFF_R0) + 8192;
#pragma unroll
                for (int c0 = 0; c0 < kC; c0 += 16) {
                    float gv[16];
                    tmem_ld16f(tmem + lane_base + TM_G + c0, gv);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int sidx = c0 + i;
                        const bool keep = (t < 64) ? (sidx < r) : (sidx <= r);
                        float f;
                        if (span_ok) f = fr * gj[192 + sidx];
                        else f = (t < 64 ? gj[64 + r] : 1.f) * __expf(keep ? gr - gj[sidx] : 0.f);
                        gv[i] = keep ? f * gv[i] : 0.f;
                    }
                    if (t < 64) {
                        float4 *dst = reinterpret_cast<float4 *>(Ab + r * L::LDA + c0);
                        dst[0] = make_float4(gv[0], gv[1], gv[2], gv[3]);
                        dst[1] = make_float4(gv[4], gv[5], gv[6], gv[7]);
                        dst[2] = make_float4(gv[8], gv[9], gv[10], gv[11]);
                        dst[3] = make_float4(gv[12], gv[13], gv[14], gv[15]);
                    } else {
                        put_row16(Pt, r, c0, gv);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(2, 128);
            if (t == 0) mbar_arrive(bar + B_GFREE);
            // (c) T = (I + A)^{-1}
            if (w < 2) {
                // 16x16 diagonal blocks, one column per thread, right-looking
                const int blk = t >> 4, c = t & 15, o = blk * 16;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < 16; ++s2) {
#pragma unroll
                    for (int r = s2 + 1; r < 16; ++r)
                        x[r] = fmaf(-Ab[(o + r) * L::LDA + o + s2], x[s2], x[r]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tb[(o + r) * L::LDA + o + c] = x[r];
            } else {
                // zero the six strictly upper 16x16 blocks
                for (int i = t - 64; i < 6 * 256; i += 64) {
                    const int b = i >> 8, e = i & 255;
                    const int bi = b < 3 ? 0 : (b < 5 ? 1 : 2);
                    const int bj = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
                    Tb[(bi * 16 + (e >> 4)) * L::LDA + bj * 16 + (e & 15)] = 0.f;
                }
            }
            named_bar(2, 128);
            {
                // 16 -> 32: T_{2p+1,2p} = -D_{2p+1} A_{2p+1,2p} D_{2p}
                const int pr = w >> 1, nh = w & 1;
                const int ro = 32 * pr + 16, co = 32 * pr;
                float *Xw = Xb + w * 16 * 9;
                float c4[4];
                tile_mma<16>(c4, Ab + ro * L::LDA + co, L::LDA, Tb + co * L::LDA + co + 8 * nh,
                             L::LDA, lane);
                store_tile(Xw, 9, c4, lane, 1.f);
                __syncwarp();
                tile_mma<16>(c4, Tb + ro * L::LDA + ro, L::LDA, Xw, 9, lane);
                __syncwarp();
                store_tile(Tb + ro * L::LDA + co + 8 * nh, L::LDA, c4, lane, -1.f);
            }
            named_bar(2, 128);
            {
                // 32 -> 64: T_{1,0} = -E1 (A_{1,0} E0), 32x32 blocks
                const int mt = w >> 1, nt0 = 2 * (w & 1);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float c4[4];
                    tile_mma<32>(c4, Ab + (32 + 16 * mt) * L::LDA, L::LDA, Tb + 8 * (nt0 + q),
                                 L::LDA, lane);
                    store_tile(Xb + 16 * mt * L::LDX + 8 * (nt0 + q), L::LDX, c4, lane, 1.f);
                }
                named_bar(2, 128);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float c4[4];
                    tile_mma<32>(c4, Tb + (32 + 16 * mt) * L::LDA + 32, L::LDA,
                                 Xb + 8 * (nt0 + q), L::LDX, lane);
                    store_tile(Tb + (32 + 16 * mt) * L::LDA + 8 * (nt0 + q), L::LDA, c4, lane,
                               -1.f);
                }
            }
            named_bar(2, 128);
            {
                // T_u = T diag(beta) (rows 0-63), T_w = T diag(beta gamma) (rows 64-127)
                const int r = t & 63;
                uint8_t *TT = sm + L::OFF_TT;
                const float *Tr = Tb + r * L::LDA;
#pragma unroll
                for (int c0 = 0; c0 < kC; c0 += 16) {
                    float x[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int sidx = c0 + i;
                        float sc = gj[64 + sidx];
                        if (t >= 64) sc *= gj[128 + sidx];
                        x[i] = sidx <= r ? Tr[sidx] * sc : 0.f;
                    }
                    put_row16(TT, t, c0, x);
                }
            }
            fence_proxy_async_smem();
            named_bar(2, 128);
            if (t == 0) mbar_arrive(bar + B_T);
            // (d) gamma-scaled Q into the chain operand (after the previous
            //     chain MMA has read it)
            if (!named_bar_and(2, 128, j == 0 || ctl.wait(B_M2, (j - 1) & 1))) break;
            if (t < 64) {
                const float gam = gj[128 + t];
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    const uint8_t *src = stg + blk * 16384 + 8192;
                    uint8_t *dst = sm + L::OFF_WQ + blk * 16384 + 8192;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint32_t off = sw128_offset(t, ch);
                        uint4 v = *reinterpret_cast<const uint4 *>(src + off);
                        uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&wv[e]);
                            float2 f2 = __bfloat1622float2(b2);
                            wv[e] = pack_bf16(f2.x * gam, f2.y * gam);
                        }
                        st16(dst + off, wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            }
            // (e) W rows (TMEM lanes 64-127) into the chain operand
            if (!named_bar_and(2, 128, ctl.wait(B_UW, j & 1))) break;
            tc_fence_after();
            if (t >= 64) {
                const int r = t - 64;
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    uint8_t *dst = sm + L::OFF_WQ + blk * 16384;
#pragma unroll
                    for (int c0 = 0; c0 < 64; c0 += 16) {
                        float x[16];
                        tmem_ld16f(tmem + lane_base + TM_W + blk * 64 + c0, x);
                        put_row16(dst, r, c0, x);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(2, 128);
            if (t == 0) {
                mbar_arrive(bar + B_WQ);
                mbar_arrive(bar + B_FREE + s);
            }
        }
    } else if (warp == 8) {
        // ================================================= TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;
            for (int j = 0; j < nch; ++j) {
                const int s = j % kNS;
                if (j >= kNS && !ctl.wait(B_FREE + s, ((j / kNS) - 1) & 1)) break;
                uint8_t *stg = sm + L::OFF_STAGE + s * L::STAGE;
                uint64_t *fb = bar + B_FULL + s;
                mbar_arrive_expect_tx(fb, (uint32_t)L::STAGE);
                const int y = ytok0 + j * kC;
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    tma_load_3d(stg + blk * 16384, &tm_k, fb, blk * 64, y, zcoord);
                    tma_load_3d(stg + blk * 16384 + 8192, &tm_q, fb, blk * 64, y, zcoord);
                }
                tma_load_3d(stg + L::OFF_V, &tm_v, fb, dv0, y, zcoord);
                issued = j + 1;
            }
            // on abort, let copies still in flight land before the CTA exits
            if (*abort_flag) {
                for (int j = max(0, issued - kNS); j < issued; ++j)
                    mbar_wait(bar + B_FULL + j % kNS, (j / kNS) & 1, ctl.limit);
            }
        }
    } else {
        // ==================================================== MMA issuer
        if (lane == 0 && nch > 0) {
            constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);   // [K;Q] K^T
            constexpr uint32_t idU = make_idesc_bf16(128, 64, false, true);    // TT V
            constexpr uint32_t idW = make_idesc_bf16(128, DK, false, true);    // TT K
            constexpr uint32_t idM2 = make_idesc_bf16(128, kNV, false, true);  // [W;gQ] H
            constexpr uint32_t idM3 = make_idesc_bf16(128, kNV, true, true);   // K^T V~
            constexpr uint32_t idM4 = make_idesc_bf16(128, kNV, false, true);  // [x;P] V'
            const uint32_t sbase = smem_u32(sm);
            auto stage_addr = [&](int j) { return sbase + L::OFF_STAGE + (j % kNS) * L::STAGE; };
            auto issue_m1 = [&](int j) {
                const uint32_t st = stage_addr(j);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_G, make_sdesc(st + off, 16, 1024, kSwizzle128B),
                             make_sdesc(st + off, 16, 1024, kSwizzle128B), idG, kk > 0);
                }
                mma_commit(bar + B_G);
            };
            auto issue_uw = [&](int j) {
                const uint32_t st = stage_addr(j);
                const uint32_t tt = sbase + L::OFF_TT;
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    const uint64_t a = make_sdesc(tt + kk * 32, 16, 1024, kSwizzle128B);
                    mma_bf16(tmem + TM_U,
                             a, make_sdesc(st + L::OFF_V + kk * 2048, 16, 1024, kSwizzle128B),
                             idU, kk > 0);
                    mma_bf16(tmem + TM_W,
                             a, make_sdesc(st + kk * 2048, 16384, 1024, kSwizzle128B), idW,
                             kk > 0);
                }
                mma_commit(bar + B_UW);
            };
            if (ctl.wait(B_READY, 0)) issue_m1(0);
            if (ctl.wait(B_T, 0)) issue_uw(0);
            for (int j = 0; j < nch; ++j) {
                if (*abort_flag) break;
                const uint32_t st = stage_addr(j);
                // 1. chain MMA  [W; gamma Q] H
                if (!ctl.wait(B_H, j & 1) || !ctl.wait(B_WQ, j & 1)) break;
                tc_fence_after();
                {
                    const uint32_t wq = sbase + L::OFF_WQ, hs = sbase + L::OFF_H;
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_bf16(tmem + TM_M2, make_sdesc(wq + off, 16, 1024, kSwizzle128B),
                                 make_sdesc(hs + kk * 2048, 16, 1024, kSwizzle128B), idM2,
                                 kk > 0);
                    }
                    mma_commit(bar + B_M2);
                }
                // 2. next chunk's Gram
                if (j + 1 < nch) {
                    if (!ctl.wait(B_READY + (j + 1) % kNS, ((j + 1) / kNS) & 1) ||
                        !ctl.wait(B_GFREE, j & 1))
                        break;
                    tc_fence_after();
                    issue_m1(j + 1);
                }
                // 3. dH = K^T V~ and O += P V'
                if (!ctl.wait(B_VN, j & 1)) break;
                tc_fence_after();
                {
                    const uint32_t vt = sbase + L::OFF_R0, vn = sbase + L::OFF_R1;
                    const uint32_t pr = sbase + ((j & 1) ? L::OFF_R1 : L::OFF_R0);
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk) {
                        mma_bf16(tmem + TM_H,
                                 make_sdesc(st + kk * 2048, 16384, 1024, kSwizzle128B),
                                 make_sdesc(vt + kk * 2048, 16, 1024, kSwizzle128B), idM3,
                                 kk > 0);
                        mma_bf16(tmem + TM_M2, make_sdesc(pr + kk * 32, 16, 1024, kSwizzle128B),
                                 make_sdesc(vn + kk * 2048, 16, 1024, kSwizzle128B), idM4, 1u);
                    }
                    mma_commit(bar + B_M34);
                    mma_commit(bar + B_FREE + (j % kNS));
                }
                // 4. next chunk's WY factors
                if (j + 1 < nch) {
                    if (!ctl.wait(B_T, (j + 1) & 1)) break;
                    tc_fence_after();
                    issue_uw(j + 1);
                }
            }
            // every issued MMA has finished before TMEM is released
            mma_commit(bar + B_DRAIN);
            mbar_wait(bar + B_DRAIN, 0, ctl.limit);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

// -------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 3-D view [z][y][x] of a bf16 tensor with rows of `d` elements; box 64 x 64 x 1,
// 128-byte swizzle, out-of-range rows read as zero.
bool make_map(CUtensorMap *m, const void *base, int d, long long ydim, long long zdim) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)ydim, (cuuint64_t)zdim};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)ydim};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool device_is_sm10x() {
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return false;
    return major == 10;
}

template <int DK>
gdn_status launch_tc(const FwdArgs &a) {
    using L = Lay<DK>;
    const long long ydim = a.sm.cu ? a.sm.T_total : a.sm.T;
    const long long zdim = a.sm.cu ? a.sm.H : (long long)a.sm.N * a.sm.H;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, DK, ydim, zdim) || !make_map(&mk, a.k, DK, ydim, zdim) ||
        !make_map(&mv, a.v, a.dv, ydim, zdim))
        return GDN_ERR_CUDA;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(k_gdn_tc<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::ALLOC) != cudaSuccess)
            return GDN_ERR_CUDA;
        attr_set = true;
    }
    TcParams p;
    p.sm = a.sm;
    p.log_alpha = a.log_alpha;
    p.beta = a.beta;
    p.h0 = a.h0;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.hT = a.hT;
    p.err = device_error_word();
    p.dv = a.dv;
    const long long lim = option(GDN_OPT_WAIT_LIMIT);
    p.wait_limit = lim > 0 ? (uint32_t)(lim > 0x7fffffffLL ? 0x7fffffffLL : lim) : (1u << 22);
    dim3 grid(a.dv / kNV, a.sm.H, a.sm.N);
    const int slot = timer_begin(a.stream, "k_gdn_tc");
    k_gdn_tc<DK><<<grid, kThreadsTC, L::ALLOC, a.stream>>>(mq, mk, mv, p);
    timer_end(slot, a.stream);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

bool tc_supported(const FwdArgs &a) {
    if (a.dt != GDN_BF16) return false;
    if (a.dk != 64 && a.dk != 128) return false;
    if (a.dv % kNV != 0 || a.dv > 256) return false;
    if (a.sm.N > 65535 || a.sm.H > 65535) return false;
    if (a.rows <= 0) return false;   // nothing but h0 -> hT: the plain path covers it
    static int ok = -1;
    if (ok < 0) ok = (device_is_sm10x() && encode_fn() != nullptr) ? 1 : 0;
    return ok == 1;
}

gdn_status tc_forward(const FwdArgs &a) {
    return a.dk == 128 ? launch_tc<128>(a) : launch_tc<64>(a);
}

}  // namespace gdn
