// gdn_prep.cu -- chunk-prep kernel of the tensor-core path: the in-chunk gate
// cumsum, the decayed beta-weighted Gram and its unit-lower-triangular inverse,
// for every chunk of every (sequence, head) at once.
//
// For one chunk of C = 64 tokens (g_r = sum_{i<=r} log_alpha_i inside the chunk):
//
//   A_rs = beta_r exp(g_r - g_s) (k_r . k_s)   for s < r, else 0
//   T    = (I + A)^{-1}
//
// T turns the chunk's delta-rule updates into the WY form used by the fused
// kernel, U = T diag(beta) V and W = T diag(beta gamma) K; neither depends on
// the state, so all chunks are independent ("Gated DeltaNet GPU并行实现",
// section 3.2: everything inside a chunk is parallel, only the state pass is
// serial).  The kernel writes T_u = T diag(beta) ([rows][64]) and
// W = T diag(beta gamma) K ([rows][d_k]) as bf16 rows indexed like the token
// rows of the inputs, so the fused kernel loads them with the same kind of
// bulk tensor copy as K.  For the backward pass it can also write T itself
// ([rows][64], fp32) and the gate cumsum g ([rows], fp32).
//
// Arithmetic: the Gram and W run on bf16 mma.sync tiles (fragments by
// ldmatrix) with fp32 accumulation (the inputs are bf16 already); the inverse
// solves the four 16x16 diagonal blocks by forward substitution in fp32 and
// merges them (16 -> 32 -> 64) with tf32 mma.sync products,
// T_{10} = -T_11 A_10 T_00 at each level.  The decay exp(g_r - g_s) is formed
// only where s < r (never overflows); when the chunk's total decay is moderate
// it is factored as exp(g_r) exp(-g_s).
//
// The work is small and latency-bound, so the kernel is persistent with four
// CTAs per SM (52 KB of shared memory each at d_k = 128), and every CTA loads
// its next chunk's K tile and gates into registers while it computes the
// current one.
#include <cuda_bf16.h>

#include "gdn_bwd_tc.h"
#include "gdn_internal.h"
#include "gdn_inv.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using ptx::griddep_launch_dependents;
using inv::LDA;
using inv::ldsm4;
using inv::saddr;
using inv::tf32;

constexpr int kCp = 64;
constexpr int LDT = 72;   // bf16 row stride of the T_w tile

template <int DK>
struct PrepLay {
    static constexpr int LDK = DK + 8;                   // bf16 row stride of the K tile
    static constexpr int KBYTES = kCp * LDK * 2;
    static constexpr int TBYTES = kCp * LDA * 4;
    // K stays for W = T_w K.  T's upper-right 32x32 block is never part of
    // T (T is lower triangular and the merges read only its two diagonal
    // 32x32 blocks), so it holds the merge products; once T is final, A's
    // space holds bf16 T_w and T's space the bf16 W tile on its way out.
    static constexpr int OFF_K = 0;
    static constexpr int OFF_T = KBYTES;                 // fp32 [64][68]
    static constexpr int OFF_A = OFF_T + TBYTES;         // fp32 [64][68]
    static constexpr int OFF_G = OFF_A + TBYTES;         // g, beta, beta gamma, 1/gamma
    static constexpr int TOTAL = OFF_G + 4 * kCp * 4;
    static constexpr int KV = kCp * DK / 8 / 128;        // 16-byte K vectors per thread
    static_assert(OFF_A % 16 == 0 && OFF_G % 16 == 0, "align");
    static_assert(kCp * LDT * 2 <= TBYTES && kCp * LDK * 2 <= TBYTES, "staging fits");
};

// D += A(16x16, row) * B(16x8, col), bf16 inputs (two per register), fp32 accumulate.
__device__ __forceinline__ void mma_bf16x16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Persistent: CTA b takes the (chunk slot, head) units b, b + grid, ...  The
// next unit's K tile and gates are loaded into registers while the current
// one is computed.
template <int DK>
__global__ void __launch_bounds__(128, 4)
k_gdn_prep(const __nv_bfloat16 *__restrict__ k, const float *__restrict__ log_alpha,
           const float *__restrict__ beta, SeqMap sm, const int2 *__restrict__ table,
           int max_chunks, int slots, int units, __nv_bfloat16 *__restrict__ Tu_out,
           __nv_bfloat16 *__restrict__ W_out, float *__restrict__ T_out,
           float *__restrict__ G_out, int *err) {
    using L = PrepLay<DK>;
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_K);
    float *Ab = reinterpret_cast<float *>(smem + L::OFF_A);
    float *Tb = reinterpret_cast<float *>(smem + L::OFF_T);
    float *gs = reinterpret_cast<float *>(smem + L::OFF_G);   // g, beta, beta gamma, 1/gamma
    __nv_bfloat16 *Tw = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_A);
    __nv_bfloat16 *Ws = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_T);

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    constexpr int VPR = DK / 8;   // 16-byte vectors per K row

    // unit u -> first token row r0 and token count Lc (0: nothing to do)
    auto decode = [&](long long u, long long &r0, int &Lc) {
        r0 = 0;
        Lc = 0;
        if (u >= units) return;
        const int slot = (int)(u % slots), h = (int)(u / slots);
        int n, c;
        if (table) {
            const int2 e = table[slot];
            n = e.x;
            c = e.y;
            if (n < 0) return;
        } else {
            n = slot / max_chunks;
            c = slot % max_chunks;
        }
        long long row0;
        int len;
        if (sm.cu) {
            const int a = __ldg(sm.cu + n), b = __ldg(sm.cu + n + 1);
            if (!(a >= 0 && a <= b && b <= sm.T_total)) {
                if (tid == 0) atomicCAS(err, 0, kErrBadIndex);
                return;
            }
            row0 = (long long)h * sm.T_total + a;
            len = b - a;
        } else {
            row0 = ((long long)n * sm.H + h) * (long long)sm.T;
            len = sm.T;
        }
        const int t0 = c * kCp;
        if (t0 >= len) return;
        Lc = min(kCp, len - t0);
        r0 = row0 + t0;
    };

    // token rows of the inputs (element counts for the bounds-check build)
    const long long nrows =
        sm.cu ? (long long)sm.H * sm.T_total : (long long)sm.N * sm.H * sm.T;
    (void)nrows;
    uint4 kr[L::KV];
    float la0 = 0.f, la1 = 0.f, b0 = 0.f, b1 = 0.f;
    // K rows past the chunk and the gates there read as zero
    auto fetch = [&](long long r0, int Lc) {
#pragma unroll
        for (int j = 0; j < L::KV; ++j) {
            const int i = tid + 128 * j, r = i / VPR, q = i % VPR;
            kr[j] = (r < Lc && GDN_IDX_OK((r0 + r) * DK + 8 * q, 8, nrows * DK))
                        ? __ldg(reinterpret_cast<const uint4 *>(k + (r0 + r) * DK) + q)
                           : make_uint4(0u, 0u, 0u, 0u);
        }
        if (w == 0) {
            const bool in0 = lane < Lc && GDN_IDX_OK(r0 + lane, 1, nrows);
            const bool in1 = lane + 32 < Lc && GDN_IDX_OK(r0 + lane + 32, 1, nrows);
            la0 = in0 ? __ldg(log_alpha + r0 + lane) : 0.f;
            la1 = in1 ? __ldg(log_alpha + r0 + lane + 32) : 0.f;
            b0 = in0 ? __ldg(beta + r0 + lane) : 0.f;
            b1 = in1 ? __ldg(beta + r0 + lane + 32) : 0.f;
        }
    };

    long long u = blockIdx.x;
    long long r0;
    int Lc;
    decode(u, r0, Lc);
    fetch(r0, Lc);
    for (; u < units; u += gridDim.x) {
        // ---- this unit's K tile and gates into shared memory (every thread
        //      finished the previous unit's reads of Ks, gs and A's space
        //      before the barrier that ended its W product)
#pragma unroll
        for (int j = 0; j < L::KV; ++j) {
            const int i = tid + 128 * j, r = i / VPR, q = i % VPR;
            *reinterpret_cast<uint4 *>(Ks + r * L::LDK + 8 * q) = kr[j];
        }
        if (w == 0) {
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
            gs[lane] = la0;
            gs[lane + 32] = la1;
            gs[64 + lane] = b0;
            gs[96 + lane] = b1;
            gs[128 + lane] = b0 * __expf(la0);
            gs[160 + lane] = b1 * __expf(la1);
            gs[192 + lane] = __expf(-la0);
            gs[224 + lane] = __expf(-la1);
            if (G_out) {
                if (lane < Lc && GDN_IDX_OK(r0 + lane, 1, nrows)) G_out[r0 + lane] = la0;
                if (lane + 32 < Lc && GDN_IDX_OK(r0 + lane + 32, 1, nrows))
                    G_out[r0 + lane + 32] = la1;
            }
        }
        __syncthreads();
        long long r0n;
        int Lcn;
        decode(u + gridDim.x, r0n, Lcn);
        const bool live = Lc > 0;   // uniform over the CTA

        // ---- A = strictly lower (beta_r exp(g_r - g_s) K K^T) from the three
        //      32x32 blocks of the Gram on or below the diagonal: warp 0 rows
        //      and columns 0-31, warp 1 rows 32-63 x columns 0-31, warp 2 rows
        //      and columns 32-63.  A is stored tf32-rounded outside its 16x16
        //      diagonal blocks (only the merges read it there).  Warp 3 zeroes
        //      the upper 16x16 blocks inside T's two diagonal 32x32 blocks.
        if (live && w < 3) {
            const float gC = gs[63];
            const bool span_ok = gC > -80.f;
            const int rb0 = w == 0 ? 0 : 32, cb0 = w == 2 ? 32 : 0;
            const bool diag = w != 1;   // rows 0-15 x columns 16-31 of the block are zero
            const uint32_t a_addr = saddr(Ks + (rb0 + (lane & 15)) * L::LDK + 8 * (lane >> 4));
            const uint32_t b_addr =
                saddr(Ks + (cb0 + (lane & 7) + 8 * (lane >> 4)) * L::LDK + 8 * ((lane >> 3) & 1));
            float acc[2][4][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
#pragma unroll
            for (int k0 = 0; k0 < DK; k0 += 16) {
                uint32_t af[2][4], bf[2][4];
                ldsm4(af[0], a_addr + 2 * k0);
                ldsm4(af[1], a_addr + 2 * (k0 + 16 * L::LDK));
                ldsm4(bf[0], b_addr + 2 * k0);
                ldsm4(bf[1], b_addr + 2 * (k0 + 16 * L::LDK));
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (diag && i == 0 && j >= 2) continue;
                        mma_bf16x16(acc[i][j], af[i], bf[j >> 1][2 * (j & 1)],
                                    bf[j >> 1][2 * (j & 1) + 1]);
                    }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = rb0 + 16 * i + g + 8 * hr;
                    const float br = gs[64 + r], bgr = gs[128 + r], gr = gs[r];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int s = cb0 + 8 * j + 2 * t;
                        const float2 ig = *reinterpret_cast<const float2 *>(gs + 192 + s);
                        float v[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            v[e] = 0.f;
                            if (s + e < r) {
                                const float f = span_ok ? bgr * (e ? ig.y : ig.x)
                                                        : br * __expf(gr - gs[s + e]);
                                v[e] = f * acc[i][j][2 * hr + e];
                                if ((r >> 4) != ((s + e) >> 4)) v[e] = tf32(v[e]);
                            }
                        }
                        *reinterpret_cast<float2 *>(Ab + r * LDA + s) = make_float2(v[0], v[1]);
                    }
                }
        } else if (live) {
            inv::clear_upper16(Tb, lane, 32);
        }
        fetch(r0n, Lcn);   // next unit's loads fly during the rest of this one
        if (live) {
            __syncthreads();

            // ---- T = (I + A)^{-1}
            inv::invert64(Ab, Tb, tid, [] { __syncthreads(); });

            // ---- T_u = T diag(beta) rows out (bf16), and T_w = T diag(beta gamma)
            //      as the bf16 A operand of W = T_w K (in A's space): lane l
            //      takes columns 2l, 2l+1 of rows 16w..16w+15
            {
                const int s = 2 * lane;
                const float2 bs = *reinterpret_cast<const float2 *>(gs + 64 + s);
                const float2 bg = *reinterpret_cast<const float2 *>(gs + 128 + s);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 16 * w + i;
                    float2 tv = *reinterpret_cast<const float2 *>(Tb + r * LDA + s);
                    if (r < 32 && s >= 32) tv = make_float2(0.f, 0.f);   // T's upper-right block
                    if (r < Lc && GDN_IDX_OK((r0 + r) * kCp + s, 2, nrows * kCp)) {
                        *reinterpret_cast<uint32_t *>(Tu_out + (r0 + r) * kCp + s) =
                            pack2(tv.x * bs.x, tv.y * bs.y);
                        if (T_out) *reinterpret_cast<float2 *>(T_out + (r0 + r) * kCp + s) = tv;
                    }
                    *reinterpret_cast<uint32_t *>(Tw + r * LDT + s) = pack2(tv.x * bg.x, tv.y * bg.y);
                }
            }
            __syncthreads();

            // ---- W = T_w K (64 x d_k): warp w owns columns [w d_k/4, (w+1) d_k/4)
            //      for all rows; T_w is lower triangular, so row block mb only
            //      needs k blocks 0..mb.  Result staged as bf16 in T's space.
            {
                constexpr int NP = DK / 64;   // 16-column pairs of n-tiles per warp
#pragma unroll
                for (int np = 0; np < NP; ++np) {
                    const int c0 = w * (DK / 4) + 16 * np;
                    float acc[4][2][4];
#pragma unroll
                    for (int mb = 0; mb < 4; ++mb)
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2)
                            acc[mb][h2][0] = acc[mb][h2][1] = acc[mb][h2][2] = acc[mb][h2][3] = 0.f;
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq) {
                        uint32_t bf[4];
                        ldsm4t(bf, saddr(Ks + (16 * kq + (lane & 7) + 8 * ((lane >> 3) & 1)) * L::LDK +
                                         c0 + 8 * (lane >> 4)));
#pragma unroll
                        for (int mb = kq; mb < 4; ++mb) {
                            uint32_t af[4];
                            ldsm4(af, saddr(Tw + (16 * mb + (lane & 15)) * LDT + 16 * kq +
                                            8 * (lane >> 4)));
                            mma_bf16x16(acc[mb][0], af, bf[0], bf[1]);
                            mma_bf16x16(acc[mb][1], af, bf[2], bf[3]);
                        }
                    }
#pragma unroll
                    for (int mb = 0; mb < 4; ++mb)
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int col = c0 + 8 * h2 + 2 * t;
                            const int ra = 16 * mb + g;
                            *reinterpret_cast<uint32_t *>(Ws + ra * L::LDK + col) =
                                pack2(acc[mb][h2][0], acc[mb][h2][1]);
                            *reinterpret_cast<uint32_t *>(Ws + (ra + 8) * L::LDK + col) =
                                pack2(acc[mb][h2][2], acc[mb][h2][3]);
                        }
                }
            }
            __syncthreads();
            // ---- W rows of the real tokens out, 16-byte vectors
#pragma unroll
            for (int j = 0; j < L::KV; ++j) {
                const int i = tid + 128 * j, r = i / VPR, q = i % VPR;
                if (r < Lc && GDN_IDX_OK((r0 + r) * DK + 8 * q, 8, nrows * DK))
                    *reinterpret_cast<uint4 *>(W_out + (r0 + r) * DK + 8 * q) =
                        *reinterpret_cast<const uint4 *>(Ws + r * L::LDK + 8 * q);
            }
        }
        r0 = r0n;
        Lc = Lcn;
    }
    // the chunk loop that follows may launch once every CTA is here (it waits
    // for this grid's completion before reading T_u / W); triggered at the
    // start, its CTAs were placed on SMs as this grid's left them, which
    // measured slower than the launch's own placement
    griddep_launch_dependents();
}

// Gated linear attention (no erase term): A = 0, so T = I, T_u = diag(beta)
// and W = 0.  One CTA of 64 threads per (chunk slot, head); thread r writes
// row r of the chunk.
template <int DK>
__global__ void __launch_bounds__(64)
k_gla_prep(const float *__restrict__ beta, SeqMap sm, const int2 *__restrict__ table,
           int max_chunks, __nv_bfloat16 *__restrict__ Tu_out, __nv_bfloat16 *__restrict__ W_out,
           int *err) {
    int n, c;
    if (table) {
        const int2 e = table[blockIdx.x];
        n = e.x;
        c = e.y;
        if (n < 0) return;
    } else {
        n = blockIdx.x / max_chunks;
        c = blockIdx.x % max_chunks;
    }
    const int h = blockIdx.y, r = threadIdx.x;
    long long row0;
    int len;
    if (sm.cu) {
        const int a = __ldg(sm.cu + n), b = __ldg(sm.cu + n + 1);
        if (!(a >= 0 && a <= b && b <= sm.T_total)) {
            if (r == 0) atomicCAS(err, 0, kErrBadIndex);
            return;
        }
        row0 = (long long)h * sm.T_total + a;
        len = b - a;
    } else {
        row0 = ((long long)n * sm.H + h) * (long long)sm.T;
        len = sm.T;
    }
    const int t0 = c * kCp;
    if (t0 + r >= len) return;
    const long long row = row0 + t0 + r;
    const uint32_t bb = pack2(__ldg(beta + row), 0.f) & 0xffffu;   // bf16 beta in the low half
    uint4 *tu = reinterpret_cast<uint4 *>(Tu_out + row * kCp);
#pragma unroll
    for (int q = 0; q < kCp / 8; ++q) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        const int e = r - 8 * q;   // position of the diagonal element in this 8-wide piece
        if (e >= 0 && e < 8) w[e >> 1] = (e & 1) ? (bb << 16) : bb;
        tu[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint4 *wr = reinterpret_cast<uint4 *>(W_out + row * DK);
#pragma unroll
    for (int q = 0; q < DK / 8; ++q) wr[q] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

size_t tc_prep_smem(int dk) {
    return dk == 128 ? (size_t)PrepLay<128>::TOTAL : (size_t)PrepLay<64>::TOTAL;
}

namespace {
template <int DK>
gdn_status launch_prep(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                       __nv_bfloat16 *W, float *T_out, float *G_out) {
    const int smem = PrepLay<DK>::TOTAL;
    if (cudaFuncSetAttribute(k_gdn_prep<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    // resident CTAs of the whole device, per device
    static std::atomic<int> memo[kMaxDeviceMemo];
    const int resident = per_device(
        memo,
        [smem](int dev) {
            int nb = 0, nsm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_gdn_prep<DK>, 128, smem) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return -1;
            return max(1, nb) * max(1, nsm);
        },
        0);
    if (resident <= 0) return GDN_ERR_CUDA;
    const long long units = (long long)a.chunk_slots * a.sm.H;
    if (units > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    const int grid = (int)(units < resident ? units : (long long)resident);
    k_gdn_prep<DK><<<grid, 128, smem, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.k), a.log_alpha, a.beta, a.sm, table, a.max_chunks,
        a.chunk_slots, (int)units, Tu, W, T_out, G_out, device_error_word());
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
}  // namespace

gdn_status enqueue_tc_prep(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                           __nv_bfloat16 *W) {
    if (a.chunk_slots <= 0 || a.sm.H <= 0) return GDN_OK;
    if (a.no_erase) {
        dim3 grid(a.chunk_slots, a.sm.H);
        if (a.dk == 128)
            k_gla_prep<128><<<grid, 64, 0, a.stream>>>(a.beta, a.sm, table, a.max_chunks, Tu, W,
                                                        device_error_word());
        else
            k_gla_prep<64><<<grid, 64, 0, a.stream>>>(a.beta, a.sm, table, a.max_chunks, Tu, W,
                                                       device_error_word());
        count_launch();
        return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    return a.dk == 128 ? launch_prep<128>(a, table, Tu, W, nullptr, nullptr)
                       : launch_prep<64>(a, table, Tu, W, nullptr, nullptr);
}

gdn_status enqueue_tc_prep_bwd(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                               __nv_bfloat16 *W, float *T_out, float *G_out) {
    if (a.no_erase || a.vector_gate || a.dt != GDN_BF16 || (a.dk != 64 && a.dk != 128))
        return GDN_ERR_UNSUPPORTED;
    if (a.chunk_slots <= 0 || a.sm.H <= 0) return GDN_OK;
    return a.dk == 128 ? launch_prep<128>(a, table, Tu, W, T_out, G_out)
                       : launch_prep<64>(a, table, Tu, W, T_out, G_out);
}

}  // namespace gdn
