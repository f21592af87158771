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
// bulk tensor copy as K.
//
// Arithmetic: the Gram runs on bf16 mma.sync tiles with fp32 accumulation
// (the inputs are bf16 already); the inverse solves the four 16x16 diagonal
// blocks by forward substitution in fp32 and merges them (16 -> 32 -> 64) with
// tf32 mma.sync products, T_{10} = -T_11 A_10 T_00 at each level.  The decay
// exp(g_r - g_s) is formed only where s < r (never overflows); when the chunk's
// total decay is moderate it is factored as exp(g_r) exp(-g_s).
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kCp = 64;
constexpr int LDA = 68;   // fp32 row stride of A / T
constexpr int LDX = 36;

template <int DK>
struct PrepLay {
    static constexpr int LDK = DK + 8;                   // bf16 row stride of the K tile
    static constexpr int KBYTES = kCp * LDK * 2;
    static constexpr int TBYTES = kCp * LDA * 4;
    // K stays for W = T_w K; once T is final, A's space holds bf16 T_w and
    // T's space holds the bf16 W tile on its way out
    static constexpr int OFF_K = 0;
    static constexpr int OFF_T = KBYTES;                 // fp32 [64][68]
    static constexpr int OFF_A = OFF_T + TBYTES;         // fp32 [64][68]
    static constexpr int OFF_X = OFF_A + TBYTES;         // fp32 [32][36]
    static constexpr int OFF_G = OFF_X + 32 * LDX * 4;   // g, beta, gamma, 1/gamma
    static constexpr int TOTAL = OFF_G + 4 * kCp * 4;
    static_assert(OFF_A % 16 == 0 && OFF_X % 16 == 0, "align");
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

// D += A(16x16, row) * B(16x8, col), bf16 inputs (two per register), fp32 accumulate.
__device__ __forceinline__ void mma_bf16x16(float (&d)[4], const uint32_t (&a)[4],
                                            const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
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

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int DK>
__global__ void __launch_bounds__(128)
k_gdn_prep(const __nv_bfloat16 *__restrict__ k, const float *__restrict__ log_alpha,
           const float *__restrict__ beta, SeqMap sm, const int2 *__restrict__ table,
           int max_chunks, __nv_bfloat16 *__restrict__ Tu_out, __nv_bfloat16 *__restrict__ W_out,
           int *err) {
    using L = PrepLay<DK>;
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_K);
    float *Ab = reinterpret_cast<float *>(smem + L::OFF_A);
    float *Tb = reinterpret_cast<float *>(smem + L::OFF_T);
    float *Xb = reinterpret_cast<float *>(smem + L::OFF_X);
    float *gs = reinterpret_cast<float *>(smem + L::OFF_G);   // g, beta, gamma, 1/gamma

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
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
    const int h = blockIdx.y;
    long long row0;
    int len;
    if (sm.cu) {
        const int a = __ldg(sm.cu + n), b = __ldg(sm.cu + n + 1);
        if (!(a >= 0 && a <= b && b <= sm.T_total)) {
            if (tid == 0) atomicCAS(err, 0, kErrSeqlens);
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
    const int Lc = min(kCp, len - t0);
    const long long r0 = row0 + t0;

    // ---- K tile (rows past the sequence are zero) and gates
    constexpr int VPR = DK / 8;   // 16-byte vectors per row
    for (int i = tid; i < kCp * VPR; i += 128) {
        const int r = i / VPR, q = i % VPR;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < Lc) v = __ldg(reinterpret_cast<const uint4 *>(k + (r0 + r) * DK) + q);
        *reinterpret_cast<uint4 *>(Ks + r * L::LDK + 8 * q) = v;
    }
    if (w == 0) {
        float la0 = lane < Lc ? __ldg(log_alpha + r0 + lane) : 0.f;
        float la1 = lane + 32 < Lc ? __ldg(log_alpha + r0 + lane + 32) : 0.f;
        const float b0 = lane < Lc ? __ldg(beta + r0 + lane) : 0.f;
        const float b1 = lane + 32 < Lc ? __ldg(beta + r0 + lane + 32) : 0.f;
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
        gs[128 + lane] = __expf(la0);
        gs[160 + lane] = __expf(la1);
        gs[192 + lane] = __expf(-la0);
        gs[224 + lane] = __expf(-la1);
    }
    __syncthreads();

    // ---- A = strictly lower (beta_r exp(g_r - g_s) K K^T): warp w owns rows
    //      16w..16w+15 and the column tiles left of its diagonal block's end
    {
        const int g = lane >> 2, t = lane & 3;
        const float gC = gs[63];
        const bool span_ok = gC > -80.f;
        const int ra = 16 * w + g, rb = ra + 8;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            if (nt > 2 * w + 1) break;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k0 = 0; k0 < DK; k0 += 16) {
                uint32_t a[4], b[2];
                a[0] = *reinterpret_cast<const uint32_t *>(Ks + ra * L::LDK + k0 + 2 * t);
                a[1] = *reinterpret_cast<const uint32_t *>(Ks + rb * L::LDK + k0 + 2 * t);
                a[2] = *reinterpret_cast<const uint32_t *>(Ks + ra * L::LDK + k0 + 2 * t + 8);
                a[3] = *reinterpret_cast<const uint32_t *>(Ks + rb * L::LDK + k0 + 2 * t + 8);
                const int nrow = 8 * nt + g;
                b[0] = *reinterpret_cast<const uint32_t *>(Ks + nrow * L::LDK + k0 + 2 * t);
                b[1] = *reinterpret_cast<const uint32_t *>(Ks + nrow * L::LDK + k0 + 2 * t + 8);
                mma_bf16x16(acc, a, b);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = (e < 2) ? ra : rb;
                const int s = 8 * nt + 2 * t + (e & 1);
                float v = 0.f;
                if (s < r) {
                    const float f = span_ok ? gs[128 + r] * gs[192 + s] : __expf(gs[r] - gs[s]);
                    v = gs[64 + r] * f * acc[e];
                }
                Ab[r * LDA + s] = v;
            }
        }
    }
    __syncthreads();

    // ---- T = (I + A)^{-1}
    if (w < 2) {
        // 16x16 diagonal blocks, one column per thread, right-looking
        const int blk = tid >> 4, cc = tid & 15, o = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 16; ++s2) {
#pragma unroll
            for (int r = s2 + 1; r < 16; ++r) x[r] = fmaf(-Ab[(o + r) * LDA + o + s2], x[s2], x[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[(o + r) * LDA + o + cc] = x[r];
    } else {
        // zero the six strictly upper 16x16 blocks
        for (int i = tid - 64; i < 6 * 256; i += 64) {
            const int b = i >> 8, e = i & 255;
            const int bi = b < 3 ? 0 : (b < 5 ? 1 : 2);
            const int bj = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
            Tb[(bi * 16 + (e >> 4)) * LDA + bj * 16 + (e & 15)] = 0.f;
        }
    }
    __syncthreads();
    {
        // 16 -> 32: T_{2p+1,2p} = -D_{2p+1} A_{2p+1,2p} D_{2p}
        const int pr = w >> 1, nh = w & 1;
        const int ro = 32 * pr + 16, co = 32 * pr;
        float *Xw = Xb + w * 16 * 9;
        float c4[4];
        tile_mma<16>(c4, Ab + ro * LDA + co, LDA, Tb + co * LDA + co + 8 * nh, LDA, lane);
        store_tile(Xw, 9, c4, lane, 1.f);
        __syncwarp();
        tile_mma<16>(c4, Tb + ro * LDA + ro, LDA, Xw, 9, lane);
        store_tile(Tb + ro * LDA + co + 8 * nh, LDA, c4, lane, -1.f);
    }
    __syncthreads();
    {
        // 32 -> 64: T_{1,0} = -E1 (A_{1,0} E0), 32x32 blocks
        const int mt = w >> 1, nt0 = 2 * (w & 1);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float c4[4];
            tile_mma<32>(c4, Ab + (32 + 16 * mt) * LDA, LDA, Tb + 8 * (nt0 + q), LDA, lane);
            store_tile(Xb + 16 * mt * LDX + 8 * (nt0 + q), LDX, c4, lane, 1.f);
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float c4[4];
            tile_mma<32>(c4, Tb + (32 + 16 * mt) * LDA + 32, LDA, Xb + 8 * (nt0 + q), LDX, lane);
            store_tile(Tb + (32 + 16 * mt) * LDA + 8 * (nt0 + q), LDA, c4, lane, -1.f);
        }
    }
    __syncthreads();

    // ---- T_u = T diag(beta) rows out (bf16), and T_w = T diag(beta gamma) as
    //      the bf16 A operand of W = T_w K (in A's space, row stride LDK)
    __nv_bfloat16 *Tw = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_A);
    {
        const int r = tid >> 1, hf = tid & 1;
        const float4 *src = reinterpret_cast<const float4 *>(Tb + r * LDA + 32 * hf);
        const float4 *sb = reinterpret_cast<const float4 *>(gs + 64 + 32 * hf);
        const float4 *sg = reinterpret_cast<const float4 *>(gs + 128 + 32 * hf);
        uint32_t u[16], wv[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a = src[2 * q], b = src[2 * q + 1];
            const float4 s0 = sb[2 * q], s1 = sb[2 * q + 1];
            const float4 g0 = sg[2 * q], g1 = sg[2 * q + 1];
            u[4 * q] = pack2(a.x * s0.x, a.y * s0.y);
            u[4 * q + 1] = pack2(a.z * s0.z, a.w * s0.w);
            u[4 * q + 2] = pack2(b.x * s1.x, b.y * s1.y);
            u[4 * q + 3] = pack2(b.z * s1.z, b.w * s1.w);
            wv[4 * q] = pack2(a.x * s0.x * g0.x, a.y * s0.y * g0.y);
            wv[4 * q + 1] = pack2(a.z * s0.z * g0.z, a.w * s0.w * g0.w);
            wv[4 * q + 2] = pack2(b.x * s1.x * g1.x, b.y * s1.y * g1.y);
            wv[4 * q + 3] = pack2(b.z * s1.z * g1.z, b.w * s1.w * g1.w);
        }
        if (r < Lc) {
            uint4 *dst = reinterpret_cast<uint4 *>(Tu_out + (r0 + r) * kCp + 32 * hf);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
        }
        uint4 *tw = reinterpret_cast<uint4 *>(Tw + r * L::LDK + 32 * hf);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            tw[q] = make_uint4(wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
    }
    __syncthreads();
    // ---- W = T_w K (64 x d_k): warp w owns rows 16w..16w+15; bf16 mma.sync,
    //      fp32 accumulation, result staged as bf16 in T's space
    __nv_bfloat16 *Ws = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_T);
    {
        const int g = lane >> 2, t = lane & 3;
        const int ra = 16 * w + g, rb = ra + 8;
        uint32_t af[4][4];
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
            const int k0 = 16 * kq;
            af[kq][0] = *reinterpret_cast<const uint32_t *>(Tw + ra * L::LDK + k0 + 2 * t);
            af[kq][1] = *reinterpret_cast<const uint32_t *>(Tw + rb * L::LDK + k0 + 2 * t);
            af[kq][2] = *reinterpret_cast<const uint32_t *>(Tw + ra * L::LDK + k0 + 2 * t + 8);
            af[kq][3] = *reinterpret_cast<const uint32_t *>(Tw + rb * L::LDK + k0 + 2 * t + 8);
        }
        const unsigned short *Ku = reinterpret_cast<const unsigned short *>(Ks);
#pragma unroll
        for (int nt = 0; nt < DK / 8; ++nt) {
            const int n = 8 * nt + g;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                const int k0 = 16 * kq;
                uint32_t b[2];
                b[0] = (uint32_t)Ku[(k0 + 2 * t) * L::LDK + n] |
                       ((uint32_t)Ku[(k0 + 2 * t + 1) * L::LDK + n] << 16);
                b[1] = (uint32_t)Ku[(k0 + 2 * t + 8) * L::LDK + n] |
                       ((uint32_t)Ku[(k0 + 2 * t + 9) * L::LDK + n] << 16);
                mma_bf16x16(acc, af[kq], b);
            }
            const int col = 8 * nt + 2 * t;
            *reinterpret_cast<uint32_t *>(Ws + ra * L::LDK + col) = pack2(acc[0], acc[1]);
            *reinterpret_cast<uint32_t *>(Ws + rb * L::LDK + col) = pack2(acc[2], acc[3]);
        }
    }
    __syncthreads();
    // ---- W rows of the real tokens out, 16-byte vectors
    for (int i = tid; i < kCp * (DK / 8); i += 128) {
        const int r = i / (DK / 8), q = i % (DK / 8);
        if (r < Lc)
            *reinterpret_cast<uint4 *>(W_out + (r0 + r) * DK + 8 * q) =
                *reinterpret_cast<const uint4 *>(Ws + r * L::LDK + 8 * q);
    }
}

}  // namespace

size_t tc_prep_smem(int dk) {
    return dk == 128 ? (size_t)PrepLay<128>::TOTAL : (size_t)PrepLay<64>::TOTAL;
}

gdn_status enqueue_tc_prep(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                           __nv_bfloat16 *W) {
    if (a.chunk_slots <= 0) return GDN_OK;
    int *err = device_error_word();
    const size_t smem = tc_prep_smem(a.dk);
    dim3 grid(a.chunk_slots, a.sm.H);
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
    if (a.dk == 128) {
        if (cudaFuncSetAttribute(k_gdn_prep<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return GDN_ERR_CUDA;
        k_gdn_prep<128><<<grid, 128, smem, a.stream>>>(k, a.log_alpha, a.beta, a.sm, table,
                                                        a.max_chunks, Tu, W, err);
    } else {
        if (cudaFuncSetAttribute(k_gdn_prep<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return GDN_ERR_CUDA;
        k_gdn_prep<64><<<grid, 128, smem, a.stream>>>(k, a.log_alpha, a.beta, a.sm, table,
                                                       a.max_chunks, Tu, W, err);
    }
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
