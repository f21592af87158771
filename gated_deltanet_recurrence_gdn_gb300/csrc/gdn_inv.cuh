// gdn_inv.cuh -- the unit-lower-triangular inverse T = (I + A)^{-1} of one
// chunk's 64 x 64 block, shared by the chunk-prep kernels (gdn_prep.cu,
// gdn_ut.cu).
//
// A is strictly lower triangular (A_rs = beta_r exp(g_r - g_s) k_r . k_s for
// s < r inside a chunk of 64 tokens, "Gated DeltaNet GPU并行实现", section 3.2),
// so I + A is unit lower triangular and so is its inverse.  The four 16 x 16
// diagonal blocks are solved by forward substitution in fp32, one column per
// thread; the off-diagonal blocks follow from T_10 = -T_11 A_10 T_00, merging
// 16 -> 32 -> 64 with tf32 mma.sync products (every fp32 matrix they read holds
// tf32-rounded values, so the products read it without conversion).
#pragma once
#include <cstdint>

#include "gdn_check.cuh"

namespace gdn {
namespace inv {

constexpr int LDA = 68;   // fp32 row stride of A and T (4 mod 8: conflict-free fragments)

__device__ __forceinline__ float tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// D += A(16x8, row) * B(8x8, col), tf32 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const float (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(__float_as_uint(b[0])),
          "r"(__float_as_uint(b[1])));
}

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Four 8x8 b16 matrices from shared memory (lanes 8i..8i+7 give the row
// addresses of matrix i).
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// One 16x8 output tile of  Y = Am * Bm  over the 8-wide k steps [kb, ke),
// operands tf32 values stored as fp32 in smem (row-major, strides lda / ldb;
// Am 16-byte aligned with lda a multiple of 4).  The A fragment of a k step is
// one ldmatrix: its 8x8 b16 matrices are 8x4 fp32 blocks, which hand thread
// (g, t) element (g, t) -- the tf32 fragment layout.
template <int K>
__device__ __forceinline__ void tile_mma(float (&c)[4], const float *Am, int lda, const float *Bm,
                                         int ldb, int lane, int kb = 0, int ke = K / 8) {
    const int g = lane >> 2, t = lane & 3;
    c[0] = c[1] = c[2] = c[3] = 0.f;
    const uint32_t a_addr = saddr(Am + (lane & 15) * lda + 4 * (lane >> 4));
#pragma unroll
    for (int ks = 0; ks < K / 8; ++ks) {
        if (ks < kb || ks >= ke) continue;
        const int k0 = 8 * ks;
        uint32_t a[4];
        ldsm4(a, a_addr + 4 * k0);
        const float b[2] = {Bm[(k0 + t) * ldb + g], Bm[(k0 + t + 4) * ldb + g]};
        mma_tf32(c, a, b);
    }
}

// Stores scale * C rounded to tf32.
__device__ __forceinline__ void store_tile(float *D, int ldd, const float (&c)[4], int lane,
                                           float scale) {
    const int g = lane >> 2, t = lane & 3;
    if (GDN_SMEM_OK(saddr(D + g * ldd + 2 * t), 8))
        *reinterpret_cast<float2 *>(D + g * ldd + 2 * t) =
            make_float2(tf32(scale * c[0]), tf32(scale * c[1]));
    if (GDN_SMEM_OK(saddr(D + (g + 8) * ldd + 2 * t), 8))
        *reinterpret_cast<float2 *>(D + (g + 8) * ldd + 2 * t) =
            make_float2(tf32(scale * c[2]), tf32(scale * c[3]));
}

// Zeroes the upper 16x16 blocks inside T's two diagonal 32x32 blocks (the
// merges read those blocks whole).  Any number of threads: thread i of n.
__device__ __forceinline__ void clear_upper16(float *Tb, int i, int n) {
    for (int e = i; e < 2 * 256; e += n) {
        const int b = e >> 8, x = e & 255;
        float *d = Tb + (32 * b + (x >> 4)) * LDA + 32 * b + 16 + (x & 15);
        if (GDN_SMEM_OK(saddr(d), 4)) *d = 0.f;
    }
}

// T = (I + A)^{-1}, computed by 128 threads (tid 0..127, four whole warps).
// On entry: Ab holds A (strictly lower; entries outside the 16x16 diagonal
// blocks rounded to tf32, the upper triangle ignored), and clear_upper16(Tb)
// has run.  On exit Tb holds T's lower triangle (unit diagonal); its
// upper-right 32x32 block (rows 0-31, columns 32-63) holds scratch and is not
// part of T.  `bar` is a barrier over the 128 threads.
template <typename Bar>
__device__ __forceinline__ void invert64(const float *Ab, float *Tb, int tid, Bar bar) {
    const int w = tid >> 5, lane = tid & 31;
    if (w < 2) {
        // 16x16 diagonal blocks, one column cc per thread: row by row,
        // x_r = delta_{r,cc} - sum_{s<r} A_rs x_s, A's rows read as float4 broadcasts
        const int blk = tid >> 4, cc = tid & 15, o = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float4 *row = reinterpret_cast<const float4 *>(Ab + (o + r) * LDA + o);
            float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
            for (int q = 0; 4 * q < r; ++q) {
                const float4 a4 = row[q];
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q + e < r) acc = fmaf(-av[e], x[4 * q + e], acc);
            }
            x[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (GDN_SMEM_OK(saddr(Tb + (o + r) * LDA + o + cc), 4))
                Tb[(o + r) * LDA + o + cc] = tf32(x[r]);
    }
    bar();
    {
        // 16 -> 32: T_{2p+1,2p} = -D_{2p+1} A_{2p+1,2p} D_{2p}  (D_{2p} is lower
        // triangular: its columns 8-15 have zero rows 0-7)
        const int pr = w >> 1, nh = w & 1;
        const int ro = 32 * pr + 16, co = 32 * pr;
        float *Xw = Tb + (16 * pr) * LDA + 32 + 8 * nh;
        float c4[4];
        tile_mma<16>(c4, Ab + ro * LDA + co, LDA, Tb + co * LDA + co + 8 * nh, LDA, lane, nh);
        store_tile(Xw, LDA, c4, lane, 1.f);
        __syncwarp();
        tile_mma<16>(c4, Tb + ro * LDA + ro, LDA, Xw, LDA, lane);
        store_tile(Tb + ro * LDA + co + 8 * nh, LDA, c4, lane, -1.f);
    }
    bar();
    {
        // 32 -> 64: T_{1,0} = -E1 (A_{1,0} E0), 32x32 blocks; E0 and E1 are lower
        // triangular, so k steps of zero operand rows or columns are skipped
        float *Xb = Tb + 32;
        const int mt = w >> 1, nt0 = 2 * (w & 1);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float c4[4];
            tile_mma<32>(c4, Ab + (32 + 16 * mt) * LDA, LDA, Tb + 8 * (nt0 + q), LDA, lane,
                         nt0 + q);
            store_tile(Xb + 16 * mt * LDA + 8 * (nt0 + q), LDA, c4, lane, 1.f);
        }
        bar();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float c4[4];
            tile_mma<32>(c4, Tb + (32 + 16 * mt) * LDA + 32, LDA, Xb + 8 * (nt0 + q), LDA, lane,
                         0, 2 + 2 * mt);
            store_tile(Tb + (32 + 16 * mt) * LDA + 8 * (nt0 + q), LDA, c4, lane, -1.f);
        }
    }
    bar();
}

// T = (I + A)^{-1} in place: on entry AT holds A with every row written in
// full (zeros on and above the diagonal, entries outside the 16x16 diagonal
// blocks rounded to tf32); on exit it holds T's lower triangle, and its
// upper-right 32x32 block (rows 0-31, columns 32-63: zeros of A) holds the
// merges' scratch, as invert64 leaves it.  Each step overwrites only entries
// of A that no later step reads: a diagonal block's 16 threads (one warp)
// sync before writing T over it, and the 16 -> 32 merge completes every
// X = A_10 T_00 before any T_10 = -T_11 X lands on A_10.
template <typename Bar>
__device__ __forceinline__ void invert64_inplace(float *AT, int tid, Bar bar) {
    const int w = tid >> 5, lane = tid & 31;
    if (w < 2) {
        const int blk = tid >> 4, cc = tid & 15, o = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float4 *row = reinterpret_cast<const float4 *>(AT + (o + r) * LDA + o);
            float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
            for (int q = 0; 4 * q < r; ++q) {
                const float4 a4 = row[q];
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q + e < r) acc = fmaf(-av[e], x[4 * q + e], acc);
            }
            x[r] = acc;
        }
        __syncwarp();   // the block's 16 threads (this warp) have read it
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (GDN_SMEM_OK(saddr(AT + (o + r) * LDA + o + cc), 4))
                AT[(o + r) * LDA + o + cc] = tf32(x[r]);
    }
    bar();
    {
        const int pr = w >> 1, nh = w & 1;
        const int ro = 32 * pr + 16, co = 32 * pr;
        float *Xw = AT + (16 * pr) * LDA + 32 + 8 * nh;
        float c4[4];
        tile_mma<16>(c4, AT + ro * LDA + co, LDA, AT + co * LDA + co + 8 * nh, LDA, lane, nh);
        store_tile(Xw, LDA, c4, lane, 1.f);
        bar();   // both halves of X read all of A_10
        tile_mma<16>(c4, AT + ro * LDA + ro, LDA, Xw, LDA, lane);
        store_tile(AT + ro * LDA + co + 8 * nh, LDA, c4, lane, -1.f);
    }
    bar();
    {
        float *Xb = AT + 32;
        const int mt = w >> 1, nt0 = 2 * (w & 1);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float c4[4];
            tile_mma<32>(c4, AT + (32 + 16 * mt) * LDA, LDA, AT + 8 * (nt0 + q), LDA, lane,
                         nt0 + q);
            store_tile(Xb + 16 * mt * LDA + 8 * (nt0 + q), LDA, c4, lane, 1.f);
        }
        bar();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float c4[4];
            tile_mma<32>(c4, AT + (32 + 16 * mt) * LDA + 32, LDA, Xb + 8 * (nt0 + q), LDA, lane,
                         0, 2 + 2 * mt);
            store_tile(AT + (32 + 16 * mt) * LDA + 8 * (nt0 + q), LDA, c4, lane, -1.f);
        }
    }
    bar();
}

// Element (r, s) of T from the buffer invert64 leaves (zero above the diagonal
// and in the scratch block).
__device__ __forceinline__ float t_at(const float *Tb, int r, int s) {
    return (s > r || (r < 32 && s >= 32)) ? 0.f : Tb[r * LDA + s];
}

}  // namespace inv
}  // namespace gdn
