// gdn_mma.cuh -- warp-level tf32 tensor-core products for the general path's
// kernels (mma.sync m16n8k8, fp32 operands in shared memory, fp32 accumulate).
//
// A warp computes a 16-row block of an output C (M x N) over NT 8-column
// tiles: C[m0 + 0..15][8 nt + 0..7] += sum_k A(m, k) B(k, n), where A and B
// are element accessors (lambdas over shared memory), so a transposed operand
// is an accessor with its indices swapped.  Fragment layout of m16n8k8 tf32
// (thread lane = 4 g + t): A holds (g, t), (g + 8, t), (g, t + 4),
// (g + 8, t + 4); B holds (t, g), (t + 4, g); the accumulator holds
// (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
//
// The tensor cores read a tf32 operand from the upper 19 bits of an fp32
// register (sign, exponent, 10 mantissa bits), so an fp32 value passed as is
// is truncated to tf32.  SPLIT = true keeps fp32 accuracy with three tf32
// products per step: each operand x is split into hi = x with its low 13
// bits cleared (exact) and lo = x - hi (exact in fp32, truncated to tf32 by
// the hardware), and hi*hi + hi*lo + lo*hi is accumulated -- the "3xTF32"
// emulation of an fp32 product on tf32 tensor cores (the dropped lo*lo term
// and the truncation of lo are about 2^-20 relative).  SPLIT = false takes x
// alone (about 2^-10 relative per operand), which is enough for bf16 outputs.
//
// Shared-memory strides: row-wise operand reads (A(m, k) = S[m * ld + k],
// B(k, n) = S[n * ld + k]) are free of bank conflicts when ld is 4 modulo 8;
// transposed reads then see two-way conflicts.
//
// Row-wise operands also load by ldmatrix: an 8 x 8 matrix of 16-bit
// elements is an 8 x 4 block of fp32 values, which ldmatrix hands out so that
// thread (g, t) holds element (g, t) -- the tf32 fragment layout.  One x4 load
// gives a whole A fragment, or the B fragments of two 8-column tiles, where
// the scalar path takes four loads.
#pragma once
#include <cstdint>

namespace gdn {
namespace mma {

__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                     uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <bool SPLIT>
struct Op {
    uint32_t hi, lo;
    __device__ __forceinline__ explicit Op(float x) {
        if (SPLIT) {
            hi = __float_as_uint(x) & 0xffffe000u;
            lo = __float_as_uint(x - __uint_as_float(hi));
        } else {
            hi = __float_as_uint(x);
            lo = 0u;
        }
    }
};

template <bool SPLIT>
struct AFrag {
    uint32_t hi[4], lo[4];
    template <typename FA>
    __device__ __forceinline__ void load(FA A, int m0, int k0, int g, int t) {
        const float v[4] = {A(m0 + g, k0 + t), A(m0 + g + 8, k0 + t), A(m0 + g, k0 + t + 4),
                            A(m0 + g + 8, k0 + t + 4)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const Op<SPLIT> o(v[i]);
            hi[i] = o.hi;
            lo[i] = o.lo;
        }
    }
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Four 8 x 8 b16 matrices; lanes 8i .. 8i + 7 give the 16-byte row addresses
// of matrix i.
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// A fragment of rows m0 .. m0 + 15, k0 .. k0 + 7 of a row-major fp32 tile:
// `addr` = address of element (m0 + (lane & 15), k0 + 4 (lane >> 4)).
template <bool SPLIT>
__device__ __forceinline__ void lda_ldsm(AFrag<SPLIT> &a, uint32_t addr) {
    uint32_t r[4];
    ldsm4(r, addr);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const Op<SPLIT> o(__uint_as_float(r[i]));
        a.hi[i] = o.hi;
        a.lo[i] = o.lo;
    }
}

// Lane address for the B fragments of the 8-column tiles n0 and n1 of a
// column-wise tile (B(k, n) = S[n * ld + k]) at k0: the x4 load then gives
// (b0, b1) of tile n0 in r[0], r[1] and of tile n1 in r[2], r[3].
__device__ __forceinline__ const float *ldb_pair_ptr(const float *S, int ld, int n0, int n1,
                                                     int k0, int lane) {
    return S + ((lane >> 4 ? n1 : n0) + (lane & 7)) * ld + k0 + 4 * ((lane >> 3) & 1);
}

template <bool SPLIT>
__device__ __forceinline__ void mma_step(float (&d)[4], const AFrag<SPLIT> &a, float b0,
                                         float b1) {
    const Op<SPLIT> x(b0), y(b1);
    mma8(d, a.hi, x.hi, y.hi);
    if (SPLIT) {
        mma8(d, a.hi, x.lo, y.lo);
        mma8(d, a.lo, x.hi, y.hi);
    }
}

// acc[i] covers columns 8 * (nt0 + i * nstep) .. +7 for i < NT while that
// tile starts below n_end; rows m0 .. m0 + 15; k over [0, K) in steps of 8.
template <int NT, bool SPLIT, typename FA, typename FB>
__device__ __forceinline__ void warp_gemm(float (&acc)[NT][4], FA A, FB B, int m0, int nt0,
                                          int nstep, int n_end, int K, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll 1
    for (int k0 = 0; k0 < K; k0 += 8) {
        AFrag<SPLIT> a;
        a.load(A, m0, k0, g, t);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int n = 8 * (nt0 + i * nstep);
            if (n < n_end) mma_step<SPLIT>(acc[i], a, B(k0 + t, n + g), B(k0 + t + 4, n + g));
        }
    }
}

// The same product with strided operands: A(m, k) = pa[m * sam + k * sak]
// (times ascale[k] when ascale is non-null) and B(k, n) = pb[k * sbk + n * sbn],
// k over [kb, K) (both multiples of 8: a triangular operand skips its zero
// blocks); the per-thread element pointers are formed once, the k loop only
// adds.
template <int NT, bool SPLIT>
__device__ __forceinline__ void gemm_s(float (&acc)[NT][4], const float *pa, int sam, int sak,
                                       const float *ascale, const float *pb, int sbk, int sbn,
                                       int m0, int nt0, int nstep, int n_end, int K, int lane,
                                       int kb = 0) {
    const int g = lane >> 2, t = lane & 3;
    if (sak == 1 && sbk == 1 && ((sam | sbn) & 3) == 0 &&
        ((smem_addr(pa) | smem_addr(pb)) & 15) == 0) {
        // rows of A and columns of B contiguous in k, 16-byte aligned: fragments
        // by ldmatrix; B tiles in pairs (the second of an odd count repeats the
        // first, its products skipped)
        constexpr int NP = (NT + 1) / 2;
        const uint32_t a_addr = smem_addr(pa + (m0 + (lane & 15)) * sam + kb + 4 * (lane >> 4));
        uint32_t b_addr[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const int n0 = 8 * (nt0 + 2 * q * nstep), n1 = 8 * (nt0 + (2 * q + 1) * nstep);
            const bool second = 2 * q + 1 < NT && n1 < n_end;
            b_addr[q] = smem_addr(ldb_pair_ptr(pb, sbn, n0, second ? n1 : n0, kb, lane));
        }
#pragma unroll 2
        for (int k0 = kb; k0 < K; k0 += 8) {
            const uint32_t ko = 4u * (uint32_t)(k0 - kb);
            AFrag<SPLIT> a;
            if (ascale) {
                uint32_t r[4];
                ldsm4(r, a_addr + ko);
                const float s0 = ascale[k0 + t], s1 = ascale[k0 + t + 4];
                const float v[4] = {__uint_as_float(r[0]) * s0, __uint_as_float(r[1]) * s0,
                                    __uint_as_float(r[2]) * s1, __uint_as_float(r[3]) * s1};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const Op<SPLIT> o(v[i]);
                    a.hi[i] = o.hi;
                    a.lo[i] = o.lo;
                }
            } else {
                lda_ldsm(a, a_addr + ko);
            }
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const int n0 = 8 * (nt0 + 2 * q * nstep), n1 = 8 * (nt0 + (2 * q + 1) * nstep);
                if (n0 < n_end) {
                    uint32_t b[4];
                    ldsm4(b, b_addr[q] + ko);
                    mma_step<SPLIT>(acc[2 * q], a, __uint_as_float(b[0]), __uint_as_float(b[1]));
                    if (2 * q + 1 < NT && n1 < n_end)
                        mma_step<SPLIT>(acc[2 * q + 1 < NT ? 2 * q + 1 : 2 * q], a,
                                        __uint_as_float(b[2]), __uint_as_float(b[3]));
                }
            }
        }
        return;
    }
    const float *a0 = pa + (m0 + g) * sam + (kb + t) * sak;
    const float *a1 = a0 + 8 * sam;
    const float *bp[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) bp[i] = pb + (kb + t) * sbk + (8 * (nt0 + i * nstep) + g) * sbn;
    const int ak4 = 4 * sak, bk4 = 4 * sbk, ak8 = 8 * sak, bk8 = 8 * sbk;
#pragma unroll 2
    for (int k0 = kb; k0 < K; k0 += 8) {
        float v0 = a0[0], v1 = a1[0], v2 = a0[ak4], v3 = a1[ak4];
        if (ascale) {
            const float s0 = ascale[k0 + t], s1 = ascale[k0 + t + 4];
            v0 *= s0;
            v1 *= s0;
            v2 *= s1;
            v3 *= s1;
        }
        AFrag<SPLIT> a;
        {
            const Op<SPLIT> o0(v0), o1(v1), o2(v2), o3(v3);
            a.hi[0] = o0.hi; a.hi[1] = o1.hi; a.hi[2] = o2.hi; a.hi[3] = o3.hi;
            a.lo[0] = o0.lo; a.lo[1] = o1.lo; a.lo[2] = o2.lo; a.lo[3] = o3.lo;
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            if (8 * (nt0 + i * nstep) < n_end) mma_step<SPLIT>(acc[i], a, bp[i][0], bp[i][bk4]);
            bp[i] += bk8;
        }
        a0 += ak8;
        a1 += ak8;
    }
}

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// Calls f(m, n, value&) for every accumulator element this thread holds.
template <int NT, typename F>
__device__ __forceinline__ void for_each(float (&acc)[NT][4], int m0, int nt0, int nstep,
                                         int n_end, int lane, F f) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        const int n = 8 * (nt0 + i * nstep);
        if (n < n_end) {
#pragma unroll
            for (int e = 0; e < 4; ++e) f(m0 + g + 8 * (e >> 1), n + 2 * t + (e & 1), acc[i][e]);
        }
    }
}

}  // namespace mma
}  // namespace gdn
