// gdn_mma.cuh -- warp-level tf32 tensor-core products for the CUDA-core
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
// SPLIT = true keeps fp32 accuracy with three tf32 products per step: each
// operand is split into its tf32 rounding hi and the tf32 rounding of the
// remainder lo, and hi*hi + hi*lo + lo*hi is accumulated (the lo*lo term,
// about 2^-22 relative, is dropped) -- the "3xTF32" emulation of an fp32
// product on tf32 tensor cores.  SPLIT = false takes hi*hi alone (about
// 2^-11 relative per product), which is enough for bf16 outputs.
//
// Shared-memory strides: row-wise operand reads (A(m, k) = S[m * ld + k],
// B(k, n) = S[n * ld + k]) are free of bank conflicts when ld is 4 modulo 8;
// transposed reads then see two-way conflicts.
#pragma once
#include <cstdint>

namespace gdn {
namespace mma {

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

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
        const float h = to_tf32(x);
        hi = __float_as_uint(h);
        lo = SPLIT ? __float_as_uint(to_tf32(x - h)) : 0u;
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
