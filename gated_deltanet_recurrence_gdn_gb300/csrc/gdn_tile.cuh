// gdn_tile.cuh -- register-staged loads of 64-row chunk tiles for the general
// path's kernels.
//
// A chunk tile is 64 rows of `width` consecutive elements (width a multiple
// of 8) at a row stride of `stride` elements.  A block of 256 threads loads it
// in 8-element groups (two 16-byte loads of fp32, one of bf16): thread tid
// takes groups tid, tid + 256, ...  load() only issues the global loads into
// registers, so a serial chunk loop can start the next chunk's loads before
// it computes the current one and store() them into shared memory (fp32, row
// stride ld, a multiple of 4) when it gets there.  Rows at or past `rows` and
// columns at or past `cols` are zero.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

namespace gdn {

__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int MAXG>   // groups per thread: 64 * width / 8 / 256 <= MAXG
struct TileRegs {
    float v[MAXG][8];

    // cols: columns present in memory (a multiple of 8, at most width); the
    // rest of each row is zero
    template <typename T>
    __device__ __forceinline__ void load(const T *base, long long stride, int width, int rows,
                                         int cols, int tid) {
        const int gpr = width >> 3;   // groups per row
#pragma unroll
        for (int m = 0; m < MAXG; ++m) {
            const int i = tid + 256 * m;
            const int r = i / gpr, c8 = i - r * gpr;
            if (r < 64 && r < rows && 8 * c8 < cols) {
                load8(base + r * stride + 8 * c8, v[m]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[m][e] = 0.f;
            }
        }
    }

    // nrows: rows the destination holds (rows past it are not written)
    __device__ __forceinline__ void store(float *s, int ld, int width, int tid,
                                          int nrows = 64) const {
        const int gpr = width >> 3;
#pragma unroll
        for (int m = 0; m < MAXG; ++m) {
            const int i = tid + 256 * m;
            const int r = i / gpr, c8 = i - r * gpr;
            if (r < 64 && r < nrows) {
                float4 *d = reinterpret_cast<float4 *>(s + r * ld + 8 * c8);
                d[0] = make_float4(v[m][0], v[m][1], v[m][2], v[m][3]);
                d[1] = make_float4(v[m][4], v[m][5], v[m][6], v[m][7]);
            }
        }
    }
};

}  // namespace gdn
