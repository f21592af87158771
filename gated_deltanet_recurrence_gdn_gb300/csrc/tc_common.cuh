// tc_common.cuh -- pieces shared by the tcgen05 kernels (gdn_tc.cu,
// gdn_bwd_tc.cu): the bounded-wait control block every role waits through,
// writers of bf16 rows into 128-byte-swizzled operand tiles, and the host
// side's bulk-tensor-copy descriptors.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace tcx {

using namespace ptx;

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
    // Bounded poll of a release/acquire counter until it reaches `target`.
    __device__ __forceinline__ bool flag(const uint32_t *f, uint32_t target) const {
        if (*abort) return false;
        if (flag_wait(f, target, limit)) return true;
        *abort = 1;
        atomicCAS(err, 0, kErrTimeout);
        return false;
    }
    // The same on a global flag that another CTA sets (gpu scope).
    __device__ __forceinline__ bool gflag(const uint32_t *f, uint32_t target) const {
        if (*abort) return false;
        if (gflag_wait(f, target, limit)) return true;
        *abort = 1;
        atomicCAS(err, 0, kErrTimeout);
        return false;
    }
};

// 16-byte store to shared memory
__device__ __forceinline__ void st16(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    if (!GDN_SMEM_OK(smem_u32(p), 16)) return;
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// Writes 8 fp32 values (columns 8*ch .. 8*ch+7 of a 64-wide row) as bf16 into
// chunk `ch` of a 128-byte-swizzled row.
__device__ __forceinline__ void put8(uint8_t *tile, int row, int ch, const float *x) {
    st16(tile + sw128_offset(row, ch), pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
         pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

__device__ __forceinline__ void put_row64(uint8_t *tile, int row, const float (&x)[64]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) put8(tile, row, ch, x + 8 * ch);
}

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// Bulk tensor stores (shared -> global) of a 128-byte-swizzled fp32 tile,
// tracked by this thread's bulk groups.  The tile's writers make it visible
// to the async proxy (fence.proxy.async) before the storing thread issues.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x,
                                             int y) {
    if (!GDN_SMEM_OK(smem_u32(src), 8192)) return;   // the box's first 8 KiB
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::
                     "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x,
                                             int y, int z) {
    if (!GDN_SMEM_OK(smem_u32(src), 8192)) return;
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until every committed store has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Until every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Row `row` of a 64-column fp32 tile staged for bulk stores: two 32-column
// halves, each `rows` rows of 128 bytes, 128-byte swizzled.
__device__ __forceinline__ void put_row64_f32(uint8_t *tile, int rows, int row,
                                              const float (&x)[64]) {
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        float4 *d = reinterpret_cast<float4 *>(tile + (q >> 3) * rows * 128 +
                                               sw128_offset(row, q & 7));
        if (!GDN_SMEM_OK(smem_u32(d), 16)) continue;
        *d = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
}

// -------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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
inline bool make_map(CUtensorMap *m, const void *base, int d, long long ydim, long long zdim) {
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

// Views of an fp32 row-major tensor with rows of `d` elements for bulk tensor
// stores of 32-column, 128-byte-swizzled boxes: 2-D [ydim][d] with boxes of
// `box_rows` rows, or 3-D [zdim][ydim][d] with boxes of 64 rows.
inline bool make_map_f32(CUtensorMap *m, const void *base, int d, long long ydim, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)ydim};
    cuuint64_t strides[1] = {(cuuint64_t)d * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}
inline bool make_map_f32_3d(CUtensorMap *m, const void *base, int d, long long ydim,
                            long long zdim) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)ydim, (cuuint64_t)zdim};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)d * 4 * (cuuint64_t)ydim};
    cuuint32_t box[3] = {32, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

inline bool device_is_sm10x() {
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return false;
    return major == 10;
}

}  // namespace tcx
}  // namespace gdn
