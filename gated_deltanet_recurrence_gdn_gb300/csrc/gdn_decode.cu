// gdn_decode.cu -- one decode step of the gated delta rule for a batch of
// (sequence, head) states ("Gated DeltaNet GPU并行实现", sections 2.1-2.2).
//
// With the old state S (d_v x d_k, fp32) and the token's q, k, v, alpha, beta:
//
//   S (I - beta k k^T) alpha + beta v k^T  =  alpha S + d k^T,
//   d = beta (v - alpha S k),   o = (alpha S + d k^T) q = alpha S q + d (k . q).
//
// Row i of the new state needs only row i of the old one (through (S k)_i
// and (S q)_i), so one warp streams a row in, reduces its two dot products
// across the lanes, and streams the updated row out: one read and one write
// of the state, with no scratch.  Rows are taken four at a time per warp so
// that four loads are in flight before the first reduction.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kDecWarps = 8;
constexpr int kDecRows = 4;   // rows in flight per warp

// VEC consecutive elements starting at p (VEC * sizeof(element) bytes aligned).
template <int VEC>
__device__ __forceinline__ void load_vec(const float *p, float (&r)[VEC]) {
    if constexpr (VEC == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        r[0] = t.x; r[1] = t.y; r[2] = t.z; r[3] = t.w;
    } else if constexpr (VEC == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        r[0] = t.x; r[1] = t.y;
    } else {
        r[0] = *p;
    }
}
template <int VEC>
__device__ __forceinline__ void load_vec(const __nv_bfloat16 *p, float (&r)[VEC]) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) r[e] = __bfloat162float(p[e]);
}
// State rows: streamed once, so read and write with evict-first hints.
template <int VEC>
__device__ __forceinline__ void load_row(const float *p, float (&r)[VEC]) {
    if constexpr (VEC == 4) {
        const float4 t = __ldcs(reinterpret_cast<const float4 *>(p));
        r[0] = t.x; r[1] = t.y; r[2] = t.z; r[3] = t.w;
    } else if constexpr (VEC == 2) {
        const float2 t = __ldcs(reinterpret_cast<const float2 *>(p));
        r[0] = t.x; r[1] = t.y;
    } else {
        r[0] = __ldcs(p);
    }
}
template <int VEC>
__device__ __forceinline__ void store_row(float *p, const float (&r)[VEC]) {
    if constexpr (VEC == 4)
        __stcs(reinterpret_cast<float4 *>(p), make_float4(r[0], r[1], r[2], r[3]));
    else if constexpr (VEC == 2)
        __stcs(reinterpret_cast<float2 *>(p), make_float2(r[0], r[1]));
    else
        __stcs(p, r[0]);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void put(float *p, float x) { *p = x; }
__device__ __forceinline__ void put(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// One CTA per (sequence, head); warp w takes rows w, w + 8, ... of its state.
template <int VEC, typename TIn>
__global__ void __launch_bounds__(kDecWarps * 32)
k_gdn_decode(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
             const float *__restrict__ log_alpha, const float *__restrict__ beta,
             float *__restrict__ state, const int32_t *__restrict__ slots, int n_slots,
             TIn *__restrict__ o, int H, int dv, int *err) {
    constexpr int DK = 32 * VEC;
    const int bh = blockIdx.x, b = bh / H, h = bh - b * H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long sidx = b;
    if (slots) {
        const int s = __ldg(slots + b);
        if (s < 0 || s >= n_slots) {
            if (threadIdx.x == 0) atomicCAS(err, 0, kErrBadIndex);
            return;
        }
        sidx = s;
    }
    float kr[VEC], qr[VEC];
    load_vec<VEC>(k + (long long)bh * DK + VEC * lane, kr);
    load_vec<VEC>(q + (long long)bh * DK + VEC * lane, qr);
    float kq = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) kq = fmaf(kr[e], qr[e], kq);
    kq = warp_sum(kq);
    const float alpha = __expf(__ldg(log_alpha + bh)), bet = __ldg(beta + bh);
    float *S = state + (sidx * H + h) * (long long)dv * DK + VEC * lane;
    const TIn *vrow = v + (long long)bh * dv;
    TIn *orow = o + (long long)bh * dv;

    for (int r0 = warp * kDecRows; r0 < dv; r0 += kDecWarps * kDecRows) {
        float s[kDecRows][VEC];
#pragma unroll
        for (int i = 0; i < kDecRows; ++i)
            if (r0 + i < dv) load_row<VEC>(S + (long long)(r0 + i) * DK, s[i]);
        float sk[kDecRows], sq[kDecRows];
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            sk[i] = 0.f;
            sq[i] = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                sk[i] = fmaf(s[i][e], kr[e], sk[i]);
                sq[i] = fmaf(s[i][e], qr[e], sq[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            sk[i] = warp_sum(sk[i]);
            sq[i] = warp_sum(sq[i]);
        }
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            const int r = r0 + i;
            if (r < dv) {
                const float d = bet * (to_f(vrow[r]) - alpha * sk[i]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) s[i][e] = fmaf(alpha, s[i][e], d * kr[e]);
                store_row<VEC>(S + (long long)r * DK, s[i]);
                if (lane == 0) put(orow + r, fmaf(alpha, sq[i], d * kq));
            }
        }
    }
}

template <int VEC, typename TIn>
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *la,
                          const float *beta, float *state, const int32_t *slots, int n_slots,
                          void *o, int B, int H, int dv, cudaStream_t st) {
    const TIn *qi = static_cast<const TIn *>(q);
    const TIn *ki = static_cast<const TIn *>(k);
    const TIn *vi = static_cast<const TIn *>(v);
    const int slot = timer_begin(st, "k_gdn_decode");
    k_gdn_decode<VEC, TIn><<<B * H, kDecWarps * 32, 0, st>>>(
        qi, ki, vi, la, beta, state, slots, n_slots, static_cast<TIn *>(o), H, dv,
        device_error_word());
    timer_end(slot, st);
    count_launch();
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t decode_dispatch(int dk, const void *q, const void *k, const void *v, const float *la,
                            const float *beta, float *state, const int32_t *slots, int n_slots,
                            void *o, int B, int H, int dv, cudaStream_t st) {
    switch (dk) {
        case 32: return launch_decode<1, TIn>(q, k, v, la, beta, state, slots, n_slots, o, B, H, dv, st);
        case 64: return launch_decode<2, TIn>(q, k, v, la, beta, state, slots, n_slots, o, B, H, dv, st);
        default: return launch_decode<4, TIn>(q, k, v, la, beta, state, slots, n_slots, o, B, H, dv, st);
    }
}

bool aligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_decode(const void *q, const void *k, const void *v,
                                 const float *log_alpha, const float *beta, float *state,
                                 const int32_t *slots, int n_slots, void *o, int B, int H,
                                 int d_k, int d_v, gdn_dtype dt, void *stream) {
    using namespace gdn;
    if (B < 0 || H < 0 || d_v < 1) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (d_k != 32 && d_k != 64 && d_k != 128) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    if (slots && n_slots < 1) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (!q || !k || !v || !log_alpha || !beta || !state || !o) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, log_alpha, beta, state, slots, o};
    for (const void *p : ptrs)
        if (p && !aligned(p)) return GDN_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        dt == GDN_BF16
            ? decode_dispatch<__nv_bfloat16>(d_k, q, k, v, log_alpha, beta, state, slots, n_slots,
                                             o, B, H, d_v, st)
            : decode_dispatch<float>(d_k, q, k, v, log_alpha, beta, state, slots, n_slots, o, B,
                                     H, d_v, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
