// gdn_simt.cu -- the general path: fp32 I/O, widths the tcgen05 kernels do
// not cover, the allocation-free entry point, gates per key dimension, and
// the backward pass's recomputation.
//
// It follows the chunked method of "Gated DeltaNet GPU并行实现" section 3.2:
// inside a chunk everything is a small dense product, across chunks a serial
// pass carries the state.  The products run on the tensor cores as warp-level
// tf32 mma.sync (gdn_mma.cuh; three products per step, the 3xTF32 split, for
// fp32 I/O).  Two kernels per gate kind:
//
//   prep  (one CTA per (chunk, head), all chunks in parallel):
//         g_r   = sum_{i<=r} log_alpha_i inside the chunk        (gate cumsum)
//         A_rs  = beta_r exp(g_r - g_s) (k_r . k_s),  s < r        (decayed Gram)
//         T     = (I + A)^{-1}  (16 x 16 blocks, then merged)
//         W     = T diag(beta exp(g)) K,   U = T diag(beta) V       (WY factors)
//   state (one CTA per (sequence, head, 64-wide d_v tile), chunks in order):
//         with H = S^T (d_k x d_v) at the chunk start,
//         V'    = U - W H
//         O     = diag(exp(g)) Q H + [mask_{s<=r} exp(g_r - g_s) Q K^T] V'
//         H    <- exp(g_C) H + K^T diag(exp(g_C - g_r)) V'
//
// Derivation (the affine form of section 2.2 unrolled over one chunk): with
// u_r = beta_r (v_r - alpha_r S_{r-1} k_r) the update is S_r = alpha_r S_{r-1}
// + u_r k_r^T, so S_r = gamma_r S_0 + sum_{s<=r} (gamma_r/gamma_s) u_s k_s^T
// (gamma = exp(g)).  Substituting into u_r gives (I + A) U' = diag(beta) V -
// diag(beta gamma) K S_0^T, i.e. U' = U - W S_0^T; the chunk-end state and the
// outputs follow by summing the same expansion.
//
// Rows past the end of a sequence are padding with k = v = q = 0, beta = 0
// and log_alpha = 0, which leaves every real row unchanged.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "gdn_bwd_tc.h"
#include "gdn_internal.h"
#include "gdn_mma.cuh"
#include "gdn_tile.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;

// Two adjacent outputs (columns c, c + 1 of a row, c even) in one store.
__device__ __forceinline__ void st_out2(float *p, float x, float y) {
    *reinterpret_cast<float2 *>(p) = make_float2(x, y);
}
__device__ __forceinline__ void st_out2(__nv_bfloat16 *p, float x, float y) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x, y);
}

// The accumulator block's column pairs (2t, 2t + 1 of each 8-column tile
// below n_end) into rows r < L of dst (row stride ld), one store a pair.
template <int NT, typename T>
__device__ __forceinline__ void store_pairs(const float (&acc)[NT][4], int m0, int nt0, int nstep,
                                            int n_end, int lane, int L, T *dst, long long ld) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        const int n = 8 * (nt0 + i * nstep);
        if (n < n_end) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = m0 + g + 8 * hr;
                if (r < L) st_out2(dst + r * ld + n + 2 * t, acc[i][2 * hr], acc[i][2 * hr + 1]);
            }
        }
    }
}

__device__ __forceinline__ void set_error(int *err, int code) { atomicCAS(err, 0, code); }

// Validates one packed sequence's range; dense maps are valid by construction.
__device__ __forceinline__ bool seq_ok(const SeqMap &sm, int n) {
    if (!sm.cu) return true;
    int a = __ldg(sm.cu + n), b = __ldg(sm.cu + n + 1);
    return a >= 0 && a <= b && b <= sm.T_total;
}

// One block lists every (sequence, chunk) pair of a packed batch; unused
// slots get n = -1.  Also validates cu_seqlens.
__global__ void k_chunk_table(const int32_t *cu, int N, int T_total, int2 *table, int slots,
                              int *err) {
    __shared__ int s_scan[1024];
    __shared__ int s_base;
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_base = 0;
        s_bad = (__ldg(cu) != 0 || __ldg(cu + N) != T_total) ? 1 : 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int cnt = 0;
        if (n < N) {
            int a = __ldg(cu + n), b = __ldg(cu + n + 1);
            if (b < a || a < 0 || b > T_total) atomicExch(&s_bad, 1);
            else cnt = (b - a + kChunk - 1) / kChunk;
        }
        s_scan[tid] = cnt;
        __syncthreads();
        for (int off = 1; off < 1024; off <<= 1) {  // inclusive Hillis-Steele scan
            int x = tid >= off ? s_scan[tid - off] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        const int start = s_base + s_scan[tid] - cnt;
        for (int c = 0; c < cnt; ++c)
            if (start + c < slots) table[start + c] = make_int2(n, c);
        __syncthreads();
        if (tid == 1023) s_base += s_scan[1023];
        __syncthreads();
    }
    const int used = s_bad ? 0 : min(s_base, slots);
    for (int i = used + tid; i < slots; i += 1024) table[i] = make_int2(-1, -1);
    if (tid == 0 && s_bad) set_error(err, kErrBadIndex);
}

// The state pass for a scalar gate with its products on the tensor cores
// (mma.sync tf32, gdn_mma.cuh: three products per step for fp32 I/O, one for
// bf16 I/O).  One CTA per (sequence, head, 64-wide d_v tile); the next
// chunk's K, W, Q and U are loaded into registers while the current chunk is
// computed.  P and O are skipped when no output is wanted (the backward
// pass's recomputation).
constexpr int kDvm = 64;           // d_v columns per CTA
constexpr int kLdh = kDvm + 8;     // d_k x 64 state tile: transposed reads conflict-free
constexpr int kLdc = kChunk + 4;   // 64 x 64 tiles

size_t state_mma_smem(int dk, bool out) {
    const size_t ldk = dk + 4;
    return sizeof(float) * ((size_t)dk * kLdh + 2 * kChunk * ldk + 2 * kChunk * kLdc +
                            3 * kChunk + (out ? kChunk * ldk + kChunk * kLdc : 0));
}

template <typename TIn, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
k_state_mma(FwdArgs a, const float *__restrict__ W, const float *__restrict__ U,
            const float *__restrict__ G, float *__restrict__ Hst, float *__restrict__ Vout,
            int *err) {
    extern __shared__ float smem[];
    const int dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int n = blockIdx.x, h = blockIdx.y, dv0 = blockIdx.z * kDvm;
    const int nv = min(kDvm, dv - dv0);
    if (!seq_ok(a.sm, n)) {
        if (tid == 0) set_error(err, kErrBadIndex);
        return;
    }
    long long row0;
    int len;
    a.sm.get(n, h, row0, len);
    const int ldk = dk + 4;
    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    TIn *op = static_cast<TIn *>(a.o);
    float *Hs = smem;                    // [dk][72]   H = S^T tile
    float *Ks = Hs + dk * kLdh;          // [64][dk+4]
    float *Ws = Ks + kChunk * ldk;       // [64][dk+4]
    float *Us = Ws + kChunk * ldk;       // [64][68]
    float *Vn = Us + kChunk * kLdc;      // [64][68]
    float *g = Vn + kChunk * kLdc;       // [64]
    float *e = g + kChunk;               // [64] exp(g_C - g_r)
    float *gm = e + kChunk;              // [64] exp(g_r)
    float *Qs = gm + kChunk;             // [64][dk+4]  (with an output only)
    float *P = Qs + kChunk * ldk;        // [64][68]    (with an output only)
    const long long sbase = ((long long)n * a.sm.H + h) * dv;
    const int m0 = 16 * (warp >> 1), nh = warp & 1;
    const int ntask = 2 * ((dk + 15) / 16);

    for (int i = tid; i < dk * kDvm; i += kThreads) {
        const int j = i / kDvm, cc = i - j * kDvm;
        Hs[j * kLdh + cc] = (a.h0 && cc < nv) ? __ldg(a.h0 + (sbase + dv0 + cc) * dk + j) : 0.f;
    }
    TileRegs<4> rk, rw, rq;
    TileRegs<2> ru;
    float gnext = 0.f;
    auto issue = [&](int c) {
        const int L = min(kChunk, len - c * kChunk);
        const long long r0 = row0 + (long long)c * kChunk;
        rk.load(kp + r0 * dk, dk, dk, L, dk, tid);
        rw.load(W + r0 * dk, dk, dk, L, dk, tid);
        if (op) rq.load(qp + r0 * dk, dk, dk, L, dk, tid);
        ru.load(U + r0 * dv + dv0, dv, kDvm, L, nv, tid);
        if (tid < kChunk) gnext = __ldg(G + r0 + min(tid, L - 1));
    };
    const int nch = (len + kChunk - 1) / kChunk;
    if (nch > 0) issue(0);
    for (int c = 0; c < nch; ++c) {
        const int t0 = c * kChunk, L = min(kChunk, len - t0);
        const long long r0 = row0 + t0;
        __syncthreads();  // previous chunk fully consumed
        if (Hst) {
            float *dst = Hst + ((long long)h * a.chunk_slots + a.chunk_slot(n, c)) * dk * dv;
            for (int i = tid; i < dk * kDvm; i += kThreads) {
                const int j = i / kDvm, cc = i - j * kDvm;
                if (cc < nv) dst[(long long)j * dv + dv0 + cc] = Hs[j * kLdh + cc];
            }
        }
        rk.store(Ks, ldk, dk, tid);
        rw.store(Ws, ldk, dk, tid);
        if (op) rq.store(Qs, ldk, dk, tid);
        ru.store(Us, kLdc, kDvm, tid);
        if (tid < kChunk) g[tid] = gnext;
        if (c + 1 < nch) issue(c + 1);
        __syncthreads();
        const float gl = g[kChunk - 1];
        if (tid < kChunk) {
            e[tid] = expf(gl - g[tid]);
            gm[tid] = expf(g[tid]);
        }
        if (op) {   // P_rs = G_rs q_r . k_s, s <= r
            float acc[4][4];
            mma::zero(acc);
            // tiles right of this warp's diagonal block are masked: not formed
            mma::gemm_s<4, SPLIT>(acc, Qs, ldk, 1, nullptr, Ks, 1, ldk, m0, nh, 2, m0 + 16, dk,
                                  lane);
            mma::for_each(acc, m0, nh, 2, m0 + 16, lane, [&](int r, int s, float &x) {
                P[r * kLdc + s] = s <= r ? expf(g[r] - g[s]) * x : 0.f;
            });
        }
        {   // V' = U - W H
            float acc[4][4];
            mma::zero(acc);
            mma::gemm_s<4, SPLIT>(acc, Ws, ldk, 1, nullptr, Hs, kLdh, 1, m0, nh, 2, kDvm, dk,
                                  lane);
            mma::for_each(acc, m0, nh, 2, kDvm, lane, [&](int r, int cc, float &x) {
                const float val = Us[r * kLdc + cc] - x;
                Vn[r * kLdc + cc] = val;
                if (Vout && r < L && cc < nv) Vout[(r0 + r) * dv + dv0 + cc] = val;
            });
        }
        __syncthreads();
        if (op) {   // O = diag(gamma) Q H + P V'
            float a1[4][4], a2[4][4];
            mma::zero(a1);
            mma::zero(a2);
            mma::gemm_s<4, SPLIT>(a1, Qs, ldk, 1, nullptr, Hs, kLdh, 1, m0, nh, 2, kDvm, dk,
                                  lane);
            mma::gemm_s<4, SPLIT>(a2, P, kLdc, 1, nullptr, Vn, kLdc, 1, m0, nh, 2, kDvm, m0 + 16,
                                  lane);
            const int gq = lane >> 2;   // accumulator rows m0 + gq and m0 + gq + 8
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    a1[i][q] = fmaf(gm[m0 + gq + 8 * (q >> 1)], a1[i][q], a2[i][q]);
            store_pairs(a1, m0, nh, 2, nv, lane, L, op + r0 * dv + dv0, dv);
            __syncthreads();  // every read of H for this chunk is done
        }
        // H <- exp(g_C) H + K^T diag(exp(g_C - g)) V'
        const float decay = expf(gl);
        for (int task = warp; task < ntask; task += kThreads / 32) {
            const int j0 = 16 * (task >> 1), th = task & 1;
            float acc[4][4];
            mma::zero(acc);
            mma::gemm_s<4, SPLIT>(acc, Ks, 1, ldk, e, Vn, kLdc, 1, j0, th, 2, kDvm, kChunk,
                                  lane);
            mma::for_each(acc, j0, th, 2, kDvm, lane, [&](int j, int cc, float &x) {
                if (j < dk) Hs[j * kLdh + cc] = fmaf(decay, Hs[j * kLdh + cc], x);
            });
        }
    }
    __syncthreads();
    if (a.hT) {
        for (int i = tid; i < dk * kDvm; i += kThreads) {
            const int j = i / kDvm, cc = i - j * kDvm;
            if (cc < nv) a.hT[(sbase + dv0 + cc) * dk + j] = Hs[j * kLdh + cc];
        }
    }
}

// Chunk prep for a scalar gate with its products on the tensor cores
// (mma.sync tf32; three products per step for fp32 I/O).  One CTA per
// (chunk, head): the gate cumsum, A = strictly_lower(diag(beta) G * K K^T),
// T = (I + A)^{-1} by blocks -- the four 16 x 16 diagonal blocks by forward
// substitution, then T21 = -T22 A21 T11 merges 16 -> 32 -> 64 -- and
// W = T diag(beta gamma) K, U = T diag(beta) V.  With Tout non-null it also
// stores T as [rows][64], with Tub and Wb non-null T diag(beta) and W as bf16
// rows (the backward pass reads them).
size_t prep_mma_smem(int dk, int dv) {
    return sizeof(float) * ((size_t)kChunk * (dk + 4) + (size_t)kChunk * (dv + 4) +
                            2 * kChunk * kLdc + 32 * 36 + 3 * kChunk);
}

template <typename TIn, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
k_prep_mma(FwdArgs a, const int2 *__restrict__ table, float *__restrict__ W,
           float *__restrict__ U, float *__restrict__ G, float *__restrict__ Tout,
           __nv_bfloat16 *__restrict__ Tub, __nv_bfloat16 *__restrict__ Wb, int *err) {
    extern __shared__ float smem[];
    const int dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    int n, c;
    if (table) {
        int2 e = table[blockIdx.x];
        n = e.x;
        c = e.y;
        if (n < 0) return;
    } else {
        n = blockIdx.x / a.max_chunks;
        c = blockIdx.x % a.max_chunks;
    }
    const int h = blockIdx.y;
    if (!seq_ok(a.sm, n)) {
        if (tid == 0) set_error(err, kErrBadIndex);
        return;
    }
    long long row0;
    int len;
    a.sm.get(n, h, row0, len);
    const int t0 = c * kChunk;
    if (t0 >= len) return;
    const int L = min(kChunk, len - t0);
    const long long r0 = row0 + t0;
    const bool erase = !a.no_erase;
    const int ldk = dk + 4, ldv = dv + 4;
    float *Ks = smem;                 // [64][dk+4]
    float *Vs = Ks + kChunk * ldk;    // [64][dv+4]
    float *A = Vs + kChunk * ldv;     // [64][68]
    float *Tm = A + kChunk * kLdc;    // [64][68]
    float *X = Tm + kChunk * kLdc;    // [32][36] merge scratch
    float *g = X + 32 * 36;           // [64] gate cumsum
    float *bb = g + kChunk;           // [64] beta
    float *wb = bb + kChunk;          // [64] beta * exp(g)
    const int m0 = 16 * (warp >> 1), nh = warp & 1;
    {
        TileRegs<4> rk;
        TileRegs<8> rv;
        rk.load(static_cast<const TIn *>(a.k) + r0 * dk, dk, dk, L, dk, tid);
        rv.load(static_cast<const TIn *>(a.v) + r0 * dv, dv, dv, L, dv, tid);
        if (tid < kChunk) {
            const bool ok = tid < L;
            g[tid] = ok ? __ldg(a.log_alpha + r0 + tid) : 0.f;
            bb[tid] = ok ? __ldg(a.beta + r0 + tid) : 0.f;
        }
        for (int i = tid; i < kChunk * kLdc; i += kThreads) Tm[i] = 0.f;
        rk.store(Ks, ldk, dk, tid);
        rv.store(Vs, ldv, dv, tid);
    }
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int r = 0; r < kChunk; ++r) {
            s += g[r];
            g[r] = s;
        }
    }
    __syncthreads();
    if (tid < kChunk) wb[tid] = bb[tid] * expf(g[tid]);
    if (erase) {   // A = strictly_lower(diag(beta) G * K K^T)
        float acc[4][4];
        mma::zero(acc);
        // only the strictly lower part of A is ever read: tiles right of this
        // warp's diagonal block are not formed
        mma::gemm_s<4, SPLIT>(acc, Ks, ldk, 1, nullptr, Ks, 1, ldk, m0, nh, 2, m0 + 16, dk, lane);
        mma::for_each(acc, m0, nh, 2, m0 + 16, lane, [&](int r, int s, float &x) {
            A[r * kLdc + s] = s < r ? bb[r] * expf(g[r] - g[s]) * x : 0.f;
        });
    } else {
        for (int i = tid; i < kChunk * kLdc; i += kThreads) A[i] = 0.f;
    }
    __syncthreads();
    if (tid < kChunk) {   // the 16 x 16 diagonal blocks, one column per thread
        const int o = 16 * (tid >> 4), cc = tid & 15;
        Tm[(o + cc) * kLdc + o + cc] = 1.f;
        for (int r = cc + 1; r < 16; ++r) {
            float acc = 0.f;
            for (int s = cc; s < r; ++s)
                acc = fmaf(A[(o + r) * kLdc + o + s], Tm[(o + s) * kLdc + o + cc], acc);
            Tm[(o + r) * kLdc + o + cc] = -acc;
        }
    }
    __syncthreads();
    // 16 -> 32: T21 = -T22 (A21 T11) for the blocks at 0 and 32
    if (warp < 2) {
        const int o = 32 * warp;
        float acc[2][4];
        mma::zero(acc);
        mma::warp_gemm<2, SPLIT>(
            acc, [&](int m, int k) { return A[(o + 16 + m) * kLdc + o + k]; },
            [&](int k, int nn) { return Tm[(o + k) * kLdc + o + nn]; }, 0, 0, 1, 16, 16, lane);
        mma::for_each(acc, 0, 0, 1, 16, lane,
                      [&](int m, int nn, float &x) { X[(16 * warp + m) * 36 + nn] = x; });
    }
    __syncthreads();
    if (warp < 2) {
        const int o = 32 * warp;
        float acc[2][4];
        mma::zero(acc);
        mma::warp_gemm<2, SPLIT>(
            acc, [&](int m, int k) { return Tm[(o + 16 + m) * kLdc + o + 16 + k]; },
            [&](int k, int nn) { return X[(16 * warp + k) * 36 + nn]; }, 0, 0, 1, 16, 16, lane);
        mma::for_each(acc, 0, 0, 1, 16, lane,
                      [&](int m, int nn, float &x) { Tm[(o + 16 + m) * kLdc + o + nn] = -x; });
    }
    __syncthreads();
    // 32 -> 64: T21 = -T22 (A21 T11), 32 x 32 blocks
    if (warp < 4) {
        float acc[2][4];
        mma::zero(acc);
        mma::warp_gemm<2, SPLIT>(
            acc, [&](int m, int k) { return A[(32 + m) * kLdc + k]; },
            [&](int k, int nn) { return Tm[k * kLdc + nn]; }, 16 * (warp >> 1), warp & 1, 2, 32,
            32, lane);
        mma::for_each(acc, 16 * (warp >> 1), warp & 1, 2, 32, lane,
                      [&](int m, int nn, float &x) { X[m * 36 + nn] = x; });
    }
    __syncthreads();
    if (warp < 4) {
        float acc[2][4];
        mma::zero(acc);
        mma::warp_gemm<2, SPLIT>(
            acc, [&](int m, int k) { return Tm[(32 + m) * kLdc + 32 + k]; },
            [&](int k, int nn) { return X[k * 36 + nn]; }, 16 * (warp >> 1), warp & 1, 2, 32, 32,
            lane);
        mma::for_each(acc, 16 * (warp >> 1), warp & 1, 2, 32, lane,
                      [&](int m, int nn, float &x) { Tm[(32 + m) * kLdc + nn] = -x; });
    }
    __syncthreads();
    {   // W = T diag(beta gamma) K (zero without the erase term)
        float acc[8][4];
        mma::zero(acc);
        if (erase)
            mma::gemm_s<8, SPLIT>(acc, Tm, kLdc, 1, wb, Ks, ldk, 1, m0, nh, 2, dk, m0 + 16, lane);
        // adjacent column pairs of the accumulator, stored as pairs
        const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int n8 = 8 * (nh + 2 * i);
            if (n8 < dk) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = m0 + gq + 8 * hr;
                    if (r < L) {
                        const long long o = (r0 + r) * dk + n8 + 2 * tq;
                        const float x0 = acc[i][2 * hr], x1 = acc[i][2 * hr + 1];
                        *reinterpret_cast<float2 *>(W + o) = make_float2(x0, x1);
                        if (Wb)
                            *reinterpret_cast<__nv_bfloat162 *>(Wb + o) =
                                __floats2bfloat162_rn(x0, x1);
                    }
                }
            }
        }
    }
    for (int c0 = 0; c0 < dv; c0 += 128) {   // U = T diag(beta) V
        float acc[8][4];
        mma::zero(acc);
        const int ne = min(dv, c0 + 128);
        mma::gemm_s<8, SPLIT>(acc, Tm, kLdc, 1, bb, Vs, ldv, 1, m0, c0 / 8 + nh, 2, ne, m0 + 16,
                              lane);
        store_pairs(acc, m0, c0 / 8 + nh, 2, ne, lane, L, U + r0 * dv, dv);
    }
    if (tid < L) G[r0 + tid] = g[tid];
    if (Tout)
        for (int i = tid; i < kChunk * kChunk; i += kThreads) {
            const int r = i >> 6, s = i & 63;
            if (r < L) Tout[(r0 + r) * kChunk + s] = Tm[r * kLdc + s];
        }
    if (Tub)   // T diag(beta), column pairs
        for (int i = tid; i < kChunk * kChunk / 2; i += kThreads) {
            const int r = i >> 5, s = 2 * (i & 31);
            if (r < L)
                *reinterpret_cast<__nv_bfloat162 *>(Tub + (r0 + r) * kChunk + s) =
                    __floats2bfloat162_rn(Tm[r * kLdc + s] * bb[s], Tm[r * kLdc + s + 1] * bb[s + 1]);
        }
}

// ------------------------------------------------ a gate per key dimension
//
// With log alpha a d_k-vector the decay between rows s <= r of a chunk is
// exp(G_rj - G_sj) per key dimension j (G the in-chunk cumsum), inside every
// contraction.  On the tensor cores it is split at 16-row blocks: for s and r
// in the same block the pair terms are formed directly; for s in an earlier
// block than r, with m the first row of r's block,
//     exp(G_rj - G_sj) = exp(G_rj - G_mj) exp(G_mj - G_sj),
// both factors <= 1 (G only decreases down the chunk), so
//     sum_j x_rj k_sj exp(G_rj - G_sj) = (x_r * exp(G_r - G_m)) . (k_s * exp(G_m - G_s))
// is a product of two bounded operands and nothing can overflow whatever the
// decay.  The other contractions take one bounded factor each:
// W = T diag(beta) (K * exp(G)), O = (Q * exp(G)) H + P V',
// H_j <- exp(G_Cj) H_j + sum_s k_sj exp(G_Cj - G_sj) V'_s.

// Prep: G [rows][d_k], A and T, W, U, and P [rows][64] (s <= r, zero above).
size_t prep_vg_smem(int dk, int dv) {
    const size_t ldk = dk + 4, ldv = dv + 4;
    const size_t region = std::max(64 * ldk + 32 * ldk + 48 * ldk, 64 * ldv);
    return sizeof(float) * (2 * 64 * ldk + 3 * (size_t)kChunk * kLdc + 32 * 36 + kChunk + region);
}

template <typename TIn, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
k_prep_vg(FwdArgs a, const int2 *__restrict__ table, float *__restrict__ W,
          float *__restrict__ U, float *__restrict__ G, float *__restrict__ Pout, int *err) {
    extern __shared__ float smem[];
    const int dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    int n, c;
    if (table) {
        int2 e = table[blockIdx.x];
        n = e.x;
        c = e.y;
        if (n < 0) return;
    } else {
        n = blockIdx.x / a.max_chunks;
        c = blockIdx.x % a.max_chunks;
    }
    const int h = blockIdx.y;
    if (!seq_ok(a.sm, n)) {
        if (tid == 0) set_error(err, kErrBadIndex);
        return;
    }
    long long row0;
    int len;
    a.sm.get(n, h, row0, len);
    const int t0 = c * kChunk;
    if (t0 >= len) return;
    const int L = min(kChunk, len - t0);
    const long long r0 = row0 + t0;
    const bool erase = !a.no_erase;
    const int ldk = dk + 4, ldv = dv + 4;
    float *Ks = smem;                   // [64][dk+4]  K, later K * exp(G)
    float *Gs = Ks + kChunk * ldk;      // [64][dk+4]  in-chunk cumsum of log alpha
    float *A = Gs + kChunk * ldk;       // [64][68]
    float *Tm = A + kChunk * kLdc;      // [64][68]
    float *Pm = Tm + kChunk * kLdc;     // [64][68]
    float *X = Pm + kChunk * kLdc;      // [32][36] merge scratch
    float *bb = X + 32 * 36;            // [64] beta
    float *Rg = bb + kChunk;            // Q and the staging tiles, then V
    float *Qs = Rg;                     // [64][dk+4]
    float *Xr = Qs + kChunk * ldk;      // [32][dk+4] rows of r's block: k-side 0..15, q-side 16..31
    float *Xs = Xr + 32 * ldk;          // [48][dk+4] rows s of the earlier blocks
    float *Vs = Rg;                     // [64][dv+4] (after the products above)
    const int m0 = 16 * (warp >> 1), nh = warp & 1;
    const bool want_p = Pout != nullptr;
    {
        TileRegs<4> rk, rq, rg;
        rk.load(static_cast<const TIn *>(a.k) + r0 * dk, dk, dk, L, dk, tid);
        if (want_p) rq.load(static_cast<const TIn *>(a.q) + r0 * dk, dk, dk, L, dk, tid);
        rg.load(a.log_alpha + r0 * dk, dk, dk, L, dk, tid);
        if (tid < kChunk) bb[tid] = tid < L ? __ldg(a.beta + r0 + tid) : 0.f;
        for (int i = tid; i < kChunk * kLdc; i += kThreads) {
            Tm[i] = 0.f;
            A[i] = 0.f;
            Pm[i] = 0.f;
        }
        rk.store(Ks, ldk, dk, tid);
        if (want_p) rq.store(Qs, ldk, dk, tid);
        rg.store(Gs, ldk, dk, tid);
    }
    __syncthreads();
    for (int j = tid; j < dk; j += kThreads) {   // column cumsums
        float acc = 0.f;
        for (int r = 0; r < kChunk; ++r) {
            acc += Gs[r * ldk + j];
            Gs[r * ldk + j] = acc;
        }
    }
    __syncthreads();
    // pairs inside the 16-row diagonal blocks, formed directly
    for (int i = tid; i < 2 * 4 * 136; i += kThreads) {
        const int which = i / (4 * 136), rem = i - which * 4 * 136;   // 0: A, 1: P
        const int blk = rem / 136;
        int p = rem - blk * 136, rl = 0;
        while (p > rl) {   // pair index -> (rl, sl) with sl <= rl
            p -= rl + 1;
            ++rl;
        }
        const int r = 16 * blk + rl, sc = 16 * blk + p;
        if (which == 0 && (sc == r || !erase)) continue;
        if (which == 1 && !want_p) continue;
        // four key dimensions per shared-memory load (rows are 16-byte
        // aligned: ldk is a multiple of 4)
        const float4 *xr = reinterpret_cast<const float4 *>(which == 0 ? Ks + r * ldk
                                                                       : Qs + r * ldk);
        const float4 *gr = reinterpret_cast<const float4 *>(Gs + r * ldk);
        const float4 *gs = reinterpret_cast<const float4 *>(Gs + sc * ldk);
        const float4 *ks = reinterpret_cast<const float4 *>(Ks + sc * ldk);
        float acc = 0.f;
        for (int j4 = 0; j4 < dk / 4; ++j4) {
            const float4 x = xr[j4], a = gr[j4], b = gs[j4], k = ks[j4];
            acc = fmaf(x.x * __expf(a.x - b.x), k.x, acc);
            acc = fmaf(x.y * __expf(a.y - b.y), k.y, acc);
            acc = fmaf(x.z * __expf(a.z - b.z), k.z, acc);
            acc = fmaf(x.w * __expf(a.w - b.w), k.w, acc);
        }
        if (which == 0) A[r * kLdc + sc] = bb[r] * acc;
        else Pm[r * kLdc + sc] = acc;
    }
    // earlier blocks, through the first row m of r's block
    for (int m = 16; m < kChunk; m += 16) {
        __syncthreads();   // staging free
        for (int row = warp; row < 32 + m; row += kThreads / 32)   // a warp per row
            for (int j = lane; j < dk; j += 32) {
                const float gm_ = Gs[m * ldk + j];
                if (row < 16) {
                    Xr[row * ldk + j] =
                        Ks[(m + row) * ldk + j] * __expf(Gs[(m + row) * ldk + j] - gm_);
                } else if (row < 32) {
                    const int rr = m + row - 16;
                    Xr[row * ldk + j] =
                        want_p ? Qs[rr * ldk + j] * __expf(Gs[rr * ldk + j] - gm_) : 0.f;
                } else {
                    const int sr = row - 32;
                    Xs[sr * ldk + j] = Ks[sr * ldk + j] * __expf(gm_ - Gs[sr * ldk + j]);
                }
            }
        __syncthreads();
        const int ntile = m / 8;
        for (int task = warp; task < 2 * ntile; task += kThreads / 32) {
            const int which = task / ntile, tile = task - which * ntile;
            if ((which == 0 && !erase) || (which == 1 && !want_p)) continue;
            float acc[1][4];
            mma::zero(acc);
            mma::gemm_s<1, SPLIT>(acc, Xr + 16 * which * ldk, ldk, 1, nullptr, Xs, 1, ldk, 0,
                                  tile, 1, m, dk, lane);
            mma::for_each(acc, 0, tile, 1, m, lane, [&](int i, int sc, float &x) {
                if (which == 0) A[(m + i) * kLdc + sc] = bb[m + i] * x;
                else Pm[(m + i) * kLdc + sc] = x;
            });
        }
    }
    __syncthreads();
    // T = (I + A)^{-1}: 16 x 16 diagonal blocks, then 16 -> 32 -> 64 merges
    if (tid < kChunk) {
        const int o = 16 * (tid >> 4), cc = tid & 15;
        Tm[(o + cc) * kLdc + o + cc] = 1.f;
        for (int r = cc + 1; r < 16; ++r) {
            float acc = 0.f;
            for (int q = cc; q < r; ++q)
                acc = fmaf(A[(o + r) * kLdc + o + q], Tm[(o + q) * kLdc + o + cc], acc);
            Tm[(o + r) * kLdc + o + cc] = -acc;
        }
    }
    __syncthreads();
    if (warp < 2) {
        const int o = 32 * warp;
        float acc[2][4];
        mma::zero(acc);
        mma::gemm_s<2, SPLIT>(acc, A + (o + 16) * kLdc + o, kLdc, 1, nullptr, Tm + o * kLdc + o,
                              kLdc, 1, 0, 0, 1, 16, 16, lane);
        mma::for_each(acc, 0, 0, 1, 16, lane,
                      [&](int i, int nn, float &x) { X[(16 * warp + i) * 36 + nn] = x; });
    }
    __syncthreads();
    if (warp < 2) {
        const int o = 32 * warp;
        float acc[2][4];
        mma::zero(acc);
        mma::gemm_s<2, SPLIT>(acc, Tm + (o + 16) * kLdc + o + 16, kLdc, 1, nullptr,
                              X + 16 * warp * 36, 36, 1, 0, 0, 1, 16, 16, lane);
        mma::for_each(acc, 0, 0, 1, 16, lane,
                      [&](int i, int nn, float &x) { Tm[(o + 16 + i) * kLdc + o + nn] = -x; });
    }
    __syncthreads();
    if (warp < 4) {
        float acc[2][4];
        mma::zero(acc);
        mma::gemm_s<2, SPLIT>(acc, A + 32 * kLdc, kLdc, 1, nullptr, Tm, kLdc, 1,
                              16 * (warp >> 1), warp & 1, 2, 32, 32, lane);
        mma::for_each(acc, 16 * (warp >> 1), warp & 1, 2, 32, lane,
                      [&](int i, int nn, float &x) { X[i * 36 + nn] = x; });
    }
    __syncthreads();
    if (warp < 4) {
        float acc[2][4];
        mma::zero(acc);
        mma::gemm_s<2, SPLIT>(acc, Tm + 32 * kLdc + 32, kLdc, 1, nullptr, X, 36, 1,
                              16 * (warp >> 1), warp & 1, 2, 32, 32, lane);
        mma::for_each(acc, 16 * (warp >> 1), warp & 1, 2, 32, lane,
                      [&](int i, int nn, float &x) { Tm[(32 + i) * kLdc + nn] = -x; });
    }
    // K * exp(G) (each factor <= 1)
    for (int r = warp; r < kChunk; r += kThreads / 32)
        for (int j = lane; j < dk; j += 32) Ks[r * ldk + j] *= __expf(Gs[r * ldk + j]);
    __syncthreads();
    {   // W = T diag(beta) (K * exp(G)) (zero without the erase term)
        float acc[8][4];
        mma::zero(acc);
        if (erase)
            mma::gemm_s<8, SPLIT>(acc, Tm, kLdc, 1, bb, Ks, ldk, 1, m0, nh, 2, dk, m0 + 16, lane);
        store_pairs(acc, m0, nh, 2, dk, lane, L, W + r0 * dk, dk);
    }
    {
        TileRegs<8> rv;
        rv.load(static_cast<const TIn *>(a.v) + r0 * dv, dv, dv, L, dv, tid);
        rv.store(Vs, ldv, dv, tid);
    }
    __syncthreads();
    for (int c0 = 0; c0 < dv; c0 += 128) {   // U = T diag(beta) V
        float acc[8][4];
        mma::zero(acc);
        const int ne = min(dv, c0 + 128);
        mma::gemm_s<8, SPLIT>(acc, Tm, kLdc, 1, bb, Vs, ldv, 1, m0, c0 / 8 + nh, 2, ne, m0 + 16,
                              lane);
        store_pairs(acc, m0, c0 / 8 + nh, 2, ne, lane, L, U + r0 * dv, dv);
    }
    for (int r = warp; r < L; r += kThreads / 32)
        for (int j = lane; j < dk; j += 32) G[(r0 + r) * dk + j] = Gs[r * ldk + j];
    if (want_p)
        for (int i = tid; i < L * kChunk; i += kThreads) {
            const int r = i >> 6, sc = i & 63;
            Pout[(r0 + r) * kChunk + sc] = Pm[r * kLdc + sc];
        }
}

// State pass with a gate per key dimension: one CTA per (sequence, head,
// 64-wide d_v tile), chunks in order, reading P from the prep.
size_t state_vg_smem(int dk) {
    const size_t ldk = dk + 4;
    return sizeof(float) * ((size_t)dk * kLdh + 4 * (size_t)kChunk * ldk +
                            3 * (size_t)kChunk * kLdc + 128);
}

template <typename TIn, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
k_state_vg(FwdArgs a, const float *__restrict__ W, const float *__restrict__ U,
           const float *__restrict__ G, const float *__restrict__ Pg, int *err) {
    extern __shared__ float smem[];
    const int dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int n = blockIdx.x, h = blockIdx.y, dv0 = blockIdx.z * kDvm;
    const int nv = min(kDvm, dv - dv0);
    if (!seq_ok(a.sm, n)) {
        if (tid == 0) set_error(err, kErrBadIndex);
        return;
    }
    long long row0;
    int len;
    a.sm.get(n, h, row0, len);
    const int ldk = dk + 4;
    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    TIn *op = static_cast<TIn *>(a.o);
    float *Hs = smem;                    // [dk][72]   H = S^T tile
    float *Ks = Hs + dk * kLdh;          // [64][dk+4] K * exp(G_C - G)
    float *Ws = Ks + kChunk * ldk;       // [64][dk+4]
    float *Qs = Ws + kChunk * ldk;       // [64][dk+4] Q * exp(G)
    float *Gt = Qs + kChunk * ldk;       // [64][dk+4] cumulative gates
    float *Us = Gt + kChunk * ldk;       // [64][68]
    float *Vn = Us + kChunk * kLdc;      // [64][68]
    float *P = Vn + kChunk * kLdc;       // [64][68]
    float *gce = P + kChunk * kLdc;      // [128] exp(G_C)
    const long long sbase = ((long long)n * a.sm.H + h) * dv;
    const int m0 = 16 * (warp >> 1), nh = warp & 1;

    for (int i = tid; i < dk * kDvm; i += kThreads) {
        const int j = i / kDvm, cc = i - j * kDvm;
        Hs[j * kLdh + cc] = (a.h0 && cc < nv) ? __ldg(a.h0 + (sbase + dv0 + cc) * dk + j) : 0.f;
    }
    const int nch = (len + kChunk - 1) / kChunk;
    for (int c = 0; c < nch; ++c) {
        const int t0 = c * kChunk, L = min(kChunk, len - t0);
        const long long r0 = row0 + t0;
        __syncthreads();  // previous chunk fully consumed
        {
            TileRegs<4> t;
            t.load(kp + r0 * dk, dk, dk, L, dk, tid);
            t.store(Ks, ldk, dk, tid);
            t.load(W + r0 * dk, dk, dk, L, dk, tid);
            t.store(Ws, ldk, dk, tid);
            t.load(qp + r0 * dk, dk, dk, L, dk, tid);
            t.store(Qs, ldk, dk, tid);
            t.load(G + r0 * dk, dk, dk, L, dk, tid);
            t.store(Gt, ldk, dk, tid);
        }
        {
            TileRegs<2> t;
            t.load(U + r0 * dv + dv0, dv, kDvm, L, nv, tid);
            t.store(Us, kLdc, kDvm, tid);
            t.load(Pg + r0 * kChunk, kChunk, kChunk, L, kChunk, tid);
            t.store(P, kLdc, kChunk, tid);
        }
        __syncthreads();
        // rows past L hold zeros (K = Q = 0), so their factors do not matter
        for (int r = warp; r < kChunk; r += kThreads / 32)
            for (int j = lane; j < dk; j += 32) {
                const float gr = Gt[r * ldk + j], gc = Gt[(L - 1) * ldk + j];
                Qs[r * ldk + j] *= __expf(gr);
                Ks[r * ldk + j] *= __expf(gc - gr);
            }
        for (int j = tid; j < dk; j += kThreads) gce[j] = __expf(Gt[(L - 1) * ldk + j]);
        {   // V' = U - W H
            float acc[4][4];
            mma::zero(acc);
            mma::gemm_s<4, SPLIT>(acc, Ws, ldk, 1, nullptr, Hs, kLdh, 1, m0, nh, 2, kDvm, dk,
                                  lane);
            mma::for_each(acc, m0, nh, 2, kDvm, lane, [&](int r, int cc, float &x) {
                Vn[r * kLdc + cc] = Us[r * kLdc + cc] - x;
            });
        }
        __syncthreads();
        {   // O = (Q * exp(G)) H + P V'
            float a1[4][4], a2[4][4];
            mma::zero(a1);
            mma::zero(a2);
            mma::gemm_s<4, SPLIT>(a1, Qs, ldk, 1, nullptr, Hs, kLdh, 1, m0, nh, 2, kDvm, dk,
                                  lane);
            mma::gemm_s<4, SPLIT>(a2, P, kLdc, 1, nullptr, Vn, kLdc, 1, m0, nh, 2, kDvm, m0 + 16,
                                  lane);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) a1[i][q] += a2[i][q];
            store_pairs(a1, m0, nh, 2, nv, lane, L, op + r0 * dv + dv0, dv);
        }
        __syncthreads();  // every read of H for this chunk is done
        // H_j <- exp(G_Cj) H_j + sum_s k_sj exp(G_Cj - G_sj) V'_s
        for (int j0 = 16 * warp; j0 < dk; j0 += 16 * (kThreads / 32)) {
            float acc[8][4];
            mma::zero(acc);
            mma::gemm_s<8, SPLIT>(acc, Ks, 1, ldk, nullptr, Vn, kLdc, 1, j0, 0, 1, kDvm, kChunk,
                                  lane);
            mma::for_each(acc, j0, 0, 1, kDvm, lane, [&](int j, int cc, float &x) {
                if (j < dk) Hs[j * kLdh + cc] = fmaf(gce[j], Hs[j * kLdh + cc], x);
            });
        }
    }
    __syncthreads();
    if (a.hT) {
        for (int i = tid; i < dk * kDvm; i += kThreads) {
            const int j = i / kDvm, cc = i - j * kDvm;
            if (cc < nv) a.hT[(sbase + dv0 + cc) * dk + j] = Hs[j * kLdh + cc];
        }
    }
}


// Launches the chunk prep (P: the intra-chunk P rows a gate per key
// dimension needs, else unused).
template <typename TIn>
cudaError_t run_prep(const FwdArgs &a, const int2 *table, float *W, float *U, float *G,
                     float *Tout, float *P, int *err, __nv_bfloat16 *Tub = nullptr,
                     __nv_bfloat16 *Wb = nullptr) {
    constexpr bool kSplit = std::is_same<TIn, float>::value;   // fp32 I/O: 3xTF32
    const dim3 grid(a.chunk_slots, a.sm.H);
    cudaError_t e;
    if (a.vector_gate) {
        const size_t psm = prep_vg_smem(a.dk, a.dv);
        e = cudaFuncSetAttribute(k_prep_vg<TIn, kSplit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psm);
        if (e != cudaSuccess) return e;
        k_prep_vg<TIn, kSplit><<<grid, kThreads, psm, a.stream>>>(a, table, W, U, G, P, err);
    } else {
        const size_t psm = prep_mma_smem(a.dk, a.dv);
        e = cudaFuncSetAttribute(k_prep_mma<TIn, kSplit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psm);
        if (e != cudaSuccess) return e;
        k_prep_mma<TIn, kSplit><<<grid, kThreads, psm, a.stream>>>(a, table, W, U, G, Tout, Tub,
                                                                  Wb, err);
    }
    count_launch();
    return cudaGetLastError();
}

// Launches the state pass (P as for run_prep).
template <typename TIn>
cudaError_t run_state(const FwdArgs &a, const float *W, const float *U, const float *G,
                      float *Hst, float *Vn, const float *P, int *err) {
    constexpr bool kSplit = std::is_same<TIn, float>::value;   // fp32 I/O: 3xTF32
    const dim3 grid(a.sm.N, a.sm.H, (a.dv + kDvm - 1) / kDvm);
    cudaError_t e;
    if (a.vector_gate) {
        const size_t ssm = state_vg_smem(a.dk);
        e = cudaFuncSetAttribute(k_state_vg<TIn, kSplit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
        if (e != cudaSuccess) return e;
        const int slot = timer_begin(a.stream, "k_state_vg");
        k_state_vg<TIn, kSplit><<<grid, kThreads, ssm, a.stream>>>(a, W, U, G, P, err);
        timer_end(slot, a.stream);
    } else {
        const size_t ssm = state_mma_smem(a.dk, a.o != nullptr);
        e = cudaFuncSetAttribute(k_state_mma<TIn, kSplit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)state_mma_smem(a.dk, true));
        if (e != cudaSuccess) return e;
        // timed only as a forward call's dominant kernel: the backward pass's
        // recomputation (no output) is not its most expensive launch
        const int slot = a.o ? timer_begin(a.stream, "k_state_mma") : -1;
        k_state_mma<TIn, kSplit><<<grid, kThreads, ssm, a.stream>>>(a, W, U, G, Hst, Vn, err);
        timer_end(slot, a.stream);
    }
    count_launch();
    return cudaGetLastError();
}

template <typename TIn>
gdn_status launch(const FwdArgs &a) {
    int *err = device_error_word();
    cudaStream_t st = a.stream;
    float *W = nullptr, *U = nullptr, *G = nullptr, *P = nullptr;
    int2 *table = nullptr;
    const size_t rows = (size_t)a.rows > 0 ? (size_t)a.rows : 1;
    if (scratch_alloc((void **)&W, rows * a.dk * sizeof(float), st) != cudaSuccess ||
        scratch_alloc((void **)&U, rows * a.dv * sizeof(float), st) != cudaSuccess ||
        scratch_alloc((void **)&G, rows * (a.vector_gate ? a.dk : 1) * sizeof(float), st) !=
            cudaSuccess ||
        (a.vector_gate &&
         scratch_alloc((void **)&P, rows * kChunk * sizeof(float), st) != cudaSuccess)) {
        if (W) scratch_free(W, st);
        if (U) scratch_free(U, st);
        if (G) scratch_free(G, st);
        return GDN_ERR_CUDA;
    }
    gdn_status rc = GDN_OK;
    if (a.chunk_slots > 0) {
        if (a.sm.cu) {
            if (scratch_alloc((void **)&table, sizeof(int2) * (size_t)a.chunk_slots, st) !=
                cudaSuccess) {
                rc = GDN_ERR_CUDA;
            } else {
                k_chunk_table<<<1, 1024, 0, st>>>(a.sm.cu, a.sm.N, a.sm.T_total, table,
                                                 a.chunk_slots, err);
                count_launch();
            }
        }
        if (rc == GDN_OK && a.sm.H > 0 &&
            run_prep<TIn>(a, table, W, U, G, nullptr, P, err) != cudaSuccess)
            rc = GDN_ERR_CUDA;
    }
    if (rc == GDN_OK && a.sm.N > 0 && a.sm.H > 0 &&
        run_state<TIn>(a, W, U, G, nullptr, nullptr, P, err) != cudaSuccess)
        rc = GDN_ERR_CUDA;
    if (rc == GDN_OK && cudaGetLastError() != cudaSuccess) rc = GDN_ERR_CUDA;
    scratch_free(W, st);
    scratch_free(U, st);
    scratch_free(G, st);
    if (P) scratch_free(P, st);
    if (table) scratch_free(table, st);
    return rc;
}

}  // namespace

gdn_status simt_forward(const FwdArgs &a) {
    return a.dt == GDN_F32 ? launch<float>(a) : launch<__nv_bfloat16>(a);
}

template <typename TIn>
gdn_status enqueue_state_t(const FwdArgs &a, const float *W, const float *U, const float *G,
                           float *Hst, float *Vn) {
    if (a.sm.N > 0 && a.sm.H > 0 &&
        run_state<TIn>(a, W, U, G, Hst, Vn, nullptr, device_error_word()) != cudaSuccess)
        return GDN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename TIn>
gdn_status enqueue_prep_t(const FwdArgs &a, const int2 *table, float *W, float *U, float *G,
                          float *Tout, __nv_bfloat16 *Tub = nullptr, __nv_bfloat16 *Wb = nullptr) {
    if (a.chunk_slots > 0 && a.sm.H > 0 &&
        run_prep<TIn>(a, table, W, U, G, Tout, nullptr, device_error_word(), Tub, Wb) !=
            cudaSuccess)
        return GDN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status enqueue_simt_prep(const FwdArgs &a, const int2 *table, float *W, float *U, float *G,
                             float *Tout) {
    if (a.vector_gate) return GDN_ERR_UNSUPPORTED;
    return a.dt == GDN_F32 ? enqueue_prep_t<float>(a, table, W, U, G, Tout)
                           : enqueue_prep_t<__nv_bfloat16>(a, table, W, U, G, Tout);
}

gdn_status enqueue_simt_prep_tc(const FwdArgs &a, const int2 *table, float *W, float *U,
                                float *G, float *Tout, __nv_bfloat16 *Tub, __nv_bfloat16 *Wb) {
    if (a.vector_gate || a.dt != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    return enqueue_prep_t<__nv_bfloat16>(a, table, W, U, G, Tout, Tub, Wb);
}

gdn_status enqueue_simt_state(const FwdArgs &a, const float *W, const float *U, const float *G,
                              float *Hst, float *Vn) {
    if (a.vector_gate) return GDN_ERR_UNSUPPORTED;
    return a.dt == GDN_F32 ? enqueue_state_t<float>(a, W, U, G, Hst, Vn)
                           : enqueue_state_t<__nv_bfloat16>(a, W, U, G, Hst, Vn);
}

gdn_status enqueue_chunk_table(const FwdArgs &a, int2 *table) {
    k_chunk_table<<<1, 1024, 0, a.stream>>>(a.sm.cu, a.sm.N, a.sm.T_total, table, a.chunk_slots,
                                             device_error_word());
    count_launch();
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn

// ------------------------------------------------- allocation-free variant
//
// gdn_fwd_noalloc runs the same two kernels (prep, state pass) on a
// dense batch, but its W / U / gate-cumsum scratch lives in this fixed device
// array instead of the library's scratch pool.  The array belongs to every
// GPU that loads the library, for as long as the library stays loaded.  All
// calls share it and it keeps whatever the previous call left: nothing in it
// needs to start at zero, because the prep kernel writes every row the state
// kernel later reads.  Two calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on it and may both be wrong.
static __device__ __align__(256) float gdn_noalloc_scratch[gdn::kNoallocScratchBytes / sizeof(float)];

namespace gdn {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name only stands in for the symbol, so the address is looked
// up once per device (with that device current) and cached.
gdn_status noalloc_scratch(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, gdn_noalloc_scratch) != cudaSuccess || !p)
            return GDN_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return GDN_OK;
}

template <typename TIn>
gdn_status launch_noalloc(const FwdArgs &a, float *scratch) {
    int *err = device_error_word();
    const size_t rows = (size_t)a.rows;
    float *W = scratch;
    float *U = W + rows * a.dk;
    float *G = U + rows * a.dv;
    if (a.chunk_slots > 0 &&
        run_prep<TIn>(a, nullptr, W, U, G, nullptr, nullptr, err) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (run_state<TIn>(a, W, U, G, nullptr, nullptr, nullptr, err) != cudaSuccess)
        return GDN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

gdn_status simt_forward_noalloc(const FwdArgs &a) {
    if (a.sm.cu) return GDN_ERR_UNSUPPORTED;   // dense batches only
    const size_t need =
        (size_t)a.rows * (size_t)(a.dk + a.dv + (a.vector_gate ? a.dk : 1)) * sizeof(float);
    if (need > kNoallocScratchBytes) return GDN_ERR_TOO_LARGE;
    float *scratch = nullptr;
    gdn_status rc = noalloc_scratch(&scratch);
    if (rc != GDN_OK) return rc;
    return a.dt == GDN_F32 ? launch_noalloc<float>(a, scratch)
                           : launch_noalloc<__nv_bfloat16>(a, scratch);
}

}  // namespace gdn
