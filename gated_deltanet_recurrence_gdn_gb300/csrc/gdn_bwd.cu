// gdn_bwd.cu -- backward pass of the chunked gated delta rule on warp-level
// tf32 mma.sync products (three per step for fp32 I/O), fp32 accumulation.
//
// The gradient of L = sum dO . o + <dhT, hT> with respect to q, k, v,
// log_alpha, beta and h0.  The recurrent state is recomputed, not stored by
// the forward pass (the recomputation of "企业官网建设流程全解析", sections 2
// and 4.3); the chunked algebra is that of the forward ("Gated DeltaNet
// GPU并行实现" section 3.2), differentiated.  Per chunk, with g the gate
// cumsum, gamma = exp(g), G_rs = exp(g_r - g_s), e_r = exp(g_C - g_r),
// S0 the chunk's starting state (d_v x d_k) and dSC the adjoint of its end
// state, the forward is
//
//     A  = strictly_lower(diag(beta) (G * K K^T)),  T = (I + A)^{-1}
//     W  = T diag(beta gamma) K,   U = T diag(beta) V,   V' = U - W S0^T
//     O  = diag(gamma) Q S0^T + (mask * G * Q K^T) V'
//     SC = gamma_C S0 + V'^T diag(e) K
//
// and its adjoint, chunk by chunk in reverse (serial in the state):
//
//     dV'  = (mask * G * Q K^T)^T dO + diag(e) K dSC^T
//     dS0  = gamma_C dSC + dO^T diag(gamma) Q - dV'^T W
//
// then, all chunks in parallel, with dP = mask * G * (dO V'^T):
//
//     dQ   = diag(gamma) dO S0 + dP K
//     dK   = dP^T Q + diag(e) V' dSC + diag(beta gamma) T^T dW + (A terms)
//     dV   = diag(beta) T^T dV',            dW = -dV' S0
//     dT   = dV' (diag(beta) V)^T + dW (diag(beta gamma) K)^T
//     dA   = -T^T dT T^T  (strictly lower part)
//     dbeta, dg from every place beta and g enter; dlog_alpha is the
//     reverse cumsum of dg inside the chunk.
//
// Kernels: the forward prep and state pass (gdn_simt.cu) recompute W, U, the
// gate cumsum, every chunk's starting state and V'; k_bwd_dstate carries the
// state adjoint backwards (for bf16 I/O on shapes it takes, the tcgen05
// kernel of gdn_bwd_tc.cu does instead); k_bwd_chunk forms every gradient of
// one chunk.
// Without the erase term A = 0, T = I and W = 0, and the A and W terms drop.
#include <cuda_bf16.h>

#include <type_traits>

#include "gdn_bwd_tc.h"
#include "gdn_internal.h"
#include "gdn_mma.cuh"
#include "gdn_tile.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kDvt = 32;     // d_v columns per tile

// Two adjacent outputs (columns c, c + 1 of a row, c even) in one store.
__device__ __forceinline__ void st_out2(float *p, float x, float y) {
    *reinterpret_cast<float2 *>(p) = make_float2(x, y);
}
__device__ __forceinline__ void st_out2(__nv_bfloat16 *p, float x, float y) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x, y);
}
__device__ __forceinline__ void set_error(int *err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ bool seq_ok(const SeqMap &sm, int n) {
    if (!sm.cu) return true;
    int a = __ldg(sm.cu + n), b = __ldg(sm.cu + n + 1);
    return a >= 0 && a <= b && b <= sm.T_total;
}

// ---------------------------------------------------------------- dS pass
//
// One CTA per (sequence, head, 64-wide d_v tile), chunks in reverse order.
// dH = dS^T (d_k x 64) lives in shared memory.  For each chunk it stores
// dH (the adjoint of the chunk's end state) as [H][chunk_slots][d_k][d_v]
// and the rows of dV', then steps dH back to the chunk's start.  The products
// run on the tensor cores (mma.sync tf32, gdn_mma.cuh); the next (earlier)
// chunk's K, Q, W and dO are loaded into registers while the current one is
// computed.

constexpr int kDvm = 64;           // d_v columns per dS-pass CTA
constexpr int kLdh = kDvm + 8;     // d_k x 64 state tiles: transposed reads conflict-free
constexpr int kLdc = kChunk + 4;   // 64 x 64 tiles
constexpr int kLdt = kDvt + 4;     // 64 x 32 tiles (chunk kernel)

size_t dstate_smem(int dk) {
    return sizeof(float) * ((size_t)dk * kLdh + 3 * (size_t)kChunk * (dk + 4) +
                            3 * kChunk * kLdc + 3 * kChunk);
}

template <typename TIn, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
k_bwd_dstate(FwdArgs a, BwdArgs b, const float *__restrict__ W, const float *__restrict__ G,
             float *__restrict__ dVn, float *__restrict__ dHc, int *err) {
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
    float *dH = smem;                    // [dk][72]
    float *Ks = dH + dk * kLdh;          // [64][dk+4]
    float *Qs = Ks + kChunk * ldk;       // [64][dk+4]
    float *Ws = Qs + kChunk * ldk;       // [64][dk+4]
    float *dOs = Ws + kChunk * ldk;      // [64][68]
    float *dVs = dOs + kChunk * kLdc;    // [64][68]
    float *P = dVs + kChunk * kLdc;      // [64][68]  P_rs = G_rs q_r . k_s, s <= r
    float *g = P + kChunk * kLdc;        // [64]
    float *e = g + kChunk;               // [64] exp(g_C - g_r)
    float *gm = e + kChunk;              // [64] exp(g_r)
    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *dop = static_cast<const TIn *>(b.dout);
    const long long sbase = ((long long)n * a.sm.H + h) * dv;
    const int m0 = 16 * (warp >> 1), nh = warp & 1;
    const int ntask = 2 * ((dk + 15) / 16);   // (16-row block, column half) tasks of d_k x 64

    for (int i = tid; i < dk * kDvm; i += kThreads) {
        const int j = i / kDvm, cc = i - j * kDvm;
        dH[j * kLdh + cc] = (b.dhT && cc < nv) ? __ldg(b.dhT + (sbase + dv0 + cc) * dk + j) : 0.f;
    }
    TileRegs<4> rk, rq, rw;
    TileRegs<2> ro;
    float gnext = 0.f;
    auto issue = [&](int c) {
        const int L = min(kChunk, len - c * kChunk);
        const long long r0 = row0 + (long long)c * kChunk;
        rk.load(kp + r0 * dk, dk, dk, L, dk, tid);
        rq.load(qp + r0 * dk, dk, dk, L, dk, tid);
        rw.load(W + r0 * dk, dk, dk, L, dk, tid);
        ro.load(dop + r0 * dv + dv0, dv, kDvm, L, nv, tid);
        if (tid < kChunk) gnext = __ldg(G + r0 + min(tid, L - 1));
    };
    const int nch = (len + kChunk - 1) / kChunk;
    if (nch > 0) issue(nch - 1);
    for (int c = nch - 1; c >= 0; --c) {
        const int t0 = c * kChunk, L = min(kChunk, len - t0);
        const long long r0 = row0 + t0;
        __syncthreads();  // the previous (later) chunk is fully consumed
        float *dst = dHc + ((long long)h * a.chunk_slots + a.chunk_slot(n, c)) * dk * dv;
        for (int i = tid; i < dk * kDvm; i += kThreads) {
            const int j = i / kDvm, cc = i - j * kDvm;
            if (cc < nv) dst[(long long)j * dv + dv0 + cc] = dH[j * kLdh + cc];
        }
        rk.store(Ks, ldk, dk, tid);
        rq.store(Qs, ldk, dk, tid);
        rw.store(Ws, ldk, dk, tid);
        ro.store(dOs, kLdc, kDvm, tid);
        if (tid < kChunk) g[tid] = gnext;
        if (c > 0) issue(c - 1);
        __syncthreads();
        const float gl = g[kChunk - 1];
        if (tid < kChunk) {
            e[tid] = expf(gl - g[tid]);
            gm[tid] = expf(g[tid]);
        }
        {
            float acc[4][4];
            mma::zero(acc);
            // tiles right of this warp's diagonal block are masked: not formed
            // (the P^T dO below reads rows s >= r only, which are)
            mma::gemm_s<4, SPLIT>(acc, Qs, ldk, 1, nullptr, Ks, 1, ldk, m0, nh, 2, m0 + 16, dk,
                                  lane);
            mma::for_each(acc, m0, nh, 2, m0 + 16, lane, [&](int r, int s, float &x) {
                P[r * kLdc + s] = s <= r ? expf(g[r] - g[s]) * x : 0.f;
            });
        }
        __syncthreads();
        {   // dV'_r = sum_{s >= r} P_sr dO_s + e_r dS k_r
            float a1[4][4], a2[4][4];
            mma::zero(a1);
            mma::zero(a2);
            mma::gemm_s<4, SPLIT>(a1, P, 1, kLdc, nullptr, dOs, kLdc, 1, m0, nh, 2, kDvm, kChunk,
                                  lane, m0);
            mma::gemm_s<4, SPLIT>(a2, Ks, ldk, 1, nullptr, dH, kLdh, 1, m0, nh, 2, kDvm, dk,
                                  lane);
            const int gl4 = lane >> 2, tl = lane & 3;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = m0 + gl4 + 8 * (q >> 1), cc = 8 * (nh + 2 * i) + 2 * tl + (q & 1);
                    const float val = r < L ? fmaf(e[r], a2[i][q], a1[i][q]) : 0.f;
                    dVs[r * kLdc + cc] = val;
                    if (r < L && cc < nv) dVn[(r0 + r) * dv + dv0 + cc] = val;
                }
        }
        __syncthreads();
        // dS <- gamma_C dS + dO^T diag(gamma) Q - dV'^T W   (as dH = dS^T)
        const float decay = expf(gl);
        for (int task = warp; task < ntask; task += kThreads / 32) {
            const int j0 = 16 * (task >> 1), th = task & 1;
            float acc[4][4], acw[4][4];
            mma::zero(acc);
            mma::zero(acw);
            mma::gemm_s<4, SPLIT>(acc, Qs, 1, ldk, gm, dOs, kLdc, 1, j0, th, 2, kDvm, kChunk,
                                  lane);
            mma::gemm_s<4, SPLIT>(acw, Ws, 1, ldk, nullptr, dVs, kLdc, 1, j0, th, 2, kDvm,
                                  kChunk, lane);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][q] -= acw[i][q];
            mma::for_each(acc, j0, th, 2, kDvm, lane, [&](int j, int cc, float &x) {
                if (j < dk) dH[j * kLdh + cc] = fmaf(decay, dH[j * kLdh + cc], x);
            });
        }
    }
    __syncthreads();
    if (b.dh0) {
        for (int i = tid; i < dk * kDvm; i += kThreads) {
            const int j = i / kDvm, cc = i - j * kDvm;
            if (cc < nv) b.dh0[(sbase + dv0 + cc) * dk + j] = dH[j * kLdh + cc];
        }
    }
}

// ------------------------------------------------------------ chunk kernel
//
// One CTA per (chunk, head), 8 warps; every product runs on the tensor
// cores through mma.sync tf32 (gdn_mma.cuh; three products per step for fp32
// I/O, one for bf16 I/O).  Warp w owns rows 16 (w / 2) .. +15 of every
// 64-row output and the 8-column tiles w % 2, w % 2 + 2, ... of it.
// Phase 1 loads T (written by the prep) and forms K K^T.  Phase 2 walks d_v in
// 32-wide tiles: dO S0, V' dSC and dV' S0 (64 x d_k) and dO V'^T,
// dV' V^T (64 x 64) accumulate in registers; dV = diag(beta) T^T dV' and the
// U part of dbeta are written per tile.  Phase 3 forms dQ, dK, dbeta and
// dlog_alpha.

constexpr int kNtK = 8;            // 8-column tiles per warp of a 64 x d_k output (d_k <= 128)
constexpr int kNtC = 4;            // ... of a 64 x 64 output
constexpr int kNtV = 2;            // ... of a 64 x 32 output

struct ChunkLay {
    int ldk, region;
    int oK, oR, oWm, oT, oB1, oB2, oB3, oV;
    size_t bytes;
};

__host__ __device__ inline ChunkLay chunk_lay(int dk) {
    ChunkLay l;
    l.ldk = dk + 4;
    const int tiles = 4 * kChunk * kLdt + 2 * dk * kLdt;
    const int qsz = kChunk * l.ldk;
    l.region = tiles > qsz ? tiles : qsz;
    l.oK = 0;
    l.oR = l.oK + kChunk * l.ldk;
    l.oWm = l.oR + l.region;
    l.oT = l.oWm + kChunk * l.ldk;
    l.oB1 = l.oT + kChunk * kLdc;
    l.oB2 = l.oB1 + kChunk * kLdc;
    l.oB3 = l.oB2 + kChunk * kLdc;
    l.oV = l.oB3 + kChunk * kLdc;
    l.bytes = sizeof(float) * ((size_t)l.oV + 12 * kChunk + 32);
    return l;
}

// Row sums (over this thread's columns and the four lanes of a row) of an
// accumulator block, added to v[row] with weight w(row).
template <int NT, typename F, typename W>
__device__ __forceinline__ void add_row_sums(float (&acc)[NT][4], int m0, int nt0, int nstep,
                                             int n_end, int lane, F value, float *v, W w) {
    float r0 = 0.f, r1 = 0.f;
    mma::for_each(acc, m0, nt0, nstep, n_end, lane, [&](int m, int n, float &x) {
        const float y = value(m, n, x);
        if (((m - m0) >> 3) == 0) r0 += y; else r1 += y;
    });
    r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
    r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
    if ((lane & 3) == 0) {
        const int m = m0 + (lane >> 2);
        atomicAdd(v + m, w(m) * r0);
        atomicAdd(v + m + 8, w(m + 8) * r1);
    }
}

// Column sums (over the 16 rows of the block) added to v[col] times scale.
template <int NT, typename F>
__device__ __forceinline__ void add_col_sums(float (&acc)[NT][4], int m0, int nt0, int nstep,
                                             int n_end, int lane, F value, float *v,
                                             float scale) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        const int n = 8 * (nt0 + i * nstep);
        if (n < n_end) {
            float c0 = value(m0 + g, n + 2 * t, acc[i][0]) + value(m0 + g + 8, n + 2 * t, acc[i][2]);
            float c1 = value(m0 + g, n + 2 * t + 1, acc[i][1]) +
                       value(m0 + g + 8, n + 2 * t + 1, acc[i][3]);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                c0 += __shfl_xor_sync(0xffffffffu, c0, o);
                c1 += __shfl_xor_sync(0xffffffffu, c1, o);
            }
            if (g == 0) {
                atomicAdd(v + n + 2 * t, scale * c0);
                atomicAdd(v + n + 2 * t + 1, scale * c1);
            }
        }
    }
}

template <typename TIn, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
k_bwd_chunk(FwdArgs a, BwdArgs b, const int2 *__restrict__ table, const float *__restrict__ Tg,
            const float *__restrict__ Hst, const float *__restrict__ dHc,
            const float *__restrict__ Vn, const float *__restrict__ dVn, int *err) {
    extern __shared__ float smem[];
    const int dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    int n, c;
    if (table) {
        const int2 en = table[blockIdx.x];
        n = en.x;
        c = en.y;
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
    const long long st_off = ((long long)h * a.chunk_slots + a.chunk_slot(n, c)) * dk * dv;

    const ChunkLay ly = chunk_lay(dk);
    const int ldk = ly.ldk;
    float *Ks = smem + ly.oK;     // [64][ldk]
    float *Rg = smem + ly.oR;     // phase 2 tiles, then Q
    float *Wm = smem + ly.oWm;    // [64][ldk]  dV' S0 (= -dW)
    float *Tm = smem + ly.oT;     // [64][68]   T
    float *B1 = smem + ly.oB1;    // [64][68]   dP, then dT T^T
    float *B2 = smem + ly.oB2;    // [64][68]   dV' (diag(beta) V)^T, then dT, then X = dA * G
    float *B3 = smem + ly.oB3;    // [64][68]   K K^T
    float *g = smem + ly.oV;      // [64] gate cumsum
    float *bb = g + kChunk;       // [64] beta
    float *gm = bb + kChunk;      // [64] exp(g)
    float *ed = gm + kChunk;      // [64] exp(g_C - g)
    float *dbU = ed + kChunk;     // [64] dbeta from U
    float *dgE = dbU + kChunk;    // [64] dg from the intra-chunk output term
    float *dgQ = dgE + kChunk;    // [64] dg from the inter-chunk output term
    float *Fv = dgQ + kChunk;     // [64] e_s k_s . (V' dSC)_s
    float *tv = Fv + kChunk;      // [64] gamma_s k_s . (T^T dW)_s
    float *dgA = tv + kChunk;     // [64] dg from A
    float *dbA = dgA + kChunk;    // [64] dbeta from A
    float *dlv = dbA + kChunk;    // [64] dg total
    float *red = dlv + kChunk;    // [32]
    float *dOs = Rg;                       // [64][36]
    float *Vns = dOs + kChunk * kLdt;      // [64][36]  V'
    float *dVs = Vns + kChunk * kLdt;      // [64][36]  dV'
    float *Vs = dVs + kChunk * kLdt;       // [64][36]  V
    float *S0t = Vs + kChunk * kLdt;       // [dk][36]  S0^T tile
    float *dSt = S0t + dk * kLdt;          // [dk][36]  dSC^T tile
    float *Qs = Rg;                        // phase 3: [64][ldk]

    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *vp = static_cast<const TIn *>(a.v);
    const TIn *dop = static_cast<const TIn *>(b.dout);

    const int m0 = 16 * (warp >> 1), nh = warp & 1;

    // ---- phase 1: K, gates, T (from the prep), K K^T
    {
        TileRegs<4> rk;
        TileRegs<2> rt;
        rk.load(kp + r0 * dk, dk, dk, L, dk, tid);
        rt.load(Tg + r0 * kChunk, kChunk, kChunk, L, kChunk, tid);
        rk.store(Ks, ldk, dk, tid);
        rt.store(Tm, kLdc, kChunk, tid, L);
    }
    for (int i = tid; i < kChunk * kChunk; i += kThreads) {   // rows past L: identity
        const int r = i >> 6, s = i & 63;
        if (r >= L) Tm[r * kLdc + s] = r == s ? 1.f : 0.f;
    }
    if (tid < kChunk) {
        const bool ok = tid < L;
        g[tid] = ok ? __ldg(a.log_alpha + r0 + tid) : 0.f;
        bb[tid] = ok ? __ldg(a.beta + r0 + tid) : 0.f;
        dbU[tid] = dgE[tid] = dgQ[tid] = Fv[tid] = tv[tid] = dgA[tid] = dbA[tid] = 0.f;
    }
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int r = 0; r < kChunk; ++r) {
            s += g[r];
            g[r] = s;
        }
    }
    if (erase) {   // K K^T
        float acc[kNtC][4];
        mma::zero(acc);
        // K K^T is read below the diagonal only: tiles right of this warp's
        // diagonal block are not formed
        mma::gemm_s<kNtC, SPLIT>(acc, Ks, ldk, 1, nullptr, Ks, 1, ldk, m0, nh, 2, m0 + 16, dk,
                                 lane);
        mma::for_each(acc, m0, nh, 2, m0 + 16, lane,
                      [&](int m, int nn, float &x) { B3[m * kLdc + nn] = x; });
    }
    __syncthreads();
    const float gC = g[L - 1];
    if (tid < kChunk) {
        gm[tid] = expf(g[tid]);
        ed[tid] = expf(gC - g[tid]);
    }

    // ---- phase 2: the d_v contractions, tile by tile
    float aQ[kNtK][4], aK[kNtK][4], aW[kNtK][4], aP[kNtC][4], aT[kNtC][4];
    mma::zero(aQ);
    mma::zero(aK);
    mma::zero(aW);
    mma::zero(aP);
    mma::zero(aT);
    float sC = 0.f;
    const int gl = lane >> 2, tl = lane & 3;
    for (int dv0 = 0; dv0 < dv; dv0 += kDvt) {
        const int nv = min(kDvt, dv - dv0);
        {   // all of this tile's loads in flight at once
            TileRegs<1> t1, t2, t3, t4, s0a, s0b, dsa, dsb;
            const long long o = r0 * dv + dv0;
            t1.load(dop + o, dv, kDvt, L, nv, tid);
            t2.load(Vn + o, dv, kDvt, L, nv, tid);
            t3.load(dVn + o, dv, kDvt, L, nv, tid);
            t4.load(vp + o, dv, kDvt, L, nv, tid);
            const float *hs = Hst + st_off + dv0, *hd = dHc + st_off + dv0;
            s0a.load(hs, dv, kDvt, dk, nv, tid);
            dsa.load(hd, dv, kDvt, dk, nv, tid);
            s0b.load(hs + 64LL * dv, dv, kDvt, dk - 64, nv, tid);
            dsb.load(hd + 64LL * dv, dv, kDvt, dk - 64, nv, tid);
            __syncthreads();  // T ready / the previous tile consumed
            t1.store(dOs, kLdt, kDvt, tid);
            t2.store(Vns, kLdt, kDvt, tid);
            t3.store(dVs, kLdt, kDvt, tid);
            t4.store(Vs, kLdt, kDvt, tid);
            s0a.store(S0t, kLdt, kDvt, tid, dk);
            dsa.store(dSt, kLdt, kDvt, tid, dk);
            if (dk > 64) {
                s0b.store(S0t + 64 * kLdt, kLdt, kDvt, tid, dk - 64);
                dsb.store(dSt + 64 * kLdt, kLdt, kDvt, tid, dk - 64);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                sC = fmaf(s0a.v[0][e], dsa.v[0][e], fmaf(s0b.v[0][e], dsb.v[0][e], sC));
        }
        __syncthreads();
        // dO S0, V' dSC, dV' S0 sharing the S0 / dSC fragments; every operand
        // here is row-wise in the d_v index, so fragments load by ldmatrix
        // (B tiles in pairs 16 columns apart; past d_k the pair repeats its
        // first tile, whose second products are skipped)
        {
            const int ao = (m0 + (lane & 15)) * kLdt + 4 * (lane >> 4);
            const uint32_t a_o = mma::smem_addr(dOs + ao), a_v = mma::smem_addr(Vns + ao),
                           a_d = mma::smem_addr(dVs + ao);
#pragma unroll
            for (int k0 = 0; k0 < kDvt; k0 += 8) {
                mma::AFrag<SPLIT> fo, fv, fd;
                mma::lda_ldsm(fo, a_o + 4 * k0);
                mma::lda_ldsm(fv, a_v + 4 * k0);
                if (erase) mma::lda_ldsm(fd, a_d + 4 * k0);
#pragma unroll
                for (int i = 0; i < kNtK; i += 2) {
                    const int n0 = 8 * (nh + 2 * i), n1 = 8 * (nh + 2 * i + 2);
                    if (n0 < dk) {
                        const int n1c = n1 < dk ? n1 : n0;
                        uint32_t bs[4], bd[4];
                        mma::ldsm4(bs, mma::smem_addr(mma::ldb_pair_ptr(S0t, kLdt, n0, n1c, k0,
                                                                         lane)));
                        mma::ldsm4(bd, mma::smem_addr(mma::ldb_pair_ptr(dSt, kLdt, n0, n1c, k0,
                                                                         lane)));
                        const float s0[4] = {__uint_as_float(bs[0]), __uint_as_float(bs[1]),
                                             __uint_as_float(bs[2]), __uint_as_float(bs[3])};
                        const float d0[4] = {__uint_as_float(bd[0]), __uint_as_float(bd[1]),
                                             __uint_as_float(bd[2]), __uint_as_float(bd[3])};
                        mma::mma_step<SPLIT>(aQ[i], fo, s0[0], s0[1]);
                        mma::mma_step<SPLIT>(aK[i], fv, d0[0], d0[1]);
                        if (erase) mma::mma_step<SPLIT>(aW[i], fd, s0[0], s0[1]);
                        if (n1 < dk) {
                            mma::mma_step<SPLIT>(aQ[i + 1], fo, s0[2], s0[3]);
                            mma::mma_step<SPLIT>(aK[i + 1], fv, d0[2], d0[3]);
                            if (erase) mma::mma_step<SPLIT>(aW[i + 1], fd, s0[2], s0[3]);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < kNtC; i += 2) {
                    const int n0 = 8 * (nh + 2 * i), n1 = 8 * (nh + 2 * i + 2);
                    uint32_t bv[4];
                    mma::ldsm4(bv, mma::smem_addr(mma::ldb_pair_ptr(Vns, kLdt, n0, n1, k0, lane)));
                    mma::mma_step<SPLIT>(aP[i], fo, __uint_as_float(bv[0]), __uint_as_float(bv[1]));
                    mma::mma_step<SPLIT>(aP[i + 1], fo, __uint_as_float(bv[2]),
                                         __uint_as_float(bv[3]));
                    if (erase) {
                        uint32_t bw[4];
                        mma::ldsm4(bw, mma::smem_addr(mma::ldb_pair_ptr(Vs, kLdt, n0, n1, k0,
                                                                         lane)));
                        mma::mma_step<SPLIT>(aT[i], fd, __uint_as_float(bw[0]),
                                             __uint_as_float(bw[1]));
                        mma::mma_step<SPLIT>(aT[i + 1], fd, __uint_as_float(bw[2]),
                                             __uint_as_float(bw[3]));
                    }
                }
            }
        }
        // dV = diag(beta) T^T dV' and the U part of dbeta
        {
            float acc[kNtV][4];
            mma::zero(acc);
            mma::gemm_s<kNtV, SPLIT>(acc, Tm, 1, kLdc, nullptr, dVs, kLdt, 1, m0, nh, 2, kDvt,
                                     kChunk, lane, m0);
            TIn *dvp = static_cast<TIn *>(b.dv);
            // the accumulator's adjacent column pairs, one store each
#pragma unroll
            for (int i = 0; i < kNtV; ++i) {
                const int cc = 8 * (nh + 2 * i) + 2 * tl;
                if (8 * (nh + 2 * i) < kDvt && cc < nv) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int s = m0 + gl + 8 * hr;
                        if (s < L)
                            st_out2(dvp + (r0 + s) * dv + dv0 + cc, bb[s] * acc[i][2 * hr],
                                    bb[s] * acc[i][2 * hr + 1]);
                    }
                }
            }
            add_row_sums(acc, m0, nh, 2, kDvt, lane,
                         [&](int s, int cc, float x) { return x * Vs[s * kLdt + cc]; }, dbU,
                         [](int) { return 1.f; });
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sC += __shfl_xor_sync(0xffffffffu, sC, o);
    __syncthreads();  // tiles consumed; B1 (A) no longer needed; Rg becomes Q
    if (lane == 0) red[warp] = sC;
    if (erase)
        mma::for_each(aW, m0, nh, 2, dk, lane,
                      [&](int m, int j, float &x) { Wm[m * ldk + j] = x; });
    mma::for_each(aP, m0, nh, 2, kChunk, lane, [&](int r, int s, float &x) {
        B1[r * kLdc + s] = s <= r ? x * expf(g[r] - g[s]) : 0.f;   // dP
    });
    if (erase)
        mma::for_each(aT, m0, nh, 2, kChunk, lane,
                      [&](int r, int s, float &x) { B2[r * kLdc + s] = s < r ? x * bb[s] : 0.f; });
    {
        TileRegs<4> rq;
        rq.load(qp + r0 * dk, dk, dk, L, dk, tid);
        rq.store(Qs, ldk, dk, tid);
    }
    __syncthreads();

    // ---- phase 3
    {   // E = dP * (Q K^T): row sums into dg_r, column sums out of dg_s
        float acc[kNtC][4];
        mma::zero(acc);
        mma::gemm_s<kNtC, SPLIT>(acc, Qs, ldk, 1, nullptr, Ks, 1, ldk, m0, nh, 2, m0 + 16, dk,
                                 lane);
        auto ev = [&](int r, int s, float x) { return B1[r * kLdc + s] * x; };
        add_row_sums(acc, m0, nh, 2, m0 + 16, lane, ev, dgE, [](int) { return 1.f; });
        add_col_sums(acc, m0, nh, 2, m0 + 16, lane, ev, dgE, -1.f);
    }
    float tmp[kNtK][4];
    {   // dQ = diag(gamma) dO S0 + dP K;  dg_r += gamma_r q_r . (dO S0)_r
        mma::zero(tmp);
        mma::gemm_s<kNtK, SPLIT>(tmp, B1, kLdc, 1, nullptr, Ks, ldk, 1, m0, nh, 2, dk, m0 + 16,
                                 lane);
        TIn *dqp = static_cast<TIn *>(b.dq);
#pragma unroll
        for (int i = 0; i < kNtK; ++i) {
            const int j = 8 * (nh + 2 * i) + 2 * tl;
            if (8 * (nh + 2 * i) < dk) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = m0 + gl + 8 * hr;
                    if (r < L)
                        st_out2(dqp + (r0 + r) * dk + j,
                                fmaf(gm[r], aQ[i][2 * hr], tmp[i][2 * hr]),
                                fmaf(gm[r], aQ[i][2 * hr + 1], tmp[i][2 * hr + 1]));
                }
            }
        }
        add_row_sums(aQ, m0, nh, 2, dk, lane,
                     [&](int r, int j, float x) { return Qs[r * ldk + j] * x; }, dgQ,
                     [&](int r) { return gm[r]; });
    }
    {   // dK = e_s (V' dSC)_s + (dP^T Q)_s + beta_s gamma_s (T^T dW)_s
        add_row_sums(aK, m0, nh, 2, dk, lane,
                     [&](int s, int j, float x) { return Ks[s * ldk + j] * x; }, Fv,
                     [&](int s) { return ed[s]; });
        mma::for_each(aK, m0, nh, 2, dk, lane, [&](int s, int, float &x) { x *= ed[s]; });
        mma::zero(tmp);
        mma::gemm_s<kNtK, SPLIT>(tmp, B1, 1, kLdc, nullptr, Qs, ldk, 1, m0, nh, 2, dk, kChunk,
                                 lane, m0);
#pragma unroll
        for (int i = 0; i < kNtK; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) aK[i][e] += tmp[i][e];
        if (erase) {
            mma::zero(tmp);
            mma::gemm_s<kNtK, SPLIT>(tmp, Tm, 1, kLdc, nullptr, Wm, ldk, 1, m0, nh, 2, dk, kChunk,
                                     lane, m0);
            // T^T dW = -tmp
            add_row_sums(tmp, m0, nh, 2, dk, lane,
                         [&](int s, int j, float x) { return -Ks[s * ldk + j] * x; }, tv,
                         [&](int s) { return gm[s]; });
            mma::for_each(tmp, m0, nh, 2, dk, lane, [&](int s, int, float &x) {
                x *= -bb[s] * gm[s];
            });
#pragma unroll
            for (int i = 0; i < kNtK; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) aK[i][e] += tmp[i][e];
        }
    }
    __syncthreads();  // B1 (dP) consumed
    if (erase) {
        {   // dT = dV'(diag(beta)V)^T - Wm (diag(beta gamma) K)^T, strictly lower part
            float acc[kNtC][4];
            mma::zero(acc);
            // strictly lower part only; B2 is already zero right of the diagonal
            mma::gemm_s<kNtC, SPLIT>(acc, Wm, ldk, 1, nullptr, Ks, 1, ldk, m0, nh, 2, m0 + 16, dk,
                                     lane);
            mma::for_each(acc, m0, nh, 2, m0 + 16, lane, [&](int r, int s, float &x) {
                B2[r * kLdc + s] = s < r ? B2[r * kLdc + s] - bb[s] * gm[s] * x : 0.f;
            });
        }
        __syncthreads();
        {   // Z = dT T^T  (B1)
            float acc[kNtC][4];
            mma::zero(acc);
            mma::gemm_s<kNtC, SPLIT>(acc, B2, kLdc, 1, nullptr, Tm, 1, kLdc, m0, nh, 2, kChunk,
                                     m0 + 16, lane);
            mma::for_each(acc, m0, nh, 2, kChunk, lane,
                          [&](int r, int s, float &x) { B1[r * kLdc + s] = x; });
        }
        __syncthreads();
        {   // X = dA * G with dA = -T^T Z (strictly lower), into B2; Y = X * K K^T
            float acc[kNtC][4];
            mma::zero(acc);
            // strictly lower part only; B2 (dT) is already zero right of the diagonal
            mma::gemm_s<kNtC, SPLIT>(acc, Tm, 1, kLdc, nullptr, B1, kLdc, 1, m0, nh, 2, m0 + 16,
                                     kChunk, lane, m0);
            mma::for_each(acc, m0, nh, 2, m0 + 16, lane, [&](int r, int s, float &x) {
                x = s < r ? -x * expf(g[r] - g[s]) : 0.f;
                B2[r * kLdc + s] = x;
            });
            auto yv = [&](int r, int s, float x) { return x * B3[r * kLdc + s]; };
            add_row_sums(acc, m0, nh, 2, m0 + 16, lane, yv, dbA, [](int) { return 1.f; });
            add_row_sums(acc, m0, nh, 2, m0 + 16, lane, yv, dgA, [&](int r) { return bb[r]; });
            add_col_sums(acc, m0, nh, 2, m0 + 16, lane,
                         [&](int r, int s, float x) { return bb[r] * x * B3[r * kLdc + s]; },
                         dgA, -1.f);
        }
        __syncthreads();
        {   // dK_r += beta_r (X K)_r + ((X * beta_row)^T K)_r
            mma::zero(tmp);
            mma::gemm_s<kNtK, SPLIT>(tmp, B2, kLdc, 1, nullptr, Ks, ldk, 1, m0, nh, 2, dk, m0 + 16,
                                     lane);
            mma::for_each(tmp, m0, nh, 2, dk, lane, [&](int r, int, float &x) { x *= bb[r]; });
#pragma unroll
            for (int i = 0; i < kNtK; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) aK[i][e] += tmp[i][e];
            mma::zero(tmp);
            mma::gemm_s<kNtK, SPLIT>(tmp, B2, 1, kLdc, bb, Ks, ldk, 1, m0, nh, 2, dk, kChunk,
                                     lane, m0);
#pragma unroll
            for (int i = 0; i < kNtK; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) aK[i][e] += tmp[i][e];
        }
    }
    {
        TIn *dkp = static_cast<TIn *>(b.dk);
#pragma unroll
        for (int i = 0; i < kNtK; ++i) {
            const int j = 8 * (nh + 2 * i) + 2 * tl;
            if (8 * (nh + 2 * i) < dk) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = m0 + gl + 8 * hr;
                    if (r < L) st_out2(dkp + (r0 + r) * dk + j, aK[i][2 * hr], aK[i][2 * hr + 1]);
                }
            }
        }
    }
    __syncthreads();
    // dg and dbeta per row; dlog_alpha is the reverse cumsum of dg
    if (tid < kChunk) {
        float x = dgE[tid] + dgQ[tid] - Fv[tid] + dgA[tid];
        if (erase) x = fmaf(bb[tid], tv[tid], x);
        dlv[tid] = x;
        if (tid < L) b.dbeta[r0 + tid] = dbU[tid] + dbA[tid] + (erase ? tv[tid] : 0.f);
    }
    __syncthreads();
    if (tid == 0) {
        float fs = 0.f, sc = 0.f;
        for (int s = 0; s < kChunk; ++s) fs += Fv[s];
        for (int w = 0; w < kThreads / 32; ++w) sc += red[w];
        float acc = fs + gm[L - 1] * sc;   // every place g_C enters
        for (int r = L - 1; r >= 0; --r) {
            acc += dlv[r];
            b.dlog_alpha[r0 + r] = acc;
        }
    }
}

template <typename TIn>
gdn_status launch_bwd(const FwdArgs &a, const BwdArgs &b, bool tc_dstate) {
    cudaStream_t st = a.stream;
    int *err = device_error_word();
    const size_t rows = (size_t)a.rows > 0 ? (size_t)a.rows : 1;
    const size_t states = (size_t)a.sm.H * (size_t)a.chunk_slots * a.dk * a.dv;
    const size_t dsm = dstate_smem(a.dk);
    const ChunkLay ly = chunk_lay(a.dk);
    constexpr bool kSplit = std::is_same<TIn, float>::value;   // fp32 I/O: 3xTF32
    if (cudaFuncSetAttribute(k_bwd_dstate<TIn, kSplit>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dsm) != cudaSuccess ||
        cudaFuncSetAttribute(k_bwd_chunk<TIn, kSplit>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ly.bytes) != cudaSuccess)
        return GDN_ERR_CUDA;
    float *W = nullptr, *U = nullptr, *G = nullptr, *Vn = nullptr, *dVn = nullptr;
    float *Hst = nullptr, *dHc = nullptr, *Tg = nullptr;
    // bf16 T diag(beta) [rows][64] then W [rows][d_k]: the tensor-core kernels' input
    __nv_bfloat16 *Tb = nullptr;
    int2 *table = nullptr;
    // with the erase term the tensor-core path's prep (gdn_prep.cu) gives
    // every input the tensor-core kernels and k_bwd_chunk read: no fp32 W, U
    const bool tc_prep = tc_dstate && !a.no_erase;
    float **bufs[] = {&W, &U, &G, &Vn, &dVn, &Hst, &dHc, &Tg};
    const size_t sizes[] = {rows * a.dk, rows * a.dv, rows, rows * a.dv, rows * a.dv,
                            states > 0 ? states : 1, states > 0 ? states : 1, rows * kChunk};
    gdn_status rc = GDN_OK;
    for (int i = tc_prep ? 2 : 0; i < 8 && rc == GDN_OK; ++i)
        if (scratch_alloc((void **)bufs[i], sizes[i] * sizeof(float), st) != cudaSuccess)
            rc = GDN_ERR_CUDA;
    if (rc == GDN_OK && tc_dstate &&
        scratch_alloc((void **)&Tb, rows * (kChunk + a.dk) * sizeof(__nv_bfloat16), st) !=
            cudaSuccess)
        rc = GDN_ERR_CUDA;
    __nv_bfloat16 *Wb = Tb ? Tb + rows * kChunk : nullptr;
    if (rc == GDN_OK && a.sm.cu && a.chunk_slots > 0) {
        if (scratch_alloc((void **)&table, sizeof(int2) * (size_t)a.chunk_slots, st) !=
            cudaSuccess)
            rc = GDN_ERR_CUDA;
        else
            rc = enqueue_chunk_table(a, table);
    }
    if (rc == GDN_OK)
        rc = tc_prep     ? enqueue_tc_prep_bwd(a, table, Tb, Wb, Tg, G)
             : tc_dstate ? enqueue_simt_prep_tc(a, table, W, U, G, Tg, Tb, Wb)
                         : enqueue_simt_prep(a, table, W, U, G, Tg);
    if (rc == GDN_OK) {
        FwdArgs f = a;
        f.o = nullptr;
        f.hT = nullptr;
        // the states and V' from the forward's fused kernel where the
        // tensor-core adjoint runs (the same bf16-operand products), else
        // from the general path's state pass
        rc = tc_dstate ? tc_state_pass(f, Tb, Hst, Vn) : enqueue_simt_state(f, W, U, G, Hst, Vn);
    }
    if (rc == GDN_OK && tc_dstate) {
        rc = tc_bwd_dstate(a, b, Wb, G, dVn, dHc);
    } else if (rc == GDN_OK && a.sm.N > 0 && a.sm.H > 0) {
        dim3 grid(a.sm.N, a.sm.H, (a.dv + kDvm - 1) / kDvm);
        k_bwd_dstate<TIn, kSplit><<<grid, kThreads, dsm, st>>>(a, b, W, G, dVn, dHc, err);
        count_launch();
    }
    if (rc == GDN_OK && a.chunk_slots > 0 && a.sm.H > 0) {
        const int slot = timer_begin(st, "k_bwd_chunk");
        k_bwd_chunk<TIn, kSplit><<<dim3(a.chunk_slots, a.sm.H), kThreads, ly.bytes, st>>>(
            a, b, table, Tg, Hst, dHc, Vn, dVn, err);
        timer_end(slot, st);
        count_launch();
    }
    if (rc == GDN_OK && cudaGetLastError() != cudaSuccess) rc = GDN_ERR_CUDA;
    for (float **p : bufs)
        if (*p) scratch_free(*p, st);
    if (Tb) scratch_free(Tb, st);
    if (table) scratch_free(table, st);
    return rc;
}

}  // namespace

gdn_status run_backward(const FwdArgs &a, const BwdArgs &b, long long impl, int *used) {
    if (a.vector_gate) return GDN_ERR_UNSUPPORTED;
    if (chunk_lay(a.dk).bytes > 227 * 1024 || dstate_smem(a.dk) > 227 * 1024)
        return GDN_ERR_UNSUPPORTED;
    const bool tc = impl != GDN_IMPL_SIMT && tc_bwd_supported(a) && tc_supported(a);
    if ((impl == GDN_IMPL_TC || impl == GDN_IMPL_TC_FUSED) && !tc) return GDN_ERR_UNSUPPORTED;
    const gdn_status rc = a.dt == GDN_F32 ? launch_bwd<float>(a, b, false)
                                          : launch_bwd<__nv_bfloat16>(a, b, tc);
    if (used) *used = tc ? GDN_IMPL_TC : GDN_IMPL_SIMT;
    return rc;
}

gdn_status simt_backward(const FwdArgs &a, const BwdArgs &b) {
    return run_backward(a, b, GDN_IMPL_SIMT, nullptr);
}

}  // namespace gdn
