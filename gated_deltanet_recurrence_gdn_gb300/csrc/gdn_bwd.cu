// gdn_bwd.cu -- backward pass of the chunked gated delta rule, CUDA cores,
// fp32 arithmetic.
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
// state adjoint backwards; k_bwd_chunk forms every gradient of one chunk.
// Without the erase term A = 0, T = I and W = 0, and the A and W terms drop.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kDvt = 32;     // d_v columns per tile
constexpr int kRegJ = 32;    // key columns a thread owns in k_bwd_chunk (d_k <= 128)

__device__ __forceinline__ float ld_in(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void set_error(int *err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ bool seq_ok(const SeqMap &sm, int n) {
    if (!sm.cu) return true;
    int a = __ldg(sm.cu + n), b = __ldg(sm.cu + n + 1);
    return a >= 0 && a <= b && b <= sm.T_total;
}

// ---------------------------------------------------------------- dS pass
//
// One CTA per (sequence, head, 32-wide d_v tile), chunks in reverse order.
// dH = dS^T (d_k x 32) lives in shared memory.  For each chunk it stores
// dH (the adjoint of the chunk's end state) as [H][chunk_slots][d_k][d_v]
// and the rows of dV', then steps dH back to the chunk's start.

size_t dstate_smem(int dk) {
    return sizeof(float) * ((size_t)dk * kDvt + 3 * (size_t)kChunk * (dk + 1) +
                            2 * kChunk * (kDvt + 1) + kChunk * 65 + 3 * kChunk);
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads)
k_bwd_dstate(FwdArgs a, BwdArgs b, const float *__restrict__ W, const float *__restrict__ G,
             float *__restrict__ dVn, float *__restrict__ dHc, int *err) {
    extern __shared__ float smem[];
    const int dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int n = blockIdx.x, h = blockIdx.y, dv0 = blockIdx.z * kDvt;
    const int nv = min(kDvt, dv - dv0);
    if (!seq_ok(a.sm, n)) {
        if (tid == 0) set_error(err, kErrBadIndex);
        return;
    }
    long long row0;
    int len;
    a.sm.get(n, h, row0, len);
    const int ks = dk + 1, us = kDvt + 1;
    float *dH = smem;                    // [dk][32]
    float *Ks = dH + dk * kDvt;          // [64][dk+1]
    float *Qs = Ks + kChunk * ks;        // [64][dk+1]
    float *Ws = Qs + kChunk * ks;        // [64][dk+1]
    float *dOs = Ws + kChunk * ks;       // [64][33]
    float *dVs = dOs + kChunk * us;      // [64][33]
    float *P = dVs + kChunk * us;        // [64][65]  P_rs = G_rs q_r . k_s, s <= r
    float *g = P + kChunk * 65;          // [64]
    float *e = g + kChunk;               // [64] exp(g_C - g_r)
    float *gm = e + kChunk;              // [64] exp(g_r)
    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *dop = static_cast<const TIn *>(b.dout);
    const long long sbase = ((long long)n * a.sm.H + h) * dv;

    for (int i = tid; i < dk * kDvt; i += kThreads) {
        const int j = i / kDvt, cc = i - j * kDvt;
        dH[i] = (b.dhT && cc < nv) ? __ldg(b.dhT + (sbase + dv0 + cc) * dk + j) : 0.f;
    }
    const int nch = (len + kChunk - 1) / kChunk;
    for (int c = nch - 1; c >= 0; --c) {
        const int t0 = c * kChunk, L = min(kChunk, len - t0);
        const long long r0 = row0 + t0;
        __syncthreads();  // the previous (later) chunk is fully consumed
        float *dst = dHc + ((long long)h * a.chunk_slots + a.chunk_slot(n, c)) * dk * dv;
        for (int i = tid; i < dk * kDvt; i += kThreads) {
            const int j = i / kDvt, cc = i - j * kDvt;
            if (cc < nv) dst[(long long)j * dv + dv0 + cc] = dH[i];
        }
        for (int i = tid; i < kChunk * dk; i += kThreads) {
            const int r = i / dk, j = i - r * dk;
            const bool ok = r < L;
            Ks[r * ks + j] = ok ? ld_in(kp + (r0 + r) * dk + j) : 0.f;
            Qs[r * ks + j] = ok ? ld_in(qp + (r0 + r) * dk + j) : 0.f;
            Ws[r * ks + j] = ok ? __ldg(W + (r0 + r) * dk + j) : 0.f;
        }
        for (int i = tid; i < kChunk * kDvt; i += kThreads) {
            const int r = i / kDvt, cc = i - r * kDvt;
            dOs[r * us + cc] = (r < L && cc < nv) ? ld_in(dop + (r0 + r) * dv + dv0 + cc) : 0.f;
        }
        if (tid < kChunk) g[tid] = __ldg(G + r0 + min(tid, L - 1));
        __syncthreads();
        const float gl = g[kChunk - 1];
        if (tid < kChunk) {
            e[tid] = expf(gl - g[tid]);
            gm[tid] = expf(g[tid]);
        }
        for (int i = tid; i < kChunk * kChunk; i += kThreads) {
            const int r = i >> 6, s = i & 63;
            float val = 0.f;
            if (s <= r) {
                float acc = 0.f;
                for (int j = 0; j < dk; ++j) acc = fmaf(Qs[r * ks + j], Ks[s * ks + j], acc);
                val = expf(g[r] - g[s]) * acc;
            }
            P[r * 65 + s] = val;
        }
        __syncthreads();
        // dV'_r = sum_{s >= r} P_sr dO_s + e_r dS k_r
        for (int i = tid; i < kChunk * kDvt; i += kThreads) {
            const int r = i / kDvt, cc = i - r * kDvt;
            float a1 = 0.f, a2 = 0.f;
            for (int s = r; s < kChunk; ++s) a1 = fmaf(P[s * 65 + r], dOs[s * us + cc], a1);
            for (int j = 0; j < dk; ++j) a2 = fmaf(Ks[r * ks + j], dH[j * kDvt + cc], a2);
            const float val = r < L ? fmaf(e[r], a2, a1) : 0.f;
            dVs[r * us + cc] = val;
            if (r < L && cc < nv) dVn[(r0 + r) * dv + dv0 + cc] = val;
        }
        __syncthreads();
        // dS <- gamma_C dS + dO^T diag(gamma) Q - dV'^T W   (as dH = dS^T)
        const float decay = expf(gl);
        for (int i = tid; i < dk * kDvt; i += kThreads) {
            const int j = i / kDvt, cc = i - j * kDvt;
            float acc = 0.f;
            for (int r = 0; r < kChunk; ++r) {
                acc = fmaf(gm[r] * Qs[r * ks + j], dOs[r * us + cc], acc);
                acc = fmaf(-Ws[r * ks + j], dVs[r * us + cc], acc);
            }
            dH[i] = fmaf(decay, dH[i], acc);
        }
    }
    __syncthreads();
    if (b.dh0) {
        for (int i = tid; i < dk * kDvt; i += kThreads) {
            const int j = i / kDvt, cc = i - j * kDvt;
            if (cc < nv) b.dh0[(sbase + dv0 + cc) * dk + j] = dH[i];
        }
    }
}

// ------------------------------------------------------------ chunk kernel
//
// One CTA per (chunk, head).  Phase 1 rebuilds A and T from K, beta and the
// gates.  Phase 2 walks d_v in 32-wide tiles and accumulates the d_v
// contractions: dO S0 and V' dSC in registers (thread (r, j mod 4) owns
// row r, key columns j = j0 + 4m), dV' S0 in shared memory, dO V'^T and
// dV' (diag(beta) V)^T as C x C tiles; it also writes dV and collects the
// U part of dbeta.  Phase 3 forms dQ, dK, dbeta and dlog_alpha.

struct ChunkLay {
    int ks, region;
    int oK, oR, oWm, oT, oB1, oB2, oB3, oV;
    size_t bytes;
};

__host__ __device__ inline ChunkLay chunk_lay(int dk) {
    ChunkLay l;
    l.ks = dk + 1;
    const int tiles = 4 * kChunk * (kDvt + 1) + 2 * dk * (kDvt + 1);
    const int qsz = kChunk * l.ks;
    l.region = tiles > qsz ? tiles : qsz;
    l.oK = 0;
    l.oR = l.oK + kChunk * l.ks;
    l.oWm = l.oR + l.region;
    l.oT = l.oWm + kChunk * l.ks;
    l.oB1 = l.oT + kChunk * 65;
    l.oB2 = l.oB1 + kChunk * 65;
    l.oB3 = l.oB2 + kChunk * 65;
    l.oV = l.oB3 + kChunk * 65;
    l.bytes = sizeof(float) * ((size_t)l.oV + 12 * kChunk + 32);
    return l;
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
k_bwd_chunk(FwdArgs a, BwdArgs b, const int2 *__restrict__ table, const float *__restrict__ Hst,
            const float *__restrict__ dHc, const float *__restrict__ Vn,
            const float *__restrict__ dVn, int *err) {
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
    const int ks = ly.ks, us = kDvt + 1;
    float *Ks = smem + ly.oK;     // [64][dk+1]
    float *Rg = smem + ly.oR;     // phase 2 tiles, then Q
    float *Wm = smem + ly.oWm;    // [64][dk+1]  dV' S0 (= -dW)
    float *Tm = smem + ly.oT;     // [64][65]    T
    float *B1 = smem + ly.oB1;    // [64][65]    dO V'^T, then dP, then dT T^T
    float *B2 = smem + ly.oB2;    // [64][65]    dV'(diag(beta)V)^T, then dT, then dA
    float *B3 = smem + ly.oB3;    // [64][65]    A, then dP * (Q K^T), then dA * G * K K^T
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
    // phase 2 tiles
    float *dOs = Rg;                       // [64][33]
    float *Vns = dOs + kChunk * us;        // [64][33]  V'
    float *dVs = Vns + kChunk * us;        // [64][33]  dV'
    float *Vs = dVs + kChunk * us;         // [64][33]  V
    float *S0t = Vs + kChunk * us;         // [dk][33]  S0^T tile
    float *dSt = S0t + dk * us;            // [dk][33]  dSC^T tile
    float *Qs = Rg;                        // phase 3: [64][dk+1]

    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *vp = static_cast<const TIn *>(a.v);
    const TIn *dop = static_cast<const TIn *>(b.dout);

    // ---- phase 1: K, gates, A, T
    for (int i = tid; i < kChunk * dk; i += kThreads) {
        const int r = i / dk, j = i - r * dk;
        Ks[r * ks + j] = r < L ? ld_in(kp + (r0 + r) * dk + j) : 0.f;
        Wm[r * ks + j] = 0.f;
    }
    if (tid < kChunk) {
        const bool ok = tid < L;
        g[tid] = ok ? __ldg(a.log_alpha + r0 + tid) : 0.f;
        bb[tid] = ok ? __ldg(a.beta + r0 + tid) : 0.f;
        dbU[tid] = 0.f;
    }
    for (int i = tid; i < kChunk * 65; i += kThreads) {
        B1[i] = 0.f;
        B2[i] = 0.f;
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
    const float gC = g[L - 1];
    if (tid < kChunk) {
        gm[tid] = expf(g[tid]);
        ed[tid] = expf(gC - g[tid]);
    }
    for (int i = tid; i < kChunk * kChunk; i += kThreads) {
        const int r = i >> 6, s = i & 63;
        float val = 0.f;
        if (s < r && erase) {
            float acc = 0.f;
            for (int j = 0; j < dk; ++j) acc = fmaf(Ks[r * ks + j], Ks[s * ks + j], acc);
            val = bb[r] * expf(g[r] - g[s]) * acc;
        }
        B3[r * 65 + s] = val;
    }
    __syncthreads();
    if (tid < kChunk) {  // column tid of T = (I + A)^{-1}
        const int cc = tid;
        for (int r = 0; r <= cc; ++r) Tm[r * 65 + cc] = (r == cc) ? 1.f : 0.f;
        for (int r = cc + 1; r < kChunk; ++r) {
            float acc = 0.f;
            for (int s = cc; s < r; ++s) acc = fmaf(B3[r * 65 + s], Tm[s * 65 + cc], acc);
            Tm[r * 65 + cc] = -acc;
        }
    }

    // ---- phase 2: the d_v contractions, tile by tile
    const int rr = tid >> 2, jq = tid & 3;
    float aQ[kRegJ], aK[kRegJ];
#pragma unroll
    for (int m = 0; m < kRegJ; ++m) {
        aQ[m] = 0.f;
        aK[m] = 0.f;
    }
    float sC = 0.f;
    for (int dv0 = 0; dv0 < dv; dv0 += kDvt) {
        const int nv = min(kDvt, dv - dv0);
        __syncthreads();  // T ready / the previous tile consumed
        for (int i = tid; i < kChunk * kDvt; i += kThreads) {
            const int r = i / kDvt, cc = i - r * kDvt;
            const bool ok = r < L && cc < nv;
            const long long o = (r0 + r) * dv + dv0 + cc;
            dOs[r * us + cc] = ok ? ld_in(dop + o) : 0.f;
            Vns[r * us + cc] = ok ? __ldg(Vn + o) : 0.f;
            dVs[r * us + cc] = ok ? __ldg(dVn + o) : 0.f;
            Vs[r * us + cc] = ok ? ld_in(vp + o) : 0.f;
        }
        for (int i = tid; i < dk * kDvt; i += kThreads) {
            const int j = i / kDvt, cc = i - j * kDvt;
            const bool ok = cc < nv;
            const long long o = st_off + (long long)j * dv + dv0 + cc;
            const float s0 = ok ? __ldg(Hst + o) : 0.f;
            const float ds = ok ? __ldg(dHc + o) : 0.f;
            S0t[j * us + cc] = s0;
            dSt[j * us + cc] = ds;
            sC = fmaf(s0, ds, sC);
        }
        __syncthreads();
        // dO S0 and V' dSC (registers), dV' S0 (shared, thread-owned elements)
#pragma unroll
        for (int m = 0; m < kRegJ; ++m) {
            const int j = jq + 4 * m;
            if (j < dk) {
                float q1 = 0.f, k1 = 0.f, w1 = 0.f;
                #pragma unroll 4
                for (int cc = 0; cc < kDvt; ++cc) {
                    const float s0 = S0t[j * us + cc];
                    q1 = fmaf(dOs[rr * us + cc], s0, q1);
                    k1 = fmaf(Vns[rr * us + cc], dSt[j * us + cc], k1);
                    if (erase) w1 = fmaf(dVs[rr * us + cc], s0, w1);
                }
                aQ[m] += q1;
                aK[m] += k1;
                if (erase) Wm[rr * ks + j] += w1;
            }
        }
        // dO V'^T and dV' (diag(beta) V)^T
        for (int i = tid; i < kChunk * kChunk; i += kThreads) {
            const int r = i >> 6, s = i & 63;
            float p1 = 0.f, p2 = 0.f;
            for (int cc = 0; cc < kDvt; ++cc) {
                p1 = fmaf(dOs[r * us + cc], Vns[s * us + cc], p1);
                if (erase) p2 = fmaf(dVs[r * us + cc], Vs[s * us + cc], p2);
            }
            B1[r * 65 + s] += p1;
            if (erase) B2[r * 65 + s] += bb[s] * p2;
        }
        // dV = diag(beta) T^T dV'  and the U part of dbeta (one warp per row s)
        for (int i = tid; i < kChunk * kDvt; i += kThreads) {
            const int s = i / kDvt, cc = i - s * kDvt;
            float acc = 0.f;
            for (int r = s; r < kChunk; ++r) acc = fmaf(Tm[r * 65 + s], dVs[r * us + cc], acc);
            if (s < L && cc < nv)
                st_out(static_cast<TIn *>(b.dv) + (r0 + s) * dv + dv0 + cc, bb[s] * acc);
            float x = acc * Vs[s * us + cc];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (lane == 0) dbU[s] += x;
        }
    }
    // <dSC, S0> over the block
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sC += __shfl_xor_sync(0xffffffffu, sC, o);
    __syncthreads();  // tiles consumed; Rg becomes Q
    if (lane == 0) red[warp] = sC;
    for (int i = tid; i < kChunk * dk; i += kThreads) {
        const int r = i / dk, j = i - r * dk;
        Qs[r * ks + j] = r < L ? ld_in(qp + (r0 + r) * dk + j) : 0.f;
    }
    __syncthreads();

    // ---- phase 3
    // dP = mask * G * (dO V'^T) in B1; E = dP * (Q K^T) in B3
    for (int i = tid; i < kChunk * kChunk; i += kThreads) {
        const int r = i >> 6, s = i & 63;
        float dp = 0.f, ev = 0.f;
        if (s <= r) {
            dp = B1[r * 65 + s] * expf(g[r] - g[s]);
            float acc = 0.f;
            for (int j = 0; j < dk; ++j) acc = fmaf(Qs[r * ks + j], Ks[s * ks + j], acc);
            ev = dp * acc;
        }
        B1[r * 65 + s] = dp;
        B3[r * 65 + s] = ev;
    }
    __syncthreads();
    if (tid < kChunk) {
        float x = 0.f;
        for (int s = 0; s < kChunk; ++s) x += B3[tid * 65 + s] - B3[s * 65 + tid];
        dgE[tid] = x;
    }
    // dQ = diag(gamma) dO S0 + dP K;  dg_r += gamma_r q_r . (dO S0)_r
    {
        float part = 0.f;
#pragma unroll
        for (int m = 0; m < kRegJ; ++m) {
            const int j = jq + 4 * m;
            if (j < dk) {
                float acc = 0.f;
                #pragma unroll 4
                for (int s = 0; s <= rr; ++s) acc = fmaf(B1[rr * 65 + s], Ks[s * ks + j], acc);
                part = fmaf(Qs[rr * ks + j], aQ[m], part);
                if (rr < L)
                    st_out(static_cast<TIn *>(b.dq) + (r0 + rr) * dk + j,
                           fmaf(gm[rr], aQ[m], acc));
            }
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (jq == 0) dgQ[rr] = gm[rr] * part;
    }
    // dK (registers aK, row s = rr) = e_s (V' dSC)_s + (dP^T Q)_s + beta_s gamma_s (T^T dW)_s
    {
        float fpart = 0.f, tpart = 0.f;
#pragma unroll
        for (int m = 0; m < kRegJ; ++m) {
            const int j = jq + 4 * m;
            if (j < dk) {
                const float kd = aK[m];
                fpart = fmaf(Ks[rr * ks + j], kd, fpart);
                float acc = ed[rr] * kd;
                #pragma unroll 4
                for (int r = rr; r < kChunk; ++r) acc = fmaf(B1[r * 65 + rr], Qs[r * ks + j], acc);
                if (erase) {
                    float tw = 0.f;   // (T^T dW)_sj = -sum_r T_rs Wm_rj
                    #pragma unroll 4
                    for (int r = rr; r < kChunk; ++r) tw = fmaf(-Tm[r * 65 + rr], Wm[r * ks + j], tw);
                    acc = fmaf(bb[rr] * gm[rr], tw, acc);
                    tpart = fmaf(Ks[rr * ks + j], tw, tpart);
                }
                aK[m] = acc;
            }
        }
        fpart += __shfl_xor_sync(0xffffffffu, fpart, 1);
        fpart += __shfl_xor_sync(0xffffffffu, fpart, 2);
        tpart += __shfl_xor_sync(0xffffffffu, tpart, 1);
        tpart += __shfl_xor_sync(0xffffffffu, tpart, 2);
        if (jq == 0) {
            Fv[rr] = ed[rr] * fpart;
            tv[rr] = gm[rr] * tpart;
        }
    }
    if (tid < kChunk) {
        dgA[tid] = 0.f;
        dbA[tid] = 0.f;
    }
    __syncthreads();  // B1 (dP) and B3 (E) consumed
    if (erase) {
        // dT = dV'(diag(beta)V)^T - Wm (diag(beta gamma) K)^T, strictly lower part
        for (int i = tid; i < kChunk * kChunk; i += kThreads) {
            const int r = i >> 6, s = i & 63;
            float val = 0.f;
            if (s < r) {
                float acc = 0.f;
                for (int j = 0; j < dk; ++j) acc = fmaf(Wm[r * ks + j], Ks[s * ks + j], acc);
                val = B2[r * 65 + s] - bb[s] * gm[s] * acc;
            }
            B2[r * 65 + s] = val;
        }
        __syncthreads();
        // Z = dT T^T  (B1)
        for (int i = tid; i < kChunk * kChunk; i += kThreads) {
            const int r = i >> 6, s = i & 63;
            float acc = 0.f;
            const int mmax = min(r - 1, s);
            for (int m = 0; m <= mmax; ++m) acc = fmaf(B2[r * 65 + m], Tm[s * 65 + m], acc);
            B1[r * 65 + s] = acc;
        }
        __syncthreads();
        // dA = -T^T Z, strictly lower, times G  (B2);  B3 = that times K K^T
        for (int i = tid; i < kChunk * kChunk; i += kThreads) {
            const int r = i >> 6, s = i & 63;
            float x = 0.f, y = 0.f;
            if (s < r) {
                float acc = 0.f;
                for (int m = r; m < kChunk; ++m) acc = fmaf(Tm[m * 65 + r], B1[m * 65 + s], acc);
                x = -acc * expf(g[r] - g[s]);
                float kk = 0.f;
                for (int j = 0; j < dk; ++j) kk = fmaf(Ks[r * ks + j], Ks[s * ks + j], kk);
                y = x * kk;
            }
            B2[r * 65 + s] = x;
            B3[r * 65 + s] = y;
        }
        __syncthreads();
        if (tid < kChunk) {
            float row = 0.f, col = 0.f;
            for (int s = 0; s < kChunk; ++s) {
                row += B3[tid * 65 + s];
                col += bb[s] * B3[s * 65 + tid];
            }
            dbA[tid] = row;
            dgA[tid] = bb[tid] * row - col;
        }
        // dK_r += beta_r sum_s X_rs k_s + sum_r' X_r'r beta_r' k_r'
#pragma unroll
        for (int m = 0; m < kRegJ; ++m) {
            const int j = jq + 4 * m;
            if (j < dk) {
                float a1 = 0.f, a2 = 0.f;
                #pragma unroll 4
                for (int s = 0; s < rr; ++s) a1 = fmaf(B2[rr * 65 + s], Ks[s * ks + j], a1);
                #pragma unroll 4
                for (int r = rr + 1; r < kChunk; ++r)
                    a2 = fmaf(B2[r * 65 + rr] * bb[r], Ks[r * ks + j], a2);
                aK[m] += fmaf(bb[rr], a1, a2);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kRegJ; ++m) {
        const int j = jq + 4 * m;
        if (j < dk && rr < L) st_out(static_cast<TIn *>(b.dk) + (r0 + rr) * dk + j, aK[m]);
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
gdn_status launch_bwd(const FwdArgs &a, const BwdArgs &b) {
    cudaStream_t st = a.stream;
    int *err = device_error_word();
    const size_t rows = (size_t)a.rows > 0 ? (size_t)a.rows : 1;
    const size_t states = (size_t)a.sm.H * (size_t)a.chunk_slots * a.dk * a.dv;
    const size_t dsm = dstate_smem(a.dk);
    const ChunkLay ly = chunk_lay(a.dk);
    if (cudaFuncSetAttribute(k_bwd_dstate<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dsm) != cudaSuccess ||
        cudaFuncSetAttribute(k_bwd_chunk<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ly.bytes) != cudaSuccess)
        return GDN_ERR_CUDA;
    float *W = nullptr, *U = nullptr, *G = nullptr, *Vn = nullptr, *dVn = nullptr;
    float *Hst = nullptr, *dHc = nullptr;
    int2 *table = nullptr;
    float **bufs[] = {&W, &U, &G, &Vn, &dVn, &Hst, &dHc};
    const size_t sizes[] = {rows * a.dk, rows * a.dv, rows, rows * a.dv, rows * a.dv,
                            states > 0 ? states : 1, states > 0 ? states : 1};
    gdn_status rc = GDN_OK;
    for (int i = 0; i < 7 && rc == GDN_OK; ++i)
        if (scratch_alloc((void **)bufs[i], sizes[i] * sizeof(float), st) != cudaSuccess)
            rc = GDN_ERR_CUDA;
    if (rc == GDN_OK && a.sm.cu && a.chunk_slots > 0) {
        if (scratch_alloc((void **)&table, sizeof(int2) * (size_t)a.chunk_slots, st) !=
            cudaSuccess)
            rc = GDN_ERR_CUDA;
        else
            rc = enqueue_chunk_table(a, table);
    }
    if (rc == GDN_OK) rc = enqueue_simt_prep(a, table, W, U, G);
    if (rc == GDN_OK) {
        FwdArgs f = a;
        f.o = nullptr;
        f.hT = nullptr;
        rc = enqueue_simt_state(f, W, U, G, Hst, Vn);
    }
    if (rc == GDN_OK && a.sm.N > 0 && a.sm.H > 0) {
        dim3 grid(a.sm.N, a.sm.H, (a.dv + kDvt - 1) / kDvt);
        k_bwd_dstate<TIn><<<grid, kThreads, dsm, st>>>(a, b, W, G, dVn, dHc, err);
        count_launch();
    }
    if (rc == GDN_OK && a.chunk_slots > 0 && a.sm.H > 0) {
        const int slot = timer_begin(st, "k_bwd_chunk");
        k_bwd_chunk<TIn><<<dim3(a.chunk_slots, a.sm.H), kThreads, ly.bytes, st>>>(
            a, b, table, Hst, dHc, Vn, dVn, err);
        timer_end(slot, st);
        count_launch();
    }
    if (rc == GDN_OK && cudaGetLastError() != cudaSuccess) rc = GDN_ERR_CUDA;
    for (float **p : bufs)
        if (*p) scratch_free(*p, st);
    if (table) scratch_free(table, st);
    return rc;
}

}  // namespace

gdn_status simt_backward(const FwdArgs &a, const BwdArgs &b) {
    if (a.vector_gate) return GDN_ERR_UNSUPPORTED;
    if (chunk_lay(a.dk).bytes > 227 * 1024 || dstate_smem(a.dk) > 227 * 1024)
        return GDN_ERR_UNSUPPORTED;
    return a.dt == GDN_F32 ? launch_bwd<float>(a, b) : launch_bwd<__nv_bfloat16>(a, b);
}

}  // namespace gdn
