// gdn_host.cu -- the forward pass on HOST buffers: host -> device copies, the
// device forward pass and device -> host copies, pipelined over time slices.
//
// The recurrence passes only the d_v x d_k state from one chunk to the next
// ("Gated DeltaNet GPU并行实现", section 3.2), so a dense batch can be cut
// along T into chunk-aligned slices that run one after another with the fp32
// state handed over in device memory: slice i's inputs go up while slice i-1
// is computed and slice i-2's outputs come down.  The copies of a slice are
// 2-D (one row per (batch, head), pitch T * d on the host), the device slice
// is a dense [B][H][T_slice][d] batch, and each slice is one gdn_fwd call on
// it.  With page-locked host buffers the three engines overlap and the call
// is bound by the host link; pageable buffers work but do not overlap.
#include <cstdint>
#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kSets = 3;             // device slice buffers in flight
constexpr int kSliceTarget = 512;    // tokens per slice (a multiple of the chunk)
constexpr int kMaxSlices = 32;
constexpr int kMaxDev = 64;

struct HostStreams {
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
};
std::mutex g_hs_mu;
HostStreams g_hs[kMaxDev];

cudaError_t host_streams(HostStreams *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_hs_mu);
    HostStreams &h = g_hs[dev];
    if (!h.in) {
        cudaStream_t s[3] = {};
        for (int i = 0; i < 3; ++i)
            if ((e = cudaStreamCreateWithFlags(&s[i], cudaStreamNonBlocking)) != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaStreamDestroy(s[j]);
                return e;
            }
        h.in = s[0];
        h.comp = s[1];
        h.out = s[2];
    }
    *out = h;
    return cudaSuccess;
}

// rows x width bytes between pitched buffers (a no-op for empty copies)
cudaError_t copy2d(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                   size_t rows, cudaMemcpyKind kind, cudaStream_t st) {
    if (width == 0 || rows == 0) return cudaSuccess;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, st);
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_fwd_host(const void *q, const void *k, const void *v,
                                   const float *log_alpha, const float *beta, const float *h0,
                                   void *o, float *hT, int B, int H, int T, int d_k, int d_v,
                                   int chunk, gdn_dtype dt, void *stream) {
    using namespace gdn;
    if (B < 0 || H < 0 || T < 0 || d_k <= 0 || d_v <= 0) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (chunk != kChunk) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H == 0) return GDN_OK;
    if (T > 0 && (!q || !k || !v || !log_alpha || !beta || !o)) return GDN_ERR_INVALID_ARG;
    const long long BH = (long long)B * H;
    const size_t es = dt == GDN_BF16 ? 2 : 4;
    // slices: chunk-aligned lengths, the last one possibly shorter
    const long long opt_slice = option(GDN_OPT_HOST_SLICE);
    const int target = opt_slice > 0 ? (int)((opt_slice + kChunk - 1) / kChunk * kChunk) : kSliceTarget;
    int S = T == 0 ? 1 : (T + target - 1) / target;
    S = S < 1 ? 1 : (S > kMaxSlices ? kMaxSlices : S);
    const int Ts = T == 0 ? 0 : ((T + S - 1) / S + kChunk - 1) / kChunk * kChunk;
    S = T == 0 ? 1 : (T + Ts - 1) / Ts;
    const int R = S < kSets ? S : kSets;

    HostStreams hs;
    if (host_streams(&hs) != cudaSuccess) return GDN_ERR_CUDA;
    cudaStream_t ust = static_cast<cudaStream_t>(stream);

    // device buffers: R slice sets and two state buffers (ping-pong)
    const size_t nq = (size_t)BH * Ts * d_k * es, nv = (size_t)BH * Ts * d_v * es;
    const size_t ng = (size_t)BH * Ts * sizeof(float), nst = (size_t)BH * d_v * d_k * sizeof(float);
    const size_t set_bytes = 2 * nq + 2 * nv + 2 * ng;
    uint8_t *sets = nullptr;
    float *state = nullptr;
    if (scratch_alloc((void **)&sets, set_bytes * R + 16, ust) != cudaSuccess) return GDN_ERR_CUDA;
    if (scratch_alloc((void **)&state, 2 * nst, ust) != cudaSuccess) {
        scratch_free(sets, ust);
        return GDN_ERR_CUDA;
    }
    auto dq = [&](int i) { return sets + (size_t)(i % R) * set_bytes; };
    auto dk_ = [&](int i) { return dq(i) + nq; };
    auto dv_ = [&](int i) { return dq(i) + 2 * nq; };
    auto do_ = [&](int i) { return dq(i) + 2 * nq + nv; };
    auto dla = [&](int i) { return reinterpret_cast<float *>(dq(i) + 2 * nq + 2 * nv); };
    auto dbe = [&](int i) { return reinterpret_cast<float *>(dq(i) + 2 * nq + 2 * nv + ng); };

    // events: start, end, and per slice inputs-landed / computed / outputs-read
    cudaEvent_t ev[2 + 3 * kMaxSlices] = {};
    const int n_ev = 2 + 3 * S;
    bool ok = true;
    for (int i = 0; i < n_ev && ok; ++i)
        ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    cudaEvent_t ev_start = ev[0], ev_end = ev[1];
    cudaEvent_t *ev_in = ev + 2, *ev_comp = ev + 2 + S, *ev_out = ev + 2 + 2 * S;
    gdn_status rc = ok ? GDN_OK : GDN_ERR_CUDA;
    auto chk = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == GDN_OK) rc = GDN_ERR_CUDA;
        return rc == GDN_OK;
    };

    // every internal stream starts after the caller's stream (and the allocations)
    if (rc == GDN_OK) {
        chk(cudaEventRecord(ev_start, ust));
        chk(cudaStreamWaitEvent(hs.in, ev_start, 0));
        chk(cudaStreamWaitEvent(hs.comp, ev_start, 0));
        chk(cudaStreamWaitEvent(hs.out, ev_start, 0));
    }
    if (rc == GDN_OK && h0)
        chk(cudaMemcpyAsync(state, h0, nst, cudaMemcpyHostToDevice, hs.in));
    for (int i = 0; i < S && rc == GDN_OK; ++i) {
        const int t0 = i * Ts, L = (T - t0) < Ts ? (T - t0) : Ts;
        // inputs of slice i, once slice i - R has released its set
        if (i >= R) {
            chk(cudaStreamWaitEvent(hs.in, ev_comp[i - R], 0));
            chk(cudaStreamWaitEvent(hs.in, ev_out[i - R], 0));
        }
        const size_t rq = (size_t)d_k * es, rv = (size_t)d_v * es;
        chk(copy2d(dq(i), L * rq, static_cast<const uint8_t *>(q) + (size_t)t0 * rq, (size_t)T * rq,
                   L * rq, BH, cudaMemcpyHostToDevice, hs.in));
        chk(copy2d(dk_(i), L * rq, static_cast<const uint8_t *>(k) + (size_t)t0 * rq,
                   (size_t)T * rq, L * rq, BH, cudaMemcpyHostToDevice, hs.in));
        chk(copy2d(dv_(i), L * rv, static_cast<const uint8_t *>(v) + (size_t)t0 * rv,
                   (size_t)T * rv, L * rv, BH, cudaMemcpyHostToDevice, hs.in));
        chk(copy2d(dla(i), L * 4, log_alpha + t0, (size_t)T * 4, L * 4, BH,
                   cudaMemcpyHostToDevice, hs.in));
        chk(copy2d(dbe(i), L * 4, beta + t0, (size_t)T * 4, L * 4, BH, cudaMemcpyHostToDevice,
                   hs.in));
        chk(cudaEventRecord(ev_in[i], hs.in));
        // compute: state[i % 2] -> state[(i + 1) % 2]
        chk(cudaStreamWaitEvent(hs.comp, ev_in[i], 0));
        if (rc != GDN_OK) break;
        const float *s_in = (i == 0 && !h0) ? nullptr : state + (size_t)(i & 1) * (nst / 4);
        float *s_out = state + (size_t)((i + 1) & 1) * (nst / 4);
        const gdn_status fr = gdn_fwd(dq(i), dk_(i), dv_(i), dla(i), dbe(i), s_in, do_(i), s_out,
                                      B, H, L, d_k, d_v, chunk, dt, hs.comp);
        if (fr != GDN_OK) {
            rc = fr;
            break;
        }
        chk(cudaEventRecord(ev_comp[i], hs.comp));
        // outputs of slice i
        chk(cudaStreamWaitEvent(hs.out, ev_comp[i], 0));
        chk(copy2d(static_cast<uint8_t *>(o) + (size_t)t0 * rv, (size_t)T * rv, do_(i), L * rv,
                   L * rv, BH, cudaMemcpyDeviceToHost, hs.out));
        chk(cudaEventRecord(ev_out[i], hs.out));
    }
    if (rc == GDN_OK && hT)
        chk(cudaMemcpyAsync(hT, state + (size_t)(S & 1) * (nst / 4), nst, cudaMemcpyDeviceToHost,
                            hs.out));
    // the caller's stream resumes after all three internal streams (after an
    // error, copies or kernels already queued on any of them may still use the
    // buffers); the buffers then go back to the pool in its order, and the
    // internal streams' next work comes after it
    if (ok) {
        const cudaStream_t internal[3] = {hs.in, hs.comp, hs.out};
        for (cudaStream_t s2 : internal) {
            cudaEventRecord(ev_end, s2);
            cudaStreamWaitEvent(ust, ev_end, 0);
        }
        cudaEventRecord(ev_end, ust);
        for (cudaStream_t s2 : internal) cudaStreamWaitEvent(s2, ev_end, 0);
    }
    scratch_free(sets, ust);
    scratch_free(state, ust);
    for (int i = 0; i < n_ev; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
    return rc;
}
