// gdn_api.cu -- the C ABI of libgdn: argument checks, dispatch, error word.
#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "gdn_bwd_tc.h"
#include "gdn_internal.h"

namespace gdn {

namespace {
__device__ int g_error_word = 0;

std::atomic<uint64_t> g_launches{0};
std::atomic<long long> g_opt_impl{GDN_IMPL_AUTO};
std::atomic<long long> g_opt_segments{0};
std::atomic<long long> g_opt_wait_limit{0};
std::atomic<long long> g_opt_poison{0};
std::atomic<long long> g_opt_host_slice{0};
std::atomic<long long> g_opt_prep_lead{0};
std::atomic<long long> g_opt_wide_chain{0};
std::atomic<int> g_last_impl{0};

struct TimerState {
    std::mutex mu;
    bool enabled = false;
    std::vector<cudaEvent_t> ev;  // pairs: ev[2i] start, ev[2i+1] stop
    size_t used = 0;              // pairs recorded since the last read
    const char *kernel = "";
};
TimerState &timer() {
    static TimerState t;
    return t;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_common(const void *q, const void *k, const void *v, const float *la,
                        const float *beta, const float *h0, const void *o, const float *hT,
                        int H, int d_k, int d_v, int chunk, gdn_dtype dt, bool need_tokens) {
    if (H < 0 || d_k <= 0 || d_v <= 0) return GDN_ERR_INVALID_ARG;
    if (H > 65535) return GDN_ERR_UNSUPPORTED;  // heads form a grid dimension
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (chunk != kChunk) return GDN_ERR_UNSUPPORTED;
    if (d_k % 8 || d_v % 8 || d_k > 128 || d_v > 256) return GDN_ERR_UNSUPPORTED;
    if (need_tokens && (!q || !k || !v || !la || !beta || !o)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, la, beta, h0, o, hT};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    return GDN_OK;
}

gdn_status dispatch(FwdArgs &a) {
    const long long impl = g_opt_impl.load();
    gdn_status rc;
    int used;
    if (impl == GDN_IMPL_SIMT || (impl == GDN_IMPL_AUTO && !tc_supported(a))) {
        rc = simt_forward(a);
        used = GDN_IMPL_SIMT;
    } else if (impl == GDN_IMPL_TC_FUSED) {
        if (!tc_supported(a) || !fused_supported(a)) return GDN_ERR_UNSUPPORTED;
        rc = fused_forward(a);
        used = GDN_IMPL_TC_FUSED;
    } else {
        if (!tc_supported(a)) return GDN_ERR_UNSUPPORTED;
        rc = tc_forward(a);
        used = GDN_IMPL_TC;
    }
    if (rc == GDN_OK) g_last_impl.store(used);
    return rc;
}
}  // namespace

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t scratch_pool(cudaMemPool_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;   // never hand freed blocks back on its own
        if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) !=
            cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return cudaSuccess;
}
}  // namespace

cudaError_t scratch_alloc(void **p, size_t bytes, cudaStream_t st) {
    cudaMemPool_t pool;
    cudaError_t e = scratch_pool(&pool);
    if (e != cudaSuccess) return e;
    if ((e = cudaMallocFromPoolAsync(p, bytes, pool, st)) != cudaSuccess) return e;
    if (g_opt_poison.load()) e = cudaMemsetAsync(*p, 0xFF, bytes, st);
    return e;
}

cudaError_t scratch_free(void *p, cudaStream_t st) { return cudaFreeAsync(p, st); }

int *device_error_word() {
    void *p = nullptr;
    cudaGetSymbolAddress(&p, g_error_word);
    return static_cast<int *>(p);
}

int timer_begin(cudaStream_t st, const char *kernel) {
    TimerState &t = timer();
    std::lock_guard<std::mutex> lk(t.mu);
    if (!t.enabled) return -1;
    if (t.used * 2 + 2 > t.ev.size()) {
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess) return -1;
        if (cudaEventCreate(&b) != cudaSuccess) {
            cudaEventDestroy(a);
            return -1;
        }
        t.ev.push_back(a);
        t.ev.push_back(b);
    }
    const int slot = (int)t.used++;
    t.kernel = kernel;
    cudaEventRecord(t.ev[2 * slot], st);
    return slot;
}

void timer_cancel(int slot) {
    if (slot < 0) return;
    TimerState &t = timer();
    std::lock_guard<std::mutex> lk(t.mu);
    if ((size_t)slot + 1 == t.used) --t.used;
}

void timer_end(int slot, cudaStream_t st) {
    if (slot < 0) return;
    TimerState &t = timer();
    std::lock_guard<std::mutex> lk(t.mu);
    cudaEventRecord(t.ev[2 * slot + 1], st);
}

void count_launch(int n) { g_launches.fetch_add((uint64_t)n); }

long long option(int key) {
    switch (key) {
        case GDN_OPT_IMPL: return g_opt_impl.load();
        case GDN_OPT_SEGMENTS: return g_opt_segments.load();
        case GDN_OPT_WAIT_LIMIT: return g_opt_wait_limit.load();
        case GDN_OPT_POISON_SCRATCH: return g_opt_poison.load();
        case GDN_OPT_HOST_SLICE: return g_opt_host_slice.load();
        case GDN_OPT_PREP_LEAD: return g_opt_prep_lead.load();
        case GDN_OPT_WIDE_CHAIN: return g_opt_wide_chain.load();
        default: return -1;
    }
}

// Readers of the violation words of the translation units built with
// GDN_BOUNDS_CHECK (gdn_check.cuh); empty in a normal build.
namespace {
std::mutex g_bounds_mu;
std::vector<int (*)(bool)> &bounds_readers() {
    static std::vector<int (*)(bool)> v;
    return v;
}
}  // namespace

void register_bounds_word(int (*read_clear)(bool clear)) {
    std::lock_guard<std::mutex> lk(g_bounds_mu);
    bounds_readers().push_back(read_clear);
}

// Source line of the first failed bounds check on the current device in any
// translation unit (0: none); clears every word if asked.
int bounds_line(bool clear) {
    std::lock_guard<std::mutex> lk(g_bounds_mu);
    int first = 0;
    for (auto fn : bounds_readers()) {
        const int v = fn(clear);
        if (first == 0) first = v;
    }
    return first;
}

}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                   const float *beta, const float *h0, void *o, float *hT, int B, int H, int T,
                   int d_k, int d_v, int chunk, gdn_dtype dt, void *stream) {
    return gdn_fwd_ex(q, k, v, log_alpha, beta, h0, o, hT, B, H, T, d_k, d_v, chunk, dt, 0u,
                      stream);
}

gdn_status gdn_fwd_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                      const float *beta, const float *h0, void *o, float *hT, int B, int H,
                      int T, int d_k, int d_v, int chunk, gdn_dtype dt, unsigned flags,
                      void *stream) {
    if (flags & ~(unsigned)(GDN_FLAG_NO_ERASE | GDN_FLAG_VECTOR_GATE)) return GDN_ERR_INVALID_ARG;
    if (B < 0 || T < 0) return GDN_ERR_INVALID_ARG;
    const bool tokens = (long long)B * H * T > 0;
    gdn_status rc = check_common(q, k, v, log_alpha, beta, h0, o, hT, H, d_k, d_v, chunk, dt,
                                 tokens);
    if (rc != GDN_OK) return rc;
    if ((long long)B * H == 0) return GDN_OK;
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.h0 = h0;
    a.o = o; a.hT = hT;
    a.sm = SeqMap{nullptr, B, H, T, 0};
    a.dk = d_k; a.dv = d_v; a.dt = dt;
    a.rows = (long long)B * H * T;
    a.max_chunks = (T + kChunk - 1) / kChunk;
    a.chunk_slots = (int)((long long)B * a.max_chunks);
    a.stream = static_cast<cudaStream_t>(stream);
    a.no_erase = (flags & GDN_FLAG_NO_ERASE) != 0;
    a.vector_gate = (flags & GDN_FLAG_VECTOR_GATE) != 0;
    if ((long long)B * a.max_chunks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    return dispatch(a);
}

gdn_status gdn_fwd_varlen(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const float *h0, void *o, float *hT,
                          const int32_t *cu_seqlens, int N, int H, int T_total, int d_k,
                          int d_v, int chunk, gdn_dtype dt, void *stream) {
    return gdn_fwd_varlen_ex(q, k, v, log_alpha, beta, h0, o, hT, cu_seqlens, N, H, T_total,
                             d_k, d_v, chunk, dt, 0u, stream);
}

gdn_status gdn_fwd_varlen_ex(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, const float *h0,
                             void *o, float *hT, const int32_t *cu_seqlens, int N, int H,
                             int T_total, int d_k, int d_v, int chunk, gdn_dtype dt,
                             unsigned flags, void *stream) {
    if (flags & ~(unsigned)(GDN_FLAG_NO_ERASE | GDN_FLAG_VECTOR_GATE)) return GDN_ERR_INVALID_ARG;
    if (N < 0 || T_total < 0) return GDN_ERR_INVALID_ARG;
    if (N > 0 && !cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (N == 0 && T_total != 0) return GDN_ERR_INVALID_ARG;
    const bool tokens = (long long)H * T_total > 0;
    gdn_status rc = check_common(q, k, v, log_alpha, beta, h0, o, hT, H, d_k, d_v, chunk, dt,
                                 tokens);
    if (rc != GDN_OK) return rc;
    if ((long long)N * H == 0) return GDN_OK;
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.h0 = h0;
    a.o = o; a.hT = hT;
    a.sm = SeqMap{cu_seqlens, N, H, 0, T_total};
    a.dk = d_k; a.dv = d_v; a.dt = dt;
    a.rows = (long long)H * T_total;
    a.max_chunks = (T_total + kChunk - 1) / kChunk;
    const long long slots = (long long)T_total / kChunk + N;
    if (slots > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    a.chunk_slots = (int)slots;
    a.stream = static_cast<cudaStream_t>(stream);
    a.no_erase = (flags & GDN_FLAG_NO_ERASE) != 0;
    a.vector_gate = (flags & GDN_FLAG_VECTOR_GATE) != 0;
    return dispatch(a);
}

gdn_status gdn_fwd_noalloc(const void *q, const void *k, const void *v, const float *log_alpha,
                           const float *beta, const float *h0, void *o, float *hT, int B, int H,
                           int T, int d_k, int d_v, int chunk, gdn_dtype dt, void *stream) {
    if (B < 0 || T < 0) return GDN_ERR_INVALID_ARG;
    const bool tokens = (long long)B * H * T > 0;
    gdn_status rc = check_common(q, k, v, log_alpha, beta, h0, o, hT, H, d_k, d_v, chunk, dt,
                                 tokens);
    if (rc != GDN_OK) return rc;
    if ((long long)B * H == 0) return GDN_OK;
    if ((long long)B * H * T * (d_k + d_v + 1) * 4 > (long long)kNoallocScratchBytes)
        return GDN_ERR_TOO_LARGE;
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.h0 = h0;
    a.o = o; a.hT = hT;
    a.sm = SeqMap{nullptr, B, H, T, 0};
    a.dk = d_k; a.dv = d_v; a.dt = dt;
    a.rows = (long long)B * H * T;
    a.max_chunks = (T + kChunk - 1) / kChunk;
    a.chunk_slots = (int)((long long)B * a.max_chunks);
    a.stream = static_cast<cudaStream_t>(stream);
    return simt_forward_noalloc(a);
}

namespace {
gdn_status check_bwd(const void *dout, const float *dhT, const void *dq, const void *dk,
                     const void *dv, const float *dla, const float *dbeta, const float *dh0,
                     bool tokens, unsigned flags) {
    if (flags & ~(unsigned)(GDN_FLAG_NO_ERASE | GDN_FLAG_VECTOR_GATE)) return GDN_ERR_INVALID_ARG;
    if (flags & GDN_FLAG_VECTOR_GATE) return GDN_ERR_UNSUPPORTED;
    if (tokens && (!dout || !dq || !dk || !dv || !dla || !dbeta)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {dout, dhT, dq, dk, dv, dla, dbeta, dh0};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    return GDN_OK;
}

gdn_status run_bwd(FwdArgs &a, const void *dout, const float *dhT, void *dq, void *dk, void *dv,
                   float *dla, float *dbeta, float *dh0) {
    BwdArgs b{};
    b.dout = dout; b.dhT = dhT; b.dq = dq; b.dk = dk; b.dv = dv;
    b.dlog_alpha = dla; b.dbeta = dbeta; b.dh0 = dh0;
    int used = 0;
    const gdn_status rc = run_backward(a, b, g_opt_impl.load(), &used);
    if (rc == GDN_OK) g_last_impl.store(used);
    return rc;
}
}  // namespace

gdn_status gdn_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                   const float *beta, const float *h0, const void *dout, const float *dhT,
                   void *dq, void *dk, void *dv, float *dlog_alpha, float *dbeta, float *dh0,
                   int B, int H, int T, int d_k, int d_v, int chunk, gdn_dtype dt,
                   unsigned flags, void *stream) {
    if (B < 0 || T < 0) return GDN_ERR_INVALID_ARG;
    const bool tokens = (long long)B * H * T > 0;
    gdn_status rc = check_common(q, k, v, log_alpha, beta, h0, dout, dhT, H, d_k, d_v, chunk,
                                 dt, tokens);
    if (rc == GDN_OK)
        rc = check_bwd(dout, dhT, dq, dk, dv, dlog_alpha, dbeta, dh0, tokens, flags);
    if (rc != GDN_OK) return rc;
    if ((long long)B * H == 0) return GDN_OK;
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.h0 = h0;
    a.sm = SeqMap{nullptr, B, H, T, 0};
    a.dk = d_k; a.dv = d_v; a.dt = dt;
    a.rows = (long long)B * H * T;
    a.max_chunks = (T + kChunk - 1) / kChunk;
    if ((long long)B * a.max_chunks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    a.chunk_slots = (int)((long long)B * a.max_chunks);
    a.stream = static_cast<cudaStream_t>(stream);
    a.no_erase = (flags & GDN_FLAG_NO_ERASE) != 0;
    return run_bwd(a, dout, dhT, dq, dk, dv, dlog_alpha, dbeta, dh0);
}

gdn_status gdn_bwd_varlen(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const float *h0, const void *dout,
                          const float *dhT, void *dq, void *dk, void *dv, float *dlog_alpha,
                          float *dbeta, float *dh0, const int32_t *cu_seqlens, int N, int H,
                          int T_total, int d_k, int d_v, int chunk, gdn_dtype dt,
                          unsigned flags, void *stream) {
    if (N < 0 || T_total < 0) return GDN_ERR_INVALID_ARG;
    if (N > 0 && !cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (N == 0 && T_total != 0) return GDN_ERR_INVALID_ARG;
    const bool tokens = (long long)H * T_total > 0;
    gdn_status rc = check_common(q, k, v, log_alpha, beta, h0, dout, dhT, H, d_k, d_v, chunk,
                                 dt, tokens);
    if (rc == GDN_OK)
        rc = check_bwd(dout, dhT, dq, dk, dv, dlog_alpha, dbeta, dh0, tokens, flags);
    if (rc != GDN_OK) return rc;
    if ((long long)N * H == 0) return GDN_OK;
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.h0 = h0;
    a.sm = SeqMap{cu_seqlens, N, H, 0, T_total};
    a.dk = d_k; a.dv = d_v; a.dt = dt;
    a.rows = (long long)H * T_total;
    a.max_chunks = (T_total + kChunk - 1) / kChunk;
    const long long slots = (long long)T_total / kChunk + N;
    if (slots > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    a.chunk_slots = (int)slots;
    a.stream = static_cast<cudaStream_t>(stream);
    a.no_erase = (flags & GDN_FLAG_NO_ERASE) != 0;
    return run_bwd(a, dout, dhT, dq, dk, dv, dlog_alpha, dbeta, dh0);
}

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: unsupported chunk, width or implementation";
        case GDN_ERR_ALIGNMENT: return "GDN_ERR_ALIGNMENT: pointer not 16-byte aligned";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA runtime error";
        case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT: bounded device wait gave up";
        case GDN_ERR_TOO_LARGE: return "GDN_ERR_TOO_LARGE: call needs more than the fixed scratch of gdn_fwd_noalloc (32 MiB)";
        case GDN_ERR_BOUNDS: return "GDN_ERR_BOUNDS: a check of the bounds-check build failed (see gdn_bounds_violation)";
        default: return "unknown gdn_status";
    }
}

gdn_status gdn_sync_check(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GDN_ERR_CUDA;
    int word = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
    if (word != 0 && cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess)
        return GDN_ERR_CUDA;
    // the debug bounds-check build: the first failed check (kept for
    // gdn_bounds_violation until it clears it)
    if (bounds_line(false) != 0) return GDN_ERR_BOUNDS;
    if (word == kErrTimeout) return GDN_ERR_DEVICE_TIMEOUT;
    if (word == kErrBadIndex) return GDN_ERR_INVALID_ARG;
    return word == 0 ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_bounds_violation(int clear) {
#ifdef GDN_BOUNDS_CHECK
    return bounds_line(clear != 0);
#else
    (void)clear;
    return -1;
#endif
}

gdn_status gdn_set_option(int key, long long value) {
    switch (key) {
        case GDN_OPT_IMPL:
            if (value < GDN_IMPL_AUTO || value > GDN_IMPL_TC_FUSED) return GDN_ERR_INVALID_ARG;
            g_opt_impl.store(value);
            return GDN_OK;
        case GDN_OPT_SEGMENTS:
            if (value < 0 || value > 4096) return GDN_ERR_INVALID_ARG;
            g_opt_segments.store(value);
            return GDN_OK;
        case GDN_OPT_WAIT_LIMIT:
            if (value < 0) return GDN_ERR_INVALID_ARG;
            g_opt_wait_limit.store(value);
            return GDN_OK;
        case GDN_OPT_POISON_SCRATCH:
            if (value != 0 && value != 1) return GDN_ERR_INVALID_ARG;
            g_opt_poison.store(value);
            return GDN_OK;
        case GDN_OPT_HOST_SLICE:
            if (value < 0 || value > (1LL << 24)) return GDN_ERR_INVALID_ARG;
            g_opt_host_slice.store(value);
            return GDN_OK;
        case GDN_OPT_PREP_LEAD:
            if (value < -1 || value > (1LL << 30)) return GDN_ERR_INVALID_ARG;
            g_opt_prep_lead.store(value);
            return GDN_OK;
        case GDN_OPT_WIDE_CHAIN:
            if (value < -1 || value > 1) return GDN_ERR_INVALID_ARG;
            g_opt_wide_chain.store(value);
            return GDN_OK;
        default:
            return GDN_ERR_INVALID_ARG;
    }
}

long long gdn_get_option(int key) { return option(key); }

gdn_status gdn_kernel_timer(int enable) {
    TimerState &t = timer();
    std::lock_guard<std::mutex> lk(t.mu);
    t.enabled = enable != 0;
    t.used = 0;
    return GDN_OK;
}

gdn_status gdn_kernel_timer_read(double *total_ms, long long *launches, const char **kernel) {
    TimerState &t = timer();
    std::lock_guard<std::mutex> lk(t.mu);
    double sum = 0.0;
    for (size_t i = 0; i < t.used; ++i) {
        float ms = 0.f;
        if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess)
            return GDN_ERR_CUDA;
        sum += ms;
    }
    if (total_ms) *total_ms = sum;
    if (launches) *launches = (long long)t.used;
    if (kernel) *kernel = t.kernel;
    t.used = 0;
    return GDN_OK;
}

uint64_t gdn_kernel_launches(void) { return g_launches.load(); }

gdn_status gdn_scratch_stats(uint64_t *used_current, uint64_t *used_high, int reset_high) {
    cudaMemPool_t pool;
    if (scratch_pool(&pool) != cudaSuccess) return GDN_ERR_CUDA;
    uint64_t cur = 0, high = 0;
    if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &cur) != cudaSuccess ||
        cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &high) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (used_current) *used_current = cur;
    if (used_high) *used_high = high;
    if (reset_high) {
        uint64_t zero = 0;   // restarts the high-water mark at the current use
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

int gdn_last_impl(void) { return g_last_impl.load(); }

gdn_status gdn_release_scratch(void) {
    cudaMemPool_t pool;
    if (gdn::scratch_pool(&pool) != cudaSuccess) return GDN_ERR_CUDA;
    return cudaMemPoolTrimTo(pool, 0) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
