// gdn_internal.h -- shared host/device declarations of libgdn (not installed).
#pragma once

#include <atomic>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;

// Device error word codes (first error wins).
// kErrBadIndex: an index read on the device (packed offsets, state slots) is out
// of range; the work that needed it is skipped.
enum : int { kErrNone = 0, kErrTimeout = 1, kErrBadIndex = 2 };

// Where the tokens of (sequence n, head h) live.  Dense tensors are
// [B][H][T][d] (sequence n = batch index); packed tensors are [H][T_total][d]
// with sequence n at tokens [cu[n], cu[n+1]).  Both reduce to "row0 + t" in a
// [rows][d] view, rows = B*H*T or H*T_total.
struct SeqMap {
    const int32_t *cu;  // device, N+1 entries; nullptr for dense
    int N;              // number of sequences (B for dense)
    int H;
    int T;              // dense sequence length
    int T_total;        // packed token count

    __device__ __forceinline__ void get(int n, int h, long long &row0, int &len) const {
        if (cu) {
            int a = __ldg(cu + n), b = __ldg(cu + n + 1);
            row0 = (long long)h * T_total + a;
            len = b - a;
        } else {
            row0 = ((long long)n * H + h) * (long long)T;
            len = T;
        }
    }
};

// Per-device memo of a small non-negative host-side value: compute(dev) runs
// until it succeeds once per device (two threads racing on a first use both
// compute the same value).  A negative result is a failure: it is returned as
// `fallback` and not remembered.  `fallback` also covers a current device
// that is unknown or past the table.
constexpr int kMaxDeviceMemo = 64;
template <typename F>
inline int per_device(std::atomic<int> (&memo)[kMaxDeviceMemo], F compute, int fallback) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDeviceMemo) return fallback;
    const int v = memo[dev].load(std::memory_order_acquire);   // value + 1; 0 = not yet known
    if (v > 0) return v - 1;
    const int c = compute(dev);
    if (c < 0) return fallback;
    memo[dev].store(c + 1, std::memory_order_release);
    return c;
}

struct FwdArgs {
    const void *q, *k, *v;
    const float *log_alpha, *beta, *h0;
    void *o;
    float *hT;
    SeqMap sm;
    int dk, dv;
    gdn_dtype dt;
    long long rows;       // rows of the [rows][d] views
    int max_chunks;       // upper bound on chunks of one sequence
    int chunk_slots;      // upper bound on chunks of all sequences
    cudaStream_t stream;
    bool no_erase;        // gated linear attention: A = 0, T = I, W = 0
    bool vector_gate;     // log_alpha [rows][d_k]: a gate per key dimension

    // Index of chunk c of sequence n among the chunk_slots per head: dense
    // batches n * max_chunks + c; packed ones floor(cu[n] / 64) + n + c, which
    // is unique because sequence n has at most (cu[n+1] - cu[n] + 63) / 64
    // chunks and floor(cu[n] / 64) + ceil(len / 64) <= floor(cu[n+1] / 64) + 1.
    __device__ __forceinline__ long long chunk_slot(int n, int c) const {
        if (sm.cu) return (long long)(__ldg(sm.cu + n) / kChunk) + n + c;
        return (long long)n * max_chunks + c;
    }
};

// Gradient pointers of a backward pass (the forward arguments say the rest).
struct BwdArgs {
    const void *dout;     // dO [rows][d_v], I/O dtype
    const float *dhT;     // [seq][H][d_v][d_k] or nullptr (zero)
    void *dq, *dk, *dv;   // [rows][d], I/O dtype
    float *dlog_alpha, *dbeta;  // [rows]
    float *dh0;           // [seq][H][d_v][d_k] or nullptr (not written)
};

// Stream-ordered scratch from the library's per-device pool, which keeps
// freed memory mapped (defined in gdn_api.cu).
cudaError_t scratch_alloc(void **p, size_t bytes, cudaStream_t st);
cudaError_t scratch_free(void *p, cudaStream_t st);

// device error word helpers (defined in gdn_api.cu)
int *device_error_word();
// dominant-kernel timer: returns a slot (or -1 when timing is off)
int timer_begin(cudaStream_t st, const char *kernel);
void timer_end(int slot, cudaStream_t st);
// Forgets `slot` (the last begun) when its launch did not start.
void timer_cancel(int slot);
void count_launch(int n = 1);
long long option(int key);

// The general path (GDN_IMPL_SIMT): every supported shape and dtype, warp-level
// tf32 mma.sync products with fp32 accumulation.
gdn_status simt_forward(const FwdArgs &a);

// Pieces of that path the backward pass reuses.  Prep: W [rows][d_k],
// U [rows][d_v], gate cumsum G [rows] and, with Tout non-null (scalar gates
// only), T = (I + A)^{-1} of every chunk as [rows][64] (table: packed
// batches only).  State pass: with Hst non-null it also stores each chunk's
// starting state H = S^T as [H][chunk_slots][d_k][d_v] and with Vn non-null
// the rows of V' = U - W H as [rows][d_v]; with a.o null it writes no output.
gdn_status enqueue_simt_prep(const FwdArgs &a, const int2 *table, float *W, float *U, float *G,
                             float *Tout);
gdn_status enqueue_simt_state(const FwdArgs &a, const float *W, const float *U, const float *G,
                              float *Hst, float *Vn);

// Backward pass of the scalar-gate recurrence (with or without the erase
// term) on the general path's products; defined in gdn_bwd.cu.
gdn_status simt_backward(const FwdArgs &a, const BwdArgs &b);

// The same path on a dense batch with its scratch in a fixed device array of
// kNoallocScratchBytes (needs rows * (d_k + d_v + 1) * 4 bytes); no allocation.
constexpr size_t kNoallocScratchBytes = size_t(32) << 20;
gdn_status simt_forward_noalloc(const FwdArgs &a);

// Lists every (sequence, chunk) of a packed batch into table[chunk_slots]
// (unused slots get n = -1) and validates cu_seqlens.
gdn_status enqueue_chunk_table(const FwdArgs &a, int2 *table);

// Chunk-prep kernel of the tensor-core path: with T = (I + A)^{-1} per chunk,
// writes T diag(beta) as bf16 rows [rows][64] into Tu and
// W = T diag(beta gamma) K as bf16 rows [rows][d_k] into W
// (table: packed batches only, else nullptr).
size_t tc_prep_smem(int dk);
gdn_status enqueue_tc_prep(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                           __nv_bfloat16 *W);

// Chunk-prep kernel of the fused forward (gdn_ut.cu): T_u = (I + A)^{-1} diag(beta)
// and T_w = (I + A)^{-1} diag(beta gamma) of every chunk as bf16
// [H][chunk_slots][T_u | T_w][64][64] (slot of chunk c of sequence n: dense
// n * max_chunks + c, packed floor(cu[n] / 64) + n + c; table: packed batches
// only).  The fused forward (gdn_fused.cu) reads it and forms W, U,
// the state pass and the output in one kernel per (sequence, head, d_v tile).
gdn_status enqueue_ut(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu);
// The same chunk prep (bf16, scalar gates, erase; d_k 64 or 128) in the layout
// of enqueue_tc_prep: T_u as [rows][64] and W = T_w K (formed on tcgen05 from
// the staged K tile) as [rows][d_k], rows indexed like the token rows of the
// inputs.  GDN_ERR_UNSUPPORTED outside those shapes.
gdn_status enqueue_ut_w(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                        __nv_bfloat16 *W);
// The same over chunks 0 .. lead - 1 of every (sequence, head) of a dense
// batch only (the chain kernel's overlapped launch prepares the rest); it
// first clears the n_done ready flags at `done` that the overlapped launch
// sets.  GDN_ERR_UNSUPPORTED where enqueue_ut_w is, for packed batches and
// for lead outside 1 .. max_chunks.
gdn_status enqueue_ut_w_lead(const FwdArgs &a, __nv_bfloat16 *Tu, __nv_bfloat16 *W, int lead,
                             uint32_t *done, long long n_done);
bool fused_supported(const FwdArgs &a);
gdn_status fused_forward(const FwdArgs &a);

// tcgen05 tensor-core path (bf16 I/O).  Returns GDN_ERR_UNSUPPORTED when the
// call does not fit it; the caller then decides whether to fall back.
bool tc_supported(const FwdArgs &a);
gdn_status tc_forward(const FwdArgs &a);

}  // namespace gdn
