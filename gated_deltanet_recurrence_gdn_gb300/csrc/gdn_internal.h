// gdn_internal.h -- shared host/device declarations of libgdn (not installed).
#pragma once

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
void count_launch(int n = 1);
long long option(int key);

// SIMT (CUDA-core, fp32 arithmetic) path: every supported shape and dtype.
gdn_status simt_forward(const FwdArgs &a);

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

// tcgen05 tensor-core path (bf16 I/O).  Returns GDN_ERR_UNSUPPORTED when the
// call does not fit it; the caller then decides whether to fall back.
bool tc_supported(const FwdArgs &a);
gdn_status tc_forward(const FwdArgs &a);

}  // namespace gdn
