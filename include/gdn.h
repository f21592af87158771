/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta rule forward library
 * (libgdn.so).
 *
 * The operation ("Gated DeltaNet GPU并行实现", sections 2.1-2.2): for every
 * (sequence, head) a state S of shape d_v x d_k evolves over tokens as
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t,            alpha_t = exp(log_alpha_t),
 *
 * starting from h0 (or zero) and ending in hT.  The library computes it in the
 * chunked form of section 3.2 (chunks of `chunk` tokens: matrix products inside
 * a chunk, a serial state pass across chunks), with the dual-parallel
 * segment scan of section 3.3 over the affine maps of section 2.3 when there
 * are too few independent (sequence, head) problems to fill the GPU.
 *
 * Layouts (all row-major, innermost dimension contiguous, section 4.1):
 *   dense:  q, k [B][H][T][d_k]; v, o [B][H][T][d_v];
 *           log_alpha, beta [B][H][T] (fp32); h0, hT [B][H][d_v][d_k] (fp32).
 *   packed: q, k [H][T_total][d_k]; v, o [H][T_total][d_v];
 *           log_alpha, beta [H][T_total] (fp32); h0, hT [N][H][d_v][d_k] (fp32);
 *           sequence n occupies tokens [cu_seqlens[n], cu_seqlens[n+1]).
 *   hT[.., i, j] is S_{i j}: i indexes d_v, j indexes d_k.
 *
 * Ownership: every pointer argument is a DEVICE pointer owned by the caller;
 * the library keeps no reference after the call returns.  Scratch memory is
 * taken, stream-ordered on `stream`, from a memory pool the library creates
 * per device on first use; the pool keeps freed memory mapped, so a call
 * after a synchronisation reuses it instead of mapping it again
 * (gdn_release_scratch gives it back).  All work is enqueued on `stream` (a cudaStream_t; NULL is
 * the legacy default stream); calls return before the GPU finishes.
 *
 * Errors: arguments are checked synchronously and a non-GDN_OK status is
 * returned before anything is enqueued.  Pointers must be 16-byte aligned
 * (section 5.2, second pitfall: misaligned or non-contiguous inputs break
 * bulk tensor copies), otherwise GDN_ERR_ALIGNMENT.  A failed launch returns
 * GDN_ERR_CUDA.  Errors found by the kernels while running (a bounded wait
 * that gave up, an invalid cu_seqlens entry) are recorded in a device error
 * word and reported by gdn_sync_check().  Values are not checked for NaN.
 * There is no CPU fallback.
 */
#ifndef GDN_H
#define GDN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,    /* NULL pointer, bad size, bad cu_seqlens */
    GDN_ERR_UNSUPPORTED = 2,    /* chunk != 64, d_k / d_v outside the supported set */
    GDN_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned */
    GDN_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    GDN_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait gave up */
    GDN_ERR_TOO_LARGE = 6,      /* gdn_fwd_noalloc: the call needs more than its fixed scratch */
    GDN_ERR_BOUNDS = 7          /* bounds-check build only: an index check failed */
} gdn_status;

typedef enum {
    GDN_F32 = 0,   /* q, k, v, o are fp32 */
    GDN_BF16 = 1   /* q, k, v, o are bf16 */
} gdn_dtype;

/*
 * Dense forward pass.  See the layouts above.
 *   q, k, v     inputs of `dt`; log_alpha, beta fp32 gates (alpha = exp(log_alpha)).
 *   h0          initial state or NULL (= zero state).
 *   o           output of `dt`, [B][H][T][d_v].
 *   hT          final state or NULL (= not written).
 *   B, H, T     batch, heads, tokens per sequence (T = 0 gives hT = h0).
 *   d_k, d_v    key and value widths: multiples of 8 with 8 <= d_k <= 128 and
 *               8 <= d_v <= 256.
 *   chunk       chunk length; only 64 is supported (GDN_ERR_UNSUPPORTED else).
 *   stream      cudaStream_t to enqueue on.
 */
gdn_status gdn_fwd(const void *q, const void *k, const void *v,
                   const float *log_alpha, const float *beta, const float *h0,
                   void *o, float *hT,
                   int B, int H, int T, int d_k, int d_v, int chunk,
                   gdn_dtype dt, void *stream);

/*
 * Packed variable-length forward pass.  cu_seqlens is a DEVICE int32 array of
 * N+1 non-decreasing offsets with cu_seqlens[0] = 0 and cu_seqlens[N] =
 * T_total (checked on the device; a violation is reported by
 * gdn_sync_check() as GDN_ERR_INVALID_ARG and leaves o / hT unspecified).
 * Sequences never interact; each starts from its own h0[n] (or zero).
 */
gdn_status gdn_fwd_varlen(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, const float *h0,
                          void *o, float *hT, const int32_t *cu_seqlens,
                          int N, int H, int T_total, int d_k, int d_v, int chunk,
                          gdn_dtype dt, void *stream);

/*
 * Dense forward pass that allocates no device memory (the paper has no
 * counterpart: this is a deployment variant of the same computation).
 *
 * Some callers cannot allocate while they run: a serving process that hands
 * all of the GPU's memory to its own pool at start-up and forbids any other
 * allocation afterwards, or a latency-critical loop in which an allocation
 * that stalls or fails is not acceptable.  gdn_fwd_noalloc takes the same
 * arguments and has the same layouts as gdn_fwd, but keeps its scratch in a
 * fixed 32 MiB array that is part of the library's device code; it never
 * calls an allocator and never takes memory from the scratch pool.
 *
 *   When the 32 MiB are taken: the CUDA driver loads a library's device code
 *   onto a device lazily, at its first use there (the default since CUDA
 *   12.2), so the array is mapped on a device by the first gdn_fwd_noalloc
 *   call there (or by an earlier general-path call, which shares that code).
 *   That first call therefore needs 32 MiB of free device memory: make one
 *   call on each device before the process reserves its device memory for
 *   itself, and before any stream capture.  Later calls map nothing.
 *
 *   Limit: B*H*T*(d_k + d_v + 1)*4 bytes must not exceed 32 MiB (for
 *   d_k = d_v = 128, about 32 000 token-heads), otherwise GDN_ERR_TOO_LARGE
 *   is returned and nothing is enqueued.  It always runs the general path's
 *   kernels (GDN_IMPL_SIMT; bf16 or fp32 I/O).
 *   Sharing: every call uses the same array.  Calls whose kernels overlap on
 *   the GPU (other streams, other host threads) race on it and give wrong
 *   results; serialise them.
 */
gdn_status gdn_fwd_noalloc(const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta, const float *h0,
                           void *o, float *hT,
                           int B, int H, int T, int d_k, int d_v, int chunk,
                           gdn_dtype dt, void *stream);

/* Static, human-readable name of a status. */
const char *gdn_status_string(gdn_status s);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns GDN_OK, GDN_ERR_DEVICE_TIMEOUT, GDN_ERR_INVALID_ARG
 * (bad cu_seqlens seen by a kernel), GDN_ERR_BOUNDS (a library built with
 * -DGDN_BOUNDS_CHECK recorded a failed index check; see gdn_bounds_violation)
 * or GDN_ERR_CUDA.
 */
gdn_status gdn_sync_check(void *stream);

/*
 * The debug bounds-check build (-DGDN_BOUNDS_CHECK): the tcgen05 and
 * chunk-prep kernels check their shared-memory, tensor-memory and global
 * indices, skip any access that fails and record the source line of the first
 * failure ("Gated DeltaNet GPU并行实现", section 5.2, second pitfall: index and
 * alignment errors in bulk-copy inputs are otherwise silent).  Returns that
 * line on the current device (0: no failure; the caller synchronises first),
 * clearing it if `clear` != 0; -1 in a normal build, which checks nothing.
 */
int gdn_bounds_violation(int clear);

/*
 * Implementation selection (process-wide; for tests and benchmarks).
 *   GDN_OPT_IMPL:      GDN_IMPL_AUTO (default), GDN_IMPL_SIMT (the general
 *                      path: every supported shape; warp-level tf32 mma.sync
 *                      products, three per step for fp32 I/O so they keep
 *                      fp32 accuracy), GDN_IMPL_TC (tcgen05
 *                      tensor-core kernels; GDN_ERR_UNSUPPORTED when the call
 *                      does not fit them), GDN_IMPL_TC_FUSED (the
 *                      alternative tcgen05 forward: a warp-specialised
 *                      chunk-prep kernel, then one kernel per (sequence, head,
 *                      64-wide d_v tile) that runs the whole chunk recurrence
 *                      with H in registers and every product on tcgen05;
 *                      bf16 I/O, scalar gates with erase, d_k 64 or 128,
 *                      d_v a multiple of 64 up to 256, else
 *                      GDN_ERR_UNSUPPORTED).  AUTO never picks it.
 *   GDN_OPT_SEGMENTS:  0 = automatic; s > 0 forces s sequence segments per
 *                      (sequence, head) in the tensor-core path's segment scan;
 *                      1 disables the scan.
 *   GDN_OPT_WAIT_LIMIT: iteration cap of device-side bounded waits (0 = default).
 *   GDN_OPT_POISON_SCRATCH: 1 fills every scratch block with 0xFF bytes (NaN
 *                      in bf16 and fp32) when it is handed out, so that a read
 *                      of scratch no kernel wrote shows up in the results; 0
 *                      (default) leaves it as the pool returns it.
 *   GDN_OPT_HOST_SLICE: target tokens per time slice of gdn_fwd_host (0 =
 *                      default; rounded up to a multiple of the chunk).
 *                      Shorter slices overlap the copies of neighbouring
 *                      slices better and cost more launches.
 *   GDN_OPT_PREP_LEAD: the tensor-core forward's overlap of chunk prep and
 *                      chain (dense batches without the segment scan, bf16,
 *                      scalar gates with erase, d_k 64 or 128).  0 =
 *                      automatic (default); -1 = off (the chunk prep is one
 *                      launch before the chain); n >= 1: the prep launch
 *                      covers chunks 0 .. n - 1 of every sequence and the
 *                      chain's launch prepares the rest on the SMs its chain
 *                      CTAs leave free (n >= the chunk count: no overlap).
 *   GDN_OPT_WIDE_CHAIN: at d_v = 128 (dense bf16 batches), whether the
 *                      tensor-core forward runs the chunk loop with both
 *                      64-column halves of d_v in one CTA (one CTA per
 *                      (sequence, head) instead of two, each slower): 0 =
 *                      automatic (default: where the two-CTA form needs more
 *                      CTAs than the device has SMs), 1 = always, -1 = never.
 * Returns GDN_ERR_INVALID_ARG for an unknown key or value.
 */
enum {
    GDN_OPT_IMPL = 0,
    GDN_OPT_SEGMENTS = 1,
    GDN_OPT_WAIT_LIMIT = 2,
    GDN_OPT_POISON_SCRATCH = 3,
    GDN_OPT_HOST_SLICE = 4,
    GDN_OPT_PREP_LEAD = 5,
    GDN_OPT_WIDE_CHAIN = 6
};
enum { GDN_IMPL_AUTO = 0, GDN_IMPL_SIMT = 1, GDN_IMPL_TC = 2, GDN_IMPL_TC_FUSED = 3 };
gdn_status gdn_set_option(int key, long long value);
long long gdn_get_option(int key);

/*
 * Live timing of the dominant kernel, for benchmarks.  While enabled, every
 * forward call records a pair of CUDA events around each launch of its most
 * expensive kernel (once per call; twice for a segment scan, whose map pass
 * and output pass are launches of the same chunk-loop kernel), on the
 * call's stream.  gdn_kernel_timer_read() waits for
 * those events, returns the summed duration in milliseconds, the number of
 * timed launches and the kernel's name (a static string), and clears the
 * record.  Not thread-safe; meant for one benchmarking thread.
 */
gdn_status gdn_kernel_timer(int enable);
gdn_status gdn_kernel_timer_read(double *total_ms, long long *launches, const char **kernel);

/* Number of kernels this library has launched since it was loaded. */
uint64_t gdn_kernel_launches(void);

/*
 * The current device's scratch pool (the stream-ordered pool every entry point
 * but gdn_fwd_noalloc takes its temporary buffers from): bytes in use now and
 * the high-water mark of bytes in use (either pointer may be null).  With
 * reset_high != 0 the high-water mark then restarts from the current use.
 * Creates the pool if the device had none.  GDN_ERR_CUDA if the pool cannot be
 * queried.
 */
gdn_status gdn_scratch_stats(uint64_t *used_current, uint64_t *used_high, int reset_high);

/* Implementation the last successful gdn_fwd / gdn_fwd_varlen / gdn_bwd /
 * gdn_bwd_varlen call used (GDN_IMPL_SIMT, GDN_IMPL_TC or GDN_IMPL_TC_FUSED;
 * for the backward, GDN_IMPL_TC when its state adjoint ran on tcgen05, where
 * GDN_IMPL_TC_FUSED selects the same backward as GDN_IMPL_TC), 0 before the
 * first call. */
int gdn_last_impl(void);

/*
 * Forward passes with variant flags (otherwise as gdn_fwd / gdn_fwd_varlen).
 *   GDN_FLAG_NO_ERASE: gated linear attention -- the recurrence without the
 *   delta rule's erase term ("线性注意力机制与Gated DeltaNet的优化实践",
 *   sections 2.2-2.3, with a scalar forget gate alpha and update gate beta):
 *       S_t = alpha_t S_{t-1} + beta_t v_t k_t^T,    o_t = S_t q_t;
 *   alpha = beta = 1 is plain linear attention.  In the chunked form the
 *   erase term is what makes A, T and W; without it T = I and W = 0, and the
 *   same kernels run with the in-chunk inverse skipped.
 *   GDN_FLAG_VECTOR_GATE: the forget gate is a vector over the key dimension
 *   ("Gated DeltaNet GPU并行实现：拆解线性注意力循环的两种高效方案", section
 *   2.2: a per-dimension gate puts an extra diagonal factor in the affine
 *   map).  log_alpha is then [B][H][T][d_k] (varlen: [H][T_total][d_k]),
 *   and the step decays the state's key columns before the erase:
 *       S_t = (S_{t-1} diag(alpha_t)) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
 *   With all d_k entries of a row equal this is the scalar-gate recurrence.
 *   Both flags together give gated linear attention with a vector gate.
 *   Vector gates run on the general path only: with GDN_IMPL_TC forced the
 *   call returns GDN_ERR_UNSUPPORTED, with GDN_IMPL_AUTO it takes that path.
 * Unknown flag bits give GDN_ERR_INVALID_ARG.
 */
enum { GDN_FLAG_NO_ERASE = 1, GDN_FLAG_VECTOR_GATE = 2 };
gdn_status gdn_fwd_ex(const void *q, const void *k, const void *v,
                      const float *log_alpha, const float *beta, const float *h0,
                      void *o, float *hT,
                      int B, int H, int T, int d_k, int d_v, int chunk,
                      gdn_dtype dt, unsigned flags, void *stream);
gdn_status gdn_fwd_varlen_ex(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, const float *h0,
                             void *o, float *hT, const int32_t *cu_seqlens,
                             int N, int H, int T_total, int d_k, int d_v, int chunk,
                             gdn_dtype dt, unsigned flags, void *stream);

/*
 * Backward pass: the gradient of
 *     L = sum_t dO_t . o_t + sum <dhT, hT>
 * with respect to q, k, v, log_alpha, beta and h0, for the forward pass
 * gdn_fwd_ex computes with the same inputs and flags.  No page writes the
 * delta rule's gradient out; the one on linear-attention training
 * ("企业官网建设流程全解析", sections 2 and 4.3) recomputes the recurrent state
 * in the backward pass rather than storing it, and so does this call: it
 * reruns the chunked forward (without writing o), carries the adjoint of the
 * state backwards chunk by chunk, then forms every chunk's gradients in
 * parallel.  For bf16 I/O with d_k 64 or 128 and d_v a multiple of 64 the
 * chunk prep, the state pass and the state adjoint run on the tcgen05 kernels
 * (bf16 operands, fp32 accumulation and fp32 states; the state pass is the
 * forward's fused kernel); the per-chunk gradients, and every step of other
 * shapes and of fp32 I/O, on warp-level tf32 mma.sync products (three per
 * step for fp32 I/O), fp32 accumulation.
 *   q, k, v, log_alpha, beta, h0, B, H, T, d_k, d_v, chunk, dt: as gdn_fwd.
 *   dout   [B][H][T][d_v] dtype dt: the weights dO of the outputs.
 *   dhT    [B][H][d_v][d_k] fp32, or NULL for zero weight on the final state.
 *   dq, dk [B][H][T][d_k] and dv [B][H][T][d_v], dtype dt (outputs).
 *   dlog_alpha, dbeta [B][H][T] fp32 (outputs).
 *   dh0    [B][H][d_v][d_k] fp32 (output; the gradient at the zero state when
 *          h0 is NULL), or NULL to skip it.
 *   flags  GDN_FLAG_NO_ERASE differentiates gated linear attention;
 *          GDN_FLAG_VECTOR_GATE gives GDN_ERR_UNSUPPORTED (not built).
 * Device memory, caller-owned; scratch (about 4 (d_k + 3 d_v + 65) bytes
 * per token-head plus 8 d_k d_v bytes per chunk-head) comes from the
 * library's pool.  Errors as gdn_fwd.  GDN_IMPL_SIMT forces the mma.sync
 * kernels throughout; GDN_IMPL_TC forced returns GDN_ERR_UNSUPPORTED where
 * the tcgen05 kernels do not take the call.
 */
gdn_status gdn_bwd(const void *q, const void *k, const void *v,
                   const float *log_alpha, const float *beta, const float *h0,
                   const void *dout, const float *dhT,
                   void *dq, void *dk, void *dv, float *dlog_alpha, float *dbeta,
                   float *dh0,
                   int B, int H, int T, int d_k, int d_v, int chunk,
                   gdn_dtype dt, unsigned flags, void *stream);

/* Packed backward pass: layouts as gdn_fwd_varlen ([H][T_total][d] tokens,
 * [H][T_total] gates, [N][H][d_v][d_k] states), otherwise as gdn_bwd. */
gdn_status gdn_bwd_varlen(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, const float *h0,
                          const void *dout, const float *dhT,
                          void *dq, void *dk, void *dv, float *dlog_alpha,
                          float *dbeta, float *dh0,
                          const int32_t *cu_seqlens, int N, int H, int T_total,
                          int d_k, int d_v, int chunk, gdn_dtype dt,
                          unsigned flags, void *stream);

/*
 * Dense forward pass on HOST buffers (no paper counterpart: the same
 * computation as gdn_fwd with the host <-> device traffic inside the call).
 * Arguments and layouts as gdn_fwd, but q, k, v, log_alpha, beta, h0 (or
 * NULL) are host inputs and o, hT (or NULL) host outputs.  The call cuts T
 * into chunk-aligned slices of about 512 tokens and pipelines, on internal
 * streams, the upload of slice i + 1, the device pass over slice i (the fp32
 * state handed over in device memory) and the download of slice i - 1; it
 * returns once everything is enqueued, with `stream` made to wait for the
 * last download: synchronise `stream` before reading o / hT, and keep every
 * buffer alive and unchanged until then.  Page-locked host memory lets the
 * copies overlap; pageable memory works without overlap.  Device scratch
 * (three slice buffers and two states) comes from the library's pool.
 */
gdn_status gdn_fwd_host(const void *q, const void *k, const void *v,
                        const float *log_alpha, const float *beta, const float *h0,
                        void *o, float *hT,
                        int B, int H, int T, int d_k, int d_v, int chunk,
                        gdn_dtype dt, void *stream);

/*
 * One decode step for a batch of sequences ("Gated DeltaNet GPU并行实现",
 * sections 2.1-2.2: the per-token update with the scalar gate absorbed into
 * the state): for every (sequence b, head h), with S the d_v x d_k state and
 * one new token,
 *     S <- alpha S (I - beta k k^T) + beta v k^T,    o = S q,
 * alpha = exp(log_alpha) -- gdn_fwd with T = 1 and h0 = hT = the state.
 * Each row of S is updated independently (row i needs only its own S k and
 * S q), so the step is one read and one write of the state: bound by HBM.
 *   q, k        [B][H][d_k] of `dt`;   v, o  [B][H][d_v] of `dt`.
 *   log_alpha, beta  [B][H] fp32.
 *   state       fp32 states, read and overwritten in place: [B][H][d_v][d_k]
 *               when slots is NULL, else a pool [n_slots][H][d_v][d_k] in
 *               which sequence b uses state slots[b] (slots: DEVICE int32
 *               [B], distinct; a slot outside [0, n_slots) is reported by
 *               gdn_sync_check() as GDN_ERR_INVALID_ARG and that sequence is
 *               left untouched).
 *   d_k         32, 64 or 128 (GDN_ERR_UNSUPPORTED else); d_v >= 1.
 * Pointers 16-byte aligned (GDN_ERR_ALIGNMENT).  No scratch memory.
 */
gdn_status gdn_decode(const void *q, const void *k, const void *v,
                      const float *log_alpha, const float *beta, float *state,
                      const int32_t *slots, int n_slots, void *o,
                      int B, int H, int d_k, int d_v, gdn_dtype dt, void *stream);

/* Returns the scratch memory the current device's pool holds (memory of
 * calls still in flight stays until they finish) to the driver.  No paper
 * counterpart: a memory-management hook.  GDN_OK, or GDN_ERR_CUDA. */
gdn_status gdn_release_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
