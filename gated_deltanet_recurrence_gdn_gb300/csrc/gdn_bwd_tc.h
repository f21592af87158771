// gdn_bwd_tc.h -- the backward pass's tcgen05 stages and its implementation
// choice: the preps' extra outputs for it (gdn_simt.cu, gdn_prep.cu), the
// forward's fused kernel as its state pass (gdn_tc.cu), the state adjoint
// (gdn_bwd_tc.cu) and the backward's entry (gdn_bwd.cu).
#pragma once
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {

// The general path's chunk prep (as enqueue_simt_prep, bf16 I/O only) that
// also writes, for the tensor-core kernels, T diag(beta) as bf16 rows
// [rows][64] into Tub and W as bf16 rows [rows][d_k] into Wb.
gdn_status enqueue_simt_prep_tc(const FwdArgs &a, const int2 *table, float *W, float *U,
                                float *G, float *Tout, __nv_bfloat16 *Tub, __nv_bfloat16 *Wb);

// The tensor-core path's chunk prep (gdn_prep.cu) for the backward pass with
// the erase term: T diag(beta) and W as bf16 rows into Tu and W (as for the
// forward), T itself as fp32 rows [rows][64] into T_out and the in-chunk gate
// cumsum [rows] into G_out.  GDN_ERR_UNSUPPORTED without the erase term or
// outside bf16 I/O with d_k 64 or 128.
gdn_status enqueue_tc_prep_bwd(const FwdArgs &a, const int2 *table, __nv_bfloat16 *Tu,
                               __nv_bfloat16 *W, float *T_out, float *G_out);

// The forward's fused tcgen05 kernel as the backward's state pass: no output,
// every chunk's starting state H = S^T into Hst [H][chunk_slots][d_k][d_v] and
// the rows of V' into Vst [rows][d_v] (fp32).  Tbuf holds T diag(beta) then W
// (bf16, as enqueue_simt_prep_tc writes them, Wb = Tbuf + rows * 64).
// GDN_ERR_UNSUPPORTED where the fused kernel does not take the call.
gdn_status tc_state_pass(const FwdArgs &a, const __nv_bfloat16 *Tbuf, float *Hst, float *Vst);

// Whether the tensor-core state adjoint takes this call: bf16 I/O, a scalar
// gate, d_k 64 or 128, d_v a multiple of 64 (at most 256), an sm_10x device.
bool tc_bwd_supported(const FwdArgs &a);

// The state adjoint dS carried backwards through every sequence's chunks on
// tcgen05 products (bf16 operands, fp32 accumulation): stores the adjoint of
// each chunk's end state as dHc [H][chunk_slots][d_k][d_v] (transposed, dH =
// dS^T) and the rows of dV' as dVn [rows][d_v] (fp32), and dh0 when the
// backward arguments ask for it.  G is the in-chunk gate cumsum [rows] and Wb
// the bf16 W of the prep.
gdn_status tc_bwd_dstate(const FwdArgs &a, const BwdArgs &b, const __nv_bfloat16 *Wb,
                         const float *G, float *dVn, float *dHc);

// The backward pass (gdn_bwd.cu) under an implementation choice: GDN_IMPL_SIMT
// keeps every kernel on warp-level mma.sync; GDN_IMPL_AUTO takes the
// tensor-core state adjoint where it fits; GDN_IMPL_TC requires it
// (GDN_ERR_UNSUPPORTED otherwise).  *used (optional) gets the choice taken.
gdn_status run_backward(const FwdArgs &a, const BwdArgs &b, long long impl, int *used);

}  // namespace gdn
