// frn_kernels.cuh -- the two kernel families and the per-variant launchers.
//
//  * frn_rows.cuh   row kernel: one token row per CTA, per thread-block
//                   cluster, or several short rows per CTA; all of a thread's
//                   loads in flight at once (in stages of two for R > 8); every
//                   row that fits one CTA, at any T.  Its two-tiles-a-warp
//                   variant holds a row of 9..64 tiles on one CTA at many
//                   rows (partials in stages of four for R > 4).
//  * frn_stream.cuh stream kernel: persistent, TMA bulk copies into a shared-
//                   memory ring, warp-specialised; for the other rows wider
//                   than one CTA.
//  * frn_unfused.cuh the 3-kernel / 2-kernel comparison stages.
// Both run the per-vector arithmetic of frn_common.cuh, so a row gives the
// same bits whichever of them computes it.
#pragma once

#include "frn_rows.cuh"
#include "frn_stream.cuh"
#include "frn_unfused.cuh"

namespace frn {

// Defined (instantiated) in one translation unit per output variant so that
// the build compiles them in parallel.
cudaError_t launch_rows_norm(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_rows_quant_a(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_rows_quant_b(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_stream_norm(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_stream_quant_a(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_stream_quant_b(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_rows_mx_a(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_rows_mx_b(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_stream_mx_a(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_stream_mx_b(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl);

// The unfused comparison stages (frn_launch_unfused.cu).
cudaError_t launch_reduce(const Params& p, float4* xsum, int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_addnorm(const Params& p, const float4* xsum, uint4* y, cudaStream_t stream, bool pdl);
cudaError_t launch_quant(const Params& p, const uint4* y, int num_sms, cudaStream_t stream, bool pdl);

}  // namespace frn
