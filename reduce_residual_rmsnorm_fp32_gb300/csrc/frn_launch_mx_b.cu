// Instantiates the MXFP4 b output variant of both kernel families (one
// translation unit per variant so that the build compiles them in parallel).
#include "frn_kernels.cuh"

namespace frn {

cudaError_t launch_rows_mx_b(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl) {
    return launch_rows<kMxB>(p, plan, stream, pdl);
}

cudaError_t launch_stream_mx_b(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl) {
    return launch_stream<kMxB>(p, plan, stream, pdl);
}

}  // namespace frn
