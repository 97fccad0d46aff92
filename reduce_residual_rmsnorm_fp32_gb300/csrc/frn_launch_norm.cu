// Instantiates the norm output variant of both kernel families (one
// translation unit per variant so that the build compiles them in parallel).
#include "frn_kernels.cuh"

namespace frn {

cudaError_t launch_rows_norm(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl) {
    return launch_rows<kNorm>(p, plan, stream, pdl);
}

cudaError_t launch_stream_norm(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl) {
    return launch_stream<kNorm>(p, plan, stream, pdl);
}

}  // namespace frn
