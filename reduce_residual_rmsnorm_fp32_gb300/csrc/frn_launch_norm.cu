// Instantiates the norm variant of the row kernel (one translation
// unit per variant so that the build compiles them in parallel).
#include "frn_kernels.cuh"

namespace frn {

cudaError_t launch_norm(const Params& p, const Plan& plan, cudaStream_t stream, bool pdl) {
    return launch_rows<kNorm>(p, plan, stream, pdl);
}

}  // namespace frn
