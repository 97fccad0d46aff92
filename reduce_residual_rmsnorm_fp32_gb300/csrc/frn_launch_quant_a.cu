// Instantiates the quant a variant of the row kernel (one translation
// unit per variant so that the build compiles them in parallel).
#include "frn_kernels.cuh"

namespace frn {

cudaError_t launch_quant_a(const Params& p, const Plan& plan, cudaStream_t stream, bool pdl) {
    return launch_rows<kQuantA>(p, plan, stream, pdl);
}

}  // namespace frn
