// Launchers of the unfused comparison stages (frn_unfused.cuh).
#include "frn_kernels.cuh"

namespace frn {

namespace {

cudaLaunchConfig_t config(unsigned grid, unsigned block, cudaStream_t stream, bool pdl, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.stream = stream;
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

unsigned grid_for(long long work_items, long long per_cta, long long cap) {
    long long g = (work_items + per_cta - 1) / per_cta;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<unsigned>(g);
}

}  // namespace

cudaError_t launch_reduce(const Params& p, float4* xsum, int num_sms, cudaStream_t stream, bool pdl) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = config(grid_for(p.T * p.nvec, 256, 8LL * num_sms), 256, stream, pdl, &attr);
    if (p.R <= 2) return cudaLaunchKernelEx(&cfg, frn_reduce_kernel<2>, p, xsum);
    if (p.R <= 4) return cudaLaunchKernelEx(&cfg, frn_reduce_kernel<4>, p, xsum);
    if (p.R <= 8) return cudaLaunchKernelEx(&cfg, frn_reduce_kernel<8>, p, xsum);
    return cudaLaunchKernelEx(&cfg, frn_reduce_kernel<16>, p, xsum);
}

cudaError_t launch_addnorm(const Params& p, const float4* xsum, uint4* y, cudaStream_t stream, bool pdl) {
    int tpw = (p.ntiles + 15) / 16;
    tpw = tpw <= 1 ? 1 : (tpw <= 2 ? 2 : 4);
    const int nw = (p.ntiles + tpw - 1) / tpw;
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = config(static_cast<unsigned>(p.T), static_cast<unsigned>(nw * 32), stream, pdl, &attr);
    if (tpw == 1) return cudaLaunchKernelEx(&cfg, frn_addnorm_kernel<1>, p, xsum, y);
    if (tpw == 2) return cudaLaunchKernelEx(&cfg, frn_addnorm_kernel<2>, p, xsum, y);
    return cudaLaunchKernelEx(&cfg, frn_addnorm_kernel<4>, p, xsum, y);
}

cudaError_t launch_quant(const Params& p, const uint4* y, int num_sms, cudaStream_t stream, bool pdl) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = config(grid_for(p.T * p.ntiles, 8, 16LL * num_sms), 256, stream, pdl, &attr);
    return cudaLaunchKernelEx(&cfg, frn_quant_kernel<kGroup>, p, y);
}

}  // namespace frn
