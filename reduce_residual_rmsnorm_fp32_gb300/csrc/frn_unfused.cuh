// frn_unfused.cuh -- the unfused comparison paths, built from the same
// per-vector arithmetic as the fused kernels so that they return the same bits.
//
// The pages compare three ways of running the epilogue ("AMD fused
// AllReduce-RMSNorm quant kernel", SGLang PR 24651 summary, implementation
// breakdown item 2 and item 4's 3-kernel / 2-kernel / 1-kernel benchmark):
//   3 kernels: reduce -> add + RMSNorm -> per-group quant
//   2 kernels: fused reduce + add + RMSNorm -> stand-alone per-group quant
//   1 kernel : the fused quant entry point.
// Here they exist to measure what fusion saves on GB300.  The 3-kernel path's
// reduce writes the fp32 sum of the partials to a workspace (so that the add
// kernel's fp32 residual add and single rounding match the fused kernels bit
// for bit); a quant path without a bf16 y output keeps y in the workspace.
#pragma once

#include "frn_common.cuh"

namespace frn {

// Stage 1 of 3: x_hat[t, :] = sum_r f32(P[r][t, :]) in rank order (no residual),
// written as fp32.  One thread per 16-byte vector, grid-stride.
template <int RMAX>
__global__ void __launch_bounds__(256) frn_reduce_kernel(const __grid_constant__ Params p, float4* xsum) {
    grid_dependency_wait();
    const long long n = p.T * static_cast<long long>(p.nvec);
    for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += static_cast<long long>(gridDim.x) * 256) {
        uint4 raw[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) raw[r] = ld_stream(p.partials[r] + i, r < p.R);
        float acc[8];
        unpack8(raw[0], acc);
#pragma unroll
        for (int r = 1; r < RMAX; ++r)
            if (r < p.R) add8(acc, raw[r]);
        xsum[2 * i] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        xsum[2 * i + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    launch_dependents();
}

// Stage 2 of 3: residual add + RMSNorm from the fp32 workspace.  One CTA per
// row, one warp per up to four tiles (TPW), tile sums through shared memory.
template <int TPW>
__global__ void __launch_bounds__(512) frn_addnorm_kernel(const __grid_constant__ Params p, const float4* xsum,
                                                           uint4* y) {
    __shared__ float tile_sum[kMaxTiles];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const long long row = blockIdx.x;
    grid_dependency_wait();
    uint4 rov[TPW];
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
        const int tile = warp + t * nw;
        const int j = tile * kTileVecs + lane;
        const bool valid = j < p.nvec;
        const long long off = row * p.nvec + j;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (valid) {
            const float4 a = xsum[2 * off], b = xsum[2 * off + 1];
            acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
            acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
        }
        add8(acc, ld_coherent(p.residual + off, valid && p.residual != nullptr));
        rov[t] = pack8(acc);
        if (valid) p.residual_out[off] = rov[t];
        const float s = tile_sumsq(rov[t]);
        if (lane == 0 && tile < p.ntiles) tile_sum[tile] = s;
    }
    __syncthreads();
    const float lo = lane < p.ntiles ? tile_sum[lane] : 0.0f;
    const float hi = lane + 32 < p.ntiles ? tile_sum[lane + 32] : 0.0f;
    const float rstd = row_rstd(lo, hi, p.H, p.eps);
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
        const int j = (warp + t * nw) * kTileVecs + lane;
        const bool valid = j < p.nvec;
        const uint4 yb = rms_y(rov[t], rstd, ld_keep(p.gamma + (valid ? j : 0), valid));
        if (valid) y[row * p.nvec + j] = yb;
    }
    launch_dependents();
}

// Stand-alone per-group quant of a bf16 [T, H] activation: one warp per tile
// (two groups of GROUP = 128 elements), grid-stride over tiles.
template <int GROUP>
__global__ void __launch_bounds__(256) frn_quant_kernel(const __grid_constant__ Params p, const uint4* y) {
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const long long tiles_per_row = p.ntiles;
    const long long ntot = p.T * tiles_per_row;
    const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long w = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5); w < ntot;
         w += wstride) {
        const long long row = w / tiles_per_row;
        const int j = static_cast<int>(w - row * tiles_per_row) * kTileVecs + lane;
        const bool valid = j < p.nvec;
        const long long off = row * p.nvec + j;
        const uint4 yb = ld_stream(y + off, valid);
        uint2 qq;
        float sc;
        quant8(yb, qq, sc);
        if (valid) {
            p.q[off] = qq;
            if ((lane & 15) == 0) p.scales[row * (p.H / GROUP) + (j >> 4)] = sc;
        }
    }
    launch_dependents();
}

}  // namespace frn
