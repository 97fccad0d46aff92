// frn_floor.cu -- reference kernels that bound what a decode-sized call can
// cost on this GPU (measurement only: no entry point of the op uses them).
//
// A decode call moves 1-10 MB, so its time is mostly fixed cost: the launch
// and hand-off from the previous kernel on the stream, one DRAM round trip,
// and the drain of the stores.  These kernels have exactly that cost and
// nothing else, launched the way the op's kernels are (programmatic dependent
// launch, a grid-dependency wait before the first global access):
//  * empty: waits on the previous grid and releases the next one;
//  * read:  every thread loads one 16-byte vector of each source buffer, with
//           the op's load path (read-only, no L1 allocation, 256-byte L2
//           sector prefetch), and keeps the loads alive without storing;
//  * copy:  the same loads, then two 16-byte stores per thread -- the bytes a
//           fused call without quant moves (R partials + residual in,
//           residual_out + y out), with none of its arithmetic.
// "How far is a fused call from its floor" is then the ratio of the two times
// measured in the same graph shape (the benchmark does this).
#include "frn_common.cuh"
#include "../../include/frn.h"

#define FRN_EXPORT extern "C" __attribute__((visibility("default")))

namespace frn {

constexpr int kFloorMaxSources = kMaxPartials + 1;

struct FloorParams {
    const uint4* src[kFloorMaxSources];
    int nsrc;
    uint4* dst0;
    uint4* dst1;
    long long nvec;
};

__global__ void frn_floor_empty_kernel() {
    grid_dependency_wait();
    launch_dependents();
}

// up to 512 threads: the 17 source vectors stay in registers (no spills)
template <bool WRITE>
__global__ void __launch_bounds__(512) frn_floor_copy_kernel(const __grid_constant__ FloorParams p) {
    grid_dependency_wait();
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const bool valid = i < p.nvec;
    uint4 v[kFloorMaxSources];
#pragma unroll
    for (int r = 0; r < kFloorMaxSources; ++r) v[r] = ld_stream(p.src[r] + (valid ? i : 0), valid && r < p.nsrc);
    launch_dependents();
    uint4 acc = v[0];
#pragma unroll
    for (int r = 1; r < kFloorMaxSources; ++r) {
        acc.x ^= v[r].x;
        acc.y ^= v[r].y;
        acc.z ^= v[r].z;
        acc.w ^= v[r].w;
    }
    if constexpr (WRITE) {
        if (valid) {
            p.dst0[i] = acc;
            p.dst1[i] = acc;
        }
    } else {
        // never true for real data; keeps the loads from being dropped
        if (valid && p.dst0 != nullptr && acc.x == 0x9E3779B9u && acc.y == 0x7F4A7C15u && acc.z == 0x85EBCA6Bu &&
            acc.w == 0xC2B2AE35u)
            p.dst0[i] = acc;
    }
}

}  // namespace frn

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

FRN_EXPORT frn_status frn_floor_launch(int kind, const void* const* srcs, int n_src, void* dst0, void* dst1,
                                       int64_t nbytes, int threads, int64_t grid_ctas, int pdl,
                                       frn_stream_t stream) {
    if (kind < 0 || kind > 2 || threads < 32 || threads > (kind == 0 ? 1024 : 512) || threads % 32 != 0)
        return FRN_ERR_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e;
    if (kind == 0) {
        if (grid_ctas < 1 || grid_ctas > 0x7FFFFFFFLL) return FRN_ERR_INVALID_ARG;
        cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
        e = cudaLaunchKernelEx(&cfg, frn::frn_floor_empty_kernel);
    } else {
        if (!srcs || n_src < 1 || n_src > frn::kFloorMaxSources || nbytes < 16 || nbytes % 16 != 0)
            return FRN_ERR_INVALID_ARG;
        if (kind == 2 && (!dst0 || !dst1)) return FRN_ERR_INVALID_ARG;
        frn::FloorParams p = {};
        for (int r = 0; r < frn::kFloorMaxSources; ++r) {
            const void* s = srcs[r < n_src ? r : 0];
            if (!s) return FRN_ERR_INVALID_ARG;
            if (!aligned16(s)) return FRN_ERR_MISALIGNED;
            p.src[r] = static_cast<const uint4*>(s);
        }
        if ((dst0 && !aligned16(dst0)) || (dst1 && !aligned16(dst1))) return FRN_ERR_MISALIGNED;
        p.nsrc = n_src;
        p.dst0 = static_cast<uint4*>(dst0);
        p.dst1 = static_cast<uint4*>(dst1);
        p.nvec = nbytes / 16;
        const long long grid = (p.nvec + threads - 1) / threads;
        if (grid > 0x7FFFFFFFLL) return FRN_ERR_UNSUPPORTED;
        cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
        e = kind == 2 ? cudaLaunchKernelEx(&cfg, frn::frn_floor_copy_kernel<true>, p)
                      : cudaLaunchKernelEx(&cfg, frn::frn_floor_copy_kernel<false>, p);
    }
    return e == cudaSuccess ? FRN_OK : FRN_ERR_CUDA;
}
