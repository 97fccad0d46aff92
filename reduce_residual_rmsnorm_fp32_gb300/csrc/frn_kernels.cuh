// frn_kernels.cuh -- device code of the fused reduce + residual add + RMSNorm
// (+ per-group-128 dynamic FP8 e4m3) epilogue for sm_103a.
//
// The op, per token row (see include/frn.h for the full contract):
//   x_hat = sum_r f32(P[r]) (rank order) + f32(residual);  residual_out = bf16(x_hat)
//   y = bf16((x * rstd) * gamma),  rstd = 1/sqrt(sum(x^2)/H + eps),  x = f32(residual_out)
//   per 128-group of y: s = max|y| / 448, q = e4m3(y / s)
// following the replaced subgraph all_reduce -> (fused_add_)rms_norm of the
// "ROCm AITER fused all-reduce + RMSNorm" page (vLLM PR 37646 summary, key source
// snippets) and the per-1x128 quant of the normalised bf16 activation of the
// "AMD fused AllReduce-RMSNorm quant kernel" page (SGLang PR 24651 summary).
//
// Layout of the work (HBM-bound: about (R+5)*T*H flops over >= 2*(R+3)*T*H bytes):
//  * A row of H bf16 is split into 16-byte vectors of 8 elements (nvec = H/8) and
//    the vectors into "tiles" of 32 (one per warp, lane l owns vector 32*k + l).
//  * The tiles of a row are spread over C CTAs of one thread-block cluster
//    (tiles_per_cta warps each).  For decode-sized T this puts one row on up to
//    8 SMs, so a handful of tokens still engages most of the GPU; for large T
//    the same kernel runs with fewer CTAs per row.
//  * Every thread issues all of its R+1 128-bit loads (partials through the
//    read-only path, no L1 allocation, 256-byte L2 prefetch) before its first
//    add, so a thread keeps R+1 requests in flight and each byte of HBM is read
//    exactly once; the row stays in registers until y is written.
//  * Sum of squares: a fixed tree whose shape depends on H alone -- an fp32 FMA
//    chain over the 8 elements of a vector, a 32-lane xor butterfly within the
//    tile, then tile slots k and k+32 paired and a second butterfly over the 32
//    pairs (absent tiles are +0).  Tile sums cross CTAs through distributed
//    shared memory after one cluster barrier; every lane ends with the same
//    bits, and a row gives the same bits for any T, cluster size or stream.
//  * Ordering: griddepcontrol.wait precedes every global access, so with
//    programmatic dependent launch the prologue overlaps the previous kernel but
//    no partial is read before its producer has completed (the lesson of the
//    missing end_sync barrier in "Fix: add missing end_sync barrier in fused
//    allreduce+rmsnorm kernel", AITER PR 4346).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace frn {

constexpr int kMaxPartials = 16;
constexpr int kVecElems = 8;        // bf16 per 16-byte vector
constexpr int kTileVecs = 32;       // vectors per warp tile
constexpr int kMaxTilesPerCta = 16; // 512 threads
constexpr int kMaxTiles = 64;       // H <= 16384
constexpr int kMaxThreads = kMaxTilesPerCta * 32;
constexpr int kGroup = 128;         // quant group (elements)

enum Mode : int { kNorm = 0, kQuantA = 1, kQuantB = 2 };

struct Params {
    const uint4* partials[kMaxPartials];
    const uint4* residual;   // nullptr: zeros
    const uint4* gamma;
    uint4* residual_out;
    uint4* y;                // bf16 output (kNorm, kQuantB)
    uint2* q;                // e4m3 codes, 8 per vector (kQuantA, kQuantB)
    float* scales;           // [T, H/128]
    long long T;
    int R;
    int H;
    int nvec;                // H / 8
    int ntiles;              // ceil(nvec / 32)
    int tiles_per_cta;       // warps per CTA
    int ctas_per_row;        // cluster size
    float eps;
};

// ------------------------------------------------------------------ PTX ----

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Streaming 128-bit load of data that is read once: non-coherent read-only
// path, no L1 allocation, 256-byte L2 sector prefetch.  Predicated inside the
// asm so that no branch is generated; a disabled load yields zeros.
__device__ __forceinline__ uint4 ld_stream(const uint4* ptr, bool pred) {
    uint4 v;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
        "@p ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "r"((int)pred));
    return v;
}

// Coherent 128-bit load, for the residual (which residual_out may overwrite in
// place) -- same hints otherwise.
__device__ __forceinline__ uint4 ld_coherent(const uint4* ptr, bool pred) {
    uint4 v;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
        "@p ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "r"((int)pred));
    return v;
}

// gamma is re-read by every row: keep it cacheable.
__device__ __forceinline__ uint4 ld_keep(const uint4* ptr, bool pred) {
    uint4 v;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
        "@p ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "r"((int)pred));
    return v;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float from the shared memory of CTA `rank` of this cluster, at the
// address that `local` has in this CTA's shared window.
__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ------------------------------------------------------- number formats ----

// bf16 pair in one 32-bit word: element 2i in the low half, 2i+1 in the high half.
__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// cvt.rn.bf16x2.f32 d, a, b puts bf16(a) in the upper half and bf16(b) in the lower.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 v;
    v.x = pack_bf16x2(f[0], f[1]);
    v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]);
    v.w = pack_bf16x2(f[6], f[7]);
    return v;
}

// OCP e4m3 ("fn"), round to nearest even, saturating to +-448; the upper byte
// of the result holds the first source operand.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 v) {
    float f[8];
    unpack8(v, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
}

__device__ __forceinline__ float butterfly_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

// ----------------------------------------------------------------- kernel ----

// One CTA handles `tiles_per_cta` tiles of one row; a cluster of
// `ctas_per_row` CTAs handles the whole row.  CLUSTER == false is the
// single-CTA row (no cluster barriers).  RMAX is the unrolled partial count
// (R <= RMAX; loads beyond R are predicated off).
template <int RMAX, int MODE, bool CLUSTER>
__global__ void __launch_bounds__(kMaxThreads) frn_row_kernel(const __grid_constant__ Params p) {
    __shared__ float tile_sum[kMaxTilesPerCta];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int rank = 0;
    long long row;
    if constexpr (CLUSTER) {
        rank = static_cast<int>(cluster_ctarank());
        row = blockIdx.x / p.ctas_per_row;
    } else {
        row = blockIdx.x;
    }
    const int tile = rank * p.tiles_per_cta + warp;
    const int j = tile * kTileVecs + lane;              // vector index in the row
    const bool valid = j < p.nvec;
    const long long off = row * static_cast<long long>(p.nvec) + j;

    // Nothing of the previous kernel on the stream may be read (or overwritten)
    // before it has completed.
    grid_dependency_wait();

    uint4 raw[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) raw[r] = ld_stream(p.partials[r] + off, valid && r < p.R);
    const uint4 res = ld_coherent(p.residual + off, valid && p.residual != nullptr);
    const uint4 g = ld_keep(p.gamma + j, valid);
    launch_dependents();

    // a1 + a2: fp32 sum in rank order, residual last, one RNE to bf16.
    float acc[8];
    unpack8(raw[0], acc);
#pragma unroll
    for (int r = 1; r < RMAX; ++r)
        if (r < p.R) add8(acc, raw[r]);
    add8(acc, res);
    const uint4 ro = pack8(acc);
    if (valid) p.residual_out[off] = ro;

    // a3: sum of squares of the bf16 residual_out.
    float x[8];
    unpack8(ro, x);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s = __fmaf_rn(x[i], x[i], s);
    s = butterfly_sum(s);
    if (lane == 0) tile_sum[warp] = s;
    __syncwarp();

    float lo, hi;   // tile slots `lane` and `lane + 32` of the row
    if constexpr (CLUSTER) {
        cluster_arrive_release();
        cluster_wait_acquire();
        const int tpc = p.tiles_per_cta;
        lo = lane < p.ntiles ? ld_dsmem(&tile_sum[lane % tpc], lane / tpc) : 0.0f;
        hi = lane + 32 < p.ntiles ? ld_dsmem(&tile_sum[(lane + 32) % tpc], (lane + 32) / tpc) : 0.0f;
        __syncwarp();
        // Done reading the other CTAs' shared memory; they may exit once all
        // CTAs have arrived here (matching wait at the end).
        cluster_arrive_release();
    } else {
        __syncthreads();
        lo = lane < p.ntiles ? tile_sum[lane] : 0.0f;
        hi = lane + 32 < p.ntiles ? tile_sum[lane + 32] : 0.0f;
    }
    const float ss = butterfly_sum(__fadd_rn(lo, hi));
    const float rstd = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(p.H)), p.eps));

    // a4: y = bf16((x * rstd) * gamma).
    float gf[8], yv[8];
    unpack8(g, gf);
#pragma unroll
    for (int i = 0; i < 8; ++i) yv[i] = __fmul_rn(__fmul_rn(x[i], rstd), gf[i]);
    const uint4 yb = pack8(yv);
    if constexpr (MODE != kQuantA) {
        if (valid) p.y[off] = yb;
    }

    // a5: per-group-128 dynamic e4m3 of the bf16 y.  A group is 16 vectors,
    // i.e. one aligned half-warp of a tile.
    if constexpr (MODE != kNorm) {
        float yq[8];
        unpack8(yb, yq);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(yq[i]));
#pragma unroll
        for (int m = 8; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
        const float sc = __fdiv_rn(amax, 448.0f);
        uint2 qq = make_uint2(0u, 0u);
        if (sc != 0.0f) {
            float qv[8];
            if (sc >= 0x1p-64f) {
                // y / s, correctly rounded, from one reciprocal per group:
                // q0 = RN(y * RN(1/s)), then one FMA correction with the
                // residual y - s*q0 (Markstein's theorem).  Checked exhaustively
                // for every bf16 significand of y against every significand
                // s = RN(absmax / 448) can take; the scaling by powers of two
                // that separates those from real operands is exact in this range.
                const float rs = __frcp_rn(sc);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float q0 = __fmul_rn(yq[i], rs);
                    const float rem = __fmaf_rn(-sc, q0, yq[i]);
                    qv[i] = __fmaf_rn(rem, rs, q0);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) qv[i] = __fdiv_rn(yq[i], sc);
            }
            uint32_t c[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i] = pack_e4m3x2(qv[2 * i], qv[2 * i + 1]);
            qq.x = c[0] | (c[1] << 16);
            qq.y = c[2] | (c[3] << 16);
        }
        if (valid) {
            p.q[off] = qq;
            if ((lane & 15) == 0) p.scales[row * (p.H / kGroup) + (j >> 4)] = sc;
        }
    }

    if constexpr (CLUSTER) {
        __syncwarp();
        cluster_wait_acquire();
    }
}

// --------------------------------------------------------------- launch ----

struct Plan {
    int ctas_per_row;
    int tiles_per_cta;
    int threads;
    long long grid;
};

template <int RMAX, int MODE, bool CLUSTER>
cudaError_t launch_one(const Params& p, const Plan& plan, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(plan.threads), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    unsigned n = 0;
    if constexpr (CLUSTER) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = static_cast<unsigned>(plan.ctas_per_row);
        attrs[n].val.clusterDim.y = 1;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, frn_row_kernel<RMAX, MODE, CLUSTER>, p);
}

// Dispatch on the unrolled partial count and on whether the row spans a cluster.
template <int MODE>
cudaError_t launch_rows(const Params& p, const Plan& plan, cudaStream_t stream, bool pdl) {
    const bool cl = plan.ctas_per_row > 1;
#define FRN_DISPATCH_R(RM)                                                        \
    return cl ? launch_one<RM, MODE, true>(p, plan, stream, pdl)                 \
              : launch_one<RM, MODE, false>(p, plan, stream, pdl)
    if (p.R <= 1) FRN_DISPATCH_R(1);
    if (p.R <= 2) FRN_DISPATCH_R(2);
    if (p.R <= 4) FRN_DISPATCH_R(4);
    if (p.R <= 8) FRN_DISPATCH_R(8);
    FRN_DISPATCH_R(16);
#undef FRN_DISPATCH_R
}

// Defined (instantiated) in one translation unit per mode.
cudaError_t launch_norm(const Params& p, const Plan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_quant_a(const Params& p, const Plan& plan, cudaStream_t stream, bool pdl);
cudaError_t launch_quant_b(const Params& p, const Plan& plan, cudaStream_t stream, bool pdl);

}  // namespace frn
