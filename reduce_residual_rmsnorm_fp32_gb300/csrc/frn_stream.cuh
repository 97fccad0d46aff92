// frn_stream.cuh -- the stream kernel: persistent, warp-specialised, for many
// token rows.
//
// One CTA per SM walks rows blockIdx.x, blockIdx.x + gridDim.x, ...  A row is
// read as nslices contiguous slices of 2*H bytes (the R partials, then the
// residual), and each slice is one 1-D bulk copy (TMA, cp.async.bulk) into a
// ring of shared-memory slots:
//  * producer warp, one lane: wait until a slot is empty, arm its "full"
//    mbarrier with the slice's byte count, issue the bulk copy;
//  * consumer groups of warps (one to four tiles per warp): a group takes every
//    groups-th row of the CTA's sequence, so while one group runs a row's
//    epilogue the next group is already accumulating the following row.  A
//    group waits until a slot is full, accumulates its vectors from shared
//    memory in slice order (rank order, residual last), releases the slot, and
//    after the last slice runs the same per-vector epilogue as the row kernel
//    (bf16 residual_out, fixed-tree sum of squares, y, quant), with the tile
//    sums exchanged through shared memory and one named barrier (its own) per
//    row.  Each group owns its own sub-ring of slots (the producer writes row i
//    into group i % groups' sub-ring), so every slot's barriers have exactly one
//    consumer, which takes the slot's fills in order -- the property the parity
//    waits rely on (a group that could wait on a slot one fill ahead of another
//    group would see the earlier phase's parity and pass too early).
// The ring holds ~220 KB, so up to that many bytes per SM stay in flight while
// the consumers reduce, normalise and store -- independent of registers.
//
// Every mbarrier wait is bounded (wait_limit_ns, from %globaltimer).  A wait
// that runs out sets kErrWaitTimeout in the device status word and raises a
// CTA-wide abort flag; all waits then give up, the consumers leave together at
// the next per-row barrier (an OR-reduction, so the decision is uniform), and
// the producer waits -- again bounded -- for every bulk copy it issued before
// the CTA exits.
#pragma once

#include <atomic>

#include "frn_common.cuh"

namespace frn {

constexpr int kStreamMaxConsumerWarps = 16;   // one group (H > 8192)
constexpr int kStreamMaxThreads = 704;        // 22 warps
constexpr int kStreamMaxGroups = 4;
constexpr int kStreamMaxSlots = 32;
constexpr int kStreamSmemLimit = 232448;     // 227 KB opt-in per CTA on sm_100-class parts
constexpr int kStreamSmemReserve = 3072;     // barriers, tile sums, flags (<= 16*32 + 4*512 + 16)

// gamma_bytes: 2*H when gamma is kept in shared memory (four tiles a warp), else 0.
__host__ __device__ constexpr int stream_smem_bytes(int slots, int slice_bytes, int groups, int gamma_bytes) {
    // data ring | gamma | full[slots], empty[slots], gamma barrier (+pad) | tile sums [groups][2][kMaxTiles] | abort flag
    return slots * slice_bytes + gamma_bytes + 16 * slots + 16 + groups * 2 * kMaxTiles * 4 + 16;
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting or
// when this wait ran out (which starts the abort).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned long long limit_ns, unsigned int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            if (err) atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}

// Named barrier `id` over `nthreads` consumer threads, OR-reducing a predicate.
__device__ __forceinline__ bool consumers_sync_or(int id, bool pred, int nthreads) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.or.pred pout, %2, %3, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(out) : "r"((uint32_t)pred), "r"(id), "r"(nthreads) : "memory");
    return out != 0;
}

// MAXTHREADS is the launch bound: 512 (16 warps, up to 128 registers a
// thread), 544 (17 warps: one group of 16 consumer warps for H > 8192, or two
// of 8) or 704 (22 warps: three groups of 7 for H = 7168, 80 registers).
template <int TPW, int MODE, int MAXTHREADS>
__global__ void __launch_bounds__(MAXTHREADS, 1) frn_stream_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    // gamma stays in registers for 1-2 tiles a warp; with 4 it is re-read per
    // row: with a quant output from a shared-memory slice (one bulk copy, so
    // that the quant epilogue does not wait on L2 for it every row), without
    // from cache (the slice would cost a ring slot, which measured slower).
    constexpr bool kGammaInRegs = TPW < 4;
    constexpr bool gamma_in_smem = !kGammaInRegs && (mode_fp8(MODE) || mode_mx(MODE));
    const int NC = p.consumer_warps;
    const int G = p.groups;
    const int S = p.slots;
    const int SG = S / G;              // slots of each group's sub-ring
    const uint32_t slice = static_cast<uint32_t>(p.slice_bytes);
    const uint32_t gamma_bytes = gamma_in_smem ? slice : 0u;
    const uint4* gamma_s = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(S) * slice);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * slice + gamma_bytes);
    float* tsum = reinterpret_cast<float*>(bars + 2 * S + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tsum + G * 2 * kMaxTiles);
    const uint32_t data0 = smem_addr(smem);
    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = full0 + 8u * S;
    const uint32_t gbar = full0 + 16u * S;   // counts the gamma copy
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, static_cast<uint32_t>(NC));
        }
        if (gamma_in_smem) mbar_init(gbar, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    // Nothing of the previous kernel on the stream may be read (or overwritten)
    // before it has completed.
    grid_dependency_wait();

    if (warp == G * NC) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            if (gamma_in_smem) {
                mbar_arrive_expect_tx(gbar, slice);
                bulk_g2s(smem_addr(gamma_s), p.gamma, slice, gbar);
            }
            uint32_t issued = 0, issued_par = 0;
            int used[kStreamMaxGroups] = {0, 0, 0, 0};   // slices issued into each group's sub-ring
            bool ok = true;
            int i = 0;
            for (long long row = blockIdx.x; ok && row < p.T; row += gridDim.x, ++i) {
                const int grp = i % G;
                for (int k = 0; k < p.nslices; ++k) {
                    const int n = used[grp]++;
                    const int slot = grp * SG + n % SG;
                    const uint32_t ph = static_cast<uint32_t>(n / SG) & 1u;
                    if (!wait_bounded(empty0 + 8u * slot, ph ^ 1u, abort_flag, p.wait_limit_ns, p.error_word)) {
                        ok = false;
                        break;
                    }
                    const uint4* src = (k < p.R ? p.partials[k] : p.residual) + row * static_cast<long long>(p.nvec);
                    const bool skip = p.inject_stall && row == blockIdx.x && k == 0;
                    if (!skip) {
                        mbar_arrive_expect_tx(full0 + 8u * slot, slice);
                        bulk_g2s(data0 + static_cast<uint32_t>(slot) * slice, src, slice, full0 + 8u * slot);
                        issued |= 1u << slot;
                        issued_par = (issued_par & ~(1u << slot)) | (ph << slot);
                    }
                }
            }
            launch_dependents();
            // Leave no bulk copy in flight into this CTA's shared memory, on the
            // normal path (where the consumers have waited for them all) as on
            // an abort (where they may not have).
            {
                for (int s = 0; s < S; ++s) {
                    if (!((issued >> s) & 1u)) continue;
                    const uint32_t bar = full0 + 8u * s;
                    const uint32_t par = (issued_par >> s) & 1u;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(bar, par) && globaltimer_ns() - t0 <= p.wait_limit_ns) {
                    }
                }
                if (gamma_in_smem) {
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(gbar, 0u) && globaltimer_ns() - t0 <= p.wait_limit_ns) {
                    }
                }
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers --
    const int grp = warp / NC;
    const int lw = warp - grp * NC;            // warp index within the group
    int jt[TPW];
    bool vt[TPW];
    uint4 g[kGammaInRegs ? TPW : 1];
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
        const int tile = lw + t * NC;
        jt[t] = tile * kTileVecs + lane;
        vt[t] = jt[t] < p.nvec;
        if constexpr (kGammaInRegs) g[t] = ld_keep(p.gamma + (vt[t] ? jt[t] : 0), vt[t]);
    }
    float* gsum = tsum + grp * 2 * kMaxTiles;
    const int ng = p.H / kGroup;
    int lslot = 0;                     // position in this group's sub-ring
    uint32_t ph = 0;
    int prow = 0;
    bool ok = true;
    bool gamma_ready = !gamma_in_smem;   // the gamma copy has landed (waited for once)
    // this group's rows: the (grp + groups*m)-th rows of the CTA's sequence
    for (long long row = blockIdx.x + static_cast<long long>(grp) * gridDim.x; row < p.T;
         row += static_cast<long long>(G) * gridDim.x) {
        float acc[TPW][8];
        for (int k = 0; k < p.nslices; ++k) {
            const int slot = grp * SG + lslot;
            const bool got = ok && wait_bounded(full0 + 8u * slot, ph, abort_flag, p.wait_limit_ns, p.error_word);
            ok = got;
            const uint4* src = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(slot) * slice);
#pragma unroll
            for (int t = 0; t < TPW; ++t) {
                const uint4 v = (got && vt[t]) ? src[jt[t]] : make_uint4(0u, 0u, 0u, 0u);
                if (k == 0) {
                    unpack8(v, acc[t]);
                } else {
                    add8(acc[t], v);
                }
            }
            __syncwarp();
            if (lane == 0 && got) mbar_arrive(empty0 + 8u * slot);
            if (++lslot == SG) {
                lslot = 0;
                ph ^= 1u;
            }
        }
        if (p.residual == nullptr) {
#pragma unroll
            for (int t = 0; t < TPW; ++t) add8(acc[t], make_uint4(0u, 0u, 0u, 0u));   // +0, as the row kernel
        }
        const long long rbase = row * static_cast<long long>(p.nvec);
        uint4 rov[TPW];   // bf16 residual_out, re-widened for y (cheaper than keeping floats)
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
            rov[t] = pack8(acc[t]);
            if (ok && vt[t] && p.residual_out != nullptr) p.residual_out[rbase + jt[t]] = rov[t];
            const float s = tile_sumsq(rov[t]);
            if (lane == 0 && lw + t * NC < p.ntiles) gsum[prow * kMaxTiles + lw + t * NC] = s;
        }
        if (!gamma_ready) {
            gamma_ready = true;
            ok = ok && wait_bounded(gbar, 0u, abort_flag, p.wait_limit_ns, p.error_word);
        }
        if (consumers_sync_or(1 + grp, !ok || *abort_flag != 0, NC * 32)) break;
        const float lo = lane < p.ntiles ? gsum[prow * kMaxTiles + lane] : 0.0f;
        const float hi = lane + 32 < p.ntiles ? gsum[prow * kMaxTiles + lane + 32] : 0.0f;
        const float rstd = row_rstd(lo, hi, p.H, p.eps);
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
            const uint4 gt = kGammaInRegs    ? g[kGammaInRegs ? t : 0]
                           : gamma_in_smem ? (vt[t] ? gamma_s[jt[t]] : make_uint4(0u, 0u, 0u, 0u))
                                           : ld_keep(p.gamma + (vt[t] ? jt[t] : 0), vt[t]);
            const uint4 yb = rms_y<false>(rov[t], rstd, gt);   // widened form: measured faster here
            if constexpr (mode_writes_y(MODE)) {
                if (vt[t]) p.y[rbase + jt[t]] = yb;
            }
            if constexpr (mode_fp8(MODE)) {
                uint2 qq;
                float sc;
                quant8(yb, qq, sc);
                if (vt[t]) {
                    p.q[rbase + jt[t]] = qq;
                    if ((lane & 15) == 0) p.scales[row * ng + (jt[t] >> 4)] = sc;
                }
            }
            if constexpr (mode_mx(MODE)) {
                uint32_t packed, code;
                mxfp4_8(yb, packed, code);
                if (vt[t]) {
                    p.q4[rbase + jt[t]] = packed;
                    if ((lane & 3) == 0) p.mx_scales[row * (p.H / 32) + (jt[t] >> 2)] = static_cast<uint8_t>(code);
                }
            }
        }
        prow ^= 1;
    }
}

struct StreamPlan {
    int tiles_per_warp;
    int consumer_warps;   // per group
    int groups;
    int slots;
    int gamma_smem;       // four tiles a warp: gamma kept in a shared-memory slice
    int smem_bytes;
    long long grid;
};

template <int TPW, int MODE, int MAXTHREADS>
cudaError_t launch_stream_one(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl) {
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(frn_stream_kernel<TPW, MODE, MAXTHREADS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmemLimit);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>((plan.groups * plan.consumer_warps + 1) * 32), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(plan.smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, frn_stream_kernel<TPW, MODE, MAXTHREADS>, p);
}

template <int MODE>
cudaError_t launch_stream(const Params& p, const StreamPlan& plan, cudaStream_t stream, bool pdl) {
    const int threads = (plan.groups * plan.consumer_warps + 1) * 32;
    if (threads > 544) return launch_stream_one<4, MODE, kStreamMaxThreads>(p, plan, stream, pdl);
    if (threads > 512) return launch_stream_one<4, MODE, 544>(p, plan, stream, pdl);
    switch (plan.tiles_per_warp) {
        case 1: return launch_stream_one<1, MODE, 512>(p, plan, stream, pdl);
        case 2: return launch_stream_one<2, MODE, 512>(p, plan, stream, pdl);
        default: return launch_stream_one<4, MODE, 512>(p, plan, stream, pdl);
    }
}

}  // namespace frn
