// frn_rows.cuh -- the row kernel: one token row per CTA or per thread-block
// cluster, or several short rows per CTA; and its two-tiles-a-warp variant
// (frn_row2_kernel) for rows of 9..64 tiles on one CTA.
//
// The tiles of a row go to one CTA (up to 1024 threads) or are spread over C
// CTAs of one cluster (tiles_per_cta warps each, one tile per warp): a row too
// wide for one CTA, or one of a few heavy decode rows, so that a handful of
// tokens still spreads over several SMs.  Rows of at most 4 tiles, when there
// are many, share 256-thread CTAs (the MAXT == 256 instantiation), 8 / ntiles
// consecutive rows each.  Every thread issues all of its R+1
// 128-bit loads (partials through the read-only path, no L1 allocation,
// 256-byte L2 prefetch) before its first add, so each byte of HBM is read
// exactly once and the row stays in registers until y is written.
//
// In a cluster, each warp pushes its tile sum straight into every CTA's shared
// memory with st.async, counted on that CTA's row mbarrier, and each CTA waits
// (bounded) on its own barrier: one one-way hop instead of a cluster barrier
// followed by remote reads.  The barriers are armed at kernel start, and the
// cluster barrier that publishes them is waited on only after the loads, so
// its latency hides behind DRAM.  A last split barrier keeps every CTA of the
// cluster resident until all of them are done.
#pragma once

#include <atomic>

#include "frn_common.cuh"

namespace frn {

// Lanes 0..R-1 of a warp ask for the warp's tile of `row` of each partial to be
// fetched into L2, lane R for the residual's, lane R+1 for gamma's (when
// with_gamma).  Hints only: nothing reads a value from them.
__device__ __forceinline__ void prefetch_tile_span(const Params& p, long long row, int tile, int lane,
                                                   bool with_gamma) {
    if (lane > p.R + (with_gamma ? 1 : 0)) return;
    const int first = tile * kTileVecs;
    const int nv = p.nvec - first < kTileVecs ? p.nvec - first : kTileVecs;
    const long long base = row * static_cast<long long>(p.nvec) + first;
    const uint4* src = lane < p.R ? p.partials[lane] + base
                     : lane == p.R ? (p.residual != nullptr ? p.residual + base : nullptr)
                                   : p.gamma + first;
    if (src != nullptr) bulk_prefetch_l2(src, 16u * static_cast<uint32_t>(nv));
}

// Lanes 0..R-1 of the CTA's first warp ask for the CTA's span of each partial
// of row `row0` to be fetched into L2, lane R for the residual's, lane R+1 for
// gamma's (when with_gamma): one bulk prefetch of up to a row per input (for
// packed short rows, `nrows` whole consecutive rows).  Used for the prefetch
// one wave ahead and for a cluster CTA's slice of its row, where a few large
// requests cost the issuing warps less than a request per warp and input.
// Hints only: nothing reads a value from them.
__device__ __forceinline__ void prefetch_cta_span(const Params& p, long long row0, int nrows, int tile0, int lane,
                                                  bool with_gamma = false) {
    if (lane > p.R + (with_gamma ? 1 : 0)) return;
    const uint4* base = lane < p.R ? p.partials[lane] : lane == p.R ? p.residual : p.gamma;
    if (base == nullptr) return;
    if (lane <= p.R) base += row0 * static_cast<long long>(p.nvec);
    else nrows = 1;
    if (nrows > 1) {
        bulk_prefetch_l2(base, 16u * static_cast<uint32_t>(nrows * p.nvec));
        return;
    }
    const int first = tile0 * kTileVecs;
    const int end = (tile0 + p.tiles_per_cta) * kTileVecs < p.nvec ? (tile0 + p.tiles_per_cta) * kTileVecs : p.nvec;
    if (end > first) bulk_prefetch_l2(base + first, 16u * static_cast<uint32_t>(end - first));
}

// RMAX is the unrolled partial count (R <= RMAX; loads beyond R are predicated
// off).  CLUSTER == false is the single-CTA row (no cluster barriers).  MAXT is
// the launch bound: 512 threads (16 tiles), 1024 for a single-CTA row of up
// to 32 tiles (H <= 8192, R <= 8: 64 registers a thread), or 256 for packed
// short rows (R <= 2 at 32 registers, R <= 4 at 40, R <= 8 at 64).  The second bound
// holds the register count of a single-CTA row where the row count per SM
// needs it: R <= 2 at 32 registers (two wide or four 512-thread rows per SM:
// the prefill shapes live on that), R <= 4 at 40 (three 512-thread rows),
// R <= 8 at 64.  Cluster rows (H > 8192, or a few heavy decode rows) keep
// what the compiler picks.
constexpr int kPackedThreads = 256;   // the packed short-row variant

constexpr int row_min_blocks(int rmax, bool cluster, int maxt, bool staged = false) {
    return staged ? (maxt > kMaxThreads ? 2 : 4)
         : cluster ? 1
         : maxt > kMaxThreads ? (rmax <= 2 ? 2 : 1)
         : maxt == kPackedThreads ? (rmax <= 2 ? 8 : rmax <= 4 ? 6 : rmax <= 8 ? 4 : 2)
                                  : (rmax <= 2 ? 4 : rmax <= 4 ? 3 : rmax <= 8 ? 2 : 1);
}

// STAGED (single-CTA rows of at most kMaxThreads, R > 8): a thread keeps two
// stages of two partial loads in flight instead of all R at once, and sums
// them in rank order as they arrive, so that it fits 32 registers -- four
// 512-thread rows resident per SM instead of one, which keeps loads in flight
// while the other rows run their epilogues.
template <int RMAX, int MODE, bool CLUSTER, int MAXT = kMaxThreads, bool STAGED = false>
__global__ void __launch_bounds__(MAXT, row_min_blocks(RMAX, CLUSTER, MAXT, STAGED))
frn_row_kernel(const __grid_constant__ Params p) {
    static_assert(!STAGED || (!CLUSTER && MAXT != 256 && RMAX % 4 == 0), "staged loads: single-CTA rows");
    // MAXT == 256 (single CTA only): several short rows per CTA, ntiles warps each
    constexpr bool kPacked = !CLUSTER && MAXT == kPackedThreads;
    // single CTA: this CTA's tile sums; cluster: every tile sum of the row
    __shared__ float tile_sum[CLUSTER ? kMaxTiles : MAXT / 32];
    __shared__ __align__(8) uint64_t row_bar;   // cluster: counts the pushed tile sums

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int rank = 0;
    int rsub = 0;        // packed short rows: which of the CTA's rows_per_cta rows this warp works on
    long long row;
    if constexpr (CLUSTER) {
        rank = static_cast<int>(cluster_ctarank());
        row = blockIdx.x / p.ctas_per_row;
    } else if constexpr (kPacked) {
        rsub = warp / p.tiles_per_cta;
        row = static_cast<long long>(blockIdx.x) * p.rows_per_cta + rsub;
    } else {
        row = blockIdx.x;
    }
    const int tile = rank * p.tiles_per_cta + (warp - rsub * p.tiles_per_cta);
    const int j = tile * kTileVecs + lane;              // vector index in the row
    const bool in_rows = !kPacked || row < p.T;         // the last packed CTA's rows may end early
    const bool valid = j < p.nvec && in_rows;
    const long long off = row * static_cast<long long>(p.nvec) + j;

    if constexpr (CLUSTER) {
        // Arm this CTA's row barrier for the 4-byte sums of all ntiles tiles
        // before any CTA may push one: pushes start only after the cluster
        // barrier this arrival belongs to.  No global memory is touched yet.
        if (threadIdx.x == 0) {
            mbar_init(smem_addr(&row_bar), 1);
            mbar_init_fence();
            mbar_arrive_expect_tx(smem_addr(&row_bar), 4u * static_cast<uint32_t>(p.ntiles));
        }
        __syncwarp();
        cluster_arrive_release();
    }

    // When the whole grid is resident at once (decode-sized T), start the DRAM
    // fetch of this warp's tile while the previous kernel on the stream is still
    // finishing.  A prefetch hands no value to this kernel, and L2 is where the
    // previous kernel's writes land, so every value read after the wait below
    // is still the completed one.
    if (p.prefetch_l2) {
        // a cluster CTA's slice in one request per input (measured faster at
        // decode T = 16 and 32, where rows are split over 4 and 2 CTAs); a
        // whole-row CTA's by each warp for its own tile (faster for wide rows)
        if constexpr (CLUSTER) {
            if (warp == 0) prefetch_cta_span(p, row, 1, rank * p.tiles_per_cta, lane, true);
        } else {
            if (tile < p.ntiles && in_rows) prefetch_tile_span(p, row, tile, lane, true);
        }
    }
    // Many rows: ask for this CTA's span of the rows a fixed distance ahead,
    // so that the CTA which takes them finds them in L2; the first wave's
    // CTAs, which start while the previous kernel drains, first ask for their
    // own span.
    if (p.prefetch_ahead > 0 && warp == 0) {
        const long long row0 = kPacked ? static_cast<long long>(blockIdx.x) * p.rows_per_cta : row;
        if (row0 < p.prefetch_own_below) {
            const long long left = p.T - row0;
            const int nrows = kPacked ? static_cast<int>(left < p.rows_per_cta ? left : p.rows_per_cta) : 1;
            prefetch_cta_span(p, row0, nrows, rank * p.tiles_per_cta, lane, true);
        }
        const long long ahead = row0 + p.prefetch_ahead;
        if (ahead < p.T) {
            const long long left = p.T - ahead;
            const int nrows = kPacked ? static_cast<int>(left < p.rows_per_cta ? left : p.rows_per_cta) : 1;
            prefetch_cta_span(p, ahead, nrows, rank * p.tiles_per_cta, lane);
        }
    }

    // Nothing of the previous kernel on the stream may be read (or overwritten)
    // before it has completed.
    grid_dependency_wait();

    // fp32 sum in rank order, residual last (+0 when absent), one RNE to bf16.
    float acc[8];
    uint4 g;
    if constexpr (STAGED) {
        // stages (a, b) of two partials each: issue the next stage, then add
        // the one before it
        uint4 a0 = ld_stream(p.partials[0] + off, valid);
        uint4 a1 = ld_stream(p.partials[1] + off, valid && 1 < p.R);
        uint4 b0 = ld_stream(p.partials[2] + off, valid && 2 < p.R);
        uint4 b1 = ld_stream(p.partials[3] + off, valid && 3 < p.R);
        launch_dependents();
        unpack8(a0, acc);
        if (1 < p.R) add8(acc, a1);
#pragma unroll
        for (int r = 4; r < RMAX; r += 4) {
            a0 = ld_stream(p.partials[r] + off, valid && r < p.R);
            a1 = ld_stream(p.partials[r + 1] + off, valid && r + 1 < p.R);
            if (r - 2 < p.R) add8(acc, b0);
            if (r - 1 < p.R) add8(acc, b1);
            b0 = ld_stream(p.partials[r + 2] + off, valid && r + 2 < p.R);
            b1 = ld_stream(p.partials[r + 3] + off, valid && r + 3 < p.R);
            if (r < p.R) add8(acc, a0);
            if (r + 1 < p.R) add8(acc, a1);
        }
        const uint4 res = ld_coherent(p.residual + off, valid && p.residual != nullptr);
        g = ld_keep(p.gamma + j, valid);
        if (RMAX - 2 < p.R) add8(acc, b0);
        if (RMAX - 1 < p.R) add8(acc, b1);
        add8(acc, res);
    } else {
        uint4 raw[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) raw[r] = ld_stream(p.partials[r] + off, valid && r < p.R);
        const uint4 res = ld_coherent(p.residual + off, valid && p.residual != nullptr);
        g = ld_keep(p.gamma + j, valid);
        launch_dependents();
        unpack8(raw[0], acc);
#pragma unroll
        for (int r = 1; r < RMAX; ++r)
            if (r < p.R) add8(acc, raw[r]);
        add8(acc, res);
    }
    const uint4 ro = pack8(acc);

    const float s = tile_sumsq(ro);

    // x * gamma and residual_out need no rstd: they are formed and stored
    // before the row barrier (a cluster's while its tile sums travel), so
    // that this runs while the other warps or CTAs catch up -- except with a
    // quant output in the 512-thread shapes (the early store measured slower
    // at the FP8 decode workload) and the packed 256-thread shape (both, tight
    // on registers).  In a cluster the early store measured 4-9 % faster at
    // decode T = 8…32 (R = 8, H = 7168) than storing after the exchange.
    constexpr bool kQuantOut = mode_fp8(MODE) || mode_mx(MODE);
    constexpr bool kEarlyXg = CLUSTER || !(MAXT == kPackedThreads && kQuantOut);
    constexpr bool kEarlyStore = kEarlyXg && !(MAXT == kMaxThreads && kQuantOut);
    float xg[8];
    // The FP8 group's absmax of y follows from the absmax of x * gamma (see
    // xgamma_group_absmax), so its shuffles can run before rstd is known too
    // (measured 0.5-2% faster; for the 4-lane MX blocks it was a wash).
    float amax_xg = 0.0f;
    auto quant_lanes_absmax = [](const float (&v)[8]) {
        if constexpr (mode_fp8(MODE)) return xgamma_group_absmax<16>(v);
        else return 0.0f;
    };
    float lo, hi;   // tile slots `lane` and `lane + 32` of the row
    if constexpr (kEarlyStore) {
        if (valid && p.residual_out != nullptr) p.residual_out[off] = ro;
    }
    if constexpr (CLUSTER) {
        cluster_wait_acquire();   // every CTA of the cluster has armed its row barrier
        // (test hook: tile 0's sum is never pushed, so every CTA's wait runs out)
        if (tile < p.ntiles && lane < p.ctas_per_row && !(p.inject_stall && tile == 0))
            st_async_f32(cluster_addr(&tile_sum[tile], static_cast<uint32_t>(lane)), s,
                         cluster_addr(&row_bar, static_cast<uint32_t>(lane)));
        xgamma8(ro, g, xg);   // while the other CTAs' sums travel
        amax_xg = quant_lanes_absmax(xg);
        if (!mbar_wait_bounded(smem_addr(&row_bar), 0u, p.wait_limit_ns) && lane == 0 && p.error_word)
            atomicOr(p.error_word, kErrWaitTimeout);
        lo = lane < p.ntiles ? tile_sum[lane] : 0.0f;
        hi = lane + 32 < p.ntiles ? tile_sum[lane + 32] : 0.0f;
    } else {
        if constexpr (kEarlyXg) {
            xgamma8(ro, g, xg);
            amax_xg = quant_lanes_absmax(xg);
        }
        // this CTA's rows are consecutive groups of ntiles warps
        if (lane == 0) tile_sum[warp] = s;
        __syncthreads();
        const float* ts = tile_sum + rsub * p.tiles_per_cta;
        lo = lane < p.ntiles ? ts[lane] : 0.0f;
        hi = lane + 32 < p.ntiles ? ts[lane + 32] : 0.0f;
    }
    float rstd;
    if (!CLUSTER && p.rstd_one_warp) {
        // Many rows: the first warp of each row alone finishes the reduction
        // and hands rstd to the others through shared memory -- one more
        // barrier, but the butterfly, divide and square root leave every other
        // warp's issue slots free for the CTAs that share the SM.  Same tree,
        // same bits.
        __shared__ float rstd_sh[CLUSTER ? 1 : MAXT / 32];
        if (warp == rsub * p.tiles_per_cta) {
            const float r0 = row_rstd(lo, hi, p.H, p.eps);
            if (lane == 0) rstd_sh[rsub] = r0;
        }
        __syncthreads();
        rstd = rstd_sh[rsub];
    } else {
        rstd = row_rstd(lo, hi, p.H, p.eps);
    }
    if constexpr (CLUSTER) {
        // all sums pushed into this CTA have landed; the matching wait at the
        // end keeps the cluster resident until every CTA got this far
        __syncwarp();
        cluster_arrive_relaxed_after(rstd);
    }
    if constexpr (!kEarlyStore) {
        if (valid && p.residual_out != nullptr) p.residual_out[off] = ro;
    }
    if constexpr (!kEarlyXg) {
        xgamma8(ro, g, xg);
        amax_xg = quant_lanes_absmax(xg);
    }
    const uint4 yb = y_from_xgamma(xg, rstd);
    if constexpr (mode_writes_y(MODE)) {
        if (valid) p.y[off] = yb;
    }
    if constexpr (mode_fp8(MODE)) {
        uint2 qq;
        float sc;
        quant8_amax(yb, y_absmax_from_xgamma(amax_xg, rstd), qq, sc);
        if (valid) {
            p.q[off] = qq;
            if ((lane & 15) == 0) p.scales[row * (p.H / kGroup) + (j >> 4)] = sc;
        }
    }
    if constexpr (mode_mx(MODE)) {
        uint32_t packed, code;
        mxfp4_8(yb, packed, code);
        if (valid) {
            p.q4[off] = packed;
            if ((lane & 3) == 0) p.mx_scales[row * (p.H / 32) + (j >> 2)] = static_cast<uint8_t>(code);
        }
    }

    if constexpr (CLUSTER) {
        __syncwarp();
        cluster_wait_acquire();
    }
}

// Rows of 33..64 tiles (8192 < H <= 16384) on one CTA of up to 1024
// threads: warp w takes tiles w and w + nwarps, so that the row's sum of
// squares never leaves the CTA (no cluster exchange, no cluster to schedule)
// while a whole row's loads are in flight on one SM (with R > 4, in stages of
// four partials, so that they fit 64 registers).  Rows of 26..32 tiles take it
// too with R = 2..4 at many rows (at up to 512 threads two rows fit an SM,
// where the one-tile-a-warp CTA leaves room for one), rows of 17..32 tiles
// with R > 8, which no one-tile-a-warp CTA holds in registers, and rows of
// 9..16 tiles with R = 9..12 (four partials in flight a stage instead of the
// staged CTA's two).  Same
// per-vector arithmetic, tile sums and tree as frn_row_kernel, so the same
// bits.  MINB = 2 (at most 640 threads, 48 registers) fits two such CTAs of
// 608..640 threads on an SM, where the default bound's 52 registers fit one.
template <int RMAX, int MODE, int MINB = 1>
__global__ void __launch_bounds__(MINB == 1 ? 1024 : 640, MINB) frn_row2_kernel(const __grid_constant__ Params p) {
    __shared__ float tile_sum[kMaxTiles];
    __shared__ float rstd_sh;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nwarps = static_cast<int>(blockDim.x >> 5);
    const long long row = blockIdx.x;
    int tile[2], j[2];
    bool valid[2];
    long long off[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        tile[t] = warp + t * nwarps;
        j[t] = tile[t] * kTileVecs + lane;
        valid[t] = tile[t] < p.ntiles && j[t] < p.nvec;
        off[t] = row * static_cast<long long>(p.nvec) + j[t];
    }

    // decode-sized grids: this warp's tiles into L2 before the dependency wait
    if (p.prefetch_l2) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (tile[t] < p.ntiles) prefetch_tile_span(p, row, tile[t], lane, true);
    }
    // many rows: the first wave's own row, and the row a fixed distance ahead
    if (p.prefetch_ahead > 0 && warp == 0) {
        if (row < p.prefetch_own_below) prefetch_cta_span(p, row, 1, 0, lane, true);
        const long long ahead = row + p.prefetch_ahead;
        if (ahead < p.T) prefetch_cta_span(p, ahead, 1, 0, lane);
    }

    grid_dependency_wait();

    uint4 res[2], g[2];
    float accs[2][8];
    if constexpr (RMAX >= 8) {
        // stages of four partials a tile (32 registers of loads in flight);
        // the residual comes with the stage that holds the last partial
        {
            uint4 a[2][4];
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int r = 0; r < 4; ++r) a[t][r] = ld_stream(p.partials[r] + off[t], valid[t] && r < p.R);
            if (p.R <= 4) {
#pragma unroll
                for (int t = 0; t < 2; ++t) res[t] = ld_coherent(p.residual + off[t], valid[t] && p.residual != nullptr);
            }
            launch_dependents();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                unpack8(a[t][0], accs[t]);
#pragma unroll
                for (int r = 1; r < 4; ++r)
                    if (r < p.R) add8(accs[t], a[t][r]);
            }
        }
        // up to 16 partials the stages stay a loop: unrolled, they spilled 40
        // bytes a thread and ran 1-8 % slower (R = 9, H = 5120, T = 2184:
        // 48.0 vs 44.0 us)
#pragma unroll (RMAX > 8 ? 1 : RMAX / 4)
        for (int s = 1; s < RMAX / 4; ++s) {
            if (4 * s >= p.R) break;
            uint4 b[2][4];
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    b[t][r] = ld_stream(p.partials[4 * s + r] + off[t], valid[t] && 4 * s + r < p.R);
            if (4 * s + 4 >= p.R) {
#pragma unroll
                for (int t = 0; t < 2; ++t) res[t] = ld_coherent(p.residual + off[t], valid[t] && p.residual != nullptr);
            }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (4 * s + r < p.R) add8(accs[t], b[t][r]);
            }
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            add8(accs[t], res[t]);
            g[t] = ld_keep(p.gamma + j[t], valid[t]);
        }
    } else {
        // every load of both tiles in flight before the first add
        uint4 raw[2][RMAX];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int r = 0; r < RMAX; ++r) raw[t][r] = ld_stream(p.partials[r] + off[t], valid[t] && r < p.R);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            res[t] = ld_coherent(p.residual + off[t], valid[t] && p.residual != nullptr);
            g[t] = ld_keep(p.gamma + j[t], valid[t]);
        }
        launch_dependents();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            unpack8(raw[t][0], accs[t]);
#pragma unroll
            for (int r = 1; r < RMAX; ++r)
                if (r < p.R) add8(accs[t], raw[t][r]);
            add8(accs[t], res[t]);
        }
    }

    // one RNE to bf16; residual_out and the tile sums right away
    uint4 ro[2];
    float amax_xg[2] = {0.0f, 0.0f};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        ro[t] = pack8(accs[t]);
        const float s = tile_sumsq(ro[t]);
        if (lane == 0 && tile[t] < p.ntiles) tile_sum[tile[t]] = s;
        if (valid[t] && p.residual_out != nullptr) p.residual_out[off[t]] = ro[t];
        if constexpr (mode_fp8(MODE)) {
            float xg[8];
            xgamma8(ro[t], g[t], xg);
            amax_xg[t] = xgamma_group_absmax<16>(xg);
        }
    }
    __syncthreads();
    // lane k holds tile slots k and k + 32 (zeros past the row's tiles)
    if (p.rstd_one_warp) {
        if (warp == 0) {
            const float lo = lane < p.ntiles ? tile_sum[lane] : 0.0f;
            const float hi = lane + 32 < p.ntiles ? tile_sum[lane + 32] : 0.0f;
            const float r0 = row_rstd(lo, hi, p.H, p.eps);
            if (lane == 0) rstd_sh = r0;
        }
        __syncthreads();
    }
    float rstd;
    if (p.rstd_one_warp) {
        rstd = rstd_sh;
    } else {
        const float lo = lane < p.ntiles ? tile_sum[lane] : 0.0f;
        const float hi = lane + 32 < p.ntiles ? tile_sum[lane + 32] : 0.0f;
        rstd = row_rstd(lo, hi, p.H, p.eps);
    }

#pragma unroll
    for (int t = 0; t < 2; ++t) {
        float xg[8];
        xgamma8(ro[t], g[t], xg);
        const uint4 yb = y_from_xgamma(xg, rstd);
        if constexpr (mode_writes_y(MODE)) {
            if (valid[t]) p.y[off[t]] = yb;
        }
        if constexpr (mode_fp8(MODE)) {
            uint2 qq;
            float sc;
            quant8_amax(yb, y_absmax_from_xgamma(amax_xg[t], rstd), qq, sc);
            if (valid[t]) {
                p.q[off[t]] = qq;
                if ((lane & 15) == 0) p.scales[row * (p.H / kGroup) + (j[t] >> 4)] = sc;
            }
        }
        if constexpr (mode_mx(MODE)) {
            uint32_t packed, code;
            mxfp4_8(yb, packed, code);
            if (valid[t]) {
                p.q4[off[t]] = packed;
                if ((lane & 3) == 0) p.mx_scales[row * (p.H / 32) + (j[t] >> 2)] = static_cast<uint8_t>(code);
            }
        }
    }
}

struct RowPlan {
    int ctas_per_row;
    int tiles_per_cta;
    int rows_per_cta;   // single-CTA rows only: short rows share a CTA
    int threads;
    long long grid;
    int staged;         // single-CTA rows with R > 8: staged partial loads (STAGED)
    int tiles_per_warp; // 2: a row on one CTA, two tiles a warp (frn_row2_kernel), else 1
};

template <int RMAX, int MODE, bool CLUSTER, int MAXT = kMaxThreads, bool STAGED = false>
cudaError_t launch_row_one(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl) {
    if constexpr (CLUSTER) {
        if (plan.ctas_per_row > 8) {
            // clusters of 9..16 CTAs are a non-portable size: opt in once per device
            static std::atomic<int> opted[64];
            int dev = 0;
            cudaError_t e = cudaGetDevice(&dev);
            if (e != cudaSuccess) return e;
            if (dev < 0 || dev >= 64 || !opted[dev].load(std::memory_order_acquire)) {
                e = cudaFuncSetAttribute(frn_row_kernel<RMAX, MODE, CLUSTER, MAXT, STAGED>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
                if (dev >= 0 && dev < 64) opted[dev].store(1, std::memory_order_release);
            }
        }
    }
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
    return cudaLaunchKernelEx(&cfg, frn_row_kernel<RMAX, MODE, CLUSTER, MAXT, STAGED>, p);
}

template <int RMAX, int MODE, int MINB = 1>
cudaError_t launch_row2(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(plan.threads), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, frn_row2_kernel<RMAX, MODE, MINB>, p);
}

// Dispatch on the unrolled partial count and on whether the row spans a cluster.
template <int MODE>
cudaError_t launch_rows(const Params& p, const RowPlan& plan, cudaStream_t stream, bool pdl) {
    // two tiles a warp: one CTA per row of 9..64 tiles (the host plans
    // nothing else; R > 4 loads its partials in stages of four)
    if (plan.tiles_per_warp == 2) {
        // R <= 2 rows of 37..40 tiles: two CTAs an SM at 48 registers (H = 10240,
        // T = 3276, R = 1 FP8 A 52.3 -> 39.2 us, FP8 B 57.2 -> 48.7 us; R = 2
        // FP8 A 47.0 -> 38.5 us, MXFP4 B 47.4 -> 44.2 us, no quant 42.6 ->
        // 41.9 us); with R > 2 the loads need more registers
        if (p.R <= 2 && plan.threads > 576 && plan.threads <= 640) {
            if (p.R <= 1) return launch_row2<1, MODE, 2>(p, plan, stream, pdl);
            return launch_row2<2, MODE, 2>(p, plan, stream, pdl);
        }
        if (p.R <= 1) return launch_row2<1, MODE>(p, plan, stream, pdl);
        if (p.R <= 2) return launch_row2<2, MODE>(p, plan, stream, pdl);
        if (p.R <= 4) return launch_row2<4, MODE>(p, plan, stream, pdl);
        if (p.R <= 8) return launch_row2<8, MODE>(p, plan, stream, pdl);
        return launch_row2<16, MODE>(p, plan, stream, pdl);
    }
    // staged loads: one CTA of at most kMaxThreads per row, R > 8 (the host
    // plans nothing else)
    if (plan.staged) return launch_row_one<16, MODE, false, kMaxThreads, true>(p, plan, stream, pdl);
    if (plan.threads > kMaxThreads) {
        // one wide CTA per row (the host only plans this for R <= 8)
        if (p.R <= 1) return launch_row_one<1, MODE, false, 1024>(p, plan, stream, pdl);
        if (p.R <= 2) return launch_row_one<2, MODE, false, 1024>(p, plan, stream, pdl);
        if (p.R <= 4) return launch_row_one<4, MODE, false, 1024>(p, plan, stream, pdl);
        return launch_row_one<8, MODE, false, 1024>(p, plan, stream, pdl);
    }
    if (plan.rows_per_cta > 1) {
        // several short rows per CTA (the host plans this for one CTA per row
        // and at most kPackedThreads threads)
        if (p.R <= 1) return launch_row_one<1, MODE, false, kPackedThreads>(p, plan, stream, pdl);
        if (p.R <= 2) return launch_row_one<2, MODE, false, kPackedThreads>(p, plan, stream, pdl);
        if (p.R <= 4) return launch_row_one<4, MODE, false, kPackedThreads>(p, plan, stream, pdl);
        if (p.R <= 8) return launch_row_one<8, MODE, false, kPackedThreads>(p, plan, stream, pdl);
        return launch_row_one<16, MODE, false, kPackedThreads>(p, plan, stream, pdl);
    }
    const bool cl = plan.ctas_per_row > 1;
#define FRN_DISPATCH_R(RM)                                                        \
    return cl ? launch_row_one<RM, MODE, true>(p, plan, stream, pdl)             \
              : launch_row_one<RM, MODE, false>(p, plan, stream, pdl)
    if (p.R <= 1) FRN_DISPATCH_R(1);
    if (p.R <= 2) FRN_DISPATCH_R(2);
    if (p.R <= 4) FRN_DISPATCH_R(4);
    if (p.R <= 8) FRN_DISPATCH_R(8);
    FRN_DISPATCH_R(16);
#undef FRN_DISPATCH_R
}

}  // namespace frn
