// frn_api.cu -- the C ABI of libfrn (declared in include/frn.h): argument
// validation, launch-shape choice and kernel launch.  Host code only.
//
// The entry points follow the fused-op signatures of the pages: the vLLM
// custom op takes (input, residual, weight, epsilon) and returns the
// normalised activation and the sum ("ROCm AITER fused all-reduce + RMSNorm",
// vLLM PR 37646 summary, key source snippets, _aiter_ops.py), and the SGLang
// quant variant adds group_size and emit_bf16 / keep_bf16 ("AMD fused
// AllReduce-RMSNorm quant kernel", SGLang PR 24651 summary, key source snippets,
// layernorm.py).  Tuples become named output pointers, and the pages' "return
// None to fall back" becomes an error status: there is no fallback path.
#include <atomic>
#include <cstdlib>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "frn_kernels.cuh"
#include "../../include/frn.h"

#define FRN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_detail[256] = "";
std::atomic<int> g_pdl{1};
std::atomic<int> g_prefetch{0};   // 0 auto, 1 never, 2 always
std::atomic<int> g_force_ctas{0};
std::atomic<int> g_force_kernel{0};
std::atomic<int> g_force_groups{0};
std::atomic<int> g_inject_stall{0};
std::atomic<long long> g_wait_limit_ns{0};

constexpr long long kDefaultWaitLimitNs = 2000000000LL;   // 2 s per mbarrier wait
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<unsigned int*> g_status_addr[kMaxDevices];

enum Kind : int { kAuto = 0, kRows = 1, kStream = 2 };


frn_status fail(frn_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return s;
}

frn_status ok() {
    g_detail[0] = '\0';
    return FRN_OK;
}

frn_status sm_count(int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < kMaxDevices) {
        int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) { *out = c; return FRN_OK; }
    }
    int c = 0;
    e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(c, std::memory_order_relaxed);
    *out = c;
    return FRN_OK;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

// Device status word of the kernels' bounded waits (one per device).
__device__ unsigned int g_frn_status_word;

namespace {

frn_status status_word(unsigned int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < kMaxDevices) {
        unsigned int* a = g_status_addr[dev].load(std::memory_order_acquire);
        if (a) { *out = a; return FRN_OK; }
    }
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_frn_status_word);
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < kMaxDevices) g_status_addr[dev].store(static_cast<unsigned int*>(a), std::memory_order_release);
    *out = static_cast<unsigned int*>(a);
    return FRN_OK;
}

// Launch shape of the row kernel.  A row's ntiles warp tiles go to C CTAs of
// a cluster, or (wide) to one CTA of up to 1024 threads.  The results do not
// depend on this choice (the reduction tree is fixed by H).
frn::RowPlan wide_plan(long long T, int ntiles) {
    frn::RowPlan plan;
    plan.ctas_per_row = 1;
    plan.tiles_per_cta = ntiles;
    plan.rows_per_cta = 1;
    plan.threads = ntiles * 32;
    plan.grid = T;
    plan.staged = 0;
    plan.tiles_per_warp = 1;
    return plan;
}

bool wide_possible(int ntiles, int R) { return ntiles <= 2 * frn::kMaxTilesPerCta && R <= 8; }

// Rows of 33..64 tiles (8192 < H <= 16384) with R <= 8 from half a wave on: one
// CTA per row, two tiles a warp (frn_row2_kernel), instead of a cluster of
// CTAs or the stream kernel -- except MXFP4 without y at R <= 2, where the
// stream kernel (gamma in shared memory) stays ahead.  Measured on GB300
// (two-tile row / stream / clusters of 4, us): R = 2, T = 8192, H = 16384 no
// quant 192.7 / 201.2 / 244.4, FP8 A 182.3 / 287.1 / 269.5, FP8 B 213.3 /
// 280.4 / 284.6, MXFP4 B 203.0 / 246.8 / 281.6, MXFP4 A 175.9 / 167.2 /
// 259.2; R = 4, T = 4096, H = 16384 FP8 A 127.2 / 189.1 / 186.1, FP8 B
// 149.6 / 189.4 / 201.3, MXFP4 A 122.8 / 134.9 / 180.1, MXFP4 B 143.4 /
// 162.5 / 195.0, no quant 136.2 / 136.9 / 174.0; R = 3 FP8 A 108.7 / 167.7 /
// 180.1; R = 4, T = 600 FP8 A 23.9 / 35.8 / 31.5; R = 4, H = 16384, T = 80
// no quant 4.7 / 6.7 / 6.3, R = 2 at T = 80 level with clusters (3.7 vs
// 3.6-3.8), at T = 152 5.2 / 7.2 / 7.1.  With R = 5..8 (partials loaded in
// stages of four), two-tile / clusters of 4 with an FP8 output: R = 8,
// T = 2048, H = 16384 FP8 A 109.9 / 125.2 us, FP8 B 119.6 / 140.9 us; two-tile
// / stream otherwise: R = 8 MXFP4 A 105.5 / 108.0 us, MXFP4 B 114.3 / 118.3
// us, no quant 110.2 / 109.8 us (T = 200 14.9 / 16.8 us, T = 800 47.6 /
// 49.3 us), H = 12288 no quant 85.8 / 88.7 us, R = 7 no quant 100.9 / 104.8
// us, R = 5 82.2 / 87.6 us (R = 6 no quant 94.1 / 91.1 us, the one loss).
//
// Rows of 17..32 tiles with R > 8, which no one-tile-a-warp CTA holds: two
// tiles a warp in stages of four partials instead of clusters with an FP8
// output (R = 16, T = 1379, H = 5120 FP8 A 46.7 / 49.1 us; R = 12, H = 8192,
// T = 1092 FP8 A 45.7 / 57.6 us) and of the stream kernel otherwise up to 22
// tiles, where a ring slot of R + 1 slices leaves the stream kernel one row
// in flight an SM (R = 16, T = 1379, H = 5120 no quant 47.9 / 54.3 us, MXFP4
// B 48.4 / 55.2 us; H = 5632 48.5 / 51.2 us).  Wider, the stream kernel keeps
// more rows in flight and wins without FP8 (R = 16, H = 7168, T = 985 49.1 /
// 45.5 us; H = 6144 48.1 / 46.3 us).  Rows of 33..64 tiles with R > 8: the
// same with an FP8 output (R = 16, T = 431, H = 16384 FP8 A 48.1 / 55.8 us
// on clusters of 4; R = 12, H = 12288 FP8 B 50.7 / 63.9 us), the stream
// kernel otherwise (no quant 48.9 / 46.1 us).
//
// Rows of 9..16 tiles with R > 8 against the staged one-tile-a-warp CTA
// (two-tile / staged or single CTA, us): better up to R = 10 at every output
// (H = 4096, R = 10, T = 2520 no quant 44.2 / 44.5, FP8 B 46.3 / 51.3, MXFP4
// B 45.3 / 48.4, T = 315 8.0 / 9.1; R = 9, T = 2730 FP8 A 43.5 / 47.6;
// H = 2304, R = 10, T = 560 FP8 B 8.0 / 9.5), and with R = 11, 12 for a quant
// output at staged sizes (H = 3072, R = 11, T = 3120 FP8 B 46.4 / 51.9; R =
// 12, T = 2912 46.5 / 48.9), but not without one (R = 12 no quant 44.5 /
// 43.3), below three waves (H = 4096, R = 11, T = 292 FP8 B 8.5 / 8.0), or
// from R = 13 on (R = 16, T = 1724 no quant 47.6 / 42.1: the staged CTA has
// twice the warps for the same bytes in flight).
//
// Rows of 26..32 tiles (6144 < H <= 8192) with R = 3 or 4 beyond one row per
// SM: the wide CTA (832..1024 threads at 40 registers) leaves room for one
// row an SM, two-tile CTAs of half as many threads for two, so twice the
// loads are in flight.  Measured on GB300 (two-tile / wide, us): H = 7168,
// R = 4, T = 160 4.02 / 4.78, T = 304 6.01 / 6.90, FP8 A 6.13 / 7.16, T = 1171
// 19.95 / 20.74, FP8 A 20.12 / 22.38, MXFP4 B 21.16 / 22.84, T = 4096 62.3 /
// 63.5, FP8 B 68.7 / 72.8, MXFP4 A 56.2 / 65.6; R = 3, T = 304 5.18 / 6.32,
// T = 1171 FP8 A 17.5 / 20.0; H = 8192, R = 4, T = 304 6.71 / 7.29, T = 1171
// FP8 A 22.0 / 24.6 (no quant at T = 4096 72.0 / 70.4, the one loss).  At
// H <= 6144 two wide CTAs fit an SM and it gains nothing (H = 6144, R = 4,
// T = 1171 17.65 / 17.32); within one row per SM the wide CTA's extra warps
// win (H = 7168, R = 4, T = 64 2.44 / 2.35, T = 147 3.56 / 3.47).  With R = 2
// only FP8 A at 16 rows an SM and more (T = 8192, H = 7168 79.9 / 81.3; no
// quant, FP8 B and MXFP4 level; T = 586 8.63 / 8.50).  With R = 5..8 from one
// to 1.65 rows an SM, where the wide CTA runs a second, partial wave and the
// two-tile grid fits one (H = 7168, R = 8, T = 180 6.32 / 7.25, FP8 B 7.17 /
// 7.83, T = 230 7.12 / 7.71, T = 250 7.67 / 8.03; R = 5, T = 200 5.02 / 6.25;
// R = 6, T = 250 FP8 A 6.55 / 7.33; R = 7, T = 200 6.07 / 7.13; H = 8192,
// R = 8, T = 200 7.38 / 8.32), but not beyond (R = 8, T = 280 8.48 / 8.20,
// T = 1171 31.3 / 30.2).
bool two_tile_rows(long long T, int ntiles, int R, int quant, int num_sms) {
    const bool fp8 = quant == 1 || quant == 2;
    if (ntiles <= frn::kMaxTilesPerCta) {
        if (ntiles <= 8 || R <= 8 || 2 * T < num_sms) return false;
        return R <= 10 || (R <= 12 && quant != 0 && T >= 3LL * num_sms);
    }
    if (R > 8) return (fp8 || ntiles <= 22) && 2 * T >= num_sms;
    if (ntiles > 2 * frn::kMaxTilesPerCta) return !(quant == 3 && R <= 2) && 2 * T >= num_sms;
    if (ntiles >= 26)
        return ((R == 3 || R == 4) && T > num_sms) || (R == 2 && quant == 1 && T >= 16LL * num_sms) ||
               (R >= 5 && T > num_sms && 20 * T <= 33LL * num_sms);
    return false;
}

frn::RowPlan two_tile_plan(long long T, int ntiles) {
    frn::RowPlan plan = wide_plan(T, ntiles);
    plan.threads = ceil_div(ntiles, 2) * 32;
    plan.tiles_per_warp = 2;
    return plan;
}


frn::RowPlan choose_rows(long long T, int H, int R, int quant, int num_sms) {
    const int nvec = H / frn::kVecElems;
    const int ntiles = ceil_div(nvec, frn::kTileVecs);
    const int cmin = ceil_div(ntiles, frn::kMaxTilesPerCta);
    int C;
    const int forced = g_force_ctas.load(std::memory_order_relaxed);
    if (forced == 1 && wide_possible(ntiles, R)) return wide_plan(T, ntiles);
    if ((forced == 1 && ntiles > 2 * frn::kMaxTilesPerCta) ||
        (forced == 0 && two_tile_rows(T, ntiles, R, quant, num_sms)))
        return two_tile_plan(T, ntiles);
    if (forced > 0) {
        // up to 8 CTAs per cluster with at least one tile each; up to 16
        // (non-portable cluster size) with at least two tiles each
        const int cmax = ntiles < 8 ? ntiles : (forced > 8 ? (ntiles / 2 < 16 ? ntiles / 2 : 16) : 8);
        C = forced < cmin ? cmin : (forced > cmax ? cmax : forced);
    } else {
        // One CTA per row (a wide one when the row needs more than 512
        // threads), or the smallest cluster that holds the row -- except for a
        // few rows of more than 96 KB of loads each, which go to clusters so
        // that about 20 to 80 CTAs share the work: up to 7 CTAs at T <= 5, 4 up
        // to T = 16, 2 up to T = 40 (measured with the L2 prefetch at
        // H = 4096..16384, R = 2..8, T = 3..128; R = 8, H = 7168 in a chain
        // of same-size calls, clusters of 1 / 2 / 4 / 7: T = 3 2.48 / 2.06 /
        // 2.05 / 1.95 us, T = 5 2.50 / 2.08 / 2.08 / 1.86 us, T = 37 2.63 /
        // 2.45 / 2.65 / 2.64 us, T = 45 2.65 / 2.71 / 2.81 / 2.86 us; larger
        // clusters and more CTAs otherwise cost more in synchronisation than
        // they gain).
        const long long row_bytes = 2LL * H * (R + 1);
        int want = 1;
        if (row_bytes > 96 * 1024) want = T <= 5 ? 7 : T <= 16 ? 4 : T <= 40 ? 2 : 1;
        if (want <= 1) {
            if (cmin > 1 && wide_possible(ntiles, R)) return wide_plan(T, ntiles);
            C = cmin;
        } else {
            // prefer a size that splits the tiles evenly (the nearest divisor of
            // ntiles, the larger on a tie): a ragged last CTA measured up to 25%
            // slower at H = 16384
            if (want < cmin) want = cmin;
            C = want;
            int best = 0;
            for (int c = cmin; c <= want; ++c) {
                if (ntiles % c) continue;
                if (!best || std::abs(c - want) <= std::abs(best - want)) best = c;
            }
            if (best) C = best;
        }
    }
    const int tpc = ceil_div(ntiles, C);
    C = ceil_div(ntiles, tpc);   // no empty CTA
    frn::RowPlan plan;
    plan.ctas_per_row = C;
    plan.tiles_per_cta = tpc;
    plan.rows_per_cta = 1;
    // Short rows (<= 4 tiles, H <= 1024) with several rows per SM: 256-thread
    // CTAs of 8 / ntiles consecutive rows, instead of CTAs of one to four
    // warps (an SM holds at most 32 CTAs).
    if (C == 1 && ntiles <= 4 && T >= 4LL * num_sms) plan.rows_per_cta = 8 / ntiles;
    plan.threads = plan.rows_per_cta * tpc * 32;
    plan.grid = (T + plan.rows_per_cta - 1) / plan.rows_per_cta * C;
    plan.staged = 0;
    plan.tiles_per_warp = 1;
    return plan;
}

// Staged partial loads for a one-CTA row (two stages of two loads in flight,
// 32 registers, so that four 512-thread rows share an SM instead of one or
// two) for R > 8 rows of <= 16 tiles (96 registers otherwise) from three
// waves, where they measured faster on GB300: R = 16, H = 4096, T = 586 /
// 1171 / 4096: 16.8 / 29.7 / 95.8 us against 18.8 / 33.8 / 99.9 us.  Below
// three waves the second DRAM round trip of a row shows (T = 293: 10.6 vs
// 9.6 us).  For R = 5..8 wide rows with a quant output they had beaten the
// stream kernel at three to six waves (R = 8, H = 7168, T = 586: FP8 A 17.9
// vs 19.7 us), but the all-loads-at-once row with its prefetch ahead now
// beats both (17.5 us).
bool staged_window(long long T, int H, int R, int num_sms) {
    const int ntiles = ceil_div(H / frn::kVecElems, frn::kTileVecs);
    return R > 8 && ntiles <= frn::kMaxTilesPerCta && T >= 3LL * num_sms;
}

frn::RowPlan plan_rows(long long T, int H, int R, int quant, int num_sms) {
    frn::RowPlan plan = choose_rows(T, H, R, quant, num_sms);
    if (plan.tiles_per_warp == 1 && plan.ctas_per_row == 1 && plan.rows_per_cta == 1 &&
        staged_window(T, H, R, num_sms))
        plan.staged = 1;
    return plan;
}

// Launch shape of the stream kernel: 1, 2 or 4 tiles per consumer warp so that
// a group has at most 8 warps (16 for H > 8192), then as many groups (<= 4) as
// keep the CTA within its warp budget; as many row-slice slots as fit in
// 227 KB; one CTA per SM.  The budget is 22 warps (the 704-thread variant, 80
// registers) when rows have few slices (R + 1 <= 4): there the consumers'
// per-row epilogue, not HBM, sets the pace and more groups overlap more of it.
// With more slices a deeper sub-ring per group pays more: 16 warps.
frn::StreamPlan choose_stream(long long T, int H, int nslices, int quant, int num_sms) {
    const int ntiles = ceil_div(H / frn::kVecElems, frn::kTileVecs);
    const int tpw = ntiles <= 4 ? 1 : (ntiles <= 8 ? 2 : 4);
    frn::StreamPlan plan;
    plan.tiles_per_warp = tpw;
    plan.consumer_warps = ceil_div(ntiles, tpw);
    int max_warps = (tpw == 4 && nslices <= 4) ? frn::kStreamMaxThreads / 32 : 16;
    // a 17th warp (the 544-thread variant) when it buys a second group of 8 and
    // rows have at most 5 slices (H = 8192, R = 4: 80 -> 75 us without quant,
    // 114 -> 96 us with FP8 B; with R = 8 the single group's deeper sub-ring
    // measured 5% faster without quant)
    if (max_warps == 16 && plan.consumer_warps == 8 && nslices <= 5) max_warps = 17;
    int groups = g_force_groups.load(std::memory_order_relaxed);
    if (groups <= 0) groups = (max_warps - 1) / plan.consumer_warps;
    if (groups > frn::kStreamMaxGroups) groups = frn::kStreamMaxGroups;
    if (groups < 1) groups = 1;
    while (groups > 1 && (groups * plan.consumer_warps + 1) > max_warps) --groups;
    plan.groups = groups;
    const int slice = 2 * H;
    // Four tiles a warp re-read gamma every row; with a quant output the kernel
    // keeps it in a shared-memory slice (the quant epilogue sets the pace).
    // Measured on GB300: R = 8, T = 1000, H = 7168 FP8 B 32.4 -> 30.6 us;
    // R = 2, T = 8192, H = 16384 MXFP4 A 198 -> 174 us; without quant the
    // ring slot it takes cost 2-4 %.
    plan.gamma_smem = tpw == 4 && quant != 0 ? 1 : 0;
    const int gamma_bytes = plan.gamma_smem ? slice : 0;
    int slots = (frn::kStreamSmemLimit - frn::kStreamSmemReserve - gamma_bytes) / slice;
    if (slots > frn::kStreamMaxSlots) slots = frn::kStreamMaxSlots;
    plan.slots = slots;
    plan.smem_bytes = frn::stream_smem_bytes(slots, slice, groups, gamma_bytes);
    plan.grid = T < num_sms ? T : num_sms;
    return plan;
}

// Which kernel (measured on GB300 at H = 5120…8192, R = 1…8, T = 8…8192):
//  * a row that fits one CTA (H <= 8192 with R <= 8, or H <= 4096): the row
//    kernel at any T.  With one wide row per SM, its prefetch ahead and the
//    first wave's own prefetch (launch_fused) keep HBM busy between rows, and
//    it beats the stream kernel from two waves on in every output variant:
//    R = 8, H = 7168, T = 586 no quant 16.6 vs 17.7 us, FP8 B 18.5 vs 19.4,
//    MXFP4 B 17.8 vs 18.5; T = 880 23.5 vs 25.1 us; H = 8192, T = 586
//    19.0 vs 21.1 us; H = 5120 13.5 vs 15.6 us; R = 4, H = 8192, T = 1171
//    23.2 vs 24.0 us; R = 3, H = 7168, T = 1171 18.8 vs 19.7 us;
//  * a wider row, or one with R > 8: the two-tile row kernel where
//    two_tile_rows says so; else the stream kernel from one row per SM on,
//    the row kernel's clusters with an FP8 output.
int choose_kind(long long T, int H, int R, int quant, int num_sms) {
    const int forced = g_force_kernel.load(std::memory_order_relaxed);
    if (forced == kRows || forced == kStream) return forced;
    const int ntiles = ceil_div(H / frn::kVecElems, frn::kTileVecs);
    if (ntiles <= frn::kMaxTilesPerCta || wide_possible(ntiles, R)) return kRows;
    if (two_tile_rows(T, ntiles, R, quant, num_sms)) return kRows;
    // The other wider rows: the stream kernel from one row per SM on -- except
    // with an FP8 output, where its single consumer group's quant epilogue, which
    // nothing overlaps, is slower than the row kernel's clusters (R = 2,
    // T = 8192: H = 16384 FP8 A 266 vs 289 us, FP8 B 283 vs 287 us; H = 12288
    // FP8 A 203 vs 220 us; R = 8, T = 2048, H = 16384 FP8 A 136 vs 151 us;
    // without quant and with MXFP4 the stream kernel stays well ahead).
    if (quant == 1 || quant == 2) return kRows;
    return T >= num_sms ? kStream : kRows;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
    uintptr_t lo, hi;
    const char* name;
};

bool overlap(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void* p, long long bytes, const char* name) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes), name};
}

// One call's arguments.  quant: 0 = none, 1 = variant A (no bf16 y output),
// 2 = variant B.  The workspace fields are used by the unfused paths only.
struct Call {
    const void* const* partials;
    int R;
    const void* residual;
    const void* gamma;
    void* residual_out;
    void* y;
    void* q;
    float* scales;
    int64_t T;
    int H;
    float eps;
    int group_size;
    int quant;
    void* workspace;
    long long workspace_bytes;
    long long workspace_needed;
    bool no_residual_out;   // plain RMSNorm: residual_out is not written
    void* mx_scales;        // MXFP4 (quant 3, 4): E8M0 codes; q holds the packed E2M1 codes
};

bool is_mx(int quant) { return quant >= 3; }

// Everything that can be checked on the host: scalars, pointers, alignment,
// overlap.  Returns FRN_OK with *empty set when T == 0 (nothing to launch).
frn_status validate(const Call& c, bool* empty) {
    *empty = false;
    const int R = c.R, H = c.H;
    const int64_t T = c.T;
    if (R < 1) return fail(FRN_ERR_INVALID_ARG, "R=%d must be >= 1", R);
    if (R > FRN_MAX_PARTIALS) return fail(FRN_ERR_UNSUPPORTED, "R=%d exceeds %d", R, FRN_MAX_PARTIALS);
    if (T < 0) return fail(FRN_ERR_INVALID_ARG, "T=%lld must be >= 0", static_cast<long long>(T));
    if (H < 1) return fail(FRN_ERR_INVALID_ARG, "H=%d must be >= 1", H);
    if (H % 8 != 0 || H > FRN_MAX_HIDDEN)
        return fail(FRN_ERR_UNSUPPORTED, "H=%d must be a multiple of 8 and <= %d", H, FRN_MAX_HIDDEN);
    if (!std::isfinite(c.eps) || c.eps < 0.0f) return fail(FRN_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (is_mx(c.quant)) {
        if (H % 32 != 0) return fail(FRN_ERR_UNSUPPORTED, "H=%d: MXFP4 needs a multiple of 32", H);
    } else if (c.quant) {
        if (c.group_size < 1 || H % c.group_size != 0)
            return fail(FRN_ERR_INVALID_ARG, "group_size=%d must divide H=%d", c.group_size, H);
        if (c.group_size != FRN_QUANT_GROUP)
            return fail(FRN_ERR_UNSUPPORTED, "group_size=%d: only %d is built", c.group_size, FRN_QUANT_GROUP);
    }
    // Nothing to do (and zero-size buffers may legitimately be NULL).
    if (T == 0) {
        *empty = true;
        return ok();
    }
    if (!c.partials) return fail(FRN_ERR_INVALID_ARG, "partials array is NULL");
    for (int r = 0; r < R; ++r) {
        if (!c.partials[r]) return fail(FRN_ERR_INVALID_ARG, "partials[%d] is NULL", r);
        if (!aligned(c.partials[r], 16)) return fail(FRN_ERR_MISALIGNED, "partials[%d] not 16-byte aligned", r);
    }
    if (!c.gamma) return fail(FRN_ERR_INVALID_ARG, "gamma is NULL");
    if (!c.residual_out && !c.no_residual_out) return fail(FRN_ERR_INVALID_ARG, "residual_out is NULL");
    if (!c.y && !(c.quant == 1 || c.quant == 3)) return fail(FRN_ERR_INVALID_ARG, "y is NULL");
    if (c.quant && !is_mx(c.quant) && (!c.q || !c.scales)) return fail(FRN_ERR_INVALID_ARG, "q / scales is NULL");
    if (is_mx(c.quant) && (!c.q || !c.mx_scales)) return fail(FRN_ERR_INVALID_ARG, "q_fp4 / scales is NULL");
    if (!aligned(c.gamma, 16)) return fail(FRN_ERR_MISALIGNED, "gamma not 16-byte aligned");
    if (c.residual && !aligned(c.residual, 16)) return fail(FRN_ERR_MISALIGNED, "residual not 16-byte aligned");
    if (c.residual_out && !aligned(c.residual_out, 16))
        return fail(FRN_ERR_MISALIGNED, "residual_out not 16-byte aligned");
    if (c.y && !aligned(c.y, 16)) return fail(FRN_ERR_MISALIGNED, "y not 16-byte aligned");
    if (c.quant && !aligned(c.q, 16)) return fail(FRN_ERR_MISALIGNED, "q not 16-byte aligned");
    if (c.quant && !is_mx(c.quant) && !aligned(c.scales, 4))
        return fail(FRN_ERR_MISALIGNED, "scales not 4-byte aligned");
    if (T > (1LL << 40) / H) return fail(FRN_ERR_UNSUPPORTED, "T*H too large");
    if (c.workspace_needed > 0) {
        if (!c.workspace) return fail(FRN_ERR_INVALID_ARG, "workspace is NULL (%lld bytes needed)", c.workspace_needed);
        if (!aligned(c.workspace, 16)) return fail(FRN_ERR_MISALIGNED, "workspace not 16-byte aligned");
        if (c.workspace_bytes < c.workspace_needed)
            return fail(FRN_ERR_INVALID_ARG, "workspace has %lld bytes, %lld needed", c.workspace_bytes,
                        c.workspace_needed);
    }

    // Outputs (and the workspace) pairwise disjoint and disjoint from inputs,
    // except residual_out == residual (in place).
    const long long act = 2LL * T * H;
    Range outs[5];
    int nout = 0;
    if (c.residual_out) outs[nout++] = range_of(c.residual_out, act, "residual_out");
    if (c.y) outs[nout++] = range_of(c.y, act, "y");
    if (is_mx(c.quant)) {
        outs[nout++] = range_of(c.q, T * static_cast<long long>(H) / 2, "q_fp4");
        outs[nout++] = range_of(c.mx_scales, T * static_cast<long long>(H) / 32, "scales_e8m0");
    } else if (c.quant) {
        outs[nout++] = range_of(c.q, T * static_cast<long long>(H), "q");
        outs[nout++] = range_of(c.scales, 4LL * T * (H / c.group_size), "scales");
    }
    if (c.workspace_needed > 0) outs[nout++] = range_of(c.workspace, c.workspace_needed, "workspace");
    for (int a = 0; a < nout; ++a)
        for (int b = a + 1; b < nout; ++b)
            if (overlap(outs[a], outs[b]))
                return fail(FRN_ERR_INVALID_ARG, "%s and %s overlap", outs[a].name, outs[b].name);
    for (int a = 0; a < nout; ++a) {
        for (int r = 0; r < R; ++r)
            if (overlap(outs[a], range_of(c.partials[r], act, "partial")))
                return fail(FRN_ERR_INVALID_ARG, "%s overlaps partials[%d]", outs[a].name, r);
        if (overlap(outs[a], range_of(c.gamma, 2LL * H, "gamma")))
            return fail(FRN_ERR_INVALID_ARG, "%s overlaps gamma", outs[a].name);
        if (c.residual && overlap(outs[a], range_of(c.residual, act, "residual"))) {
            const bool in_place = c.residual_out != nullptr && (a == 0) && c.residual_out == c.residual;
            if (!in_place) return fail(FRN_ERR_INVALID_ARG, "%s overlaps residual", outs[a].name);
        }
    }
    return ok();
}

frn::Params make_params(const Call& c, const frn::RowPlan& rplan, const frn::StreamPlan& splan,
                        unsigned int* status) {
    frn::Params p;
    std::memset(&p, 0, sizeof(p));
    for (int r = 0; r < frn::kMaxPartials; ++r)
        p.partials[r] = static_cast<const uint4*>(c.partials[r < c.R ? r : 0]);
    p.residual = static_cast<const uint4*>(c.residual);
    p.gamma = static_cast<const uint4*>(c.gamma);
    p.residual_out = static_cast<uint4*>(c.residual_out);
    p.y = static_cast<uint4*>(c.y);
    if (is_mx(c.quant)) {
        p.q4 = static_cast<uint32_t*>(c.q);
        p.mx_scales = static_cast<uint8_t*>(c.mx_scales);
    } else {
        p.q = static_cast<uint2*>(c.q);
        p.scales = c.scales;
    }
    p.T = c.T;
    p.R = c.R;
    p.H = c.H;
    p.nvec = c.H / frn::kVecElems;
    p.ntiles = ceil_div(p.nvec, frn::kTileVecs);
    p.tiles_per_cta = rplan.tiles_per_cta;
    p.rows_per_cta = rplan.rows_per_cta;
    p.ctas_per_row = rplan.ctas_per_row;
    p.eps = c.eps;
    p.nslices = c.R + (c.residual ? 1 : 0);
    p.consumer_warps = splan.consumer_warps;
    p.groups = splan.groups;
    p.slots = splan.slots;
    p.slice_bytes = 2 * c.H;
    const long long lim = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.wait_limit_ns = static_cast<unsigned long long>(lim > 0 ? lim : kDefaultWaitLimitNs);
    p.inject_stall = g_inject_stall.load(std::memory_order_relaxed);
    p.error_word = status;
    return p;
}

// The fused epilogue (one kernel).  quant as in Call; the kernel writes c.y
// when it is not NULL.
// The L2 prefetch pays when the grid is at most about two waves (most CTAs
// start while the previous kernel on the stream drains, or while the first
// wave runs) and there is enough to fetch: a single-CTA row of at least 32 KB
// of loads, or a cluster CTA of at least 48 KB or a grid of at least 32
// cluster CTAs (with one request per input and CTA since the cluster CTAs
// prefetch their slice whole: the decode step R = 8, H = 7168, T = 8, 16, 32,
// 64 measured 9.54 -> 9.27 us per step with T = 8's 32 CTAs prefetching).
// Measured on GB300: below that, and for packed short rows (up to 2x slower
// at H = 256), the extra requests cost more than the overlap gives; beyond
// two waves it gains nothing.
// CTAs of a row-kernel launch resident on one SM: by threads (2048), CTAs
// (32) and the registers the kernel's launch bound holds (row_min_blocks).
long long row_ctas_per_sm(const frn::RowPlan& plan, int R) {
    if (plan.tiles_per_warp == 2) {
        // frn_row2_kernel: launch bound (1024, 1), so up to 64 registers a
        // thread; (640, 2), 48 registers, for R <= 2 at 608..640 threads
        const long long regs = R <= 2 && plan.threads > 576 && plan.threads <= 640 ? 48 : 64;
        const long long by_threads = 2048 / plan.threads, by_regs = 65536 / (plan.threads * regs);
        return by_threads < by_regs ? by_threads : by_regs;
    }
    const bool cluster = plan.ctas_per_row > 1;
    const int maxt = plan.rows_per_cta > 1 ? frn::kPackedThreads : (plan.threads > frn::kMaxThreads ? 1024 : frn::kMaxThreads);
    const int rmax = R <= 1 ? 1 : R <= 2 ? 2 : R <= 4 ? 4 : R <= 8 ? 8 : 16;
    int by_regs = frn::row_min_blocks(rmax, cluster, maxt);
    if (by_regs < 1) by_regs = 1;
    long long n = 2048 / plan.threads;
    if (n > 32) n = 32;
    return n < by_regs ? n : by_regs;
}

// Distance of the prefetch ahead, in rows: about 9.5 MB of loads (R = 8,
// H = 7168, one row per SM: 77 rows; R = 2, two rows per SM: 232), within a
// quarter of a wave and one wave, in whole CTA spans.  Measured on GB300 at
// H = 7168 against other fractions of a wave: R = 8 best at about half a wave
// (T = 1171: 30.5 us at 0.5, 31.5 at 1, 31.2 at 0.25; T = 4682: 106.7 /
// 108.4 / 109.4 us), R = 2 at 0.65-0.8 of a wave (T = 1024: 12.7 us at 0.65,
// 13.3 at 1; T = 8192 FP8 A 81.9 / 82.1 us); two waves ahead was 5-14 % slower.
long long ahead_rows(long long wave_rows, int rows_per_cta, int H, int nloads) {
    constexpr long long kAheadBytes = 9728LL * 1024;
    const long long row_bytes = 2LL * H * nloads;
    long long n = (kAheadBytes + row_bytes / 2) / row_bytes;
    const long long lo = wave_rows / 4 > 1 ? wave_rows / 4 : 1;
    if (n < lo) n = lo;
    if (n > wave_rows) n = wave_rows;
    n -= n % rows_per_cta;
    return n > 0 ? n : rows_per_cta;
}

bool prefetch_pays(const frn::RowPlan& plan, long long T, int H, int R, int sms) {
    if (plan.grid * plan.threads > 2048LL * sms || plan.rows_per_cta > 1) return false;
    // Wide and two-tile rows: only when the registers hold the whole grid at
    // once too (one or two rows an SM); beyond, the prefetch ahead takes over (R = 8,
    // H = 7168: T = 250 8.5 -> 8.0 us, T = 293 9.65 -> 9.1 us, T = 347
    // 12.3 -> 11.55 us).
    if ((plan.threads > frn::kMaxThreads || plan.tiles_per_warp == 2) && plan.ctas_per_row == 1 &&
        plan.grid > row_ctas_per_sm(plan, R) * sms)
        return false;
    const long long row_bytes = 2LL * H * (R + 1);
    if (plan.ctas_per_row == 1) return row_bytes >= 32 * 1024;
    return row_bytes / plan.ctas_per_row >= 48 * 1024 || T * plan.ctas_per_row >= 32;
}

frn_status launch_fused(const Call& c, int quant, int sms, frn_stream_t stream) {
    const int kind = choose_kind(c.T, c.H, c.R, quant, sms);
    const frn::RowPlan rplan = plan_rows(c.T, c.H, c.R, quant, sms);
    const frn::StreamPlan splan = choose_stream(c.T, c.H, c.R + (c.residual ? 1 : 0), quant, sms);
    if (kind == kRows && rplan.grid > 0x7FFFFFFFLL)
        return fail(FRN_ERR_UNSUPPORTED, "grid too large (T=%lld)", static_cast<long long>(c.T));
    unsigned int* status = nullptr;
    frn_status st = status_word(&status);
    if (st != FRN_OK) return st;
    frn::Params p = make_params(c, rplan, splan, status);
    // decode-sized grids (every CTA resident at once, so each starts while the
    // previous kernel drains): prefetch the row into L2 before the dependency wait
    const int pf = g_prefetch.load(std::memory_order_relaxed);
    p.prefetch_l2 = kind == kRows && (pf == 2 || (pf == 0 && prefetch_pays(rplan, c.T, c.H, c.R, sms)));
    // Beyond about two waves the row kernel is issue-bound rather than
    // latency-bound: warp 0 alone computes rstd (measured -1..4% time at
    // T = 8192, H = 7168, R = 2; +2% at T = 32, where it is left off).
    p.rstd_one_warp = kind == kRows && rplan.grid * rplan.threads > 2048LL * sms;
    // More rows than one wave holds, with R <= 2 (few loads in flight per SM)
    // or for wide and two-tile rows: each CTA prefetches its span of the rows a fixed
    // distance ahead (ahead_rows), one bulk request per input, and the first
    // wave's CTAs their own span before the dependency wait.  Measured on
    // GB300 at R = 2, H = 7168: +6% at T = 8192 without quant, +4..5% at
    // T = 512..1024; at T = 8192 FP8 A 92.1 -> 81.9 us, MXFP4 A 86.0 -> 76.6 us
    // (a request per warp and input instead measured -1% there).  Wide rows,
    // R = 8, H = 7168: T = 4682 115.0 -> 106.7 us, T = 586 19.5 -> 16.6 us,
    // T = 170 7.2 -> 7.0 us; for 512-thread rows it cost 4 %.  Cluster rows
    // with R > 2 from two waves on: R = 8, T = 2048, H = 16384 FP8 A 134.8 ->
    // 123.9 us, FP8 B 144.4 -> 137.8 us; R = 4, T = 4096 FP8 B 221.6 ->
    // 207.3 us (at T = 64 it cost 3 %).  The first wave's own prefetch, which
    // overlaps the previous kernel's tail: R = 8, T = 1171 31.7 -> 30.5 us,
    // T = 2341 58.4 -> 57.2 us.
    const long long wave_rows = row_ctas_per_sm(rplan, c.R) * sms * rplan.rows_per_cta / rplan.ctas_per_row;
    const bool wide = (rplan.threads > frn::kMaxThreads || rplan.tiles_per_warp == 2) && rplan.ctas_per_row == 1 &&
                      !rplan.staged;
    const bool cluster_waves = rplan.ctas_per_row > 1 && c.T >= 2 * wave_rows;
    if (kind == kRows && pf != 1 && (c.R <= 2 || wide || cluster_waves)) {
        if (wave_rows > 0 && c.T > wave_rows) {
            p.prefetch_ahead = ahead_rows(wave_rows, rplan.rows_per_cta, c.H, c.R + (c.residual ? 1 : 0));
            p.prefetch_own_below = wave_rows;
        }
    }
    const bool pdl = g_pdl.load(std::memory_order_relaxed) != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (kind == kStream) {
        switch (quant) {
            case 0: e = frn::launch_stream_norm(p, splan, s, pdl); break;
            case 1: e = frn::launch_stream_quant_a(p, splan, s, pdl); break;
            case 2: e = frn::launch_stream_quant_b(p, splan, s, pdl); break;
            case 3: e = frn::launch_stream_mx_a(p, splan, s, pdl); break;
            default: e = frn::launch_stream_mx_b(p, splan, s, pdl); break;
        }
    } else {
        switch (quant) {
            case 0: e = frn::launch_rows_norm(p, rplan, s, pdl); break;
            case 1: e = frn::launch_rows_quant_a(p, rplan, s, pdl); break;
            case 2: e = frn::launch_rows_quant_b(p, rplan, s, pdl); break;
            case 3: e = frn::launch_rows_mx_a(p, rplan, s, pdl); break;
            default: e = frn::launch_rows_mx_b(p, rplan, s, pdl); break;
        }
    }
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return ok();
}

frn_status run(const Call& c, frn_stream_t stream) {
    bool empty = false;
    frn_status st = validate(c, &empty);
    if (st != FRN_OK || empty) return st;
    int sms = 0;
    st = sm_count(&sms);
    if (st != FRN_OK) return st;
    return launch_fused(c, c.quant, sms, stream);
}

// ---------------------------------------------------------- unfused paths --

long long unfused_workspace(int64_t T, int H, int stages, bool quant, bool emit_y) {
    if (T <= 0 || H <= 0) return 0;
    long long b = 0;
    if (stages == 3 || !quant) b += 4LL * T * H;   // fp32 sum of the partials
    if (quant && !emit_y) b += 2LL * T * H;        // bf16 y between norm and quant
    return b;
}

frn_status run_unfused(Call c, int stages, frn_stream_t stream) {
    if (!(stages == 2 || (stages == 3 && c.quant)))
        return fail(FRN_ERR_INVALID_ARG, "stages=%d: 2, or 3 with quant", stages);
    c.workspace_needed = unfused_workspace(c.T, c.H, stages, c.quant != 0, c.y != nullptr);
    bool empty = false;
    frn_status st = validate(c, &empty);
    if (st != FRN_OK || empty) return st;
    int sms = 0;
    st = sm_count(&sms);
    if (st != FRN_OK) return st;
    const bool pdl = g_pdl.load(std::memory_order_relaxed) != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(c.workspace);
    const bool need_x = stages == 3 || !c.quant;
    float4* xsum = need_x ? reinterpret_cast<float4*>(ws) : nullptr;
    uint4* ytarget = c.y ? static_cast<uint4*>(c.y)
                         : reinterpret_cast<uint4*>(ws + (need_x ? 4LL * c.T * c.H : 0));
    Call norm = c;
    norm.y = ytarget;
    const frn::RowPlan rplan = choose_rows(c.T, c.H, c.R, 0, sms);
    const frn::StreamPlan splan = choose_stream(c.T, c.H, c.R + (c.residual ? 1 : 0), c.quant, sms);
    frn::Params p = make_params(norm, rplan, splan, nullptr);
    cudaError_t e = cudaSuccess;
    if (need_x) {
        e = frn::launch_reduce(p, xsum, sms, s, pdl);
        if (e == cudaSuccess) e = frn::launch_addnorm(p, xsum, ytarget, s, pdl);
    } else {
        st = launch_fused(norm, 0, sms, stream);
        if (st != FRN_OK) return st;
    }
    if (e == cudaSuccess && c.quant) e = frn::launch_quant(p, ytarget, sms, s, pdl);
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // namespace

FRN_EXPORT frn_status fused_reduce_rmsnorm(const void* const* partials, int R, const void* residual,
                                           const void* gamma, void* residual_out, void* y, int64_t T,
                                           int H, float eps, frn_stream_t stream) {
    const Call c{partials, R, residual, gamma, residual_out, y, nullptr, nullptr, T, H, eps, FRN_QUANT_GROUP,
                 0, nullptr, 0, 0, false};
    return run(c, stream);
}

FRN_EXPORT frn_status fused_reduce_rmsnorm_quant_per_group(const void* const* partials, int R,
                                                           const void* residual, const void* gamma,
                                                           void* residual_out, void* y, void* q_e4m3,
                                                           float* scales, int64_t T, int H, float eps,
                                                           int group_size, frn_stream_t stream) {
    const Call c{partials, R, residual, gamma, residual_out, y, q_e4m3, scales, T, H, eps, group_size,
                 y ? 2 : 1, nullptr, 0, 0, false};
    return run(c, stream);
}

FRN_EXPORT frn_status fused_reduce_rmsnorm_mxfp4(const void* const* partials, int R, const void* residual,
                                                 const void* gamma, void* residual_out, void* y, void* q_fp4,
                                                 void* scales_e8m0, int64_t T, int H, float eps,
                                                 frn_stream_t stream) {
    const Call c{partials, R, residual, gamma, residual_out, y, q_fp4, nullptr, T, H, eps, 32, y ? 4 : 3,
                 nullptr, 0, 0, false, scales_e8m0};
    return run(c, stream);
}

FRN_EXPORT frn_status frn_fused_add_rmsnorm(const void* x, const void* residual, const void* gamma,
                                            void* residual_out, void* y, int64_t T, int H, float eps,
                                            frn_stream_t stream) {
    const void* parts[1] = {x};
    const Call c{x ? parts : nullptr, 1, residual, gamma, residual_out, y, nullptr, nullptr, T, H, eps,
                 FRN_QUANT_GROUP, 0, nullptr, 0, 0, false};
    return run(c, stream);
}

FRN_EXPORT frn_status frn_rmsnorm(const void* x, const void* gamma, void* y, int64_t T, int H, float eps,
                                  frn_stream_t stream) {
    const void* parts[1] = {x};
    const Call c{x ? parts : nullptr, 1, nullptr, gamma, nullptr, y, nullptr, nullptr, T, H, eps,
                 FRN_QUANT_GROUP, 0, nullptr, 0, 0, true};
    return run(c, stream);
}

FRN_EXPORT int64_t frn_unfused_workspace_bytes(int64_t T, int H, int stages, int quant, int emit_y) {
    if (!(stages == 2 || (stages == 3 && quant))) return -1;
    return unfused_workspace(T, H, stages, quant != 0, emit_y != 0);
}

FRN_EXPORT frn_status frn_unfused_reduce_rmsnorm(const void* const* partials, int R, const void* residual,
                                                 const void* gamma, void* residual_out, void* y, void* q_e4m3,
                                                 float* scales, int64_t T, int H, float eps, int group_size,
                                                 int stages, void* workspace, int64_t workspace_bytes,
                                                 frn_stream_t stream) {
    const int quant = q_e4m3 || scales ? (y ? 2 : 1) : 0;
    const Call c{partials, R, residual, gamma, residual_out, y, q_e4m3, scales, T, H, eps,
                 quant ? group_size : FRN_QUANT_GROUP, quant, workspace, workspace_bytes, 0, false};
    return run_unfused(c, stages, stream);
}

// ------------------------------------------------ no-allocation variant --
//
// The unfused paths need scratch: the fp32 sum of the partials and, without a
// y output, the bf16 y.  Some callers cannot allocate it: code running while a
// CUDA graph is being captured in the default (global) capture mode, where
// cudaMalloc is not allowed; serving engines that give nearly all device memory
// to their own pool at start-up and forbid allocation on the hot path; plugins
// handed raw pointers and no allocator.  For them this variant keeps its
// scratch in the array below, a fixed part of the library's device image: every
// GPU that loads the library holds FRN_STATIC_WORKSPACE_BYTES of it until the
// process exits, and no call allocates or frees anything.
static __device__ __align__(256) unsigned char g_frn_static_workspace[FRN_STATIC_WORKSPACE_BYTES];

namespace {

std::atomic<void*> g_static_ws_addr[kMaxDevices];

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
frn_status static_workspace(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(FRN_ERR_UNSUPPORTED, "device %d out of range", dev);
    void* a = g_static_ws_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        e = cudaGetSymbolAddress(&a, g_frn_static_workspace);
        if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_static_ws_addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return FRN_OK;
}

}  // namespace

FRN_EXPORT frn_status frn_unfused_reduce_rmsnorm_noalloc(const void* const* partials, int R, const void* residual,
                                                         const void* gamma, void* residual_out, void* y,
                                                         void* q_e4m3, float* scales, int64_t T, int H, float eps,
                                                         int group_size, int stages, frn_stream_t stream) {
    const int quant = q_e4m3 || scales ? (y ? 2 : 1) : 0;
    if (!(stages == 2 || (stages == 3 && quant)))
        return fail(FRN_ERR_INVALID_ARG, "stages=%d: 2, or 3 with quant", stages);
    const long long need = unfused_workspace(T, H, stages, quant != 0, y != nullptr);
    if (need > FRN_STATIC_WORKSPACE_BYTES)
        return fail(FRN_ERR_UNSUPPORTED,
                    "needs %lld bytes of scratch; the static workspace holds %lld (pass your own to "
                    "frn_unfused_reduce_rmsnorm instead)",
                    need, static_cast<long long>(FRN_STATIC_WORKSPACE_BYTES));
    void* ws = nullptr;
    if (T > 0) {
        frn_status st = static_workspace(&ws);
        if (st != FRN_OK) return st;
    }
    // The array is fully overwritten before it is read (the fp32 sum, then y),
    // so nothing in it has to start at zero.
    const Call c{partials, R, residual, gamma, residual_out, y, q_e4m3, scales, T, H, eps,
                 quant ? group_size : FRN_QUANT_GROUP, quant, ws, FRN_STATIC_WORKSPACE_BYTES, 0, false};
    return run_unfused(c, stages, stream);
}

FRN_EXPORT const char* frn_status_string(frn_status s) {
    switch (s) {
        case FRN_OK: return "FRN_OK";
        case FRN_ERR_INVALID_ARG: return "FRN_ERR_INVALID_ARG";
        case FRN_ERR_UNSUPPORTED: return "FRN_ERR_UNSUPPORTED";
        case FRN_ERR_MISALIGNED: return "FRN_ERR_MISALIGNED";
        case FRN_ERR_CUDA: return "FRN_ERR_CUDA";
        case FRN_ERR_TIMEOUT: return "FRN_ERR_TIMEOUT";
    }
    return "FRN_ERR_UNKNOWN";
}

FRN_EXPORT const char* frn_last_error_detail(void) { return g_detail; }

// 2.0.0: frn_query_launch takes has_residual; frn_launch_plan has `staged`;
// frn_floor_launch added.
FRN_EXPORT int frn_version(void) { return 20000; }

FRN_EXPORT frn_status frn_set_l2_prefetch(int mode) {
    if (mode < 0 || mode > 2) return fail(FRN_ERR_INVALID_ARG, "l2 prefetch mode=%d must be 0..2", mode);
    g_prefetch.store(mode, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_set_pdl(int enable) {
    g_pdl.store(enable ? 1 : 0, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_set_ctas_per_row(int ctas_per_row) {
    if (ctas_per_row < 0 || ctas_per_row > 16)
        return fail(FRN_ERR_INVALID_ARG, "ctas_per_row=%d must be 0..16", ctas_per_row);
    g_force_ctas.store(ctas_per_row, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_set_kernel(int kernel) {
    if (kernel < 0 || kernel > 2) return fail(FRN_ERR_INVALID_ARG, "kernel=%d must be 0, 1 or 2", kernel);
    g_force_kernel.store(kernel, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_set_stream_groups(int groups) {
    if (groups < 0 || groups > frn::kStreamMaxGroups)
        return fail(FRN_ERR_INVALID_ARG, "groups=%d must be 0..%d", groups, frn::kStreamMaxGroups);
    g_force_groups.store(groups, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_set_test_hooks(int inject_stall, int64_t wait_limit_ns) {
    g_inject_stall.store(inject_stall ? 1 : 0, std::memory_order_relaxed);
    g_wait_limit_ns.store(wait_limit_ns > 0 ? static_cast<long long>(wait_limit_ns) : 0, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_device_status(int clear) {
    unsigned int* addr = nullptr;
    frn_status st = status_word(&addr);
    if (st != FRN_OK) return st;
    unsigned int word = 0;
    cudaError_t e = cudaMemcpy(&word, addr, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
    if (clear && word) {
        const unsigned int zero = 0;
        e = cudaMemcpy(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
    }
    if (word & frn::kErrWaitTimeout) return fail(FRN_ERR_TIMEOUT, "a bounded device-side wait ran out");
    return ok();
}

FRN_EXPORT frn_status frn_plan_launch(int64_t T, int H, int R, int quant, int has_residual, int num_sms,
                                      frn_launch_plan* out) {
    if (R < 1 || R > FRN_MAX_PARTIALS || T < 1 || H < 8 || H % 8 != 0 || H > FRN_MAX_HIDDEN || quant < 0 ||
        quant > 4 || num_sms < 1 || !out)
        return fail(FRN_ERR_INVALID_ARG, "bad sizes");
    std::memset(out, 0, sizeof(*out));
    const int kind = choose_kind(T, H, R, quant, num_sms);
    out->kernel = kind;
    if (kind == kStream) {
        const frn::StreamPlan plan = choose_stream(T, H, R + (has_residual ? 1 : 0), quant, num_sms);
        out->ctas_per_row = 1;
        out->rows_per_cta = 1;
        out->tiles_per_warp = plan.tiles_per_warp;
        out->groups = plan.groups;
        out->consumer_warps = plan.consumer_warps;
        out->slots = plan.slots;
        out->smem_bytes = plan.smem_bytes;
        out->threads = (plan.groups * plan.consumer_warps + 1) * 32;
        out->grid = plan.grid;
    } else {
        const frn::RowPlan plan = plan_rows(T, H, R, quant, num_sms);
        out->ctas_per_row = plan.ctas_per_row;
        out->rows_per_cta = plan.rows_per_cta;
        out->tiles_per_warp = plan.tiles_per_warp;
        out->tiles_per_cta = plan.tiles_per_cta;
        out->threads = plan.threads;
        out->grid = plan.grid;
        out->staged = plan.staged;
    }
    return ok();
}

FRN_EXPORT frn_status frn_query_launch(int64_t T, int H, int R, int quant, int has_residual, int* kernel,
                                       int* ctas_per_row, int* threads_per_cta, int64_t* grid_ctas) {
    if (R < 1 || R > FRN_MAX_PARTIALS || T < 0 || H < 8 || H % 8 != 0 || H > FRN_MAX_HIDDEN || quant < 0 ||
        quant > 4)
        return fail(FRN_ERR_INVALID_ARG, "bad sizes");
    int sms = 0;
    frn_status st = sm_count(&sms);
    if (st != FRN_OK) return st;
    // the plan of a call with these sizes on this device's SM count (T = 0
    // launches nothing; it reports the plan of one row)
    frn_launch_plan plan;
    st = frn_plan_launch(T > 0 ? T : 1, H, R, quant, has_residual, sms, &plan);
    if (st != FRN_OK) return st;
    if (kernel) *kernel = plan.kernel;
    if (ctas_per_row) *ctas_per_row = plan.ctas_per_row;
    if (threads_per_cta) *threads_per_cta = plan.threads;
    if (grid_ctas) *grid_ctas = T > 0 ? plan.grid : 0;
    return ok();
}
