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
std::atomic<int> g_force_ctas{0};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

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

// Launch shape.  A row's ntiles warp tiles go to C CTAs of a cluster.  The
// results do not depend on this choice (the reduction tree is fixed by H).
frn::Plan choose_plan(long long T, int H, int num_sms) {
    const int nvec = H / frn::kVecElems;
    const int ntiles = ceil_div(nvec, frn::kTileVecs);
    const int cmin = ceil_div(ntiles, frn::kMaxTilesPerCta);
    const int cmax = ntiles < 8 ? ntiles : 8;
    int C;
    const int forced = g_force_ctas.load(std::memory_order_relaxed);
    if (forced > 0) {
        C = forced < cmin ? cmin : (forced > cmax ? cmax : forced);
    } else {
        // Few rows: spread each row over more SMs (down to 4 warps per CTA)
        // until the rows alone give about two CTAs per SM.
        C = cmin;
        while (C < cmax && T * C < 2LL * num_sms && ceil_div(ntiles, C + 1) >= 4) ++C;
    }
    const int tpc = ceil_div(ntiles, C);
    C = ceil_div(ntiles, tpc);   // no empty CTA
    frn::Plan plan;
    plan.ctas_per_row = C;
    plan.tiles_per_cta = tpc;
    plan.threads = tpc * 32;
    plan.grid = T * C;
    return plan;
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

// Shared by both entry points.  quant: 0 = none, 1 = variant A (y NULL),
// 2 = variant B.
frn_status run(const void* const* partials, int R, const void* residual, const void* gamma,
               void* residual_out, void* y, void* q, float* scales, int64_t T, int H,
               float eps, int group_size, int quant, frn_stream_t stream) {
    // ---- scalar arguments
    if (R < 1) return fail(FRN_ERR_INVALID_ARG, "R=%d must be >= 1", R);
    if (R > FRN_MAX_PARTIALS) return fail(FRN_ERR_UNSUPPORTED, "R=%d exceeds %d", R, FRN_MAX_PARTIALS);
    if (T < 0) return fail(FRN_ERR_INVALID_ARG, "T=%lld must be >= 0", static_cast<long long>(T));
    if (H < 1) return fail(FRN_ERR_INVALID_ARG, "H=%d must be >= 1", H);
    if (H % 8 != 0 || H > FRN_MAX_HIDDEN)
        return fail(FRN_ERR_UNSUPPORTED, "H=%d must be a multiple of 8 and <= %d", H, FRN_MAX_HIDDEN);
    if (!std::isfinite(eps) || eps < 0.0f) return fail(FRN_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (quant) {
        if (group_size < 1 || H % group_size != 0)
            return fail(FRN_ERR_INVALID_ARG, "group_size=%d must divide H=%d", group_size, H);
        if (group_size != FRN_QUANT_GROUP)
            return fail(FRN_ERR_UNSUPPORTED, "group_size=%d: only %d is built", group_size, FRN_QUANT_GROUP);
    }
    // Nothing to do (and zero-size buffers may legitimately be NULL).
    if (T == 0) return ok();
    // ---- pointers
    if (!partials) return fail(FRN_ERR_INVALID_ARG, "partials array is NULL");
    for (int r = 0; r < R; ++r) {
        if (!partials[r]) return fail(FRN_ERR_INVALID_ARG, "partials[%d] is NULL", r);
        if (!aligned(partials[r], 16)) return fail(FRN_ERR_MISALIGNED, "partials[%d] not 16-byte aligned", r);
    }
    if (!gamma) return fail(FRN_ERR_INVALID_ARG, "gamma is NULL");
    if (!residual_out) return fail(FRN_ERR_INVALID_ARG, "residual_out is NULL");
    if (quant != 1 && !y) return fail(FRN_ERR_INVALID_ARG, "y is NULL");
    if (quant && (!q || !scales)) return fail(FRN_ERR_INVALID_ARG, "q / scales is NULL");
    if (!aligned(gamma, 16)) return fail(FRN_ERR_MISALIGNED, "gamma not 16-byte aligned");
    if (residual && !aligned(residual, 16)) return fail(FRN_ERR_MISALIGNED, "residual not 16-byte aligned");
    if (!aligned(residual_out, 16)) return fail(FRN_ERR_MISALIGNED, "residual_out not 16-byte aligned");
    if (y && !aligned(y, 16)) return fail(FRN_ERR_MISALIGNED, "y not 16-byte aligned");
    if (quant && !aligned(q, 16)) return fail(FRN_ERR_MISALIGNED, "q not 16-byte aligned");
    if (quant && !aligned(scales, 4)) return fail(FRN_ERR_MISALIGNED, "scales not 4-byte aligned");
    // T * H bf16 elements must be addressable and the grid must fit.
    if (T > (1LL << 40) / H) return fail(FRN_ERR_UNSUPPORTED, "T*H too large");

    // ---- overlap: outputs pairwise disjoint and disjoint from inputs, except
    // residual_out == residual (in place).
    const long long act = 2LL * T * H;
    Range outs[4];
    int nout = 0;
    outs[nout++] = range_of(residual_out, act, "residual_out");
    if (y) outs[nout++] = range_of(y, act, "y");
    if (quant) {
        outs[nout++] = range_of(q, T * static_cast<long long>(H), "q");
        outs[nout++] = range_of(scales, 4LL * T * (H / group_size), "scales");
    }
    for (int a = 0; a < nout; ++a)
        for (int b = a + 1; b < nout; ++b)
            if (overlap(outs[a], outs[b]))
                return fail(FRN_ERR_INVALID_ARG, "outputs %s and %s overlap", outs[a].name, outs[b].name);
    for (int a = 0; a < nout; ++a) {
        for (int r = 0; r < R; ++r)
            if (overlap(outs[a], range_of(partials[r], act, "partial")))
                return fail(FRN_ERR_INVALID_ARG, "output %s overlaps partials[%d]", outs[a].name, r);
        if (overlap(outs[a], range_of(gamma, 2LL * H, "gamma")))
            return fail(FRN_ERR_INVALID_ARG, "output %s overlaps gamma", outs[a].name);
        if (residual && overlap(outs[a], range_of(residual, act, "residual"))) {
            const bool in_place = (a == 0) && residual_out == residual;
            if (!in_place) return fail(FRN_ERR_INVALID_ARG, "output %s overlaps residual", outs[a].name);
        }
    }

    int sms = 0;
    frn_status st = sm_count(&sms);
    if (st != FRN_OK) return st;
    const frn::Plan plan = choose_plan(T, H, sms);
    if (plan.grid > 0x7FFFFFFFLL) return fail(FRN_ERR_UNSUPPORTED, "grid too large (T=%lld)", static_cast<long long>(T));

    frn::Params p;
    std::memset(&p, 0, sizeof(p));
    for (int r = 0; r < frn::kMaxPartials; ++r)
        p.partials[r] = static_cast<const uint4*>(partials[r < R ? r : 0]);
    p.residual = static_cast<const uint4*>(residual);
    p.gamma = static_cast<const uint4*>(gamma);
    p.residual_out = static_cast<uint4*>(residual_out);
    p.y = static_cast<uint4*>(y);
    p.q = static_cast<uint2*>(q);
    p.scales = scales;
    p.T = T;
    p.R = R;
    p.H = H;
    p.nvec = H / frn::kVecElems;
    p.ntiles = ceil_div(p.nvec, frn::kTileVecs);
    p.tiles_per_cta = plan.tiles_per_cta;
    p.ctas_per_row = plan.ctas_per_row;
    p.eps = eps;

    const bool pdl = g_pdl.load(std::memory_order_relaxed) != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (quant) {
        case 0: e = frn::launch_norm(p, plan, s, pdl); break;
        case 1: e = frn::launch_quant_a(p, plan, s, pdl); break;
        default: e = frn::launch_quant_b(p, plan, s, pdl); break;
    }
    if (e != cudaSuccess) return fail(FRN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // namespace

FRN_EXPORT frn_status fused_reduce_rmsnorm(const void* const* partials, int R, const void* residual,
                                           const void* gamma, void* residual_out, void* y, int64_t T,
                                           int H, float eps, frn_stream_t stream) {
    return run(partials, R, residual, gamma, residual_out, y, nullptr, nullptr, T, H, eps,
               FRN_QUANT_GROUP, 0, stream);
}

FRN_EXPORT frn_status fused_reduce_rmsnorm_quant_per_group(const void* const* partials, int R,
                                                           const void* residual, const void* gamma,
                                                           void* residual_out, void* y, void* q_e4m3,
                                                           float* scales, int64_t T, int H, float eps,
                                                           int group_size, frn_stream_t stream) {
    return run(partials, R, residual, gamma, residual_out, y, q_e4m3, scales, T, H, eps, group_size,
               y ? 2 : 1, stream);
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

FRN_EXPORT int frn_version(void) { return 100; }

FRN_EXPORT frn_status frn_set_pdl(int enable) {
    g_pdl.store(enable ? 1 : 0, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_set_ctas_per_row(int ctas_per_row) {
    if (ctas_per_row < 0 || ctas_per_row > 8)
        return fail(FRN_ERR_INVALID_ARG, "ctas_per_row=%d must be 0..8", ctas_per_row);
    g_force_ctas.store(ctas_per_row, std::memory_order_relaxed);
    return ok();
}

FRN_EXPORT frn_status frn_query_launch(int64_t T, int H, int R, int quant, int* ctas_per_row,
                                       int* threads_per_cta, int64_t* grid_ctas) {
    (void)quant;
    if (R < 1 || T < 0 || H < 8 || H % 8 != 0 || H > FRN_MAX_HIDDEN)
        return fail(FRN_ERR_INVALID_ARG, "bad sizes");
    int sms = 0;
    frn_status st = sm_count(&sms);
    if (st != FRN_OK) return st;
    const frn::Plan plan = choose_plan(T, H, sms);
    if (ctas_per_row) *ctas_per_row = plan.ctas_per_row;
    if (threads_per_cta) *threads_per_cta = plan.threads;
    if (grid_ctas) *grid_ctas = plan.grid;
    return ok();
}
