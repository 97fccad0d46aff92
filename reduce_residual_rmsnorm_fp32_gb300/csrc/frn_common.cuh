// frn_common.cuh -- shared device code of the fused reduce + residual add +
// RMSNorm (+ per-group-128 dynamic FP8 e4m3) epilogue for sm_103a: parameter
// block, PTX wrappers, number formats and the per-vector arithmetic that both
// kernel families (frn_rows.cuh, frn_stream.cuh) run identically.
//
// The op, per token row (include/frn.h has the full contract):
//   x_hat = sum_r f32(P[r]) (rank order) + f32(residual);  residual_out = bf16(x_hat)
//   y = bf16((x * gamma) * rstd),  rstd = 1/sqrt(sum(x^2)/H + eps),  x = f32(residual_out)
//   per 128-group of y: s = max|y| / 448, q = e4m3(y / s)
// following the replaced subgraph all_reduce -> (fused_add_)rms_norm of the
// "ROCm AITER fused all-reduce + RMSNorm" page (vLLM PR 37646 summary, key source
// snippets) and the per-1x128 quant of the normalised bf16 activation of the
// "AMD fused AllReduce-RMSNorm quant kernel" page (SGLang PR 24651 summary).
//
// Work decomposition shared by both kernels:
//  * A row of H bf16 is split into 16-byte vectors of 8 elements (nvec = H/8) and
//    the vectors into "tiles" of 32; lane l of the warp owning tile k holds
//    vector 32*k + l.  A quant group (128 elements) is an aligned half-warp.
//  * Sum of squares: a fixed tree whose shape depends on H alone -- an fp32 FMA
//    chain over the 8 elements of a vector, a 32-lane xor butterfly within the
//    tile, then tile slots k and k+32 paired and a second butterfly over the 32
//    pairs (absent tiles are +0).  Every lane ends with the same bits, and a row
//    gives the same bits whichever kernel, launch shape or T computes it.
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
constexpr int kMaxTiles = 64;       // H <= 16384 (two tile slots per lane)
constexpr int kMaxThreads = kMaxTilesPerCta * 32;
constexpr int kGroup = 128;         // quant group (elements)

// Output variants: norm only; per-group-128 e4m3 without (A) / with (B) the
// bf16 y; MXFP4 (32-blocks, E8M0 scale, E2M1) without (A) / with (B) y.
enum Mode : int { kNorm = 0, kQuantA = 1, kQuantB = 2, kMxA = 3, kMxB = 4 };

__host__ __device__ constexpr bool mode_writes_y(int m) { return m == kNorm || m == kQuantB || m == kMxB; }
__host__ __device__ constexpr bool mode_fp8(int m) { return m == kQuantA || m == kQuantB; }
__host__ __device__ constexpr bool mode_mx(int m) { return m == kMxA || m == kMxB; }

struct Params {
    const uint4* partials[kMaxPartials];
    const uint4* residual;   // nullptr: zeros
    const uint4* gamma;
    uint4* residual_out;     // nullptr: not stored (plain RMSNorm)
    uint4* y;                // bf16 output (kNorm, kQuantB)
    uint2* q;                // e4m3 codes, 8 per vector (kQuantA, kQuantB)
    float* scales;           // [T, H/128]
    uint32_t* q4;            // MXFP4: 8 E2M1 codes per vector, element 2i in the low nibble
    uint8_t* mx_scales;      // MXFP4: E8M0 codes [T, H/32]
    long long T;
    int R;
    int H;
    int nvec;                // H / 8
    int ntiles;              // ceil(nvec / 32)
    int prefetch_l2;         // row kernel: prefetch the row into L2 before the grid dependency wait
    long long prefetch_ahead;  // row kernel: also prefetch the row this many rows ahead (0: no)
    long long prefetch_own_below;  // row kernel: CTAs whose first row is below this index (the first
                                   // wave) also prefetch their own span before the dependency wait
    int rstd_one_warp;       // single-CTA row kernel: warp 0 alone computes rstd and shares it
    int tiles_per_cta;       // warps per row in a CTA (row kernel)
    int rows_per_cta;        // single-CTA row kernel: consecutive rows per CTA
    int ctas_per_row;        // cluster size (row kernel)
    float eps;
    // stream kernel
    int nslices;             // bulk copies per row: R partials, then the residual if any
    int consumer_warps;      // per consumer group
    int groups;              // consumer groups, each taking every groups-th row of the CTA
    int slots;               // shared-memory ring slots, one row slice (2*H bytes) each
    int slice_bytes;
    unsigned long long wait_limit_ns;   // bound on every mbarrier wait
    int inject_stall;        // test hook: stream kernel never issues its first copy, cluster rows
                             // never push tile 0's sum (either forces a bounded wait to run out)
    unsigned int* error_word;           // device status word, set on a timed-out wait
};

// Bits of the device status word.
constexpr unsigned kErrWaitTimeout = 1u;

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

// Relaxed arrival that must follow the computation of `after`: the dummy input
// makes the compiler keep that computation (and the loads it consumed) ahead
// of the arrival, and in-order issue keeps the hardware from reordering them.
__device__ __forceinline__ void cluster_arrive_relaxed_after(float after) {
    asm volatile("barrier.cluster.arrive.relaxed.aligned; // %0" ::"f"(after) : "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of `local` in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
    return remote;
}

// Store a float into another CTA's shared memory and count its 4 bytes against
// that CTA's mbarrier (the remote CTA waits on the barrier for the data).
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(remote_addr), "r"(__float_as_uint(v)), "r"(remote_bar) : "memory");
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

// acc[2i] += f32(lo half of w), acc[2i+1] += f32(hi half): the mixed-precision
// add takes the bf16 straight from the register half.  Widening bf16 is exact,
// so this is the same single-rounded fp32 add as unpacking first.
__device__ __forceinline__ void add2_bf16(float& a0, float& a1, uint32_t w) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\t"
        "add.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(a0), "+f"(a1) : "r"(w));
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 v) {
    add2_bf16(acc[0], acc[1], v.x);
    add2_bf16(acc[2], acc[3], v.y);
    add2_bf16(acc[4], acc[5], v.z);
    add2_bf16(acc[6], acc[7], v.w);
}

// s = fma(x_lo, x_lo, s); s = fma(x_hi, x_hi, s) with bf16 x: the product of two
// bf16 values is exact in fp32, so this is the fp32 FMA of the widened values.
__device__ __forceinline__ float sumsq2_bf16(float s, uint32_t w) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "fma.rn.f32.bf16 %0, lo, lo, %0;\n\t"
        "fma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
        : "+f"(s) : "r"(w));
    return s;
}

// max |element| of a packed bf16 pair set, as a bf16 pair (exact).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b32 a;\n\t"
        "abs.bf16x2 a, %2;\n\t"
        "max.bf16x2 %0, %1, a;\n\t}"
        : "=r"(r) : "r"(m), "r"(w));
    return r;
}

__device__ __forceinline__ float butterfly_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------- mbarrier + bulk copy ----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(bar), "r"(bytes) : "memory");
}

// One bounded try: the thread may sleep in the instruction until the phase
// completes or about `hint_ns` pass, so a waiting warp takes no issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns = 20000) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity, giving up after about
// limit_ns nanoseconds (returns false then).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// 1-D bulk copy global -> shared (TMA, non-tensor form), completing `bytes`
// transaction bytes on the mbarrier.  Both addresses 16-byte aligned, size a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Ask the TMA unit to bring [src, src + bytes) into L2 (16-byte aligned, a
// multiple of 16 bytes).  A hint only: no register receives data from it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------- per-vector arithmetic ----

// Sum of squares of one tile: an fp32 FMA chain over the 8 elements of this
// lane's bf16 vector, in element order; xor butterfly over the 32 lanes.
__device__ __forceinline__ float tile_sumsq(const uint4 ro) {
    float s = 0.0f;
    s = sumsq2_bf16(s, ro.x);
    s = sumsq2_bf16(s, ro.y);
    s = sumsq2_bf16(s, ro.z);
    s = sumsq2_bf16(s, ro.w);
    return butterfly_sum(s);
}

// rstd from the row's tile slots `lane` (lo) and `lane + 32` (hi).
__device__ __forceinline__ float row_rstd(float lo, float hi, int H, float eps) {
    const float ss = butterfly_sum(__fadd_rn(lo, hi));
    return __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(H)), eps));
}

// x * gamma for a packed bf16 pair of each, straight from the register halves:
// the mixed-precision FMA with a -0 addend (-0 keeps the sign of a zero
// product) rounds the exact product once, like an fp32 multiply of the widened
// values; inside fp32's range the product of two bf16 values is exact.
__device__ __forceinline__ void mul2_bf16(float& p0, float& p1, uint32_t xw, uint32_t gw) {
    asm("{\n\t.reg .b16 xl, xh, gl, gh;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "mov.b32 {gl, gh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, xl, gl, 0f80000000;\n\t"
        "fma.rn.f32.bf16 %1, xh, gh, 0f80000000;\n\t}"
        : "=f"(p0), "=f"(p1) : "r"(xw), "r"(gw));
}

// y = bf16(fl32((x * gamma) * rstd)) for one vector of bf16 x: x * gamma is
// exact (inside fp32's range), so y takes one fp32 rounding of x * gamma * rstd
// before the bf16 one.
// MIXED forms x * gamma with the mixed-precision FMA (fewer instructions);
// otherwise both are widened first and multiplied in fp32 (fewer live
// registers in register-capped kernels).  The two give the same bits.
template <bool MIXED = true>
__device__ __forceinline__ void xgamma8(const uint4 xb, const uint4 g, float (&xg)[8]) {
    if constexpr (MIXED) {
        mul2_bf16(xg[0], xg[1], xb.x, g.x);
        mul2_bf16(xg[2], xg[3], xb.y, g.y);
        mul2_bf16(xg[4], xg[5], xb.z, g.z);
        mul2_bf16(xg[6], xg[7], xb.w, g.w);
    } else {
        float gf[8];
        unpack8(xb, xg);
        unpack8(g, gf);
#pragma unroll
        for (int i = 0; i < 8; ++i) xg[i] = __fmul_rn(xg[i], gf[i]);
    }
}

// y from the x * gamma products (xgamma8) and rstd.
__device__ __forceinline__ uint4 y_from_xgamma(float (&xg)[8], float rstd) {
#pragma unroll
    for (int i = 0; i < 8; ++i) xg[i] = __fmul_rn(xg[i], rstd);
    return pack8(xg);
}

template <bool MIXED = true>
__device__ __forceinline__ uint4 rms_y(const uint4 xb, float rstd, const uint4 g) {
    float xg[8];
    xgamma8<MIXED>(xb, g, xg);
    return y_from_xgamma(xg, rstd);
}

// max |element| of one bf16 vector, as fp32 (exact).
__device__ __forceinline__ float vec_absmax(const uint4 yb) {
    uint32_t mp = absmax_bf16x2(0u, yb.x);
    mp = absmax_bf16x2(mp, yb.y);
    mp = absmax_bf16x2(mp, yb.z);
    mp = absmax_bf16x2(mp, yb.w);
    return fmaxf(__uint_as_float(mp << 16), __uint_as_float(mp & 0xFFFF0000u));
}

// max over an aligned group of `lanes` lanes (16: a quant group, 4: an MX block).
template <int LANES>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int m = LANES / 2; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

// The group's absmax of y from x * gamma, before rstd is known: every y is
// bf16(fl32(x*gamma * rstd)) with rstd > 0, and both roundings are monotonic
// and odd, so max |y| = bf16(fl32(max |x*gamma| * rstd)) -- the same value as
// the max over the rounded y.
template <int LANES>
__device__ __forceinline__ float xgamma_group_absmax(const float (&xg)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(xg[i]));
    return group_max<LANES>(m);
}

__device__ __forceinline__ float y_absmax_from_xgamma(float amax_xg, float rstd) {
    return __uint_as_float(pack_bf16x2(__fmul_rn(amax_xg, rstd), 0.0f) << 16);
}

// Per-group dynamic e4m3 of one bf16 y vector, given the group's absmax of y
// (fp32; a quant group of 128 elements is an aligned half-warp).
// s = absmax / 448; q = e4m3(y / s), q = 0 when s == 0.
__device__ __forceinline__ void quant8_amax(const uint4 yb, float amax, uint2& qq, float& sc) {
    float yq[8];
    unpack8(yb, yq);
    if (amax >= 0x1p-60f) {
        // absmax / 448, correctly rounded, without a divide: RN(absmax * RN(1/448))
        // and one FMA correction (Markstein's theorem); checked exhaustively for
        // every bf16 significand of absmax.
        constexpr float kInv448 = 1.0f / 448.0f;
        const float q0 = __fmul_rn(amax, kInv448);
        const float rem = __fmaf_rn(-448.0f, q0, amax);
        sc = __fmaf_rn(rem, kInv448, q0);
    } else {
        sc = __fdiv_rn(amax, 448.0f);
    }
    qq = make_uint2(0u, 0u);
    if (sc != 0.0f) {
        float qv[8];
        if (sc >= 0x1p-64f) {
            // y / s, correctly rounded, from one reciprocal per group:
            // q0 = RN(y * RN(1/s)), then one FMA correction with the residual
            // y - s*q0 (Markstein's theorem).  Checked exhaustively for every
            // bf16 significand of y against every significand s = RN(absmax/448)
            // can take; powers of two scale these exactly in this range.
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
}

// Per-group dynamic e4m3 of one bf16 y vector; all 32 lanes must call it.
__device__ __forceinline__ void quant8(const uint4 yb, uint2& qq, float& sc) {
    quant8_amax(yb, group_max<16>(vec_absmax(yb)), qq, sc);
}

// OCP Microscaling (MX v1.0) FP4: E2M1, round to nearest even, saturating to
// +-6; the low nibble of the result holds the second source operand.
__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// MXFP4 of one bf16 y vector given its block's absmax of y (fp32; a block of
// 32 elements is an aligned group of 4 lanes).  shared_exp = floor(log2(absmax)) - 2
// (2 = emax of E2M1), clamped to [-127, 127]; elements y * 2^-shared_exp (exact)
// rounded to E2M1.  An all-zero block gives scale code 0 and zero elements.
__device__ __forceinline__ void mxfp4_8_amax(const uint4 yb, float amax, uint32_t& packed, uint32_t& code) {
    packed = 0u;
    code = 0u;
    if (amax > 0.0f) {
        const uint32_t bits = __float_as_uint(amax);
        const int ef = static_cast<int>((bits >> 23) & 0xFFu);
        // floor(log2(amax)): the exponent field, or for an fp32 subnormal the
        // position of the leading mantissa bit (value = m * 2^-149)
        const int lg = ef != 0 ? ef - 127 : (31 - __clz(static_cast<int>(bits & 0x7FFFFFu))) - 149;
        int shared = lg - 2;
        shared = shared < -127 ? -127 : (shared > 127 ? 127 : shared);
        code = static_cast<uint32_t>(shared + 127);
        // 2^-shared as a bf16 pair: shared lies in [-127, 125] for bf16 y, so
        // 2^-shared is a bf16 normal (exponent field 2..254).  y * 2^-shared is
        // then one mixed-precision product per element, exact unless it falls
        // among the fp32 subnormals, where it takes the same single rounding as
        // an fp32 multiply.
        const uint32_t inv16 = static_cast<uint32_t>(127 - shared) << 7;
        const uint32_t inv2 = inv16 | (inv16 << 16);
        float v[8];
        mul2_bf16(v[0], v[1], yb.x, inv2);
        mul2_bf16(v[2], v[3], yb.y, inv2);
        mul2_bf16(v[4], v[5], yb.z, inv2);
        mul2_bf16(v[6], v[7], yb.w, inv2);
        packed = pack_e2m1x2(v[0], v[1]) | (pack_e2m1x2(v[2], v[3]) << 8) | (pack_e2m1x2(v[4], v[5]) << 16) |
                 (pack_e2m1x2(v[6], v[7]) << 24);
    }
}

// MXFP4 of one bf16 y vector; all 32 lanes must call it (a block is 4 lanes).
__device__ __forceinline__ void mxfp4_8(const uint4 yb, uint32_t& packed, uint32_t& code) {
    mxfp4_8_amax(yb, group_max<4>(vec_absmax(yb)), packed, code);
}

}  // namespace frn
