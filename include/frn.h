/*
 * frn.h -- C ABI of libfrn: fused reduce + residual add + RMSNorm
 * (+ per-group dynamic FP8 e4m3 quant) for NVIDIA GB300 (sm_103a).
 *
 * The operation is the tensor-parallel decoder-layer epilogue
 * "allreduce -> residual add -> RMSNorm (-> per-1x128 FP8 quant)" re-posed for
 * one GPU: the R per-rank partial hidden states already sit in this GPU's
 * memory, and the "allreduce" is their fixed-order fp32 sum.
 *
 * Where it comes from:
 *  - "ROCm AITER fused all-reduce + RMSNorm" (vLLM PR 37646 summary), sections
 *    "implementation breakdown" (items 1-2) and "key source snippets"
 *    (allreduce_rms_fusion.py, _aiter_ops.py): the replaced subgraph is
 *    all_reduce(input) followed by rms_norm / fused_add_rms_norm, returning the
 *    normalised activation and the un-normalised sum, and the fused op takes
 *    (input, residual, weight, eps).
 *  - "AMD fused AllReduce-RMSNorm quant kernel" (SGLang PR 24651 summary),
 *    sections "features and motivation", "implementation breakdown" (items
 *    1-3) and "key source snippets" (layernorm.py): the quant variant returns
 *    ((fp8, scale), residual) or, with keep_bf16, ((bf16, fp8, scale), residual),
 *    quantising the normalised bf16 activation per 1x128 group.
 *  - "Fix: add missing end_sync barrier in fused allreduce+rmsnorm kernel"
 *    (AITER PR 4346), "Pull request overview": a fused call must never read a
 *    partial before its producer has finished, nor let the next call reuse
 *    buffers the previous one still reads.  Here that is stream order: every
 *    kernel waits on the previous grid before its first global load or store
 *    (only L2 prefetch hints, which hand no value to the kernel, come first).
 *
 * Per token row t, with f32() the exact bf16 -> fp32 widening:
 *   x_hat        = ((f32(P0[t]) + f32(P1[t])) + ... + f32(P[R-1][t])) + f32(residual[t])
 *                  (fp32 adds, rank order 0..R-1, residual last)
 *   residual_out = bf16_rn(x_hat)
 *   x            = f32(residual_out)
 *   y            = bf16_rn((x * f32(gamma)) * rstd),  rstd = 1/sqrt(sum(x^2)/H + eps)
 *                  (x * gamma is exact in fp32; one fp32 rounding, then one to bf16)
 *   per group g of group_size consecutive elements of y:
 *     a = max |f32(y)|,  s = a / 448 (fp32),  q = e4m3fn_rn_satfinite(f32(y) / s),
 *     and q = 0 when s == 0.
 *
 * residual_out is bit-exact (fixed-order fp32 sum, one round-to-nearest-even).
 * y is within one bf16 ulp of the exact RMSNorm of residual_out: the sum of
 * squares is an fp32 tree whose shape depends only on H, so a given row gives
 * the same bits whatever T, launch shape or stream it is computed in.
 *
 * Conventions for every entry point:
 *  - Inputs (partials, residual, gamma) are device memory.  Outputs are device
 *    memory, or pinned host memory mapped into the device's address space
 *    (cudaHostAlloc), which the kernel then writes over the host link.  All
 *    are row-major, rows contiguous: bf16 tensors are [T, H] with row stride H
 *    elements, gamma is bf16 [H], q is e4m3fn bytes [T, H], scales is fp32
 *    [T, H/group].  The library does not check the memory type; a pointer the
 *    device cannot address faults.
 *  - The caller owns every buffer.  The library allocates nothing, never
 *    synchronises the host, and reads no device state on the host, so every
 *    call can be captured in a CUDA graph.
 *  - partials is a HOST array of R device pointers; it is read during the call
 *    (copied into the kernel's parameters) and may be freed on return.
 *    Partial pointers may repeat.
 *  - residual may be NULL, which means a residual of zeros.  residual_out may
 *    equal residual exactly (in-place update); any other overlap between an
 *    output and any input, or between two outputs, is rejected.
 *  - bf16 and fp8 pointers must be 16-byte aligned, scales 4-byte aligned.
 *  - Limits: 1 <= R <= FRN_MAX_PARTIALS, T >= 0, H % 8 == 0,
 *    8 <= H <= FRN_MAX_HIDDEN, eps finite >= 0, group_size == 128 with
 *    H % 128 == 0.  T == 0 checks only the scalar arguments, touches no
 *    pointer and returns FRN_OK.
 *  - Arguments are validated on the host before anything is launched; a
 *    rejected call launches nothing.  FRN_ERR_CUDA reports a launch error;
 *    errors of earlier, unrelated work on the stream are not reported here.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *    Work queued earlier on the stream (e.g. the producers of the partials)
 *    is complete before the kernel reads anything; calls on different streams
 *    that share buffers must be ordered by the caller (events).
 *  - On its first use on a device the library looks up and keeps, for the
 *    life of the process, that device's SM count and the device addresses of
 *    its own status word and static workspace.  cudaDeviceReset (or any other
 *    teardown of the device's primary context) makes the kept addresses stale:
 *    do not call the library on a device after resetting it.
 */
#ifndef FRN_H_
#define FRN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, declared here so that callers need no
 * CUDA header. */
typedef struct CUstream_st* frn_stream_t;

typedef enum frn_status {
    FRN_OK = 0,
    FRN_ERR_INVALID_ARG = 1,  /* NULL pointer, R < 1, T < 0, H < 1, bad eps, bad group, overlap */
    FRN_ERR_UNSUPPORTED = 2,  /* well-formed but outside this build's limits            */
    FRN_ERR_MISALIGNED = 3,   /* a tensor pointer breaks the alignment rule              */
    FRN_ERR_CUDA = 4,         /* a CUDA runtime call or the kernel launch failed          */
    FRN_ERR_TIMEOUT = 5       /* a bounded device-side wait ran out (frn_device_status)  */
} frn_status;

#define FRN_MAX_PARTIALS 16
#define FRN_MAX_HIDDEN 16384
#define FRN_QUANT_GROUP 128
#define FRN_E4M3_MAX 448.0f

/*
 * Sum R bf16 partials in fp32 (rank order), add the residual, write
 * residual_out (bf16) and the RMSNorm output y (bf16).
 *
 *   partials     host array [R] of device pointers, each bf16 [T, H]
 *   R            number of partials (tensor-parallel ranks), 1..16
 *   residual     bf16 [T, H] or NULL (zeros)
 *   gamma        bf16 [H] RMSNorm weight
 *   residual_out bf16 [T, H] output (may equal residual)
 *   y            bf16 [T, H] output
 *   T, H         tokens and hidden size
 *   eps          variance epsilon, added to mean(x^2) inside the square root
 *   stream       CUDA stream
 */
frn_status fused_reduce_rmsnorm(const void* const* partials, int R,
                                const void* residual, const void* gamma,
                                void* residual_out, void* y,
                                int64_t T, int H, float eps, frn_stream_t stream);

/*
 * As fused_reduce_rmsnorm, then per-group dynamic FP8 quant of y:
 *
 *   y        NULL -> variant A, outputs (fp8, scale) + residual_out and no bf16 y;
 *            bf16 [T, H] -> variant B, outputs (bf16, fp8, scale) + residual_out.
 *            q and scales are bit-identical between the two variants.
 *   q_e4m3   e4m3fn [T, H] output codes (OCP FP8 E4M3: bias 7, max 448, no inf)
 *   scales   fp32 [T, H / group_size] output, row-major; dequant = e4m3(q) * s
 *   group_size  must be 128 (FRN_QUANT_GROUP)
 */
frn_status fused_reduce_rmsnorm_quant_per_group(const void* const* partials, int R,
                                                const void* residual, const void* gamma,
                                                void* residual_out, void* y,
                                                void* q_e4m3, float* scales,
                                                int64_t T, int H, float eps, int group_size,
                                                frn_stream_t stream);

/*
 * As fused_reduce_rmsnorm, then MXFP4 of y -- the third fused output variant
 * ("Fix: add missing end_sync barrier in fused allreduce+rmsnorm kernel", AITER
 * PR 4346, Pull request overview: the MXFP4 1-stage variant).  The pages give
 * no format; this follows the OCP Microscaling Formats (MX) v1.0 conversion:
 *   blocks of 32 consecutive elements of y along H;
 *   shared_exp = floor(log2(max |y| over the block)) - 2 (the emax of E2M1),
 *     clamped to [-127, 127];  scale code = shared_exp + 127 (E8M0);
 *   element = E2M1 round-to-nearest-even, saturating to +-6, of y / 2^shared_exp;
 *   an all-zero block gets scale code 0 and zero elements.
 *
 *   y             NULL -> (fp4, scale) + residual_out;  bf16 [T, H] -> (bf16, fp4, scale)
 *   q_fp4         uint8 [T, H/2]: element 2i in the low nibble of byte i (16-byte aligned)
 *   scales_e8m0   uint8 [T, H/32]
 *   H % 32 == 0; other arguments, conventions and errors as for fused_reduce_rmsnorm.
 */
frn_status fused_reduce_rmsnorm_mxfp4(const void* const* partials, int R,
                                      const void* residual, const void* gamma,
                                      void* residual_out, void* y,
                                      void* q_fp4, void* scales_e8m0,
                                      int64_t T, int H, float eps, frn_stream_t stream);

/*
 * The adjacent steps of the same layer, on the same kernels ("ROCm AITER fused
 * all-reduce + RMSNorm", vLLM PR 37646 summary, implementation breakdown item
 * 2: the rms_norm and fused_add_rms_norm patterns).
 *
 * frn_fused_add_rmsnorm: one activation x plus the residual, i.e.
 *   fused_reduce_rmsnorm with R = 1: residual_out = bf16(f32(x) + f32(residual)),
 *   y = RMSNorm(residual_out).  residual may be NULL (zeros) and residual_out
 *   may equal residual.
 * frn_rmsnorm: y = bf16((f32(x) * rstd) * f32(gamma)), rstd over f32(x) + 0.0
 *   (so a -0.0 input element gives +0.0); nothing else is written.
 * Arguments, layouts, limits and errors as for fused_reduce_rmsnorm.
 */
frn_status frn_fused_add_rmsnorm(const void* x, const void* residual, const void* gamma,
                                 void* residual_out, void* y, int64_t T, int H, float eps,
                                 frn_stream_t stream);

frn_status frn_rmsnorm(const void* x, const void* gamma, void* y, int64_t T, int H, float eps,
                       frn_stream_t stream);

/*
 * Unfused comparison paths: the same outputs, bit for bit, computed the way an
 * unfused layer would, to measure what fusion saves ("AMD fused
 * AllReduce-RMSNorm quant kernel", SGLang PR 24651 summary, implementation
 * breakdown items 2 and 4: the 3-kernel / 2-kernel / 1-kernel comparison).
 *
 *   q_e4m3 == NULL and scales == NULL: no quant; stages must be 2
 *       (reduce -> residual add + RMSNorm).
 *   otherwise: per-group quant as fused_reduce_rmsnorm_quant_per_group
 *       (y NULL = variant A), stages 3 (reduce -> residual add + RMSNorm ->
 *       quant) or 2 (fused reduce + add + RMSNorm -> stand-alone quant).
 *
 * The reduce stage writes the fp32 sum of the partials to the workspace; a quant
 * path without a y output keeps the bf16 y there.  workspace: device memory of
 * at least frn_unfused_workspace_bytes(T, H, stages, quant, emit_y) bytes,
 * 16-byte aligned, not overlapping any argument; the caller owns it and it may
 * be reused once the call's work on `stream` has completed.  Other arguments,
 * conventions and errors as for the fused entry points.
 */
int64_t frn_unfused_workspace_bytes(int64_t T, int H, int stages, int quant, int emit_y);

frn_status frn_unfused_reduce_rmsnorm(const void* const* partials, int R,
                                      const void* residual, const void* gamma,
                                      void* residual_out, void* y,
                                      void* q_e4m3, float* scales,
                                      int64_t T, int H, float eps, int group_size,
                                      int stages, void* workspace, int64_t workspace_bytes,
                                      frn_stream_t stream);

/*
 * No-allocation variant of frn_unfused_reduce_rmsnorm.  (The pages have no
 * counterpart: it exists for callers of this library that cannot allocate
 * device memory on the call path -- code running during CUDA-graph capture in
 * the default capture mode, where cudaMalloc is not allowed; serving engines
 * that hand nearly all device memory to their own pool at start-up; plugins
 * given raw pointers and no allocator.)
 *
 * Same arguments and results as frn_unfused_reduce_rmsnorm, without the
 * workspace: the scratch is a fixed array of FRN_STATIC_WORKSPACE_BYTES (16 MiB)
 * inside the library's device image, which every GPU that loads the library
 * holds until the process exits.  Nothing is allocated or freed by any call.
 *  - Sizes whose scratch (frn_unfused_workspace_bytes) exceeds the array are
 *    rejected with FRN_ERR_UNSUPPORTED, e.g. 3 stages with quant and no y at
 *    H = 7168 fit up to T = 390.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array and leaves its last contents
 *    there (nothing needs to start at zero: each call overwrites what it reads).
 *    Calls that can overlap on the GPU -- on different streams without ordering
 *    between them, or from several host threads -- race on it; order them, or
 *    use frn_unfused_reduce_rmsnorm with separate workspaces.
 */
#define FRN_STATIC_WORKSPACE_BYTES (16LL << 20)

frn_status frn_unfused_reduce_rmsnorm_noalloc(const void* const* partials, int R,
                                              const void* residual, const void* gamma,
                                              void* residual_out, void* y,
                                              void* q_e4m3, float* scales,
                                              int64_t T, int H, float eps, int group_size,
                                              int stages, frn_stream_t stream);

/*
 * Measurement reference kernels (no entry point of the op uses them).  A
 * decode-sized call is mostly fixed cost -- launch and hand-off from the
 * previous kernel, one DRAM round trip, the drain of its stores -- so its
 * speed is judged against kernels that have that cost and nothing else,
 * launched the same way (pdl != 0: programmatic dependent launch, with the
 * grid-dependency wait before the first global access):
 *   kind 0  empty kernel: grid_ctas CTAs of `threads` threads (srcs, dst0,
 *           dst1 and nbytes unused);
 *   kind 1  read: each thread loads one 16-byte vector of each of the n_src
 *           (1..17) device buffers of nbytes bytes (a multiple of 16), through
 *           the op's load path, and stores nothing;
 *   kind 2  copy: the same loads, then stores of nbytes bytes into each of
 *           dst0 and dst1 -- the traffic of a call without quant (R partials
 *           and the residual in; residual_out and y out) without its arithmetic.
 * Kinds 1 and 2 launch ceil(nbytes / 16 / threads) CTAs (grid_ctas unused).
 * threads: a multiple of 32, up to 1024 for kind 0 and 512 for kinds 1 and 2.
 * All pointers 16-byte aligned.
 * Returns FRN_ERR_INVALID_ARG / FRN_ERR_MISALIGNED without launching on bad
 * arguments, FRN_ERR_CUDA on a launch error; frn_last_error_detail is not set.
 */
frn_status frn_floor_launch(int kind, const void* const* srcs, int n_src, void* dst0, void* dst1,
                            int64_t nbytes, int threads, int64_t grid_ctas, int pdl, frn_stream_t stream);

/* Static text for a status code. */
const char* frn_status_string(frn_status s);

/* Text describing the last error returned on the calling thread (argument name,
 * CUDA error string), or "" if none.  Valid until the thread's next call. */
const char* frn_last_error_detail(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int frn_version(void);

/*
 * Launch control.  Process-wide settings read at each call; set them before
 * concurrent use, not while other threads are launching.  Results are
 * bit-identical for every choice.
 *
 * frn_set_pdl: 1 (default) launches with programmatic dependent launch, so
 *   the kernel's prologue may overlap the tail of the previous kernel on the
 *   stream; the kernel still waits for that kernel's completion before its
 *   first global-memory load or store (only an L2 prefetch hint, which hands
 *   no value to the kernel, may precede the wait).  0 launches plainly.
 * frn_set_kernel: 0 (default) picks the kernel from T, H, R, the output and
 *   the SM count; 1 forces the row kernel (a row per CTA -- one tile a warp,
 *   or two for rows of 9..64 tiles -- per wide CTA or thread-block cluster,
 *   or several short rows per CTA; registers hold each row),
 *   2 forces the stream kernel (persistent, one CTA per SM, rows streamed
 *   through shared memory with TMA bulk copies, for many rows).
 * frn_set_ctas_per_row: row kernel only.  0 (default) chooses from T, H, R
 *   and the SM count between one CTA per row (several short rows per CTA when
 *   H <= 1024 and T is large) and a cluster of CTAs per row;
 *   1 forces one CTA per row (up to 1024 threads when H <= 8192 and R <= 8,
 *   two tiles a warp when H > 8192, else the smallest cluster that holds the
 *   row); 2..16 force a cluster of
 *   that many CTAs (rounded so that no CTA is empty; 9..16 is a non-portable
 *   cluster size, with at least two tiles a CTA).
 * frn_set_stream_groups: stream kernel only.  0 (default) chooses how many
 *   consumer groups (each taking every n-th row of a CTA, so that one group's
 *   epilogue overlaps the next group's loads) from H and the slices a row
 *   has; 1..4 forces it, reduced where the CTA would exceed its warp budget.
 * frn_set_l2_prefetch: row kernel only.  0 (default) decides from the launch
 *   shape whether each warp asks for its slice of the row to be fetched into
 *   L2 before the wait on the previous kernel, and, for grids of more than
 *   one wave, whether each CTA asks for its slice of the row about 9.5 MB of
 *   loads ahead (and the first wave's CTAs for their own, before the wait):
 *   hints that hand no value to the kernel; 1 does neither; 2 always does the
 *   first and decides the second as 0 does.
 */
frn_status frn_set_pdl(int enable);
frn_status frn_set_l2_prefetch(int mode);
frn_status frn_set_kernel(int kernel);
frn_status frn_set_ctas_per_row(int ctas_per_row);
frn_status frn_set_stream_groups(int groups);

/*
 * The launch the library plans for a call of these sizes on a device with
 * num_sms SMs, without touching a device (host code only; for inspection and
 * tests).  quant as for frn_query_launch; has_residual != 0 when a residual
 * is passed (the stream kernel then streams R + 1 slices a row).  T >= 1.
 *   kernel          1 row kernel, 2 stream kernel
 *   ctas_per_row    row kernel: CTAs of the row's cluster (1: one CTA)
 *   rows_per_cta    row kernel: consecutive short rows a CTA (1 otherwise)
 *   tiles_per_cta   row kernel: warps (32-vector tiles) a row has in a CTA
 *   tiles_per_warp  stream kernel: tiles a consumer warp holds; row kernel: 2
 *                   when one CTA holds a row at two tiles a warp (rows of
 *                   9..64 tiles), else 1
 *   threads, grid   threads per CTA, CTAs in the grid
 *   groups, consumer_warps, slots, smem_bytes
 *                   stream kernel: consumer groups, warps a group, ring slots
 *                   (one 2*H-byte row slice each), dynamic shared memory
 *   staged          row kernel: 1 when each thread loads its partials in
 *                   stages of two (two stages in flight, 32 registers) rather
 *                   than all at once, so that more rows share an SM
 * Launch controls (frn_set_kernel, frn_set_ctas_per_row, ...) apply as they
 * would to a call.
 */
typedef struct frn_launch_plan {
    int kernel;
    int ctas_per_row;
    int rows_per_cta;
    int tiles_per_cta;
    int tiles_per_warp;
    int threads;
    int64_t grid;
    int groups;
    int consumer_warps;
    int slots;
    int smem_bytes;
    int staged;
} frn_launch_plan;

frn_status frn_plan_launch(int64_t T, int H, int R, int quant, int has_residual, int num_sms,
                           frn_launch_plan* out);

/*
 * Report the launch a call with these sizes would use on the current device:
 * kernel (1 row, 2 stream), CTAs per row (cluster size; 1 for the stream
 * kernel and for a single wide CTA), threads per CTA, and CTAs in the grid --
 * frn_plan_launch with the current device's SM count.  quant: 0 no quant,
 * 1 / 2 per-group FP8 without / with y, 3 / 4 MXFP4 without / with y.
 * has_residual != 0 when the call passes a residual.  T == 0 reports the
 * shape of a one-row call with a grid of 0.  Output pointers may be NULL.
 */
frn_status frn_query_launch(int64_t T, int H, int R, int quant, int has_residual, int* kernel,
                            int* ctas_per_row, int* threads_per_cta, int64_t* grid_ctas);

/*
 * Device-side failure detection.  Every device-side wait is bounded (default
 * 2 s): the stream kernel's shared-memory pipeline and the row kernel's wait
 * for the tile sums of a row split over a cluster.  A wait that runs out sets a
 * status word on the device and the kernel finishes without waiting further;
 * the call's outputs are then incomplete.  frn_device_status reads that word for the current device --
 * synchronously, so call it after the work in question has completed (e.g.
 * after synchronising its stream) -- and returns FRN_ERR_TIMEOUT if it is set
 * (FRN_OK otherwise).  clear != 0 resets the word.
 */
frn_status frn_device_status(int clear);

/*
 * Test hook for the failure path above.  inject_stall != 0 makes every CTA of
 * the stream kernel skip its first bulk copy, and the row kernel's cluster
 * shape never push tile 0's sum, so that the waits on them run out;
 * wait_limit_ns > 0 replaces the 2 s bound (<= 0 restores it).  The kernel then
 * returns with the status word set and the context stays usable.
 */
frn_status frn_set_test_hooks(int inject_stall, int64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* FRN_H_ */
