/*
 * nvfp4_gemm.h -- C ABI of libnvfp4gemm.so, a GB300 (sm_103a) NVFP4
 * block-scaled GEMM, dense and grouped.
 *
 * The operation (stated alike on all three source pages: "nvfp4_group_gemm,
 * submission 498453", custom_kernel docstring "C = A * SFA * B * SFB for all
 * groups", and the MMA-loop comment of that page and of "nvfp4 gemm,
 * submission 125598"):
 *
 *   C[l][m][n] = fp16( sum_k e2m1(A[l][m][k]) * e4m3(SFA[l][m][k/16])
 *                           * e2m1(B[l][n][k]) * e4m3(SFB[l][n][k/16]) )
 *
 * accumulated in fp32 by the tensor cores and rounded to fp16 (RNE) once.
 *
 * Layouts (device memory, row-major, l outermost):
 *   A    [L][M][K/2]  uint8, two E2M1 codes per byte, element 2i in the low
 *                     nibble of byte i (float4_e2m1fn_x2), K-major;
 *   B    [L][N][K/2]  same as A;
 *   SFA, SFB          E4M3 (float8_e4m3fn) scales in the REPACKED layout
 *                     produced by nvfp4_gemm_repack_scales (below);
 *   C    [L][M][N]    fp16.
 *
 * Conventions for every entry point:
 *   - All pointers named "device" are device pointers on the current CUDA
 *     device; the caller owns them and keeps them alive until the work queued
 *     on `stream` has finished.  Host arrays are read before the call returns.
 *     Every device pointer is checked with cudaPointerGetAttributes: host
 *     memory (pinned or not) and memory of another GPU are refused with
 *     NVFP4_ERR_INVALID_ARG before anything is launched.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  All work is asynchronous on that stream; nothing synchronises
 *     unless stated.  The GEMM, repack and quantize kernels are launched as
 *     programmatic dependents of the work before them on the stream: they may
 *     be scheduled while that work drains, but touch no global memory until
 *     it has completed, so stream order holds as for any kernel.
 *   - Return value: NVFP4_OK or a negative nvfp4_status.  On error nothing is
 *     queued, and nvfp4_gemm_last_error_string() (per calling thread) says why.
 *     The library never aborts the process.
 *   - Every device buffer must be 16-byte aligned.
 */
#ifndef NVFP4_GEMM_H
#define NVFP4_GEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = -1,       /* null / misaligned pointer, size < 1, G outside 1..8 */
    NVFP4_ERR_UNSUPPORTED_SHAPE = -2, /* K % 64 != 0, N % 8 != 0, size beyond limits */
    NVFP4_ERR_CUDA = -3,              /* a CUDA runtime / driver call failed */
    NVFP4_ERR_DEVICE_TIMEOUT = -4,    /* a kernel's bounded wait ran out (see below) */
    NVFP4_ERR_UNSUPPORTED_DEVICE = -5 /* the current device is not sm_103 */
} nvfp4_status;

/* Largest number of problems one grouped call takes ("expected 1..8 groups",
 * "nvfp4 group gemm, submission 407526", group_gemm argument checks). */
#define NVFP4_MAX_GROUPS 8

/*
 * Size in bytes of the repacked scale buffer for a [L][rows][K/16] scale
 * tensor: L * ceil(rows/128) * (4*ceil(K/256)) * 512.
 * Returns 0 for rows < 1, K < 1, L < 1 or K % 16 != 0.
 */
NVFP4_API size_t nvfp4_gemm_repacked_scales_bytes(int rows, int K, int L);

/*
 * Repack row-major E4M3 scales into the tensor-core scale layout.
 *
 * Layout ("nvfp4 gemm, submission 125598", custom_kernel docstring: permuted
 * scales of logical shape [32, 4, rest_m, 4, rest_k, l]; "nvfp4 group gemm,
 * submission 407526", grouped_kernel TMA producer: one 512-byte atom per
 * (128-row block, 4 scale columns), 2048 bytes per 256-wide k-tile):
 *   out[l][rm][ck][r0][r1][c0] = sf[l][128*rm + 32*r1 + r0][4*ck + c0]
 * with r0 < 32, r1 < 4, c0 < 4, rm < ceil(rows/128), ck < 4*ceil(K/256);
 * positions outside the input are zero.
 *
 *   sf     device, [L][rows][K/16] bytes, row-major, 16-byte aligned
 *   out    device, nvfp4_gemm_repacked_scales_bytes(rows, K, L) bytes
 *   rows   M for SFA, N for SFB (>= 1);  K >= 16, K % 16 == 0;  L >= 1
 * Errors: INVALID_ARG (null/misaligned pointer, sizes), CUDA.
 */
NVFP4_API int nvfp4_gemm_repack_scales(const void* sf, void* out, int rows, int K, int L, void* stream);

/* Input element types of nvfp4_quantize. */
#define NVFP4_DTYPE_BF16 0
#define NVFP4_DTYPE_F16 1

/*
 * Quantize values to NVFP4 and write the scales already repacked: the step
 * that produces A (or B) and SFA (or SFB) for nvfp4_gemm_run.  The pages take
 * pre-quantized inputs and print no quantizer; this is the plainest reading of
 * the formats they name ("nvfp4 gemm, submission 125598": ab_dtype Float4E2M1FN,
 * sf_dtype Float8E4M3FN, sf_vec_size 16), in IEEE fp32:
 *   per 16 consecutive values along K:  sf = E4M3(amax / 6), round to nearest
 *   even, finite values above 448 give 448;  d = value of sf;
 *   code = E2M1(x / d), round to nearest even on {0, .5, 1, 1.5, 2, 3, 4, 6},
 *   magnitudes above 6 give 6, sign of x / d kept;  d = 0 gives code 0.
 *
 *   x            device [L][rows][K], bf16 or fp16 per x_dtype, row-major
 *   codes        device [L][rows][K/2] bytes, written (low nibble = even k)
 *   sf_repacked  device, nvfp4_gemm_repacked_scales_bytes(rows, K, L) bytes,
 *                written in full (padding rows and k-blocks as zero)
 *   rows, K, L   rows >= 1, K >= 16 with K % 16 == 0, L >= 1
 * Asynchronous on `stream`; pointers 16-byte aligned; x must not overlap the
 * outputs.  Inputs with Inf or NaN are outside the contract.
 * Errors: INVALID_ARG (null / misaligned pointer, sizes, dtype), CUDA.
 */
NVFP4_API int nvfp4_quantize(const void* x, int x_dtype, void* codes, void* sf_repacked, int rows, int K,
                             int L, void* stream);

/*
 * One problem: C = A * SFA * B * SFB ("nvfp4 gemm, submission 125598",
 * custom_kernel).  Equivalent to nvfp4_gemm_run_grouped with G = 1.
 *
 *   A    device [L][M][K/2]       SFA  device, repacked (rows = M)
 *   B    device [L][N][K/2]       SFB  device, repacked (rows = N)
 *   C    device [L][M][N] fp16, written (rows >= M and columns >= N untouched)
 * Shape contract: M, N, K, L >= 1; K % 64 == 0 (one MMA k-block; a partial
 * 256-wide k-tile reads zero codes past the end of each row and the zero
 * padding of the repacked scales); N % 8 == 0 (16-byte C rows).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, UNSUPPORTED_DEVICE, CUDA.
 */
NVFP4_API int nvfp4_gemm_run(const void* A, const void* B, const void* SFA, const void* SFB, void* C,
                   int M, int N, int K, int L, void* stream);

/*
 * G independent problems in one launch ("nvfp4 group gemm, submission
 * 407526", group_gemm; "nvfp4_group_gemm, submission 498453", custom_kernel:
 * "each group has its own a, b, c, sfa, sfb with different m, n, k, l").
 *
 *   G                1..NVFP4_MAX_GROUPS
 *   A, B, SFA, SFB, C  host arrays of G device pointers, per group as in
 *                    nvfp4_gemm_run
 *   M, N, K, L       host arrays of G sizes, per group as in nvfp4_gemm_run
 * Errors: as nvfp4_gemm_run; the first offending group is named.
 *
 * Workspace: plans whose tiles are summed from partial results in a device
 * workspace (nvfp4_gemm_plan out[7] > 1 and out[10] == 0) use one per device
 * and stream, created by the first such launch and grown (at least doubled)
 * by a launch that needs more; growing synchronises the stream and is an
 * INVALID_ARG error while the stream is being captured into a CUDA graph
 * (run the problem once on the stream before capturing it).  A replaced
 * buffer stays allocated until the process exits, so a graph captured
 * before the growth stays valid.  Launches that share a workspace must not
 * run concurrently: replay such graphs on the stream they were captured on.
 */
NVFP4_API int nvfp4_gemm_run_grouped(int G, const void* const* A, const void* const* B,
                           const void* const* SFA, const void* const* SFB, void* const* C,
                           const int* M, const int* N, const int* K, const int* L, void* stream);

/* Text of the last error on the calling thread ("" if none).  The pointer
 * stays valid until the next call from the same thread. */
NVFP4_API const char* nvfp4_gemm_last_error_string(void);

/*
 * Device-side failure detection.  Every wait inside the kernels is bounded:
 * when one runs out, the kernel records NVFP4_ERR_DEVICE_TIMEOUT in a status
 * word on the device, stops issuing work, waits for its own copies in flight,
 * frees its tensor memory and returns.  Its output is then undefined.
 *
 * nvfp4_gemm_check_device_status synchronises `stream`, reads and clears the
 * current device's status words (the one of nvfp4_gemm_run / _run_grouped
 * and the one of nvfp4_gemm_run_noalloc) and returns NVFP4_OK or
 * NVFP4_ERR_DEVICE_TIMEOUT (or CUDA if the synchronisation itself failed).
 * It makes no device allocation.
 */
NVFP4_API int nvfp4_gemm_check_device_status(void* stream);

/* Limit of every bounded wait, in nanoseconds (default 2e9; minimum 1e5).
 * Applies to launches made after the call, on all devices. */
NVFP4_API int nvfp4_gemm_set_wait_timeout_ns(uint64_t ns);

/*
 * Fault injection for tests: when `ktile` >= 0, CTA 0's producer skips the
 * arrival for its ktile-th k-tile of the next launch only, so that a consumer
 * wait runs out.  Nothing is copied for that k-tile, so no copy is left in
 * flight.  -1 disables.  Not for production use.
 */
NVFP4_API int nvfp4_gemm_debug_inject_skip(int ktile);

/*
 * Launch plan, host only (no GPU needed): how nvfp4_gemm_run_grouped would
 * decompose these sizes on a device with `num_sms` SMs.  Output tiles are
 * 128 x BN.  Tiles [0, dp_tiles) run whole, one per CTA per wave; the rest are
 * cut into equal contiguous k-tile ranges, one per CTA ("stream-K"), and a
 * tile covered by several CTAs is summed from their partial results in k
 * order.  out_len >= 8:
 *   out[0] BN            out[1] output tiles     out[2] grid (CTAs)
 *   out[3] smem stages   out[4] dp_tiles         out[5] stream-K tiles
 *   out[6] stream-K k-tile iterations            out[7] most CTAs sharing a tile
 *   out[8] (when out_len >= 9) CTAs per cluster: 2 when pairs of CTAs with the
 *          same B columns (m-tiles 2q, 2q+1) share each B tile
 *   out[9] (when out_len >= 10) 1 when such a pair runs as one 256 x BN tile of
 *          2-SM MMAs (tcgen05 cta_group::2, each CTA holding half of B), 0 when
 *          the pair shares B through cluster multicast
 *   out[10] (when out_len >= 11) 1 when the stream-K segments of each tile run
 *          as one cluster (out[8] CTAs, one segment each) and are summed in
 *          distributed shared memory instead of a device workspace
 */
NVFP4_API int nvfp4_gemm_plan(int G, const int* M, const int* N, const int* K, const int* L,
                    int num_sms, int* out, int out_len);

/*
 * The work list CTA `cta` of that plan processes, host only, for checking the
 * decomposition without a GPU.  Writes 9 ints per item while they fit in
 * out_cap ints -- group, l, m-tile, n-tile, first k-tile, end k-tile, global
 * tile index, segment index, segments of the tile -- and returns the number of
 * items (or a negative status).
 */
NVFP4_API int nvfp4_gemm_debug_schedule(int G, const int* M, const int* N, const int* K,
                                        const int* L, int num_sms, int cta, int* out, int out_cap);

/*
 * What the calling host thread's most recent successful GEMM launch
 * (nvfp4_gemm_run, _run_grouped or _run_noalloc) actually ran, after any
 * device-dependent fallback of the plan.  Writes min(out_len, 5) ints:
 *   out[0] BN    out[1] grid (CTAs)    out[2] CTAs per cluster
 *   out[3] variant: 0 one CTA per tile, 1 CTA pairs sharing B by multicast,
 *          2 CTA pairs running 2-SM MMAs, 3 stream-K segments reduced in a
 *          cluster's distributed shared memory; -1 before the first launch
 *   out[4] shared-memory stages
 * Host only, no device call.  Errors: INVALID_ARG (null out, out_len < 1).
 */
NVFP4_API int nvfp4_gemm_last_launch(int* out, int out_len);

/*
 * nvfp4_gemm_run without any device allocation.  The source pages have no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc -- code running inside a host callback or a custom allocator, a
 * runtime that owns the whole device heap, or a process held to a fixed
 * memory budget -- and so cannot let the library create its stream-K
 * workspace on first use.
 *
 * Same arguments, layouts, shape contract and result as nvfp4_gemm_run (one
 * problem).  Stream-K scratch (fp32 partial tiles, per-tile arrival counters,
 * a status word) lives in one static device array of 16 MiB + 16.25 KiB that
 * every device which loads this library holds until the process exits.  The
 * first call on a device (with that device current) looks up the array's
 * device address once; make that first call before capturing any stream.
 * Each call clears the tile counters it uses (an asynchronous memset on
 * `stream`) and calls no allocator.
 *
 * All calls share the one array: calls whose work may overlap on the GPU
 * (different streams, or different host threads) race on it and give wrong
 * results; order them on one stream.  A problem whose stream-K plan needs more
 * than the array holds returns NVFP4_ERR_UNSUPPORTED_SHAPE with the sizes in
 * the error string.  A bounded device wait that runs out ends the kernel early
 * and leaves C undefined; the timeout stays in the array's status word until
 * nvfp4_gemm_check_device_status (which reads both status words of the
 * current device) reports and clears it.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, UNSUPPORTED_DEVICE, CUDA.
 */
NVFP4_API int nvfp4_gemm_run_noalloc(const void* A, const void* B, const void* SFA, const void* SFB,
                                     void* C, int M, int N, int K, int L, void* stream);

/*
 * Descriptor encoders used by the kernel, exported for host-side checks.
 *   nvfp4_gemm_encode_idesc: tcgen05.mma kind::mxf4nvf4 instruction
 *     descriptor for E2M1 x E2M1 with E4M3 block-16 scales, K-major operands.
 *   nvfp4_gemm_encode_smem_desc: shared-memory matrix descriptor;
 *     swizzle128 = 1 for the K-major 128-byte-swizzled operand tiles
 *     (8-row stride 1024 B), 0 for the unswizzled scale atoms (stride 128 B).
 */
NVFP4_API uint32_t nvfp4_gemm_encode_idesc(int M, int N);
NVFP4_API uint64_t nvfp4_gemm_encode_smem_desc(uint32_t smem_addr, int swizzle128);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_GEMM_H */
