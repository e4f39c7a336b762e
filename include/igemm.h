/*
 * igemm.h — exact integer GEMM on packed int4 operands for NVIDIA GB300 (sm_103a).
 *
 * C-ABI of libigemm.so.  All entry points are asynchronous on `stream` and
 * return an igemm_status synchronously: argument errors are reported before
 * anything is enqueued, and nothing is launched when the return value is not
 * IGEMM_OK.  Every pointer argument is caller-owned device memory (global
 * memory of the current device), except the array arguments of the *_host
 * entry points, which are caller-owned host memory.  Device-side problems (a pipeline wait that
 * exceeded the watchdog limit) are reported later by igemm_last_status().
 *
 * Workspace.  Large GEMMs (M * N >= 2^22 and, for int4 x int4, M, N >= 512;
 * for W4A8, M >= 768 and N >= 256) first write the operands as one code byte
 * per value, with row sums, into a workspace of (rows of A + rows of B) * K
 * bytes (W4A8: N*K + 2*M*K) plus a few KB.  The library takes it from its own
 * stream-ordered memory pool on the current device (allocated and released in
 * `stream` order, so concurrent calls on different streams do not share it);
 * the pool keeps what it reserved for later calls until the process exits.  A
 * failed workspace allocation returns IGEMM_CUDA_ERROR.  w4a8_gemm_scaled (its
 * int32 product) and fp8_blockscaled_gemm (its transposed scales) take theirs
 * from the same pool; skinny shapes (M <= 64) and fp8_gemm (either format)
 * need none.
 *
 * Launch overlap.  Where a call launches a short pass before its GEMM kernel
 * (the preparation of codes, the zeroing of C, the transposed scales), the GEMM
 * kernel is launched with programmatic stream serialization: its set-up and
 * the loads that do not depend on the pass run while the pass finishes, and it
 * waits for the pass (griddepcontrol.wait) before it reads or writes what the
 * pass touches.
 *
 * Operand formats
 *   Packed int4 matrix [rows, K/2] bytes, row-major: byte j of a row holds
 *   element 2j in its low nibble and element 2j+1 in its high nibble, each a
 *   4-bit two's-complement value in [-8, 7] (TileLang tutorial page
 *   low_precision_gemm.py, pack_int4; "[Example] add w4a8 gemm kernel",
 *   tilelang PR #815, _tir_u8_to_i4_to_i8: pos 0 = low nibble).
 *   C is [M, N] int32, row-major; every element is overwritten.
 *
 * Shape and alignment rules (violations are returned, never launched)
 *   M, N, K >= 0; M == 0 or N == 0 is an empty product (no work, IGEMM_OK);
 *   K == 0 with M, N > 0 sets C to zero.
 *   K % 32 == 0 for the integer GEMMs (a packed row is a whole number of
 *   16-byte units, the TMA row-pitch rule) else IGEMM_UNSUPPORTED_SHAPE.
 *   K <= 33554431 (int4 x int4: |a b| <= 64, so |C| <= 64 K < 2^31) or
 *   K <= 2097151 (W4A8: |a b| <= 1024) else IGEMM_OVERFLOW_BOUND, the int32
 *   range of the result.  One f32 MMA accumulation is exact over at most
 *   65536 k; a longer K runs on the prepared-codes path in pieces of at most
 *   65536 k whose exact int32 results add into C (its workspace then holds
 *   (M + N) * K, or N * K + 2 * M * K, bytes of codes).
 *   Every non-empty operand base address and C must be 16-byte aligned, else
 *   IGEMM_MISALIGNED.
 */
#ifndef IGEMM_H
#define IGEMM_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define IGEMM_API __attribute__((visibility("default")))
#else
#define IGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum igemm_status {
    IGEMM_OK = 0,
    IGEMM_INVALID_ARGUMENT = 1,  /* null pointer for a non-empty operand, negative size */
    IGEMM_UNSUPPORTED_SHAPE = 2, /* K % 32 != 0 (GEMM); odd K (pack_int4) */
    IGEMM_MISALIGNED = 3,        /* a base address is not 16-byte aligned */
    IGEMM_OVERFLOW_BOUND = 4,    /* K above the int32 bound (33554431 int4 x int4, 2097151 W4A8) */
    IGEMM_CUDA_ERROR = 5,        /* tensor-map encoding, memset or launch failed */
    IGEMM_DEVICE_TIMEOUT = 6,    /* a kernel's bounded wait expired (see igemm_last_status) */
    IGEMM_WORKSPACE_LIMIT = 7    /* i4i4_gemm_noalloc: the problem needs more than its fixed workspace */
} igemm_status;

/*
 * int4 x int4 GEMM:  C[m,n] = sum_k a[m,k] * b[n,k], exact, int32.
 * Defined by "[CUDA] Support int4 T.gemm" (tilelang PR #2063),
 * examples/gemm_int4/example_tilelang_gemm_int4.py, matmul_nt_int4: A (M,K)
 * int4, B (N,K) int4, C (M,N) int32, T.gemm(A_shared, B_shared, C_local,
 * transpose_B=True); same contract as matmul_int4 of the tutorial page
 * low_precision_gemm.py.
 *   Ap  [M, K/2] packed int4 (device), read only
 *   Bp  [N, K/2] packed int4 (device), read only
 *   C   [M, N] int32 (device), written
 * Returns IGEMM_OK once the work is enqueued on `stream`.
 */
IGEMM_API int i4i4_gemm(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);

/*
 * int4 x int4 GEMM that allocates nothing: the same result as i4i4_gemm, for
 * callers that may not allocate device memory during a call (for example
 * code running where a memory allocation would block on other work, or
 * whose memory budget is fixed up front).  None of the pages describes such
 * an entry point; it is an addition of this library.
 *
 * Its workspace is a fixed array of 32 MiB (IGEMM_NOALLOC_WORKSPACE_BYTES)
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  It always takes the prepared-codes path, which needs
 * (M + N) * K bytes plus about 4 * (M + N + 1024) bytes of row sums; larger
 * problems return IGEMM_WORKSPACE_LIMIT before anything is enqueued.  The
 * call makes no cudaMalloc, cudaFree or pool allocation.
 *
 * The first call on each device does the set-up: it looks up the device
 * address of the array (cudaGetSymbolAddress, with that device current), and
 * with CUDA's lazy module loading (the default) it may be the call that loads
 * the library's device code, which is when the 32 MiB array is mapped.  So
 * make one call per device during set-up, before any stream capture; from the
 * second call on nothing is reserved.  All calls share the one array and each call
 * rewrites what it reads, so results never depend on an earlier call; but
 * calls whose work overlaps on the GPU (on different streams, or from
 * different threads without ordering) race on the array and give wrong
 * results.  Arguments and the other rules are those of i4i4_gemm.
 */
#define IGEMM_NOALLOC_WORKSPACE_BYTES (32u << 20)
IGEMM_API int i4i4_gemm_noalloc(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                                cudaStream_t stream);

/*
 * W4A8 GEMM:  C[m,n] = sum_k a[m,k] * b[n,k], a int8, b int4, exact, int32.
 * Defined by "[Example] add w4a8 gemm kernel" (tilelang PR #815): int8
 * activations times int4 weights sign-extended in the kernel
 * (_tir_u8_to_i4_to_i8), checked against an integer matmul (reviewed
 * ref_program).  The page's kernel returns C transposed; this entry point
 * returns C[M, N].
 *   A   [M, K] int8 activations (device), read only
 *   Bp  [N, K/2] packed int4 weights (device), read only
 *   C   [M, N] int32 (device), written
 */
IGEMM_API int w4a8_gemm(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);

/*
 * The same two GEMMs with A, Bp and C in HOST memory (pinned memory lets the
 * copies run asynchronously and overlap; pageable memory works but the copies
 * then block the calling thread).  The call copies Bp to the device, then A in
 * row chunks (about eight chunks of at least 1024 rows, one chunk below 2048
 * rows), runs the device entry point on each chunk in `stream`, and copies each
 * chunk of C back while later chunks compute.  The copies run on two copy
 * streams of the library's own (per device, created on first use); `stream`
 * waits for them, so C is complete on the host once `stream` has reached the
 * end of the call (e.g. after cudaStreamSynchronize(stream)).  The host buffers
 * must stay valid and unchanged until then.  Device memory for Bp, two chunks
 * of A and two chunks of C comes from the library's pool.
 *   Ap / A  [M, K/2] packed int4 / [M, K] int8 (host), read only
 *   Bp      [N, K/2] packed int4 (host), read only
 *   C       [M, N] int32 (host), written
 * Rules as for i4i4_gemm / w4a8_gemm (K % 32 == 0, the same K bounds, empty
 * shapes are no-ops, K == 0 zeroes C), except that host pointers need no
 * alignment.
 * igemm_time_next_gemm times the GEMM kernel of the first chunk only.  A CUDA
 * error after the first chunk was enqueued (IGEMM_CUDA_ERROR) leaves the earlier
 * chunks' work in the streams; the call still joins its copy streams to
 * `stream` before it returns.
 */
IGEMM_API int i4i4_gemm_host(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                             cudaStream_t stream);
IGEMM_API int w4a8_gemm_host(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                             cudaStream_t stream);

/*
 * W4A8 GEMM with per-channel dequantisation (the "scaled epilogue" step that
 * follows the integer product in W4A8 inference; the pages show scales only
 * as the per-block structure of the tutorial's gemm_blockscaled):
 *   C[m,n] = bf16_rn((float(sum_k a[m,k] * b[n,k]) * scale_a[m]) * scale_b[n])
 * with the integer sum exact (w4a8_gemm), its conversion to float32 rounded to
 * nearest, two float32 multiplications in that order, and round-to-nearest-even
 * to bfloat16.
 *   A        [M, K] int8 (device), read only
 *   Bp       [N, K/2] packed int4 (device), read only
 *   scale_a  [M] float32 (device), scale_b [N] float32 (device), read only
 *   C        [M, N] bfloat16 bit patterns (device), written
 * The int32 product is held in a workspace of M*N*4 bytes from the library's
 * pool, then a second kernel applies the scales.  Rules as for w4a8_gemm; the
 * scale arrays must be 16-byte aligned too.
 */
IGEMM_API int w4a8_gemm_scaled(const int8_t *A, const uint8_t *Bp, const float *scale_a, const float *scale_b,
                               uint16_t *C, int M, int N, int K, cudaStream_t stream);

/*
 * fp8 GEMM:  C[m,n] = sum_k a[m,k] * b[n,k] for E4M3 operands, accumulated in
 * float32 (TileLang tutorial page low_precision_gemm.py, gemm_fp8: A (M,K) and
 * B (N,K) in an fp8 dtype, float32 accumulator, C = A . B^T).  The page writes C
 * in the operands' fp8 dtype; this entry point returns the float32
 * accumulator itself (rounding it to fp8 is the caller's choice).
 *   A   [M, K] E4M3 bytes (device), read only
 *   B   [N, K] E4M3 bytes (device), read only
 *   C   [M, N] float32 (device), written
 * K % 16 == 0 (IGEMM_UNSUPPORTED_SHAPE otherwise; the TMA row pitch).  The
 * order of the float32 additions is not specified: when the launch splits K
 * (few output tiles, deep K) the partial sums meet through atomic adds, so the
 * last bits can differ from call to call.  Other rules as for i4i4_gemm
 * (K == 0 zeroes C, 16-byte alignment, empty shapes are no-ops); there is no
 * K limit.
 */
IGEMM_API int fp8_gemm(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, cudaStream_t stream);

/*
 * The same GEMM for E5M2 operands (the page's other fp8 dtype; both A and B
 * in E5M2: 5 exponent bits with bias 15, 2 mantissa bits, largest finite
 * value 57344).  Arguments, rules and rounding as for fp8_gemm.  Products and
 * sums of finite inputs stay finite in float32 for every K the int argument
 * can hold; infinities and NaNs among the inputs are not given a meaning here.
 */
IGEMM_API int fp8_gemm_e5m2(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, cudaStream_t stream);

/*
 * Block-scaled fp8 GEMM (TileLang tutorial page low_precision_gemm.py,
 * gemm_blockscaled: fp8 A (M,K) and B (N,K), float32 scale tensors SFA
 * (M, ceil(K/g)) and SFB (N, ceil(K/g)) applied along K per block of g values,
 * float32 accumulator; the page names g = 128 for sm100):
 *   C[m,n] = sum_kb SFA[m,kb] * SFB[n,kb] * sum_{k in block kb} a[m,k] * b[n,k]
 * with g = 128 and KB = ceil(K/128) blocks (the last one may be short).
 *   A    [M, K] E4M3 bytes (device), read only
 *   B    [N, K] E4M3 bytes (device), read only
 *   SFA  [M, KB] float32 (device, row-major), read only
 *   SFB  [N, KB] float32 (device, row-major), read only
 *   C    [M, N] float32 (device), written
 * Each block's partial sum comes from the tensor core (float32) and is scaled
 * and added in float32 in block order; the order of the additions inside a
 * block is not specified.  The scales are transposed into a workspace of
 * 4 * KB * (M + N rounded up to 128 each) bytes from the library's pool.
 * K % 16 == 0 (IGEMM_UNSUPPORTED_SHAPE otherwise); A, B and C 16-byte aligned,
 * SFA and SFB 4-byte aligned (IGEMM_MISALIGNED); K == 0 zeroes C; empty shapes
 * are no-ops.
 */
IGEMM_API int fp8_blockscaled_gemm(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, float *C,
                                   int M, int N, int K, cudaStream_t stream);

/*
 * The same block-scaled GEMM for E5M2 operands (A and B both E5M2); scales,
 * arguments and rules as for fp8_blockscaled_gemm.
 */
IGEMM_API int fp8_blockscaled_gemm_e5m2(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB,
                                        float *C, int M, int N, int K, cudaStream_t stream);

/*
 * Host-buffer twins of the four fp8 entry points above: A, B, C (and SFA, SFB)
 * in HOST memory, moved and computed in row chunks exactly as i4i4_gemm_host
 * does (B and SFB copied whole, A and the matching rows of SFA per chunk).
 * Arguments and rules as for the device entry points, except that host
 * pointers need no alignment; C is complete once `stream` has reached the end
 * of the call.  A chunk's GEMM may plan its split of K differently from a
 * whole-matrix call, so the last bits of a float32 C can differ from the device
 * entry point's where that call would split K.
 */
IGEMM_API int fp8_gemm_host(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, cudaStream_t stream);
IGEMM_API int fp8_gemm_e5m2_host(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K,
                                 cudaStream_t stream);
IGEMM_API int fp8_blockscaled_gemm_host(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB,
                                        float *C, int M, int N, int K, cudaStream_t stream);
IGEMM_API int fp8_blockscaled_gemm_e5m2_host(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB,
                                             float *C, int M, int N, int K, cudaStream_t stream);

/*
 * Pack logical int4 values two per byte (TileLang tutorial page
 * low_precision_gemm.py, pack_int4): packed[r, j] = (logical[r, 2j] & 0xF) |
 * ((logical[r, 2j+1] & 0xF) << 4).  Values outside [-8, 7] are masked to four
 * bits (two's-complement wrap), as on the page; this is not an error.
 *   logical [rows, K] int8 (device), read only
 *   packed  [rows, K/2] bytes (device), written
 * K must be even (IGEMM_UNSUPPORTED_SHAPE otherwise, the page's ValueError);
 * rows == 0 or K == 0 is a no-op.  Any alignment is accepted.
 */
IGEMM_API int pack_int4(const int8_t *logical, uint8_t *packed, int64_t rows, int64_t K, cudaStream_t stream);

/*
 * Number of kernels this library has launched in this process so far (all
 * devices and streams; a launch counts when it was enqueued).  One GEMM call
 * launches one kernel, or two: the preparation pass and the GEMM (prepared
 * codes), the zeroing of C and the GEMM (skinny shapes whose K slices are
 * summed with atomics), the scale transpose and the GEMM (block-scaled fp8).
 * The split K of the other paths adds a memset, which is not a kernel.
 */
IGEMM_API uint64_t igemm_kernels_launched(void);

/*
 * Planning query, host only (no GPU is touched): the split of K that a call of
 * i4i4_gemm (variant 0) or w4a8_gemm (variant 1) with 1 <= M <= 64 would use on
 * a GPU with `sms` SMs where `pairs` clusters of two and `quads` clusters of
 * four of the skinny kernel can be resident at once (0: none; the library asks
 * the driver for these on a real call).  Writes out[0] = k slices, out[1] = k
 * per slice (a multiple of 256), out[2] = CTAs launched (a multiple of the
 * slices), out[3] = cluster size (1: one slice, or slices summed with atomics
 * into C after a zeroing kernel; 2 or 4: the slices of a tile on one cluster,
 * summed through distributed shared memory).  The pages have no counterpart;
 * the kernel and the split are this library's.  IGEMM_INVALID_ARGUMENT for a
 * variant other than 0 or 1, M outside [1, 64], N < 1, K < 32, K % 32 != 0,
 * K > 65536, sms < 1, negative cluster counts or a null `out`;
 * IGEMM_UNSUPPORTED_SHAPE when no plan fits.
 */
IGEMM_API int igemm_skinny_plan(int variant, int M, int N, int K, int sms, int pairs, int quads, int *out);

/*
 * Planning query, host only: the work plan of the prepared-codes kernel (the
 * path of large products) for i4i4_gemm (variant 0) or w4a8_gemm (variant 1)
 * on a GPU where `clusters` CTA pairs of it fit at once, checked on the host by
 * enumerating every pair's units the way the kernel does.  Tiles run whole,
 * round robin over the pairs, except the last partial wave, whose k blocks are
 * dealt out evenly (stream-K): each pair takes one range of them, cut where a
 * tile ends, and the pieces add into C.  Writes out[0] = k splits of every tile
 * (K past 65536), out[1] = k blocks of 128 per split, out[2] = whole units,
 * out[3] = tiles of the stream-K tail (0: none), out[4] = k blocks per pair
 * range of the tail, out[5] = pairs launched, out[6] = 1 when every k block of
 * every tile is covered exactly once with one unit per tile starting at k 0,
 * else 0.  The pages have no counterpart; the plan is this library's.
 * IGEMM_INVALID_ARGUMENT for a variant other than 0 or 1, M or N < 1, K < 32,
 * K % 32 != 0, K past the variant's bound, clusters < 1 or a null `out`.
 */
IGEMM_API int igemm_ss_plan(int variant, int M, int N, int K, int clusters, int *out);

/*
 * Routing query, host only: the path an i4i4_gemm (variant 0) or w4a8_gemm
 * (variant 1) call of this shape takes on a GPU with `sms` SMs where `pairs`
 * clusters of two and `quads` clusters of four of the skinny kernel fit (the
 * calls use the same decisions, with the device's own counts).  Writes *route:
 * 0 = skinny kernel (M <= 64: split K, activation codes resident), 1 =
 * small-product kernel (one CTA per output tile), 2 = prepared codes (a pass
 * writes both operands' codes, then the CTA-pair kernel), 3 = in-kernel
 * unpacking kernel, 4 = prepared activation codes with the weights expanded in
 * the CTA-pair kernel (W4A8 only).  IGEMM_INVALID_ARGUMENT for a variant other
 * than 0 or 1, M or N < 1, K < 32, K % 32 != 0, K past the variant's bound,
 * sms < 1, negative cluster counts or a null `route`.
 */
IGEMM_API int igemm_route(int variant, int M, int N, int K, int sms, int pairs, int quads, int *route);

/*
 * Measurement hook: arms two caller-created CUDA events for the next GEMM call
 * (any of the GEMM entry points) made by this host thread.  That call records
 * `start` on its stream right before it launches its GEMM kernel and `stop`
 * right after, so cudaEventElapsedTime(start, stop) is that kernel's duration
 * alone (without the preparation, zeroing or transpose pass before it; while
 * the events are armed the GEMM is not launched to overlap that pass).  Calls
 * that launch no GEMM kernel (empty shapes, argument errors) leave the events
 * armed.  IGEMM_INVALID_ARGUMENT for a null event.
 */
IGEMM_API int igemm_time_next_gemm(cudaEvent_t start, cudaEvent_t stop);

/*
 * Unpack int4 values to int8, the inverse of pack_int4: logical[r, 2j + p] is
 * nibble p (p = 0: low) of packed[r, j], sign-extended from 4 bits, so every
 * value lies in [-8, 7].  This is the conversion the W4A8 page applies to the
 * weights inside its kernel ("[Example] add w4a8 gemm kernel", tilelang PR
 * #815, _tir_u8_to_i4_to_i8: pos 0 = low nibble), as a standalone pass.
 *   packed  [rows, K/2] bytes (device), read only
 *   logical [rows, K] int8 (device), written
 * K must be even (IGEMM_UNSUPPORTED_SHAPE otherwise); rows == 0 or K == 0 is a
 * no-op.  Any alignment is accepted.
 */
IGEMM_API int unpack_int4(const uint8_t *packed, int8_t *logical, int64_t rows, int64_t K, cudaStream_t stream);

/* Static, human-readable text for an igemm_status value. */
IGEMM_API const char *igemm_strerror(int code);

/*
 * Synchronizes `stream`, then returns and clears the device status word of
 * the current device: IGEMM_OK, or IGEMM_DEVICE_TIMEOUT when some kernel of
 * this library had a pipeline wait exceed the watchdog limit (that kernel then
 * stopped early and its C is not valid).  IGEMM_CUDA_ERROR if the
 * synchronization itself failed.  The limit is 2 s per wait, or
 * IGEMM_WATCHDOG_MS milliseconds from the environment (read once).
 */
IGEMM_API int igemm_last_status(cudaStream_t stream);

/*
 * Self-test of the watchdog: enqueues one single-CTA kernel whose wait can
 * never be satisfied (an mbarrier nobody arrives at) with a limit of
 * `limit_us` microseconds.  The kernel gives up, records IGEMM_DEVICE_TIMEOUT
 * in the status word and exits normally; igemm_last_status() then returns it.
 * No GPU fault or hang is involved.  limit_us must be in [1, 1000000].
 */
IGEMM_API int igemm_watchdog_selftest(uint32_t limit_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IGEMM_H */
