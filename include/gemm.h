/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * Every entry point computes C = A·B: C[i,j] = sum_k A[i,k]*B[k,j], 2*M*N*K
 * floating-point operations, with the sum accumulated in FP32 and rounded once
 * to the output type (round to nearest, ties to even).  Sources of the
 * operation:
 *   - the FP32 SGEMM and its FLOP convention: "SGEMM measured and the three
 *     ledgers" (section 2, the cuBLAS baseline in pure FP32 with TF32 off;
 *     K3 step 3, GFLOP/s = 2*M*N*K / t);
 *   - the half, column-major variant: "MTT S4000 FP16 GEMM", section 1 (the
 *     fixed contest signature gemm_optimized(d_A, d_B, d_C, M, N, K): A, B, C
 *     column-major, half in and out, FP32 accumulation);
 *   - the bf16, row-major projection: "Chapter 5 Operators and Runtime",
 *     section 5.2.1 (the FFN projection C = X·W, BF16 inputs, FP32 accumulator,
 *     the element loop over i, j, k) and figure 5-7.
 * alpha = 1 and beta = 0: C is write-only, never read.
 *
 * Pointers.  A, B and C are DEVICE pointers (cudaMalloc, torch CUDA tensors,
 * or any memory the current device can address), owned by the caller.  The
 * library keeps no reference to them after the call.  Half and bf16 elements
 * are passed as their 16-bit patterns.  Memory the library uses besides A, B,
 * C: one 4-byte status word per device (cudaMalloc on first use); and, only for
 * a 16-bit problem with M > 128, N >= 1024 whose A rows are not 16-byte
 * aligned (e.g. bf16 with K = 4100), an aligned copy of A taken from the
 * device's default stream-ordered pool (cudaMallocAsync / cudaFreeAsync on the
 * caller's stream); if that allocation fails the call uses a slower kernel
 * instead.  A 16-bit problem on the CTA-pair tensor-core kernel whose tiles
 * leave a nearly empty last wave (at most a quarter of the clusters busy, K of
 * at least 48 blocks of 64) takes FP32 partial tiles for its stream-K tail from
 * the same pool (512 KiB per participating CTA pair, at most ~39 MB), freed on
 * the stream after the call; without it the call runs whole tiles.  The
 * allocation-free entry point never allocates.
 *
 * Leading dimensions are tight:
 *   _rm (row-major):    A is [M,K] with lda = K, B is [K,N] with ldb = N,
 *                       C is [M,N] with ldc = N.
 *   _cm (column-major): A is [M,K] with lda = M, B is [K,N] with ldb = K,
 *                       C is [M,N] with ldc = M.
 * Any alignment is accepted.  Pointers or strides that are not 16-byte aligned
 * select slower kernels; they are never an error.
 *
 * Execution.  Calls are asynchronous and ordered on the calling host thread's
 * stream (gemm_set_stream; default: the legacy default stream).  A call returns
 * once its kernels are enqueued; gemm_synchronize() waits for them.  The kernels
 * are launched as programmatic dependents: one may start its set-up while the
 * kernel before it on the stream drains, but it touches global memory only once
 * that kernel has completed, so stream order holds for any producer of A or B
 * and any consumer of C, the library's or not.  (An FP32 call whose last round
 * of tiles is at most half full launches two grids; the second reads A and B
 * while the first still runs, and completes only after it.)  A call launches
 * one to three kernels, or more for a general-form batch beyond 65535 matrices;
 * gemm_kernel_launches() counts them.  Calls may be captured into CUDA
 * graphs.  Results are deterministic: the same inputs give bit-identical C on
 * every run (no atomics, fixed summation order per element).
 *
 * Errors.  Every entry point returns a status; nothing is thrown across the ABI.
 *   GEMM_ERR_INVALID_VALUE      a dimension < 0, or a null pointer needed by the
 *                               call (A and B when K > 0; C when M*N > 0), or a
 *                               forced kernel that cannot run this problem.
 *   GEMM_ERR_ALIAS              C overlaps A or B.
 *   GEMM_ERR_UNSUPPORTED_DEVICE the current device is not compute capability
 *                               10.3 (GB300).  There is no fallback to other
 *                               devices or to the CPU.
 *   GEMM_ERR_CUDA               a CUDA runtime call or kernel launch failed.
 *   GEMM_ERR_TIMEOUT            a kernel gave up waiting on one of its own
 *                               pipeline barriers (reported by gemm_synchronize).
 * M = 0 or N = 0 is a no-op returning GEMM_OK.  K = 0 fills C with zeros (the
 * empty sum).
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

#if defined(_WIN32)
#define GEMM_API __declspec(dllexport)
#else
#define GEMM_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm_status_t {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,
    GEMM_ERR_ALIAS = 2,
    GEMM_ERR_UNSUPPORTED_DEVICE = 3,
    GEMM_ERR_CUDA = 4,
    GEMM_ERR_TIMEOUT = 5
} gemm_status_t;

/* Pure FP32 row-major SGEMM on the CUDA cores: FP32 FFMA only, no TF32 and no
 * tensor cores ("SGEMM measured and the three ledgers", section 2).  A [M,K],
 * B [K,N], C [M,N], all row-major float. */
GEMM_API gemm_status_t gemm_f32_rm(const float *A, const float *B, float *C,
                                   int M, int N, int K);

/* Half column-major GEMM with FP32 accumulation ("MTT S4000 FP16 GEMM",
 * section 1).  A [M,K] (lda = M), B [K,N] (ldb = K), C [M,N] (ldc = M), all
 * column-major IEEE half bit patterns. */
GEMM_API gemm_status_t gemm_f16_cm(const uint16_t *A, const uint16_t *B, uint16_t *C,
                                   int M, int N, int K);

/* BF16 row-major projection GEMM with FP32 accumulation ("Chapter 5 Operators
 * and Runtime", section 5.2.1).  A [M,K], B [K,N], C [M,N], row-major bf16 bit
 * patterns. */
GEMM_API gemm_status_t gemm_bf16_rm(const uint16_t *A, const uint16_t *B, uint16_t *C,
                                    int M, int N, int K);

/* Fused FFN gate/up projection ("Chapter 5 Operators and Runtime", section 5.3.1
 * and example 5-4): Z = SiLU(X·W_g) ⊙ (X·W_u), with SiLU(x) = x / (1 + e^-x) and ⊙
 * the element-wise product.  All bf16 row-major with tight strides: X [M,K],
 * W_g [K,N], W_u [K,N], Z [M,N].  Both products accumulate in FP32 on the tensor
 * cores; the fused epilogue keeps the rounding points of the unfused chain
 * (section 5.3.1, figure 5-15): G and U rounded to bf16, T = bf16(SiLU(G)) with
 * SiLU evaluated in FP32, Z = bf16(T·U).  G, U and T are never written to
 * memory.  Needs X, W_g, W_u, Z 16-byte aligned and K, N multiples of 8
 * (GEMM_ERR_INVALID_VALUE otherwise); Z must not overlap an input
 * (GEMM_ERR_ALIAS).  K = 0 gives Z = 0. */
GEMM_API gemm_status_t gemm_bf16_rm_silu_mul(const uint16_t *X, const uint16_t *W_g, const uint16_t *W_u,
                                             uint16_t *Z, int M, int N, int K);

/* BF16 row-major GEMM that allocates no device memory.  The pages have no
 * counterpart to this entry point: it is an interface addition for callers that
 * cannot call cudaMalloc.  Some host applications own all device memory through
 * their own allocator (a framework's caching pool that has already reserved the
 * GPU's memory, or an embedding program with a fixed memory budget) and forbid
 * allocations made behind its back; others run on latency-critical paths where
 * cudaMalloc's implicit device-wide synchronisation is not acceptable.
 *
 * Same arguments, layout, rounding and error codes as gemm_bf16_rm, but always
 * on the tensor-core kernel, so it needs B and C 16-byte aligned with N a
 * multiple of 8, and A either 16-byte aligned with K a multiple of 8 or 8-byte
 * aligned with K a multiple of 4 (otherwise GEMM_ERR_INVALID_VALUE, with a
 * message in gemm_last_error).  The kernel's scratch -- its 4-byte pipeline-timeout status
 * word, the same for every M, N, K -- lives in a static device array of 256
 * bytes that every GPU loading this library holds until the process exits;
 * a problem needing more scratch than that would be refused with
 * GEMM_ERR_INVALID_VALUE.  No call makes cudaMalloc, cudaFree or any other
 * allocating call.
 *
 * The first call on a device does the set-up, once per device, with that device
 * current: it looks up the array's device address and zeroes the status word
 * (a synchronous cudaMemset, which allocates nothing); make that first call
 * before any stream capture.  A pipeline timeout sets the word, which stays set
 * until gemm_synchronize reads and clears it: gemm_synchronize returns
 * GEMM_ERR_TIMEOUT for it, as for the other entry points, and allocates nothing
 * itself.  All calls share the array, so calls that overlap on the GPU race on
 * it: a timeout of either is reported to whichever thread synchronises
 * first. */
GEMM_API gemm_status_t gemm_bf16_rm_noalloc(const uint16_t *A, const uint16_t *B, uint16_t *C,
                                            int M, int N, int K);

/* General form ("SGEMM measured and the three ledgers", section 2: the
 * library call with operation flags and leading dimensions, and the row- and
 * column-major readings of the same bytes; section 3, kernel K1:
 * alpha * acc + beta * C).  For b = 0 .. batch-1:
 *
 *     C_b <- alpha * op(A_b) * op(B_b) + beta * C_b
 *
 * op(X) is X (GEMM_OP_N) or its transpose (GEMM_OP_T); op(A) is M x K, op(B)
 * is K x N, C is M x N.  dtype gives the element type of A, B and C (float, or
 * IEEE half / bf16 bit patterns); alpha and beta are float.  The products are
 * accumulated in FP32; alpha * acc + beta * c is formed in FP32 and rounded
 * once to the output type.
 *
 * Storage.  A stored matrix of R x Cn elements with leading dimension ld holds
 * element (r, c) at r*ld + c (GEMM_ROW_MAJOR) or r + c*ld (GEMM_COL_MAJOR).
 * A is stored M x K for GEMM_OP_N and K x M for GEMM_OP_T; B is stored K x N or
 * N x K; C is stored M x N.  Each leading dimension must be at least the stored
 * matrix's contiguous extent (and at least 1).  Matrix b of A starts stride_a
 * elements after matrix b-1 (likewise B and C); stride_a or stride_b may be 0
 * (one matrix serves every b); stride_c must keep the C matrices apart when
 * batch > 1.  Leading dimensions and strides are in elements, int64.
 * All pointers are device pointers owned by the caller.
 *
 * Reads.  C is not read when beta == 0 (a NaN in C does not reach the result).
 * A and B are not read when alpha == 0 or K == 0; C is then scaled by beta
 * (or set to zero).
 *
 * Errors.  GEMM_ERR_INVALID_VALUE: an unknown enum value; a negative size or
 * stride; a leading dimension below the contiguous extent; overlapping C
 * matrices; a null pointer that would be read or written; sizes whose element
 * span overflows; a forced kernel family that cannot run the problem
 * ("simt" and "umma" are accepted here, the others are not).
 * GEMM_ERR_ALIAS: C's span overlaps A's or B's span.  Otherwise as the entry
 * points above.  M, N or batch == 0 is a no-op.
 *
 * Kernels.  16-bit problems whose A, B, C are 16-byte aligned and whose
 * leading dimensions (and, for batch > 1, nonzero batch strides) and stored
 * contiguous extents (K or M for A, N or K for B, N for C in row-major terms)
 * are multiples of 8 elements run on the tensor-core CTA pairs; everything
 * else, and every FP32 problem, on the SIMT kernel (float4 loads where
 * alignment allows). */
typedef enum gemm_dtype_t { GEMM_F32 = 0, GEMM_F16 = 1, GEMM_BF16 = 2 } gemm_dtype_t;
typedef enum gemm_layout_t { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;
typedef enum gemm_op_t { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op_t;

GEMM_API gemm_status_t gemm_ex(gemm_dtype_t dtype, gemm_layout_t layout, gemm_op_t op_a, gemm_op_t op_b,
                               int M, int N, int K, float alpha,
                               const void *A, int64_t lda, int64_t stride_a,
                               const void *B, int64_t ldb, int64_t stride_b,
                               float beta, void *C, int64_t ldc, int64_t stride_c, int batch);

/* Row-wise FP8 quantisation ("Chapter 5 Operators and Runtime", section 5.4.3,
 * example 5-7).  A is [M,K] row-major IEEE half; for every row i:
 *     amax_i  = max_k |a_ik|
 *     Q[i,k]  = E4M3FN(a_ik * (448 / amax_i))   nearest, ties to even, clamped to +-448
 *     scale_i = amax_i / 448
 * with 448 / amax_i, the product and amax_i / 448 each one FP32 operation, so
 * a_ik ~ Q[i,k] * scale_i.  A row of zeros gives Q = 0 and scale 0.  The whole
 * row is read before any of its codes is written (the scale depends on it).
 * E4M3FN: 1 sign, 4 exponent (bias 7), 3 fraction bits, largest finite 448,
 * no infinities.  Q [M,K] row-major bytes, scale [M] float, device pointers
 * owned by the caller.  Any alignment (16-byte aligned A and 8-byte aligned Q
 * with K % 8 == 0 use vector loads).  NaN or infinite inputs are outside the
 * contract.  K = 0 sets every scale to 0.  Errors: GEMM_ERR_INVALID_VALUE for a
 * negative size or a null pointer; GEMM_ERR_ALIAS if Q, scale and A overlap. */
GEMM_API gemm_status_t gemm_quantize_rows_e4m3(const uint16_t *A, uint8_t *Q, float *scale, int M, int K);

/* Row-scaled FP8 projection ("Chapter 5 Operators and Runtime", section 5.4.4,
 * example 5-8: FP8 input times FP8 weights, FP16 output):
 *     C[i,j] = scale_i * sum_k Q[i,k] * W[k,j]
 * on the tensor cores (E4M3 x E4M3 products, FP32 accumulation), the row scale
 * applied to the FP32 sum, one rounding to half.  Q [M,K] row-major E4M3FN codes
 * and scale [M] as written by gemm_quantize_rows_e4m3; the weights W [K,N] are
 * given transposed, Wt [N,K] row-major (each output column's K codes
 * contiguous, the layout of a linear layer's weight); C [M,N] row-major half.
 * Needs Q, Wt, C 16-byte aligned, K % 16 == 0 and N % 8 == 0
 * (GEMM_ERR_INVALID_VALUE otherwise, with a message in gemm_last_error).
 * K = 0 gives C = 0.  GEMM_ERR_ALIAS if C overlaps Q, Wt or scale. */
GEMM_API gemm_status_t gemm_e4m3_rowscale(const uint8_t *Q, const float *scale, const uint8_t *Wt, uint16_t *C,
                                          int M, int N, int K);

/* Row-scaled FP8 projection with the quantisation fused into the product's
 * load path ("Chapter 5 Operators and Runtime", section 5.4.4, example 5-8, the
 * second scheme: the row scales from a first pass over the whole input, then
 * every column block of the product reads the half input and quantises it
 * locally):
 *     amax_i  = max_k |a_ik|
 *     C[i,j]  = (amax_i / 448) * sum_k E4M3(a_ik * (448 / amax_i)) * W[k,j]
 * -- the codes and the row scale of gemm_quantize_rows_e4m3 (the same FP32
 * steps), but never written to memory: the product's loader quantises each
 * tile of A as it stages it.  A [M,K] row-major IEEE half; the weights W [K,N]
 * given transposed, Wt [N,K] row-major E4M3FN codes; C [M,N] row-major half.
 * Results equal gemm_quantize_rows_e4m3 followed by gemm_e4m3_rowscale up to
 * the summation order of the FP32 accumulation.  The rows' amax (4 bytes per
 * row) are kept in the device's default stream-ordered pool for the duration
 * of the call (cudaMallocAsync / cudaFreeAsync on the caller's stream).  Needs
 * A, Wt, C 16-byte aligned, K % 16 == 0 and N % 8 == 0
 * (GEMM_ERR_INVALID_VALUE otherwise, with a message in gemm_last_error).
 * K = 0 gives C = 0.  GEMM_ERR_ALIAS if C overlaps A or Wt.  NaN or infinite
 * inputs are outside the contract. */
GEMM_API gemm_status_t gemm_e4m3_rowscale_fused(const uint16_t *A, const uint8_t *Wt, uint16_t *C,
                                                int M, int N, int K);

/* Stream for the calling host thread's subsequent calls: a cudaStream_t passed
 * as void*.  NULL selects the legacy default stream.  The stream stays owned by
 * the caller and must outlive the calls issued on it. */
GEMM_API gemm_status_t gemm_set_stream(void *cuda_stream);

/* The calling host thread's current stream (NULL = legacy default stream). */
GEMM_API void *gemm_get_stream(void);

/* Waits for the calling thread's stream; returns GEMM_ERR_CUDA for an
 * asynchronous CUDA error and GEMM_ERR_TIMEOUT if a kernel of this library
 * recorded a pipeline timeout on the current device (the record is cleared).
 * It reads only status words that calls on this device have already set up,
 * so it allocates nothing. */
GEMM_API gemm_status_t gemm_synchronize(void);

/* Static, human-readable name of a status code. */
GEMM_API const char *gemm_status_string(gemm_status_t status);

/* Name of the kernel the calling thread's last call dispatched to, e.g.
 * "simt_f32_vec4", "umma_bf16", "gemv_bf16_vec", "zero_fill", "noop" (static
 * string; for tests and benchmarks). */
GEMM_API const char *gemm_last_kernel(void);

/* Number of CUDA kernels this library has launched in this process, on every
 * thread and device, since it was loaded (one count per launch call issued,
 * whether or not the kernel has run yet).  The difference over a span of calls
 * is the kernels those calls queued; for tests and benchmarks. */
GEMM_API unsigned long long gemm_kernel_launches(void);

/* Message of the last CUDA error seen by the calling thread ("" if none). */
GEMM_API const char *gemm_last_error(void);

/* Test and benchmark hook: forces the calling thread's later calls onto one
 * kernel family -- "simt", "simt_scalar", "gemv", "gemv_scalar", "umma",
 * "umma_skinny_wide" (16-bit, M <= 64: the skinny tensor-core kernel on
 * 256-column strips of B) -- or back to automatic dispatch with NULL or "".  A forced family that cannot run
 * a given problem makes that call return GEMM_ERR_INVALID_VALUE; an unknown
 * name is rejected here with GEMM_ERR_INVALID_VALUE.
 * "umma_stall" tests the tensor-core kernel's bounded waits: a 16-bit call whose
 * A, B and C suit the TMA kernel launches it with a producer that issues no
 * loads, every CTA gives up after about two seconds, C is left unwritten and
 * the next gemm_synchronize returns GEMM_ERR_TIMEOUT.  "umma_stall_pair" does the
 * same on the CTA-pair kernel (16-bit, M > 128, A 16-byte aligned with K a
 * multiple of 8), and "umma_stall_peer" makes the pair's second CTA give up
 * after loading one stage while the first has loaded further, so that the pair
 * ends with loads of only one CTA outstanding.  gemm_bf16_rm_noalloc
 * honours "umma_stall" (recording in its static status word) and ignores the
 * other families. */
GEMM_API gemm_status_t gemm_force_kernel(const char *family);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
