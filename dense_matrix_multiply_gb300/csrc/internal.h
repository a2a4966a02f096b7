// Internal launcher interface shared by the C-ABI layer and the kernels.
// Every problem reaching a launcher is row-major: Problem is the tight
// C[M,N] = A[M,K] · B[K,N] with M, N, K >= 1; ProblemEx the general form.
// Column-major problems are mapped onto row-major ones before dispatch
// (C^T = B^T · A^T).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace gemm_gb300 {

// Programmatic dependent launch.  Every kernel is launched with programmatic
// stream serialisation allowed: it may start while the previous kernel on the
// stream drains.  After a prologue that touches only its shared memory, tensor
// memory and parameters -- the skinny kernels add L2 prefetch hints for their
// first weight tiles, which read nothing and change no value a later load
// returns -- it waits for the previous grid to complete and its writes to
// become visible (pdl_wait) before its first global-memory access.
// The tensor-core kernels (one CTA per SM) also let their own dependents launch
// at once (pdl_launch_dependents) -- the skinny ones once every CTA has issued
// its last load, so that the dependent's CTAs prefetch their first weights
// into L2 while this grid drains; kernels with several CTAs per SM leave that
// to their CTAs' exit, so that a small grid's successor is not placed, and
// packed onto the same SMs, while the grid still runs (FP32 1000^3: 86 against
// 49 us).  The one exception is the first grid of an FP32 problem split in two,
// whose dependent is its own last round (that packing is the point).  Back to back on GB300 this hides the 2-3 us between kernels: a
// 100 MB weight stream went from 18.5 to 15.9 us.
#ifndef GEMM_PDL
#define GEMM_PDL 1
#endif
constexpr bool g_pdl = GEMM_PDL != 0;
// Kernel launches issued by the library (gemm_kernel_launches): every launch
// goes through launch_counted or calls note_launch next to its <<< >>>.
extern std::atomic<unsigned long long> g_launches;
inline void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
template <typename... KArgs, typename... Args>
inline cudaError_t launch_counted(const cudaLaunchConfig_t *cfg, void (*kern)(KArgs...), Args &&...args) {
    note_launch();
    return cudaLaunchKernelEx(cfg, kern, std::forward<Args>(args)...);
}
inline void pdl_attr(cudaLaunchAttribute &a) {
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
}
// Launch configuration with programmatic dependent launch allowed (the
// attribute array must outlive the launch call; a cluster dimension may be
// appended after it).
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    pdl_attr(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 1 : 0;
    return cfg;
}
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_launch_dependents() {
    if (g_pdl) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    if (g_pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
}
#endif

// Per-device tables of the library hold this many devices (ordinals 0 .. 63).
constexpr int kMaxDevices = 64;

enum class Elt { F32, F16, BF16 };

struct Problem {
    const void *A;
    const void *B;
    void *C;
    int M, N, K;
    Elt elt;
};

// The general form, row-major: C_b = alpha * op(A_b) * op(B_b) + beta * C_b
// for b < batch.  a_t: A is stored [K, M] (op(A) = A^T), else [M, K]; b_t: B is
// stored [N, K], else [K, N]; C is [M, N].  Leading dimensions and batch
// strides in elements; a batch stride may be 0 for A or B (one matrix for
// every b).  C is read only when beta != 0.  M, N, K, batch >= 1 and
// alpha != 0 when this reaches a launcher.
struct ProblemEx {
    const void *A;
    const void *B;
    void *C;
    int M, N, K, batch;
    bool a_t, b_t;
    long long lda, ldb, ldc;
    long long sa, sb, sc;
    float alpha, beta;
    Elt elt;
};

// FP32 (or 16-bit fallback) SIMT kernel on the CUDA cores.  vec4: float4
// global loads/stores (needs K % 4 == 0, N % 4 == 0 and 16-byte aligned bases;
// f32 only).  num_sms sizes the split of a partly filled last wave.  Returns
// the launch status.
cudaError_t launch_simt(const Problem &p, bool vec4, int num_sms, cudaStream_t s);

// The general form on the SIMT kernel (any alignment, any leading dimension;
// FP32 or 16-bit).  Vector loads where every operand allows them.
cudaError_t launch_simt_ex(const ProblemEx &p, cudaStream_t s);
bool simt_ex_vec(const ProblemEx &p);  // whether launch_simt_ex uses float4 loads

// Skinny-M kernel (M <= kGemvMaxM): streams B once, FP32 accumulation, K split
// over a thread-block cluster, fixed-order reduction in shared and distributed
// shared memory.  vec: 16-byte loads of B (needs N a multiple of the vector
// width and a 16-byte aligned B).  num_sms sizes the split.
constexpr int kGemvMaxM = 8;
cudaError_t launch_gemv(const Problem &p, bool vec, int num_sms, cudaStream_t s);

// tcgen05 tensor-core kernel for 16-bit inputs.  Needs B and C 16-byte aligned
// with N % 8 == 0 (TMA for B, vector stores for C), and A either TMA-describable
// (16-byte aligned, K % 8 == 0) or 8-byte aligned with K % 4 == 0.  num_sms:
// persistent grid size.  status: device word the kernel ORs a timeout code
// into.  may_allocate: large problems with unaligned A rows may stage A in
// stream-ordered scratch (cudaMallocAsync); without it they use cp.async.
cudaError_t launch_umma(const Problem &p, int num_sms, int *status, cudaStream_t s, bool may_allocate = true);
bool umma_supported(const Problem &p);

// Skinny 16-bit GEMM (1 <= M <= 64) on 256-column strips of B, K split over a
// cluster of up to 8 CTAs (see skinny_wide.cu).  Needs A and B 16-byte
// aligned, C 8-byte aligned, K % 8 == 0 and N % 8 == 0 (cudaErrorNotSupported
// otherwise, before any launch).  status: device word for timeout codes.
bool skinny_wide_supported(const Problem &p);
cudaError_t launch_skinny_wide(const Problem &p, int num_sms, int *status, cudaStream_t s);

// The general form on the tensor-core CTA pairs (16-bit only).  Needs A, B, C
// 16-byte aligned, every leading dimension (and, for batch > 1, every nonzero
// batch stride) and every stored matrix's contiguous extent a multiple of 8
// elements.  Returns
// cudaErrorNotSupported, before any launch, when the problem does not qualify.
bool umma_ex_supported(const ProblemEx &p);
cudaError_t launch_umma_ex(const ProblemEx &p, int *status, cudaStream_t s);

// Row-wise E4M3 quantisation of a half [M,K] row-major matrix: Q [M,K] codes,
// scale [M] (see quant_e4m3.cu).  M, K >= 1.
bool quantize_rows_vec_ok(const void *A, const void *Q, int K);
cudaError_t launch_quantize_rows_e4m3(const void *A, void *Q, float *scale, int M, int K, cudaStream_t s);

// Row-scaled FP8 product on the tensor-core CTA pairs: C [M,N] half =
// diag(scale) * Q [M,K] * Wt^T with Q and Wt [N,K] E4M3 codes, row-major.
// Needs Q, Wt, C 16-byte aligned, K % 16 == 0, N % 8 == 0; returns
// cudaErrorNotSupported, before any launch, otherwise.
bool umma_e4m3_supported(const void *Q, const void *Wt, const void *C, int N, int K);
cudaError_t launch_umma_e4m3_rowscale(const void *Q, const float *scale, const void *Wt, void *C, int M, int N,
                                      int K, int *status, cudaStream_t s);

// Row amax of a half [M,K] row-major matrix: amax[i] = max_k |a_ik| (see
// quant_e4m3.cu).  M, K >= 1.
cudaError_t launch_row_amax_f16(const void *A, float *amax, int M, int K, cudaStream_t s);

// Row-scaled FP8 product with the quantisation fused into the load path: C
// [M,N] half = diag(amax/448) E4M3(diag(448/amax) A) Wt^T, A [M,K] half, Wt
// [N,K] E4M3, row-major.  A row amax pass first (its M floats in stream-ordered
// scratch), then the CTA-pair kernel whose converter warps quantise A's tiles
// as they load them.  Needs A, Wt, C 16-byte aligned, K % 16 == 0, N % 8 == 0;
// returns cudaErrorNotSupported, before any launch, otherwise.
bool umma_e4m3_fused_supported(const void *A, const void *Wt, const void *C, int N, int K);
cudaError_t launch_umma_e4m3_fused(const void *A, const void *Wt, void *C, int M, int N, int K, int *status,
                                   cudaStream_t s);

// Test of the bounded pipeline waits: the single-CTA tensor-core kernel with a
// producer that issues no load, so every CTA takes its timeout path (~2 s) and
// records a code in *status.  Returns the launch status.
cudaError_t launch_umma_stall_test(const Problem &p, int num_sms, int *status, cudaStream_t s);
// The same on the CTA-pair kernel (16-bit, M > 128, A TMA-describable).  mode
// 1: both producers load nothing; mode 2: the peer CTA loads one stage and
// gives up (recording a timeout) while the leader has loaded further.  Either way the leader's MMA thread gives up,
// raises the abort flag of both CTAs, the leader waits until every stage either
// CTA loaded has landed, and the pair ends with its tensor memory released.
cudaError_t launch_umma_pair_stall_test(const Problem &p, int mode, int *status, cudaStream_t s);

// Fused FFN gate/up projection Z = SiLU(X W_g) * (X W_u) on the tensor-core
// CTA pairs: p.A = X [M,K], p.B = W_g [K,N], p.C = Z [M,N], w_u = W_u [K,N],
// all bf16 row-major, 16-byte aligned, K % 8 == 0, N % 8 == 0.
bool umma_silu_mul_supported(const Problem &p, const void *w_u);
cudaError_t launch_umma_silu_mul(const Problem &p, const void *w_u, int *status, cudaStream_t s);

// Allocation-free variant of launch_umma: the status word lives in a static
// device array of kNoallocScratchBytes bytes (see umma_gemm.cu).  stall: the
// bounded-wait test kernel instead (as launch_umma_stall_test).
constexpr size_t kNoallocScratchBytes = 256;
size_t umma_noalloc_scratch_need(const Problem &p);
cudaError_t launch_umma_noalloc(const Problem &p, int num_sms, cudaStream_t s, bool stall = false);
// Reads the allocation-free entry point's status word on device `dev` into
// *code and clears it; *code = 0 if that entry point was never set up there.
// Synchronous; allocates nothing.
cudaError_t take_noalloc_status(int dev, int *code);

}  // namespace gemm_gb300
