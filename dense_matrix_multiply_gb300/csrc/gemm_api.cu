// C ABI of the library: argument checks, per-thread stream, device check,
// dispatch to the kernels.  See include/gemm.h for the contract.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "gemm.h"
#include "internal.h"

using namespace gemm_gb300;

std::atomic<unsigned long long> gemm_gb300::g_launches{0};

namespace {

enum class Family { Auto, Simt, SimtScalar, Gemv, GemvScalar, Umma, UmmaSkinnyWide, UmmaStall, UmmaStallPair, UmmaStallPeer };

thread_local cudaStream_t t_stream = nullptr;
thread_local const char *t_last_kernel = "none";
thread_local char t_last_error[256] = "";
thread_local Family t_force = Family::Auto;

struct DeviceInfo {
    std::once_flag once;
    std::atomic<bool> ready{false};  // set once the status word exists
    bool supported = false;
    int num_sms = 0;
    int *status = nullptr;  // device word the tensor-core kernel reports timeouts in
    cudaError_t init_error = cudaSuccess;
};
DeviceInfo g_devices[kMaxDevices];

__global__ void zero_fill_kernel(uint4 *p, size_t n16, uint8_t *tail, size_t ntail) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
        p[i] = make_uint4(0, 0, 0, 0);
    if (blockIdx.x == 0 && threadIdx.x < ntail) tail[threadIdx.x] = 0;
}

__global__ void zero_fill_bytes_kernel(uint8_t *p, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0;
}

// Zeros `bytes` bytes at p on stream s (16-byte stores when p is aligned).
cudaError_t zero_fill(void *p, size_t bytes, int num_sms, cudaStream_t s) {
    const unsigned grid = (unsigned)(num_sms * 4);
    note_launch();
    if (((uintptr_t)p & 15u) == 0) {
        zero_fill_kernel<<<grid, 256, 0, s>>>((uint4 *)p, bytes / 16, (uint8_t *)p + (bytes & ~(size_t)15),
                                              bytes & 15);
    } else {
        zero_fill_bytes_kernel<<<grid, 256, 0, s>>>((uint8_t *)p, bytes);
    }
    return cudaGetLastError();
}

__device__ __forceinline__ float elt_to_f32(float x) { return x; }
__device__ __forceinline__ float elt_to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float elt_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void elt_from_f32(float *p, float x) { *p = x; }
__device__ __forceinline__ void elt_from_f32(__half *p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void elt_from_f32(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// The general form when the product term is absent (alpha == 0 or K == 0):
// C_b = beta * C_b over row-major [M, N] matrices with leading dimension ldc,
// and C_b = 0 without reading it when beta == 0.
template <typename T>
__global__ void scale_c_kernel(T *C, int M, int N, long long ldc, long long sc, long long batch, float beta) {
    const long long per = (long long)M * N, total = batch * per;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const long long b = i / per, r = i - b * per;
        const long long row = r / N, col = r - row * N;
        T *p = C + b * sc + row * ldc + col;
        elt_from_f32(p, beta == 0.0f ? 0.0f : beta * elt_to_f32(*p));
    }
}

void record_cuda_error(cudaError_t e) {
    strncpy(t_last_error, cudaGetErrorString(e), sizeof(t_last_error) - 1);
    t_last_error[sizeof(t_last_error) - 1] = '\0';
}

// Per-device set-up on first use: capability check, SM count, status word.
gemm_status_t device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { record_cuda_error(e); return GEMM_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    DeviceInfo &d = g_devices[dev];
    std::call_once(d.once, [&] {
        int major = 0, minor = 0;
        cudaError_t err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) { d.init_error = err; return; }
        d.supported = (major == 10 && minor == 3);
        if (!d.supported) return;
        err = cudaMalloc(&d.status, sizeof(int));
        if (err == cudaSuccess) err = cudaMemset(d.status, 0, sizeof(int));
        if (err != cudaSuccess) d.init_error = err;
        else d.ready.store(true, std::memory_order_release);
    });
    if (d.init_error != cudaSuccess) { record_cuda_error(d.init_error); return GEMM_ERR_CUDA; }
    if (!d.supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return GEMM_OK;
}

bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return an && bn && a0 < b0 + bn && b0 < a0 + an;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

gemm_status_t finish(cudaError_t e, const char *name) {
    t_last_kernel = name;
    if (e == cudaSuccess) return GEMM_OK;
    record_cuda_error(e);
    return GEMM_ERR_CUDA;
}

const char *kernel_name(const char *fam, Elt elt) {
    // Static names: family x element type.
    static const char *names[5][3] = {
        {"simt_f32_vec4", "simt_f16_scalar", "simt_bf16_scalar"},
        {"simt_f32_scalar", "simt_f16_scalar", "simt_bf16_scalar"},
        {"gemv_f32_vec", "gemv_f16_vec", "gemv_bf16_vec"},
        {"gemv_f32_scalar", "gemv_f16_scalar", "gemv_bf16_scalar"},
        {"umma_f32", "umma_f16", "umma_bf16"},
    };
    int f = 0;
    if (!strcmp(fam, "simt")) f = 0;
    else if (!strcmp(fam, "simt_scalar")) f = 1;
    else if (!strcmp(fam, "gemv")) f = 2;
    else if (!strcmp(fam, "gemv_scalar")) f = 3;
    else f = 4;
    return names[f][(int)elt];
}

// Row-major problem C[M,N] = A[M,K] B[K,N] with tight strides.
gemm_status_t run(const void *A, const void *B, void *C, int M, int N, int K, Elt elt) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    const size_t es = elt == Elt::F32 ? 4 : 2;
    if (M == 0 || N == 0) { t_last_kernel = "noop"; return GEMM_OK; }
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_VALUE;
    const size_t c_bytes = (size_t)M * N * es;
    if (overlaps(C, c_bytes, A, (size_t)M * K * es) || overlaps(C, c_bytes, B, (size_t)K * N * es))
        return GEMM_ERR_ALIAS;

    DeviceInfo *dev = nullptr;
    gemm_status_t st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = t_stream;

    if (K == 0) {
        if (t_force != Family::Auto) return GEMM_ERR_INVALID_VALUE;
        return finish(zero_fill(C, c_bytes, dev->num_sms, s), "zero_fill");
    }

    Problem p{A, B, C, M, N, K, elt};
    const int vw = elt == Elt::F32 ? 4 : 8;
    const bool gemv_vec_ok = (N % vw) == 0 && aligned16(B);
    const bool simt_vec_ok = elt == Elt::F32 && (K % 4) == 0 && (N % 4) == 0 && aligned16(A) &&
                             aligned16(B) && aligned16(C);

    switch (t_force) {
    case Family::Simt:
        if (elt == Elt::F32 && !simt_vec_ok) return GEMM_ERR_INVALID_VALUE;
        return finish(launch_simt(p, elt == Elt::F32, dev->num_sms, s), kernel_name("simt", elt));
    case Family::SimtScalar:
        return finish(launch_simt(p, false, dev->num_sms, s), kernel_name("simt_scalar", elt));
    case Family::Gemv:
        if (M > kGemvMaxM || !gemv_vec_ok) return GEMM_ERR_INVALID_VALUE;
        return finish(launch_gemv(p, true, dev->num_sms, s), kernel_name("gemv", elt));
    case Family::GemvScalar:
        if (M > kGemvMaxM) return GEMM_ERR_INVALID_VALUE;
        return finish(launch_gemv(p, false, dev->num_sms, s), kernel_name("gemv_scalar", elt));
    case Family::Umma:
        if (!umma_supported(p)) return GEMM_ERR_INVALID_VALUE;
        return finish(launch_umma(p, dev->num_sms, dev->status, s), kernel_name("umma", elt));
    case Family::UmmaSkinnyWide:
        if (!skinny_wide_supported(p)) return GEMM_ERR_INVALID_VALUE;
        return finish(launch_skinny_wide(p, dev->num_sms, dev->status, s),
                      elt == Elt::BF16 ? "umma_skinny_wide_bf16" : "umma_skinny_wide_f16");
    case Family::UmmaStall:
        if (elt == Elt::F32) return GEMM_ERR_INVALID_VALUE;
        return finish(launch_umma_stall_test(p, dev->num_sms, dev->status, s), "umma_stall");
    case Family::UmmaStallPair:
    case Family::UmmaStallPeer: {
        if (elt == Elt::F32 || M <= 128) return GEMM_ERR_INVALID_VALUE;
        const bool peer = t_force == Family::UmmaStallPeer;
        return finish(launch_umma_pair_stall_test(p, peer ? 2 : 1, dev->status, s),
                      peer ? "umma_stall_peer" : "umma_stall_pair");
    }
    case Family::Auto:
        break;
    }

    // Skinny M: the streaming GEMV for FP32 and for 16-bit problems the
    // tensor-core kernels cannot take; other 16-bit problems with M <= 8 run on
    // the tensor cores (the skinny kernels, weights as the MMA's rows), which
    // stream B faster -- for M = 1 too whenever the X rows suit TMA and the
    // 256-column strips fit on the SMs at once.  Measured back to back (bf16, W
    // from DRAM), skinny against GEMV, M = 1: N = 12288, K = 4096 17.7 vs
    // 18.8 us; N = 4096, K = 12288 19.1 vs 22.2; N = 1024, K = 4096 5.5 vs 7.3;
    // N = 28672, K = 4096 38.1 vs 48.6.
    const bool m1_tensor = M == 1 && elt != Elt::F32 && umma_supported(p) && (K % 8) == 0 && aligned16(A) &&
                           (N + 255) / 256 <= dev->num_sms;
    if (M <= kGemvMaxM && (elt == Elt::F32 || (M == 1 && !m1_tensor) || !umma_supported(p)))
        return gemv_vec_ok ? finish(launch_gemv(p, true, dev->num_sms, s), kernel_name("gemv", elt))
                           : finish(launch_gemv(p, false, dev->num_sms, s), kernel_name("gemv_scalar", elt));
    if (elt == Elt::F32)
        return simt_vec_ok ? finish(launch_simt(p, true, dev->num_sms, s), kernel_name("simt", elt))
                           : finish(launch_simt(p, false, dev->num_sms, s), kernel_name("simt_scalar", elt));
    if (umma_supported(p)) return finish(launch_umma(p, dev->num_sms, dev->status, s), kernel_name("umma", elt));
    return finish(launch_simt(p, false, dev->num_sms, s), kernel_name("simt_scalar", elt));
}

// Capability and SM count of the current device, without allocating anything
// (used only by the allocation-free entry point).
struct PlainDeviceInfo {
    std::once_flag once;
    bool supported = false;
    int num_sms = 0;
    cudaError_t err = cudaSuccess;
};
PlainDeviceInfo g_plain_devices[kMaxDevices];

gemm_status_t plain_device_info(PlainDeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { record_cuda_error(e); return GEMM_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    PlainDeviceInfo &d = g_plain_devices[dev];
    std::call_once(d.once, [&] {
        int major = 0, minor = 0;
        cudaError_t err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        d.err = err;
        d.supported = err == cudaSuccess && major == 10 && minor == 3;
    });
    if (d.err != cudaSuccess) { record_cuda_error(d.err); return GEMM_ERR_CUDA; }
    if (!d.supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return GEMM_OK;
}

void record_message(const char *msg) {
    strncpy(t_last_error, msg, sizeof(t_last_error) - 1);
    t_last_error[sizeof(t_last_error) - 1] = '\0';
}

// a * b + c for non-negative operands; false if it exceeds 2^62.
bool mul_add(long long a, long long b, long long c, long long *out) {
    const long long lim = 1LL << 62;
    if (a < 0 || b < 0 || c < 0) return false;
    if (a != 0 && b > (lim - c) / a) return false;
    *out = a * b + c;
    return true;
}

// Elements from the first to one past the last one that `batch` stored
// matrices of [outer, inner] (leading dimension ld, matrix stride `stride`)
// touch: (batch - 1) * stride + (outer - 1) * ld + inner.  false on overflow.
bool span_elems(long long batch, long long stride, long long outer, long long ld, long long inner, long long *out) {
    long long one = 0, all = 0;
    if (outer < 1 || inner < 1 || batch < 1) { *out = 0; return true; }
    if (!mul_add(outer - 1, ld, inner, &one)) return false;
    if (!mul_add(batch - 1, stride, one, &all)) return false;
    *out = all;
    return true;
}

gemm_status_t run_ex(int dtype, int layout, int op_a, int op_b, int M, int N, int K, float alpha, const void *A,
                     long long lda, long long sa, const void *B, long long ldb, long long sb, float beta, void *C,
                     long long ldc, long long sc, int batch) {
    if (dtype < GEMM_F32 || dtype > GEMM_BF16) return GEMM_ERR_INVALID_VALUE;
    if (layout != GEMM_ROW_MAJOR && layout != GEMM_COL_MAJOR) return GEMM_ERR_INVALID_VALUE;
    if ((op_a != GEMM_OP_N && op_a != GEMM_OP_T) || (op_b != GEMM_OP_N && op_b != GEMM_OP_T))
        return GEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || batch < 0 || sa < 0 || sb < 0 || sc < 0) return GEMM_ERR_INVALID_VALUE;
    const Elt elt = dtype == GEMM_F32 ? Elt::F32 : dtype == GEMM_F16 ? Elt::F16 : Elt::BF16;
    const long long es = elt == Elt::F32 ? 4 : 2;
    // Column-major C = op(A) op(B) is row-major C^T = op(B)^T op(A)^T on the
    // same buffers ("SGEMM measured and the three ledgers", section 2): swap the
    // operands, their flags, leading dimensions and strides, and M with N.
    if (layout == GEMM_COL_MAJOR) {
        const void *tp = A; A = B; B = tp;
        long long t = lda; lda = ldb; ldb = t;
        t = sa; sa = sb; sb = t;
        int ti = op_a; op_a = op_b; op_b = ti;
        ti = M; M = N; N = ti;
    }
    // Row-major from here on.  A is stored [M,K] ('N') or [K,M] ('T'); B is
    // stored [K,N] or [N,K]; C is [M,N].
    const bool a_t = op_a == GEMM_OP_T, b_t = op_b == GEMM_OP_T;
    const long long a_inner = a_t ? M : K, a_outer = a_t ? K : M;
    const long long b_inner = b_t ? K : N, b_outer = b_t ? N : K;
    const long long one = 1;
    if (ldc < (N > 1 ? N : one) || lda < (a_inner > 1 ? a_inner : one) || ldb < (b_inner > 1 ? b_inner : one))
        return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0 || batch == 0) { t_last_kernel = "noop"; return GEMM_OK; }
    const bool use_ab = alpha != 0.0f && K > 0;
    if (!C || (use_ab && (!A || !B))) return GEMM_ERR_INVALID_VALUE;
    long long c_one = 0, c_span = 0, a_span = 0, b_span = 0;
    if (!span_elems(1, 0, M, ldc, N, &c_one) || !span_elems(batch, sc, M, ldc, N, &c_span))
        return GEMM_ERR_INVALID_VALUE;
    if (batch > 1 && sc < c_one) return GEMM_ERR_INVALID_VALUE;  // the C matrices would overlap
    if (use_ab) {
        if (!span_elems(batch, sa, a_outer, lda, a_inner, &a_span) ||
            !span_elems(batch, sb, b_outer, ldb, b_inner, &b_span))
            return GEMM_ERR_INVALID_VALUE;
        if (c_span > (1LL << 62) / es || a_span > (1LL << 62) / es || b_span > (1LL << 62) / es)
            return GEMM_ERR_INVALID_VALUE;
        if (overlaps(C, (size_t)(c_span * es), A, (size_t)(a_span * es)) ||
            overlaps(C, (size_t)(c_span * es), B, (size_t)(b_span * es)))
            return GEMM_ERR_ALIAS;
    }

    DeviceInfo *dev = nullptr;
    gemm_status_t st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = t_stream;

    if (!use_ab) {
        if (t_force != Family::Auto) return GEMM_ERR_INVALID_VALUE;
        const unsigned grid = (unsigned)(dev->num_sms * 8);
        note_launch();
        switch (elt) {
        case Elt::F32: scale_c_kernel<<<grid, 256, 0, s>>>((float *)C, M, N, ldc, sc, batch, beta); break;
        case Elt::F16: scale_c_kernel<<<grid, 256, 0, s>>>((__half *)C, M, N, ldc, sc, batch, beta); break;
        case Elt::BF16: scale_c_kernel<<<grid, 256, 0, s>>>((__nv_bfloat16 *)C, M, N, ldc, sc, batch, beta); break;
        }
        return finish(cudaGetLastError(), "scale_c");
    }

    ProblemEx p = {};
    p.A = A;
    p.B = B;
    p.C = C;
    p.M = M;
    p.N = N;
    p.K = K;
    p.batch = batch;
    p.a_t = a_t;
    p.b_t = b_t;
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.sa = sa;
    p.sb = sb;
    p.sc = sc;
    p.alpha = alpha;
    p.beta = beta;
    p.elt = elt;
    static const char *simt_names[3] = {"simt_ex_f32", "simt_ex_f16", "simt_ex_bf16"};
    const char *simt_name = simt_ex_vec(p) ? "simt_ex_f32_vec4" : simt_names[(int)elt];
    const char *umma_name = elt == Elt::BF16 ? "umma_ex_bf16" : "umma_ex_f16";

    switch (t_force) {
    case Family::Simt:
        return finish(launch_simt_ex(p, s), simt_name);
    case Family::Umma: {
        if (!umma_ex_supported(p)) return GEMM_ERR_INVALID_VALUE;
        const cudaError_t e = launch_umma_ex(p, dev->status, s);
        if (e == cudaErrorNotSupported) return GEMM_ERR_INVALID_VALUE;
        return finish(e, umma_name);
    }
    case Family::Auto:
        break;
    default:
        return GEMM_ERR_INVALID_VALUE;
    }
    if (elt != Elt::F32 && umma_ex_supported(p)) {
        const cudaError_t e = launch_umma_ex(p, dev->status, s);
        if (e != cudaErrorNotSupported) return finish(e, umma_name);
    }
    return finish(launch_simt_ex(p, s), simt_name);
}

}  // namespace

extern "C" {

GEMM_API gemm_status_t gemm_ex(gemm_dtype_t dtype, gemm_layout_t layout, gemm_op_t op_a, gemm_op_t op_b, int M,
                               int N, int K, float alpha, const void *A, int64_t lda, int64_t stride_a,
                               const void *B, int64_t ldb, int64_t stride_b, float beta, void *C, int64_t ldc,
                               int64_t stride_c, int batch) {
    return run_ex((int)dtype, (int)layout, (int)op_a, (int)op_b, M, N, K, alpha, A, lda, stride_a, B, ldb,
                  stride_b, beta, C, ldc, stride_c, batch);
}

GEMM_API gemm_status_t gemm_f32_rm(const float *A, const float *B, float *C, int M, int N, int K) {
    return run(A, B, C, M, N, K, Elt::F32);
}

// Column-major C = A·B is row-major C^T = B^T·A^T on the same buffers: the
// column-major B buffer read row-major is B^T [N,K], the column-major A buffer
// read row-major is A^T [K,M], and the row-major [N,M] result is the
// column-major [M,N] C ("SGEMM measured and the three ledgers", section 2).
GEMM_API gemm_status_t gemm_f16_cm(const uint16_t *A, const uint16_t *B, uint16_t *C, int M, int N, int K) {
    return run(B, A, C, N, M, K, Elt::F16);
}

GEMM_API gemm_status_t gemm_bf16_rm(const uint16_t *A, const uint16_t *B, uint16_t *C, int M, int N, int K) {
    return run(A, B, C, M, N, K, Elt::BF16);
}

// Allocation-free bf16 entry point: the tensor-core kernel with its status word
// in a static device array instead of library-allocated memory.
GEMM_API gemm_status_t gemm_bf16_rm_noalloc(const uint16_t *A, const uint16_t *B, uint16_t *C, int M, int N,
                                            int K) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) { t_last_kernel = "noop"; return GEMM_OK; }
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_VALUE;
    const size_t c_bytes = (size_t)M * N * 2;
    if (overlaps(C, c_bytes, A, (size_t)M * K * 2) || overlaps(C, c_bytes, B, (size_t)K * N * 2))
        return GEMM_ERR_ALIAS;
    PlainDeviceInfo *dev = nullptr;
    gemm_status_t st = plain_device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = t_stream;
    if (K == 0) {
        return finish(zero_fill(C, c_bytes, dev->num_sms, s), "zero_fill");
    }
    Problem p{A, B, C, M, N, K, Elt::BF16};
    const bool stall = t_force == Family::UmmaStall;
    if (stall && !umma_supported(p)) return GEMM_ERR_INVALID_VALUE;
    if (!umma_supported(p)) {
        record_message("gemm_bf16_rm_noalloc: needs B and C 16-byte aligned with N % 8 == 0, and A 16-byte "
                       "aligned with K % 8 == 0 or 8-byte aligned with K % 4 == 0");
        return GEMM_ERR_INVALID_VALUE;
    }
    if (umma_noalloc_scratch_need(p) > kNoallocScratchBytes) {
        record_message("gemm_bf16_rm_noalloc: problem needs more scratch than the static array holds");
        return GEMM_ERR_INVALID_VALUE;
    }
    if (stall) return finish(launch_umma_noalloc(p, dev->num_sms, s, true), "umma_stall");
    return finish(launch_umma_noalloc(p, dev->num_sms, s), "umma_bf16_noalloc");
}

GEMM_API gemm_status_t gemm_bf16_rm_silu_mul(const uint16_t *X, const uint16_t *Wg, const uint16_t *Wu, uint16_t *Z,
                                             int M, int N, int K) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) { t_last_kernel = "noop"; return GEMM_OK; }
    if (!Z || (K > 0 && (!X || !Wg || !Wu))) return GEMM_ERR_INVALID_VALUE;
    const size_t z_bytes = (size_t)M * N * 2, w_bytes = (size_t)K * N * 2;
    if (overlaps(Z, z_bytes, X, (size_t)M * K * 2) || overlaps(Z, z_bytes, Wg, w_bytes) ||
        overlaps(Z, z_bytes, Wu, w_bytes))
        return GEMM_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    gemm_status_t st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = t_stream;
    if (K == 0) {  // G = U = 0, SiLU(0) * 0 = 0
        return finish(zero_fill(Z, z_bytes, dev->num_sms, s), "zero_fill");
    }
    Problem p{X, Wg, Z, M, N, K, Elt::BF16};
    if (!umma_silu_mul_supported(p, Wu)) {
        record_message("gemm_bf16_rm_silu_mul: needs X, W_g, W_u, Z 16-byte aligned and K, N multiples of 8");
        return GEMM_ERR_INVALID_VALUE;
    }
    return finish(launch_umma_silu_mul(p, Wu, dev->status, s), "umma_bf16_silu_mul");
}

GEMM_API gemm_status_t gemm_quantize_rows_e4m3(const uint16_t *A, uint8_t *Q, float *scale, int M, int K) {
    if (M < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    if (M == 0) { t_last_kernel = "noop"; return GEMM_OK; }
    if (!scale || (K > 0 && (!A || !Q))) return GEMM_ERR_INVALID_VALUE;
    const size_t a_bytes = (size_t)M * K * 2, q_bytes = (size_t)M * K, s_bytes = (size_t)M * 4;
    if (overlaps(Q, q_bytes, A, a_bytes) || overlaps(scale, s_bytes, A, a_bytes) ||
        overlaps(scale, s_bytes, Q, q_bytes))
        return GEMM_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    gemm_status_t st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = t_stream;
    if (K == 0) {  // every row is empty: amax = 0, scale 0
        const cudaError_t e = cudaMemsetAsync(scale, 0, s_bytes, s);
        return finish(e, "zero_fill");
    }
    return finish(launch_quantize_rows_e4m3(A, Q, scale, M, K, s),
                  quantize_rows_vec_ok(A, Q, K) ? "quantize_e4m3_vec" : "quantize_e4m3_scalar");
}

GEMM_API gemm_status_t gemm_e4m3_rowscale(const uint8_t *Q, const float *scale, const uint8_t *Wt, uint16_t *C,
                                          int M, int N, int K) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) { t_last_kernel = "noop"; return GEMM_OK; }
    if (!C || (K > 0 && (!Q || !scale || !Wt))) return GEMM_ERR_INVALID_VALUE;
    const size_t c_bytes = (size_t)M * N * 2;
    if (overlaps(C, c_bytes, Q, (size_t)M * K) || overlaps(C, c_bytes, Wt, (size_t)N * K) ||
        overlaps(C, c_bytes, scale, (size_t)M * 4))
        return GEMM_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    gemm_status_t st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = t_stream;
    if (K == 0) {
        return finish(zero_fill(C, c_bytes, dev->num_sms, s), "zero_fill");
    }
    if (!umma_e4m3_supported(Q, Wt, C, N, K)) {
        record_message("gemm_e4m3_rowscale: needs Q, Wt, C 16-byte aligned, K % 16 == 0 and N % 8 == 0");
        return GEMM_ERR_INVALID_VALUE;
    }
    const cudaError_t e = launch_umma_e4m3_rowscale(Q, scale, Wt, C, M, N, K, dev->status, s);
    if (e == cudaErrorNotSupported) {
        record_message("gemm_e4m3_rowscale: the tensor-core kernel cannot describe these operands");
        return GEMM_ERR_INVALID_VALUE;
    }
    return finish(e, "umma_e4m3_rowscale");
}

GEMM_API gemm_status_t gemm_e4m3_rowscale_fused(const uint16_t *A, const uint8_t *Wt, uint16_t *C, int M, int N,
                                                int K) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) { t_last_kernel = "noop"; return GEMM_OK; }
    if (!C || (K > 0 && (!A || !Wt))) return GEMM_ERR_INVALID_VALUE;
    const size_t c_bytes = (size_t)M * N * 2;
    if (overlaps(C, c_bytes, A, (size_t)M * K * 2) || overlaps(C, c_bytes, Wt, (size_t)N * K))
        return GEMM_ERR_ALIAS;
    DeviceInfo *dev = nullptr;
    gemm_status_t st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = t_stream;
    if (K == 0) {
        return finish(zero_fill(C, c_bytes, dev->num_sms, s), "zero_fill");
    }
    if (!umma_e4m3_fused_supported(A, Wt, C, N, K)) {
        record_message("gemm_e4m3_rowscale_fused: needs A, Wt, C 16-byte aligned, K % 16 == 0 and N % 8 == 0");
        return GEMM_ERR_INVALID_VALUE;
    }
    const cudaError_t e = launch_umma_e4m3_fused(A, Wt, C, M, N, K, dev->status, s);
    if (e == cudaErrorNotSupported) {
        record_message("gemm_e4m3_rowscale_fused: the tensor-core kernel cannot describe these operands");
        return GEMM_ERR_INVALID_VALUE;
    }
    return finish(e, "umma_e4m3_rowscale_fused");
}

GEMM_API gemm_status_t gemm_set_stream(void *cuda_stream) {
    t_stream = static_cast<cudaStream_t>(cuda_stream);
    return GEMM_OK;
}

GEMM_API void *gemm_get_stream(void) { return t_stream; }

GEMM_API gemm_status_t gemm_synchronize(void) {
    cudaError_t e = cudaStreamSynchronize(t_stream);
    if (e != cudaSuccess) { record_cuda_error(e); return GEMM_ERR_CUDA; }
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { record_cuda_error(e); return GEMM_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    // The status words that exist on this device: the allocating entry points'
    // (once one of them has run here) and the allocation-free entry point's
    // (once it has run here).  Reading them allocates nothing.
    int code = 0;
    DeviceInfo &d = g_devices[dev];
    if (d.ready.load(std::memory_order_acquire)) {
        e = cudaMemcpy(&code, d.status, sizeof(int), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) { record_cuda_error(e); return GEMM_ERR_CUDA; }
        if (code != 0) {
            e = cudaMemset(d.status, 0, sizeof(int));
            if (e != cudaSuccess) { record_cuda_error(e); return GEMM_ERR_CUDA; }
        }
    }
    int code_na = 0;
    e = take_noalloc_status(dev, &code_na);
    if (e != cudaSuccess) { record_cuda_error(e); return GEMM_ERR_CUDA; }
    return (code | code_na) != 0 ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

GEMM_API const char *gemm_status_string(gemm_status_t s) {
    switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE";
    case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    }
    return "GEMM_ERR_UNKNOWN";
}

GEMM_API const char *gemm_last_kernel(void) { return t_last_kernel; }

GEMM_API unsigned long long gemm_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

GEMM_API const char *gemm_last_error(void) { return t_last_error; }

GEMM_API gemm_status_t gemm_force_kernel(const char *family) {
    if (!family || !*family) { t_force = Family::Auto; return GEMM_OK; }
    if (!strcmp(family, "simt")) t_force = Family::Simt;
    else if (!strcmp(family, "simt_scalar")) t_force = Family::SimtScalar;
    else if (!strcmp(family, "gemv")) t_force = Family::Gemv;
    else if (!strcmp(family, "gemv_scalar")) t_force = Family::GemvScalar;
    else if (!strcmp(family, "umma")) t_force = Family::Umma;
    else if (!strcmp(family, "umma_skinny_wide")) t_force = Family::UmmaSkinnyWide;
    else if (!strcmp(family, "umma_stall")) t_force = Family::UmmaStall;
    else if (!strcmp(family, "umma_stall_pair")) t_force = Family::UmmaStallPair;
    else if (!strcmp(family, "umma_stall_peer")) t_force = Family::UmmaStallPeer;
    else return GEMM_ERR_INVALID_VALUE;
    return GEMM_OK;
}

}  // extern "C"
