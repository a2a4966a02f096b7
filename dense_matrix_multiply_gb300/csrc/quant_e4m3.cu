// Row-wise FP8 (E4M3FN) quantisation of a half matrix ("Chapter 5 Operators
// and Runtime", section 5.4.3, example 5-7): the scale of a row comes from the
// whole row's largest magnitude, so a row is read completely before any of its
// elements is quantised.
//     amax_i  = max_k |a_ik|
//     q_ik    = E4M3(a_ik * (448 / amax_i))   nearest, ties to even, clamped to +-448
//     scale_i = amax_i / 448
// 448 / amax_i, the product and amax_i / 448 are single FP32 operations (IEEE
// division: the library is built without fast math), so the codes are the
// ones an FP32 evaluation of these steps gives.  A row of zeros gives q = 0 and
// scale 0.
//
// Bound: HBM (read 2 bytes, write 1 byte per element).  A row (16-byte aligned,
// K % 8 == 0) is read once into registers -- all of its 16-byte loads in flight
// together -- its amax found by warp shuffles and, where several warps hold the
// row, through shared memory, and its codes written from the registers, 8 per
// 8-byte store: one warp per row up to 1024 elements, four warps (1024
// elements each, 54 registers per thread) up to 4096, two warps (4096 each, 143
// registers) up to 8192.  Longer rows take two passes (amax, then a re-read from
// L1/L2 and the codes); rows that are not 16-byte aligned use scalar loads.
// CTAs of four warps.  Measured back to back with A read from DRAM, A [4096,
// 4096]: 9.0 us with four warps per row, 9.3 with two, 10.0 with one (143
// registers: three CTAs per SM), 11.5 with one warp per row in CTAs of eight
// warps (one CTA per SM), 10.4 for the two-pass kernel; [16384, 4096] 29.4 us;
// [8192, 8192] 30.9 us against 52.3 for the two-pass kernel.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"

namespace gemm_gb300 {
namespace {

constexpr int WARPS = 4;

__device__ __forceinline__ uint16_t cvt2(float lo, float hi) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// Rows held in registers: NV 16-byte chunks per lane, WPR warps per row (warp
// part p holds elements [p NV 256, (p + 1) NV 256) of its row; K <= WPR NV 256).
// With two warps per row their amax values meet in shared memory; the largest
// magnitude does not depend on the order it is found in, so the codes are the
// one-warp kernel's.
template <int NV, int WPR>
__global__ void __launch_bounds__(WARPS * 32)
quantize_rows_reg_kernel(const __half *__restrict__ A, uint8_t *__restrict__ Q, float *__restrict__ scale, int M,
                         int K) {
    static_assert(WARPS % WPR == 0, "whole rows per CTA");
    pdl_wait();  // dependents launch as this grid's CTAs exit (several CTAs per SM: no early trigger)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long row = (long long)blockIdx.x * (WARPS / WPR) + warp / WPR;
    const int part = warp % WPR;
    const bool valid = row < M;
    if (WPR == 1 && !valid) return;
    const __half *a = A + (valid ? row : 0) * K;
    uint8_t *q = Q + (valid ? row : 0) * K;
    const int kbase = part * NV * 256;
    uint4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int k = kbase + (i * 32 + lane) * 8;
        v[i] = valid && k < K ? __ldg(reinterpret_cast<const uint4 *>(a + k)) : make_uint4(0u, 0u, 0u, 0u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&v[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(h[j]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if constexpr (WPR > 1) {
        __shared__ float part_amax[WARPS];
        if (lane == 0) part_amax[warp] = amax;
        __syncthreads();
#pragma unroll
        for (int p = 0; p < WPR; ++p) amax = fmaxf(amax, part_amax[warp - part + p]);
        if (!valid) return;
    }
    const float inv = amax == 0.0f ? 0.0f : 448.0f / amax;  // a row of zeros: codes 0
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int k = kbase + (i * 32 + lane) * 8;
        if (k >= K) break;
        const __half2 *h = reinterpret_cast<const __half2 *>(&v[i]);
        uint32_t w[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float2 f0 = __half22float2(h[2 * j]);
            const float2 f1 = __half22float2(h[2 * j + 1]);
            w[j] = (uint32_t)cvt2(f0.x * inv, f0.y * inv) | ((uint32_t)cvt2(f1.x * inv, f1.y * inv) << 16);
        }
        *reinterpret_cast<uint2 *>(q + k) = make_uint2(w[0], w[1]);
    }
    if (lane == 0 && part == 0) scale[row] = amax / 448.0f;
}

template <bool VEC>
__global__ void __launch_bounds__(WARPS * 32)
quantize_rows_kernel(const __half *__restrict__ A, uint8_t *__restrict__ Q, float *__restrict__ scale, int M,
                     int K) {
    pdl_wait();  // dependents launch as this grid's CTAs exit (several CTAs per SM: no early trigger)
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (row >= M) return;
    const __half *a = A + row * K;
    uint8_t *q = Q + row * K;

    float amax = 0.0f;
    if (VEC) {
#pragma unroll 4
        for (int k = lane * 8; k < K; k += 32 * 8) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(a + k));
            const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h[i]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    } else {
        for (int k = lane; k < K; k += 32) amax = fmaxf(amax, fabsf(__half2float(a[k])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

    if (amax == 0.0f) {
        if (VEC) {
            for (int k = lane * 8; k < K; k += 32 * 8) *reinterpret_cast<uint2 *>(q + k) = make_uint2(0u, 0u);
        } else {
            for (int k = lane; k < K; k += 32) q[k] = 0;
        }
        if (lane == 0) scale[row] = 0.0f;
        return;
    }
    const float inv = 448.0f / amax;
    if (VEC) {
#pragma unroll 4
        for (int k = lane * 8; k < K; k += 32 * 8) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(a + k));
            const __half2 *h = reinterpret_cast<const __half2 *>(&u);
            uint32_t w[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float2 f0 = __half22float2(h[2 * i]);
                const float2 f1 = __half22float2(h[2 * i + 1]);
                w[i] = (uint32_t)cvt2(f0.x * inv, f0.y * inv) | ((uint32_t)cvt2(f1.x * inv, f1.y * inv) << 16);
            }
            *reinterpret_cast<uint2 *>(q + k) = make_uint2(w[0], w[1]);
        }
    } else {
        for (int k = lane; k < K; k += 32)
            q[k] = (uint8_t)__nv_cvt_float_to_fp8(__half2float(a[k]) * inv, __NV_SATFINITE, __NV_E4M3);
    }
    if (lane == 0) scale[row] = amax / 448.0f;
}

// amax pass alone (the fused product's first step): one warp per row, the
// same loads and reduction as the first pass above.
template <bool VEC>
__global__ void __launch_bounds__(WARPS * 32)
row_amax_kernel(const __half *__restrict__ A, float *__restrict__ amax_out, int M, int K) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (row >= M) return;
    const __half *a = A + row * K;
    float amax = 0.0f;
    if (VEC) {
#pragma unroll 4
        for (int k = lane * 8; k < K; k += 32 * 8) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(a + k));
            const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h[i]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    } else {
        for (int k = lane; k < K; k += 32) amax = fmaxf(amax, fabsf(__half2float(a[k])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) amax_out[row] = amax;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

bool quantize_rows_vec_ok(const void *A, const void *Q, int K) {
    return aligned(A, 16) && aligned(Q, 8) && (K % 8) == 0;
}

cudaError_t launch_quantize_rows_e4m3(const void *A, void *Q, float *scale, int M, int K, cudaStream_t s) {
    const long long blocks = ((long long)M + WARPS - 1) / WARPS;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)blocks), dim3(WARPS * 32), 0, s, attr);
    if (quantize_rows_vec_ok(A, Q, K)) {
        const __half *a = static_cast<const __half *>(A);
        uint8_t *q = static_cast<uint8_t *>(Q);
        // WPR warps per row: WARPS / WPR rows per CTA
        auto launch_reg = [&](auto kern, int wpr) {
            const long long blocks2 = ((long long)M + WARPS / wpr - 1) / (WARPS / wpr);
            if (blocks2 > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
            cudaLaunchAttribute attr2[1];
            const cudaLaunchConfig_t cfg2 = pdl_config(dim3((unsigned)blocks2), dim3(WARPS * 32), 0, s, attr2);
            return launch_counted(&cfg2, kern, a, q, scale, M, K);
        };
        if (K <= 1024) return launch_reg(quantize_rows_reg_kernel<4, 1>, 1);
        if (K <= 4096) return launch_reg(quantize_rows_reg_kernel<4, 4>, 4);
        if (K <= 8192) return launch_reg(quantize_rows_reg_kernel<16, 2>, 2);
        return launch_counted(&cfg, quantize_rows_kernel<true>, a, q, scale, M, K);
    }
    return launch_counted(&cfg, quantize_rows_kernel<false>, static_cast<const __half *>(A),
                              static_cast<uint8_t *>(Q), scale, M, K);
}

cudaError_t launch_row_amax_f16(const void *A, float *amax, int M, int K, cudaStream_t s) {
    const long long blocks = ((long long)M + WARPS - 1) / WARPS;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)blocks), dim3(WARPS * 32), 0, s, attr);
    if (aligned(A, 16) && (K % 8) == 0)
        return launch_counted(&cfg, row_amax_kernel<true>, static_cast<const __half *>(A), amax, M, K);
    return launch_counted(&cfg, row_amax_kernel<false>, static_cast<const __half *>(A), amax, M, K);
}

}  // namespace gemm_gb300
