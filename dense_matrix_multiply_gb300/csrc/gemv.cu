// Skinny-M GEMM (M <= 8), e.g. the decode case M = 1: c[m,j] = sum_k x[m,k]*W[k,j].
//
// With one or a few rows of A the product is bound by reading B (W) once from
// HBM ("SGEMM measured and the three ledgers", the shape table: decode with
// batch 1 gains only 3.4x from the SGEMM tricks; "Chapter 5 Operators and
// Runtime", section 5.1: decode processes M = 1 token).  So the kernel is a
// streaming reduction, not a tiled contraction, sized by Little's law
// (section 5.1.5: bytes in flight = bandwidth x latency):
//   * a cluster of CS CTAs owns a strip of CW consecutive columns of W; CTA r
//     of the cluster reads rows [r*K/CS, (r+1)*K/CS) of that strip;
//   * a CTA's 256 threads form TC column-lanes x TK k-groups; a column-lane
//     reads VW consecutive elements (16 bytes) of one row per step, so TC lanes
//     read one contiguous row segment; k-group g takes every TK-th row and
//     issues UNROLL independent 16-byte loads at a time;
//   * FP32 accumulators per (m, column).  Partial sums are added in a fixed
//     order: the TK k-groups in shared memory (g = 0, 1, ...), then the CS
//     CTAs of the cluster by rank 0 reading its peers' shared memory
//     (distributed shared memory, r = 0, 1, ...).  The result is deterministic
//     and needs no atomics, no second launch and no global scratch.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace cg = cooperative_groups;

namespace gemm_gb300 {
namespace {

constexpr int THREADS = 256;
constexpr int UNROLL = 8;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// VW elements of W as one 16-byte load (VW = 16 / sizeof(T)) or VW = 1 scalar.
template <typename T, int VW>
struct Vec { T v[VW]; };

template <typename T, int VW>
__device__ __forceinline__ Vec<T, VW> load_w(const T *p) {
    Vec<T, VW> r;
    if constexpr (VW * sizeof(T) == 16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        memcpy(&r, &u, 16);
    } else {
#pragma unroll
        for (int i = 0; i < VW; ++i) r.v[i] = p[i];
    }
    return r;
}

// Dynamic shared memory: red[TK][MM][CW] partials of the k-groups, then
// part[MM][CW], this CTA's sum over its K range.
template <typename T, int VW, int TC, int MM>
__global__ void __launch_bounds__(THREADS)
gemv_kernel(const T *__restrict__ X, const T *__restrict__ W, T *__restrict__ C, int M, int N, int K)
{
    pdl_wait();  // dependents launch as this grid's CTAs exit (several CTAs per SM: no early trigger)
    constexpr int TK = THREADS / TC;
    constexpr int CW = TC * VW;
    extern __shared__ float red[];
    float *part = red + (size_t)TK * MM * CW;

    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int strip = blockIdx.x / cs;

    const int tc = threadIdx.x % TC;
    const int kg = threadIdx.x / TC;
    const int n = strip * CW + tc * VW;
    // Vector loads need the whole vector in range (N % VW == 0 when VW > 1).
    const bool active = n < N;
    const int k_begin = (int)(((long long)K * rank) / cs);
    const int k_end = (int)(((long long)K * (rank + 1)) / cs);

    float acc[MM][VW];
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[m][v] = 0.f;

    if (active) {
        const T *wp = W + n;
        int k = k_begin + kg;
        for (; k + (UNROLL - 1) * TK < k_end; k += UNROLL * TK) {
            Vec<T, VW> w[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) w[u] = load_w<T, VW>(wp + (size_t)(k + u * TK) * N);
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
#pragma unroll
                for (int m = 0; m < MM; ++m) {
                    if (m < M) {
                        const float x = to_f32(X[(size_t)m * K + k + u * TK]);
#pragma unroll
                        for (int v = 0; v < VW; ++v) acc[m][v] = fmaf(x, to_f32(w[u].v[v]), acc[m][v]);
                    }
                }
            }
        }
        for (; k < k_end; k += TK) {
            const Vec<T, VW> w = load_w<T, VW>(wp + (size_t)k * N);
#pragma unroll
            for (int m = 0; m < MM; ++m) {
                if (m < M) {
                    const float x = to_f32(X[(size_t)m * K + k]);
#pragma unroll
                    for (int v = 0; v < VW; ++v) acc[m][v] = fmaf(x, to_f32(w.v[v]), acc[m][v]);
                }
            }
        }
    }

#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
        for (int v = 0; v < VW; ++v) red[((size_t)kg * MM + m) * CW + tc * VW + v] = acc[m][v];
    __syncthreads();

    // Sum of the k-groups, in order, into this CTA's partial.
    for (int o = threadIdx.x; o < MM * CW; o += THREADS) {
        const int m = o / CW, c = o % CW;
        float s = 0.f;
        for (int g = 0; g < TK; ++g) s += red[((size_t)g * MM + m) * CW + c];
        part[o] = s;
    }
    cluster.sync();  // every CTA's partial is complete and visible cluster-wide

    if (rank == 0) {
        for (int o = threadIdx.x; o < MM * CW; o += THREADS) {
            const int m = o / CW, c = o % CW;
            const int gn = strip * CW + c;
            if (m >= M || gn >= N) continue;
            float s = 0.f;
            for (int r = 0; r < cs; ++r) s += cluster.map_shared_rank(part, r)[o];
            C[(size_t)m * N + gn] = from_f32<T>(s);
        }
    }
    cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

template <typename T, int VW, int TC, int MM>
cudaError_t launch_cfg(const Problem &p, int num_sms, cudaStream_t s) {
    constexpr int TK = THREADS / TC;
    constexpr int CW = TC * VW;
    const size_t smem = sizeof(float) * (size_t)(TK + 1) * MM * CW;
    auto kern = gemv_kernel<T, VW, TC, MM>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const long long strips = (p.N + CW - 1) / CW;
    // Split K over a cluster so that about six CTAs per SM keep loads in flight,
    // with at least UNROLL rows per k-group.
    long long cs = (6LL * num_sms + strips - 1) / strips;
    const long long cs_k = p.K / (long long)(UNROLL * TK);
    if (cs > cs_k) cs = cs_k;
    if (cs > 8) cs = 8;
    if (cs < 1) cs = 1;
    if (strips * cs > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(strips * cs), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    pdl_attr(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 2 : 1;
    return launch_counted(&cfg, kern, static_cast<const T *>(p.A), static_cast<const T *>(p.B),
                              static_cast<T *>(p.C), p.M, p.N, p.K);
}

template <typename T, int VW, int TC>
cudaError_t launch_m(const Problem &p, int num_sms, cudaStream_t s) {
    if (p.M == 1) return launch_cfg<T, VW, TC, 1>(p, num_sms, s);
    if (p.M <= 2) return launch_cfg<T, VW, TC, 2>(p, num_sms, s);
    if (p.M <= 4) return launch_cfg<T, VW, TC, 4>(p, num_sms, s);
    return launch_cfg<T, VW, TC, 8>(p, num_sms, s);
}

}  // namespace

cudaError_t launch_gemv(const Problem &p, bool vec, int num_sms, cudaStream_t s) {
    if (p.M < 1 || p.M > kGemvMaxM) return cudaErrorInvalidValue;
    switch (p.elt) {
    case Elt::F32:
        return vec ? launch_m<float, 4, 8>(p, num_sms, s) : launch_m<float, 1, 32>(p, num_sms, s);
    case Elt::F16:
        return vec ? launch_m<__half, 8, 8>(p, num_sms, s) : launch_m<__half, 1, 32>(p, num_sms, s);
    case Elt::BF16:
        return vec ? launch_m<__nv_bfloat16, 8, 8>(p, num_sms, s) : launch_m<__nv_bfloat16, 1, 32>(p, num_sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
