// SIMT GEMM on the CUDA cores: FP32 FFMA only, no tensor cores, no TF32.
//
// Design (prior art: "SGEMM measured and the three ledgers", K5/K6 -- register
// blocking and 128-bit shared loads; the 800 -> 10600 GFLOPS SGEMM blog,
// versions 2-4 -- shared tiles, register micro-tiles, double buffering; chapter
// 5 of the AI-infra book, section 5.2.3 -- bank-conflict-free layouts):
//   * CTA tile 128 x 128, K step 8, 128 threads (4 warps), 16 x 8 outputs per
//     thread held in 128 FP32 registers; two CTAs per SM (~230 registers per
//     thread), so one CTA's barrier wait overlaps the other's FFMA stream.
//   * A is stored k-major in shared memory (transposed on the way in), so one
//     128-bit shared load gives four consecutive rows; B is stored as it lies
//     (n contiguous).  Per k: four LDS.128 of A, two of B, 128 FFMA.
//   * Each warp covers a 64 x 64 sub-tile as 4 x 8 lanes; a lane owns rows
//     {4t..4t+3} + {0, 16, 32, 48} and columns {4u..4u+3} + {0, 32}, so the A
//     and B fragment loads of a warp touch 64 and 128 contiguous bytes: one
//     shared-memory wavefront each, no bank conflict.
//   * Two shared buffers; the next K tile is fetched into registers (LDG.128)
//     while the current one is computed, then stored into the other buffer: one
//     barrier per K tile.  The bounds predicates on these loads also keep them
//     at the top of the iteration, ahead of the FFMA stream that hides them.
//   * Grouped rasterisation: runs of 8 row-tiles sweep the column tiles so that
//     concurrently resident CTAs share A rows and B columns in L2.
//   * Ragged M, N, K: loads are predicated with zero fill, stores are predicated.
// The same template with 16-bit inputs (converted to FP32 when staged) and
// 16-bit outputs (rounded to nearest even once) serves as the tensor path's
// fallback for strides TMA cannot describe.  FP32 problems with float4-able
// operands run on simt_ffma2_kernel instead: the same order of operations on
// 128 x 64 tiles, issued as packed two-lane FMAs (see below).
//
// EX: the general form ("SGEMM measured and the three ledgers", section 2,
// operation flags and leading dimensions; section 3, kernel K1,
// alpha * acc + beta * C): C_b = alpha * op(A_b) op(B_b) + beta * C_b with
// blockIdx.y the batch index.  TA: A stored [K, M]; its tile is then loaded
// along m and stored k-major as it lies.  TB: B stored [N, K]; its tile is
// loaded along k and transposed into the n-contiguous layout on the way in,
// into rows padded by four floats so that the transposing stores of a warp
// fall in 32 distinct banks.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <algorithm>
#include <atomic>

#include "internal.h"

namespace gemm_gb300 {
namespace {

namespace cg = cooperative_groups;

constexpr int BM = 128, BN = 128, THREADS = 128;
constexpr int A_LD = BM + 4;  // padded row of the k-major A tile (floats)
constexpr int B_LD = BN;      // row of the B tile (floats)
constexpr int GROUP_M = 8;

// Whether FP32 problems with float4-able operands use the packed-FMA kernel.
#ifndef SIMT_FFMA2
#define SIMT_FFMA2 1
#endif
constexpr bool g_simt_ffma2 = SIMT_FFMA2 != 0;
// Whether the packed-FMA kernel's part-full last round runs as K halves.
#ifndef SIMT_SPLIT_TAIL
#define SIMT_SPLIT_TAIL 1
#endif
constexpr bool g_simt_split_tail = SIMT_SPLIT_TAIL != 0;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Linear CTA index -> (row tile, column tile), grouped along M.
__device__ __forceinline__ void raster(int pid, int tiles_m, int tiles_n, int &tm, int &tn) {
    const int per_group = GROUP_M * tiles_n;
    const int group = pid / per_group;
    const int first_m = group * GROUP_M;
    const int gsize = min(tiles_m - first_m, GROUP_M);
    const int r = pid - group * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

// Leading dimensions, batch strides (elements) and scalars of the general form.
struct SimtEx {
    long long lda, ldb, ldc;
    long long sa, sb, sc;
    float alpha, beta;
};

// BK: K step of a shared tile (8 or 16).  MINB: CTAs per SM the register
// budget is sized for (__launch_bounds__).  MT: rows of C per CTA, 128 (a whole
// 128 x 128 tile) or 64 (half a tile: CTA 2j+h computes rows 64h..64h+63 of
// tile tile_begin + j, each thread 8 x 8 outputs).  Half tiles spread a
// problem too small to fill the GPU over twice as many CTAs.
template <typename TIn, typename TOut, bool VEC, int BK, int MINB, int MT, bool EX = false, bool TA = false,
          bool TB = false>
__global__ void __launch_bounds__(THREADS, MINB)
simt_gemm_kernel(const TIn *__restrict__ A, const TIn *__restrict__ B, TOut *__restrict__ C,
                 int M, int N, int K, int tile_begin, SimtEx ex)
{
    static_assert(MT == 128 || MT == 64, "CTA covers a whole or half tile");
    pdl_wait();  // no early trigger of dependents: see launch_ffma2
    static_assert(EX || (!TA && !TB), "transposed operands need the general form");
    constexpr int RG = MT / 32;  // groups of four rows per thread
    constexpr int BLD = TB ? B_LD + 4 : B_LD;
    __shared__ __align__(16) float As[2][BK][A_LD];
    __shared__ __align__(16) float Bs[2][BK][BLD];

    const long long lda = EX ? ex.lda : K, ldb = EX ? ex.ldb : N, ldc = EX ? ex.ldc : N;
    if (EX) {
        A += (long long)blockIdx.y * ex.sa;
        B += (long long)blockIdx.y * ex.sb;
        C += (long long)blockIdx.y * ex.sc;
    }

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 1, wn = warp & 1;     // 2 x 2 warps
    const int lm = lane >> 3, ln = lane & 7;     // 4 x 8 lanes

    int tm, tn;
    const int pid = tile_begin + (MT == BM ? (int)blockIdx.x : (int)(blockIdx.x >> 1));
    raster(pid, (M + BM - 1) / BM, (N + BN - 1) / BN, tm, tn);
    const int m0 = tm * BM + (MT == BM ? 0 : (int)(blockIdx.x & 1) * MT), n0 = tn * BN;

    // Global -> register staging: LA quads of A and LB quads of B per thread.
    // A [M,K]: MT rows x QA quads of k.  A stored [K,M] (TA): BK k-rows x MT/4
    // quads of m.  B [K,N]: BK k-rows x 32 quads of n.  B stored [N,K] (TB): BN
    // rows x QA quads of k.
    constexpr int QA = BK / 4;
    constexpr int LA = MT * QA / THREADS, LB = BK * (BN / 4) / THREADS;
    static_assert(LA >= 1 && LB >= 1 && MT * QA % THREADS == 0, "tile/thread mapping");
    static_assert(BK * (MT / 4) == LA * THREADS && BN * QA == LB * THREADS, "transposed mappings");
    float ra[LA][4], rb[LB][4];
    auto load_tile = [&](int k0) {
#pragma unroll
        for (int i = 0; i < LA; ++i) {
            const int idx = tid + i * THREADS;
            // (gm, gk) of the quad's first element; the quad runs along k, or
            // along m when A is stored [K,M].
            const int gm = TA ? m0 + (idx % (MT / 4)) * 4 : m0 + idx / QA;
            const int gk = TA ? k0 + idx / (MT / 4) : k0 + (idx % QA) * 4;
            const size_t off = TA ? (size_t)gk * lda + gm : (size_t)gm * lda + gk;
            if (VEC) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (gm < M && gk < K) v = __ldg(reinterpret_cast<const float4 *>(A + off));
                ra[i][0] = v.x; ra[i][1] = v.y; ra[i][2] = v.z; ra[i][3] = v.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = TA ? (gm + j < M && gk < K) : (gm < M && gk + j < K);
                    ra[i][j] = in ? to_f32(A[off + j]) : 0.f;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < LB; ++i) {
            const int idx = tid + i * THREADS;
            // (gk, gn) of the quad's first element; the quad runs along n, or
            // along k when B is stored [N,K].
            const int gk = TB ? k0 + (idx % QA) * 4 : k0 + (idx >> 5);
            const int gn = TB ? n0 + idx / QA : n0 + (idx & 31) * 4;
            const size_t off = TB ? (size_t)gn * ldb + gk : (size_t)gk * ldb + gn;
            if (VEC) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (gk < K && gn < N) v = __ldg(reinterpret_cast<const float4 *>(B + off));
                rb[i][0] = v.x; rb[i][1] = v.y; rb[i][2] = v.z; rb[i][3] = v.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = TB ? (gk + j < K && gn < N) : (gk < K && gn + j < N);
                    rb[i][j] = in ? to_f32(B[off + j]) : 0.f;
                }
            }
        }
    };
    auto store_tile = [&](int buf) {
#pragma unroll
        for (int i = 0; i < LA; ++i) {
            const int idx = tid + i * THREADS;
            if (TA) {
                const int kr = idx / (MT / 4), mq = (idx % (MT / 4)) * 4;
                *reinterpret_cast<float4 *>(&As[buf][kr][mq]) = make_float4(ra[i][0], ra[i][1], ra[i][2], ra[i][3]);
            } else {
                const int row = idx / QA, kq = (idx % QA) * 4;
#pragma unroll
                for (int j = 0; j < 4; ++j) As[buf][kq + j][row] = ra[i][j];
            }
        }
#pragma unroll
        for (int i = 0; i < LB; ++i) {
            const int idx = tid + i * THREADS;
            if (TB) {
                const int col = idx / QA, kq = (idx % QA) * 4;
#pragma unroll
                for (int j = 0; j < 4; ++j) Bs[buf][kq + j][col] = rb[i][j];
            } else {
                const int kr = idx >> 5, nq = (idx & 31) * 4;
                *reinterpret_cast<float4 *>(&Bs[buf][kr][nq]) = make_float4(rb[i][0], rb[i][1], rb[i][2], rb[i][3]);
            }
        }
    };

    float acc[4 * RG][8];
#pragma unroll
    for (int i = 0; i < 4 * RG; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int a_off = wm * (MT / 2) + lm * 4;  // + 16 * {0 .. RG-1}
    const int b_off = wn * 64 + ln * 4;  // + {0, 32}
    const int ktiles = (K + BK - 1) / BK;

    load_tile(0);
    store_tile(0);
    __syncthreads();

    for (int t = 0; t < ktiles; ++t) {
        const int buf = t & 1;
        if (t + 1 < ktiles) load_tile((t + 1) * BK);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4 * RG], b[8];
#pragma unroll
            for (int q = 0; q < RG; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(&As[buf][kk][a_off + 16 * q]);
                a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(&Bs[buf][kk][b_off + 32 * q]);
                b[4 * q] = v.x; b[4 * q + 1] = v.y; b[4 * q + 2] = v.z; b[4 * q + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < 4 * RG; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (t + 1 < ktiles) store_tile(buf ^ 1);
        __syncthreads();
    }

    // Epilogue: each thread writes its 4*RG rows x (2 x 4) columns; the general
    // form scales by alpha and, when beta != 0, adds beta times the old C.
    const bool use_beta = EX && ex.beta != 0.0f;
#pragma unroll
    for (int i = 0; i < 4 * RG; ++i) {
        const int gm = m0 + a_off + 16 * (i >> 2) + (i & 3);
        if (gm >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gn = n0 + b_off + h * 32;
            TOut *dst = C + (size_t)gm * ldc + gn;
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = EX ? ex.alpha * acc[i][4 * h + j] : acc[i][4 * h + j];
            if (VEC && gn + 3 < N) {
                if (use_beta) {
                    const float4 o = *reinterpret_cast<const float4 *>(dst);
                    v[0] = fmaf(ex.beta, o.x, v[0]);
                    v[1] = fmaf(ex.beta, o.y, v[1]);
                    v[2] = fmaf(ex.beta, o.z, v[2]);
                    v[3] = fmaf(ex.beta, o.w, v[3]);
                }
                *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (gn + j < N) {
                        const float w = use_beta ? fmaf(ex.beta, to_f32(dst[j]), v[j]) : v[j];
                        dst[j] = from_f32<TOut>(w);
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------ packed-FMA FP32 kernel
// The FP32 kernel for float4-able operands.  The FFMA stream is issued as
// packed two-lane FMAs (fma.rn.f32x2 through __ffma2_rn): one instruction
// updates two accumulators, so the FMA pipe rather than instruction issue
// bounds the loop, and loads, stores and address work fit in the issue slots
// the pipe leaves free.
//   * CTA tile 128 x 64, 128 threads (2 x 2 warps of 64 x 32), 8 x 8 outputs
//     per thread held as 32 pairs of horizontally adjacent outputs (columns
//     c, c+1 of one row): B's fragment supplies (b_c, b_c+1) as it lies, A's
//     value is paired with itself, (a_r, a_r).  A lane (lm, ln) of the 8 x 4
//     lane grid owns rows {4lm..4lm+3} + {0, 32} and columns {4ln..4ln+3} +
//     {0, 16} of its warp's sub-tile: per k two LDS.128 of A (the 8 row groups
//     of a warp read 128 contiguous bytes), two of B, 32 packed FMAs.
//   * K step 16; B quads go to shared memory with 16-byte cp.async, A quads
//     pass through registers to be transposed into the k-major tile, whose
//     16-byte chunks are XOR-swizzled by k so that the transposing stores of
//     a warp hit 32 distinct banks (a padded tile left them 2-way conflicted:
//     61.1 against 62.5 TFLOP/s at 4096^3).
//   * A ring of three stages, one barrier per K step.  B is requested two steps
//     ahead; A is loaded into registers one step before its store, so each load
//     has a whole compute step to arrive.  148 registers: three CTAs per SM.
//   * Grouped rasterisation along M, predicated loads (zero fill) and stores.
// Every product and sum is the scalar kernel's, in the same order, so the
// results are bit-identical to it, except in a split last round (below).
//   * Split last round: the tiles past the last full round of resident CTAs
//     (a part-full round) run as a second grid of
//     two-CTA clusters, one CTA per half of the K blocks, launched as a
//     programmatic dependent that the first grid releases once all its CTAs
//     are resident; such a tile is the sum of its two halves' FP32 sums.
// Measured on GB300 (CUDA events):
// 62.5 TFLOP/s at 4096^3 against 54.4 for the scalar-FFMA 128 x 128 kernel,
// 38.9 against 24.3 at 1000^3; 128 x 128 tiles with 16 x 8 packed outputs per
// thread reached 57.6 (242 registers, two CTAs per SM); K steps 8 and 32, four
// stages and four CTAs per SM were slower.
constexpr int G_BM = 128, G_BN = 64, G_BK = 16, G_STAGES = 3;
constexpr int G_ALD = G_BM;
// 16-byte chunk c of k-row k of the A tile lives at chunk c ^ a_swz(k): the
// four k-rows one transposing store instruction writes land in different
// banks, and the eight chunks of a fragment load stay within one 128-byte row
// segment.
__device__ __forceinline__ int a_swz(int k) { return 2 * ((k >> 2) & 3); }
__device__ __forceinline__ int a_col(int k, int row) { return ((((row >> 2) ^ a_swz(k))) << 2) | (row & 3); }
// The B tile uses the same swizzle when it is transposed through registers
// (B stored [N, K]); filled by cp.async it lies unswizzled.
template <bool TB>
__device__ __forceinline__ int b_col(int k, int col) { return TB ? a_col(k, col) : col; }
struct F2Shared {
    float As[G_STAGES][G_BK][G_ALD];
    float Bs[G_STAGES][G_BK][G_BN];
};

// EX: the general form (blockIdx.y the batch index, leading dimensions,
// alpha and beta), TA: A stored [K, M] -- its tile is already k-major and goes
// to shared memory by cp.async; TB: B stored [N, K] -- its tile passes through
// registers to be transposed into the swizzled layout.
// MODE 0: every tile of the problem.  MODE 3: every tile as a cluster of two
// half-K CTAs (a problem too small for one round of resident CTAs).  A plain
// problem whose last round of resident CTAs would be part full runs as two
// grids: MODE 1 the whole tiles before tile_base, MODE 2 the rest on clusters
// of two CTAs, the first taking
// the first half of the K blocks and the second the rest; the halves' FP32
// sums are exchanged through distributed shared memory and added.
template <bool EX, bool TA, bool TB, int MODE = 0>
__global__ void __launch_bounds__(THREADS, 2)
simt_ffma2_kernel(const float *__restrict__ A, const float *__restrict__ B, float *__restrict__ C, int M,
                  int N, int K, SimtEx ex, int tile_base)
{
    static_assert(EX || (!TA && !TB), "transposed operands need the general form");
    static_assert(MODE == 0 || (!EX && !TA && !TB), "split launches are plain problems");
    // MODE 0 and 1 wait for the previous kernel on the stream; MODE 1 then lets
    // its dependent (the MODE 2 tail) launch, so the tail's CTAs take the slots
    // this grid frees.  The tail reads only A and B (complete once every MODE 1
    // CTA has passed its wait) and waits for MODE 1 before it exits, so that
    // the next kernel on the stream sees both grids' tiles of C.
    if constexpr (MODE != 2) pdl_wait();  // MODE 3, a grid of its own, waits too
    if constexpr (MODE == 1) pdl_launch_dependents();
    extern __shared__ __align__(16) uint8_t f2_smem[];
    F2Shared &sm = *reinterpret_cast<F2Shared *>(f2_smem);
    constexpr int QA = G_BK / 4;                     // quads of k per A row ([M,K] storage)
    constexpr int LA = G_BM * QA / THREADS;          // 4 A quads per thread and step
    constexpr int QB = G_BN / 4;                     // quads of n per B row ([K,N] storage)
    constexpr int LB = G_BK * QB / THREADS;          // 2 B quads per thread and step
    static_assert(LA == 4 && LB == 2, "tile/thread mapping");
    const long long lda = EX ? ex.lda : K, ldb = EX ? ex.ldb : N, ldc = EX ? ex.ldc : N;
    if (EX) {
        A += (long long)blockIdx.y * ex.sa;
        B += (long long)blockIdx.y * ex.sb;
        C += (long long)blockIdx.y * ex.sc;
    }
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 1, wn = warp & 1;
    const int lm = lane >> 2, ln = lane & 3;
    // Linear CTA index -> tile, grouped along M.
    const int tiles_m = (M + G_BM - 1) / G_BM, tiles_n = (N + G_BN - 1) / G_BN;
    int tm, tn;
    {
        const int pid = MODE >= 2 ? tile_base + (int)(blockIdx.x >> 1) : (int)blockIdx.x;
        const int per_group = GROUP_M * tiles_n;
        const int group = pid / per_group;
        const int first_m = group * GROUP_M;
        const int gsize = min(tiles_m - first_m, GROUP_M);
        const int r = pid - group * per_group;
        tm = first_m + r % gsize;
        tn = r / gsize;
    }
    const int m0 = tm * G_BM, n0 = tn * G_BN;
    const int ktiles = (K + G_BK - 1) / G_BK;
    // K blocks [kt0, kt0 + kcount) of the tile: all of them, or one half (MODE 2)
    const int khalf = MODE >= 2 ? (int)(blockIdx.x & 1) : 0;
    const int kt0 = khalf ? ktiles / 2 : 0;
    const int kcount = MODE >= 2 ? (khalf ? ktiles - ktiles / 2 : ktiles / 2) : ktiles;

    auto cp16 = [&](float *dst, const float *src, bool in) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                     "l"(in ? src : A), "r"(in ? 16 : 0)
                     : "memory");
    };
    // A stored [M,K]: 128 rows x 4 quads of k per step through registers.
    float4 ra[TA ? 1 : LA];
    auto load_a = [&](int t) {
        if constexpr (!TA) {
#pragma unroll
            for (int i = 0; i < LA; ++i) {
                const int idx = tid + i * THREADS;
                const int row = idx / QA, kq = (idx % QA) * 4;
                const int gm = m0 + row, gk = (kt0 + t) * G_BK + kq;
                ra[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (gm < M && gk < K) ra[i] = __ldg(reinterpret_cast<const float4 *>(A + (size_t)gm * lda + gk));
            }
        }
    };
    auto store_a = [&](int stage) {
        if constexpr (!TA) {
#pragma unroll
            for (int i = 0; i < LA; ++i) {
                const int idx = tid + i * THREADS;
                const int row = idx / QA, kq = (idx % QA) * 4;
                sm.As[stage][kq + 0][a_col(kq + 0, row)] = ra[i].x;
                sm.As[stage][kq + 1][a_col(kq + 1, row)] = ra[i].y;
                sm.As[stage][kq + 2][a_col(kq + 2, row)] = ra[i].z;
                sm.As[stage][kq + 3][a_col(kq + 3, row)] = ra[i].w;
            }
        }
    };
    // A stored [K,M]: 16 k-rows x 32 quads of m per step by cp.async.
    auto copy_a = [&](int t, int stage) {
        if constexpr (TA) {
#pragma unroll
            for (int i = 0; i < LA; ++i) {
                const int idx = tid + i * THREADS;
                const int kr = idx >> 5, mq = (idx & 31) * 4;
                const int gk = (kt0 + t) * G_BK + kr, gm = m0 + mq;
                cp16(&sm.As[stage][kr][a_col(kr, mq)], A + (size_t)gk * lda + gm, gk < K && gm < M);
            }
        }
    };
    // B stored [K,N]: 16 k-rows x 16 quads of n per step by cp.async.
    auto copy_b = [&](int t, int stage) {
        if constexpr (!TB) {
#pragma unroll
            for (int i = 0; i < LB; ++i) {
                const int idx = tid + i * THREADS;
                const int kr = idx / QB, nq = (idx % QB) * 4;
                const int gk = (kt0 + t) * G_BK + kr, gn = n0 + nq;
                cp16(&sm.Bs[stage][kr][nq], B + (size_t)gk * ldb + gn, gk < K && gn < N);
            }
        }
    };
    // B stored [N,K]: 64 columns x 4 quads of k per step through registers.
    float4 rb[TB ? LB : 1];
    auto load_b = [&](int t) {
        if constexpr (TB) {
#pragma unroll
            for (int i = 0; i < LB; ++i) {
                const int idx = tid + i * THREADS;
                const int col = idx / QA, kq = (idx % QA) * 4;
                const int gn = n0 + col, gk = (kt0 + t) * G_BK + kq;
                rb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (gn < N && gk < K) rb[i] = __ldg(reinterpret_cast<const float4 *>(B + (size_t)gn * ldb + gk));
            }
        }
    };
    auto store_b = [&](int stage) {
        if constexpr (TB) {
#pragma unroll
            for (int i = 0; i < LB; ++i) {
                const int idx = tid + i * THREADS;
                const int col = idx / QA, kq = (idx % QA) * 4;
                sm.Bs[stage][kq + 0][b_col<TB>(kq + 0, col)] = rb[i].x;
                sm.Bs[stage][kq + 1][b_col<TB>(kq + 1, col)] = rb[i].y;
                sm.Bs[stage][kq + 2][b_col<TB>(kq + 2, col)] = rb[i].z;
                sm.Bs[stage][kq + 3][b_col<TB>(kq + 3, col)] = rb[i].w;
            }
        }
    };

#pragma unroll
    for (int t = 0; t < G_STAGES - 1; ++t) {
        if (t < kcount) {
            copy_a(t, t);
            copy_b(t, t);
            load_a(t);
            store_a(t);
            load_b(t);
            store_b(t);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (G_STAGES - 1 < kcount) {
        load_a(G_STAGES - 1);
        load_b(G_STAGES - 1);
    }

    float2 acc[8][4];  // [row][column pair]
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);

    const int a_off = wm * 64 + lm * 4;  // rows a_off + {0..3} + {0, 32}
    const int b_off = wn * 32 + ln * 4;  // columns b_off + {0..3} + {0, 16}

    for (int t = 0; t < kcount; ++t) {
        const int stage = t % G_STAGES;
        asm volatile("cp.async.wait_group %0;" ::"n"(G_STAGES - 2) : "memory");
        __syncthreads();
        const int tr = t + G_STAGES - 1;
        if (tr < kcount) {
            const int st = tr % G_STAGES;
            copy_a(tr, st);
            copy_b(tr, st);
            store_a(st);
            store_b(st);
            if (tr + 1 < kcount) {
                load_a(tr + 1);
                load_b(tr + 1);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
        for (int kk = 0; kk < G_BK; ++kk) {
            float a[8];
            float2 b[4];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(&sm.As[stage][kk][a_col(kk, a_off + 32 * q)]);
                a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 v = *reinterpret_cast<const float4 *>(&sm.Bs[stage][kk][b_col<TB>(kk, b_off + 16 * h)]);
                b[2 * h] = make_float2(v.x, v.y);
                b[2 * h + 1] = make_float2(v.z, v.w);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(make_float2(a[i], a[i]), b[j], acc[i][j]);
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");

    // row i: a_off + 32 (i >> 2) + (i & 3); column pair j: b_off + 16 (j >> 1) + 2 (j & 1).
    if constexpr (MODE >= 2) {
        // Rows a_off + 32 q + {0..3} are stored by the CTA of rank q.  Each CTA
        // puts the rows its partner stores into its own shared memory (row
        // wm 32 + lm 4 + i of a 64-row buffer, stride 68 floats so that the
        // lanes of a store phase hit distinct banks), then adds the partner's
        // copy of its own rows.
        constexpr int PLD = G_BN + 4;
        static_assert(G_BM / 2 * PLD * 4 <= (int)sizeof(F2Shared), "partial tile fits the stage buffers");
        cg::cluster_group cluster = cg::this_cluster();
        const int q = khalf;  // cluster rank = blockIdx.x & 1
        float *part = reinterpret_cast<float *>(f2_smem);
        __syncthreads();  // every warp is done with the stage buffers
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // the partner's rows: group 1 - q (selected, not indexed, to keep acc in registers)
                const float2 lo = q ? acc[i][2 * h] : acc[4 + i][2 * h];
                const float2 hi = q ? acc[i][2 * h + 1] : acc[4 + i][2 * h + 1];
                *reinterpret_cast<float4 *>(part + (wm * 32 + (a_off & 31) + i) * PLD + b_off + 16 * h) =
                    make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        cluster.sync();
        const float *peer = cluster.map_shared_rank(part, q ^ 1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gm = m0 + a_off + 32 * q + i;
            if (gm >= M) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = b_off + 16 * h, gn = n0 + c;
                const float4 o = *reinterpret_cast<const float4 *>(peer + (wm * 32 + (a_off & 31) + i) * PLD + c);
                const float2 lo = q ? acc[4 + i][2 * h] : acc[i][2 * h];
                const float2 hi = q ? acc[4 + i][2 * h + 1] : acc[i][2 * h + 1];
                // q = 0 holds the first K half, q = 1 the second: the sum is the
                // same either way round (IEEE addition commutes).
                const float v[4] = {lo.x + o.x, lo.y + o.y, hi.x + o.z, hi.y + o.w};
                float *dst = C + (size_t)gm * ldc + gn;
                if (gn + 3 < N) {
                    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (gn + j < N) dst[j] = v[j];
                }
            }
        }
        cluster.sync();  // the partner's reads of this CTA's shared memory are done
        if constexpr (MODE == 2) pdl_wait();  // MODE 1 complete before this grid counts as complete
        return;
    }
    // The general form scales by alpha and, when beta != 0, adds beta * old C.
    const bool use_beta = EX && ex.beta != 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gm = m0 + a_off + 32 * (i >> 2) + (i & 3);
        if (gm >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gn = n0 + b_off + 16 * h;
            float *dst = C + (size_t)gm * ldc + gn;
            const float2 lo = acc[i][2 * h], hi = acc[i][2 * h + 1];
            float v[4] = {lo.x, lo.y, hi.x, hi.y};
            if (EX) {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] *= ex.alpha;
            }
            if (gn + 3 < N) {
                if (use_beta) {
                    const float4 o = *reinterpret_cast<const float4 *>(dst);
                    v[0] = fmaf(ex.beta, o.x, v[0]);
                    v[1] = fmaf(ex.beta, o.y, v[1]);
                    v[2] = fmaf(ex.beta, o.z, v[2]);
                    v[3] = fmaf(ex.beta, o.w, v[3]);
                }
                *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < N) dst[j] = use_beta ? fmaf(ex.beta, dst[j], v[j]) : v[j];
            }
        }
    }
}

// Launch of the packed-FMA kernel over `batches` batch entries (grid.y).
template <bool EX, bool TA, bool TB>
cudaError_t launch_ffma2(const float *A, const float *B, float *C, int M, int N, int K, const SimtEx &ex,
                         unsigned batches, cudaStream_t s) {
    const long long tiles = (long long)((M + G_BM - 1) / G_BM) * ((N + G_BN - 1) / G_BN);
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    constexpr int smem = (int)sizeof(F2Shared);
    static_assert(smem <= 48 * 1024, "launched without the large-shared-memory attribute");
    // Launched as a programmatic dependent (its prologue overlaps the previous
    // kernel's drain), but it does not trigger its own dependents early: with
    // three CTAs per SM, a small grid's successor would be placed while this
    // grid still runs and pack onto its SMs -- 1000^3 measured 86 us against
    // 49 us with the trigger left to the CTAs' exit (51 us without PDL).
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)tiles, batches, 1), dim3(THREADS), smem, s, attr);
    return launch_counted(&cfg, simt_ffma2_kernel<EX, TA, TB>, A, B, C, M, N, K, ex, 0);
}

// Tiles of a plain problem to run as K halves: the part-full last round of
// `slots` resident CTAs, when the problem fills at least one round and each
// half has at least 16 K blocks.  0: one launch.  A last round more than half
// full gains too, its half-K CTAs taking slots as the whole rounds drain
// (measured back to back: 2560 x 2560 x 4096, 344 of 456 slots, 874.5 against
// 957.3 us as one grid; 3072^3, 240 of 456, 944.4 against 950.3; 3328 x 3328 x
// 2048, 440 of 456, 715.7 against 716.6).
long long ffma2_tail_tiles(long long tiles, int K, long long slots) {
    if (!g_simt_split_tail || !g_pdl) return 0;
    const long long rem = tiles % slots;
    const int ktiles = (K + G_BK - 1) / G_BK;
    if (tiles < slots || rem == 0 || ktiles < 32) return 0;
    return rem;
}

// A plain problem as two grids: the whole tiles (which let the second grid
// launch as soon as they are all resident), then the last `tail` tiles as
// clusters of two half-K CTAs, which take the slots the first grid frees.
cudaError_t launch_ffma2_split(const float *A, const float *B, float *C, int M, int N, int K, long long tiles,
                               long long tail, cudaStream_t s) {
    constexpr int smem = (int)sizeof(F2Shared);
    const long long base = tiles - tail;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)base), dim3(THREADS), smem, s, attr);
    cudaError_t e = launch_counted(&cfg, simt_ffma2_kernel<false, false, false, 1>, A, B, C, M, N, K,
                                       SimtEx{}, (int)base);
    if (e != cudaSuccess) return e;
    cfg = pdl_config(dim3((unsigned)(2 * tail)), dim3(THREADS), smem, s, attr);
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = 2;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    cfg.numAttrs += 1;
    return launch_counted(&cfg, simt_ffma2_kernel<false, false, false, 2>, A, B, C, M, N, K, SimtEx{},
                              (int)base);
}

// ------------------------------------------------------------ small problems
// A plain FP32 problem whose 128 x 64 tiles would occupy at most a quarter of
// the SMs (SGEMM 256^3 is 8 such tiles on 152 SMs) runs on 32 x 32 tiles
// instead: sixteen times the CTAs, 64 threads each, 4 x 4 outputs per thread,
// K step 16.  Measured on GB300 (back to back over 64 copies of the operands,
// which at 256^3 -- 49 MB -- stay in L2), small kernel against the 128 x 64
// one: 256^3 9.3 vs 13.6 us, 512^3 22.7 vs 26.6, 300 x 520 x 272 12.8 vs 15.3,
// 64^3 3.2 vs 4.7; with more tiles the large kernel wins (1000^3: 128 tiles,
// 50.5 vs 83.9 us).  With every call's operands from DRAM, 256^3 takes 12.1-12.7
// us: one K step of lookahead leaves most of a DRAM round trip exposed per step.  The k-major A
// tile and the B tile are double-buffered in shared memory, the next K step
// loaded into registers (16-byte loads) while the current one is multiplied;
// one barrier per step.  Per k a thread makes one 16-byte shared load of A
// (its four rows) and one of B (its four columns) and 16 FFMAs, every output
// summed over k in ascending order with one rounding per step, as in the
// other SIMT kernels.
#ifndef SIMT_SMALL
#define SIMT_SMALL 1
#endif
#ifndef SIMT_SPLIT_ALL
#define SIMT_SPLIT_ALL 1
#endif
constexpr int S_BM = 32, S_BN = 32, S_BK = 16, S_THREADS = 64;

__global__ void __launch_bounds__(S_THREADS, 16)
simt_small_kernel(const float *__restrict__ A, const float *__restrict__ B, float *__restrict__ C, int M, int N,
                  int K)
{
    pdl_wait();  // several CTAs per SM: dependents launch as the CTAs exit
    __shared__ __align__(16) float As[2][S_BK][S_BM];
    __shared__ __align__(16) float Bs[2][S_BK][S_BN];
    const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
    const int tiles_n = (N + S_BN - 1) / S_BN;
    const int m0 = (int)(blockIdx.x / tiles_n) * S_BM, n0 = (int)(blockIdx.x % tiles_n) * S_BN;
    float4 ra[2], rb[2];
    auto load = [&](int k0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = tid + i * S_THREADS;
            const int row = idx >> 2, kq = (idx & 3) * 4;  // A: 32 rows x 4 quads of k
            const int gm = m0 + row, gk = k0 + kq;
            ra[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (gm < M && gk < K) ra[i] = __ldg(reinterpret_cast<const float4 *>(A + (size_t)gm * K + gk));
            const int kr = idx >> 3, nq = (idx & 7) * 4;   // B: 16 k-rows x 8 quads of n
            const int gk2 = k0 + kr, gn = n0 + nq;
            rb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (gk2 < K && gn < N) rb[i] = __ldg(reinterpret_cast<const float4 *>(B + (size_t)gk2 * N + gn));
        }
    };
    auto store = [&](int b) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = tid + i * S_THREADS;
            const int row = idx >> 2, kq = (idx & 3) * 4;
            As[b][kq + 0][row] = ra[i].x;
            As[b][kq + 1][row] = ra[i].y;
            As[b][kq + 2][row] = ra[i].z;
            As[b][kq + 3][row] = ra[i].w;
            *reinterpret_cast<float4 *>(&Bs[b][idx >> 3][(idx & 7) * 4]) = rb[i];
        }
    };
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int ktiles = (K + S_BK - 1) / S_BK;
    load(0);
    store(0);
    __syncthreads();
    for (int t = 0; t < ktiles; ++t) {
        const int b = t & 1;
        if (t + 1 < ktiles) load((t + 1) * S_BK);
#pragma unroll
        for (int kk = 0; kk < S_BK; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 4]);
            const float4 bb = *reinterpret_cast<const float4 *>(&Bs[b][kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (t + 1 < ktiles) store(b ^ 1);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gm = m0 + ty * 4 + i, gn = n0 + tx * 4;
        if (gm >= M) continue;
        float *dst = C + (size_t)gm * N + gn;
        if (gn + 3 < N) {
            *reinterpret_cast<float4 *>(dst) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (gn + j < N) dst[j] = acc[i][j];
        }
    }
}

// Tile configuration of the SIMT kernel: K step and CTAs per SM.
#ifndef SIMT_BK
#define SIMT_BK 8
#endif
#ifndef SIMT_MINB
#define SIMT_MINB 2
#endif

template <typename TIn, typename TOut, bool VEC>
cudaError_t launch_typed(const Problem &p, int num_sms, cudaStream_t s) {
    const long long tiles = (long long)((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (2 * tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const TIn *A = static_cast<const TIn *>(p.A);
    const TIn *B = static_cast<const TIn *>(p.B);
    TOut *C = static_cast<TOut *>(p.C);
    if constexpr (VEC && sizeof(TIn) == 4) {
        if (g_simt_ffma2) {
            const float *fA = static_cast<const float *>(p.A), *fB = static_cast<const float *>(p.B);
            float *fC = static_cast<float *>(p.C);
            // three packed-FMA CTAs are resident per SM
            const long long ftiles = (long long)((p.M + G_BM - 1) / G_BM) * ((p.N + G_BN - 1) / G_BN);
            if (SIMT_SMALL && 4 * ftiles <= num_sms) {
                const long long stiles = (long long)((p.M + S_BM - 1) / S_BM) * ((p.N + S_BN - 1) / S_BN);
                cudaLaunchAttribute attr[1];
                const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)stiles), dim3(S_THREADS), 0, s, attr);
                return launch_counted(&cfg, simt_small_kernel, fA, fB, fC, p.M, p.N, p.K);
            }
            // fewer tiles than one round of resident CTAs, at most half a round:
            // every tile as two half-K CTAs (1000^3: 128 tiles, 256 CTAs; on
            // GB300 48.4 against 50.3 us, 1024 x 1024 x 4096 174.5 against 191.2)
            if (SIMT_SPLIT_ALL && g_simt_split_tail && g_pdl && 2 * ftiles <= 3LL * num_sms &&
                (p.K + G_BK - 1) / G_BK >= 32) {
                cudaLaunchAttribute attr[2];
                cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)(2 * ftiles)), dim3(THREADS),
                                                    (int)sizeof(F2Shared), s, attr);
                attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
                attr[cfg.numAttrs].val.clusterDim.x = 2;
                attr[cfg.numAttrs].val.clusterDim.y = 1;
                attr[cfg.numAttrs].val.clusterDim.z = 1;
                cfg.numAttrs += 1;
                return launch_counted(&cfg, simt_ffma2_kernel<false, false, false, 3>, fA, fB, fC, p.M, p.N, p.K,
                                      SimtEx{}, 0);
            }
            const long long tail = ffma2_tail_tiles(ftiles, p.K, 3LL * num_sms);
            if (tail > 0) return launch_ffma2_split(fA, fB, fC, p.M, p.N, p.K, ftiles, tail, s);
            return launch_ffma2<false, false, false>(fA, fB, fC, p.M, p.N, p.K, SimtEx{}, 1, s);
        }
    }
    // A problem too small to fill half of one round of resident CTAs runs as
    // half tiles: twice the CTAs, half the rows each.  (Splitting only the last
    // round of a large problem into half-height tiles in a second launch
    // measured slower for this kernel: a lone CTA already runs near the SM's
    // full rate, and the second launch waited for the first to drain.  The
    // packed-FMA kernel's split above differs on both counts: half-K CTA pairs,
    // launched while the first grid still runs.)
    const long long slots = (long long)num_sms * SIMT_MINB;
    const long long split = 2 * tiles <= slots ? tiles : 0;
    const long long whole = tiles - split;
    if (whole > 0) {
        cudaLaunchAttribute attr[1];
        const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)whole), dim3(THREADS), 0, s, attr);
        const cudaError_t e = launch_counted(&cfg, simt_gemm_kernel<TIn, TOut, VEC, SIMT_BK, SIMT_MINB, 128>, A,
                                                 B, C, p.M, p.N, p.K, 0, SimtEx{});
        if (e != cudaSuccess) return e;
    }
    if (split > 0) {
        cudaLaunchAttribute attr[1];
        const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)(2 * split)), dim3(THREADS), 0, s, attr);
        const cudaError_t e = launch_counted(&cfg, simt_gemm_kernel<TIn, TOut, VEC, SIMT_BK, SIMT_MINB, 64>, A,
                                                 B, C, p.M, p.N, p.K, (int)whole, SimtEx{});
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The general form: one launch per chunk of at most 65535 batch entries
// (blockIdx.y), whole 128 x 128 tiles.
template <typename TIn, bool VEC, bool TA, bool TB>
cudaError_t launch_ex_typed(const ProblemEx &p, cudaStream_t s) {
    const long long tiles = (long long)((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const SimtEx ex = {p.lda, p.ldb, p.ldc, p.sa, p.sb, p.sc, p.alpha, p.beta};
    for (long long b0 = 0; b0 < p.batch; b0 += 65535) {
        const long long nb = std::min<long long>(65535, p.batch - b0);
        const TIn *A = static_cast<const TIn *>(p.A) + b0 * p.sa;
        const TIn *B = static_cast<const TIn *>(p.B) + b0 * p.sb;
        TIn *C = static_cast<TIn *>(p.C) + b0 * p.sc;
        cudaError_t e;
        if constexpr (VEC && sizeof(TIn) == 4) {
            // float4-able FP32: the packed-FMA kernel
            e = launch_ffma2<true, TA, TB>(A, B, C, p.M, p.N, p.K, ex, (unsigned)nb, s);
        } else {
            cudaLaunchAttribute attr[1];
            const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)tiles, (unsigned)nb, 1), dim3(THREADS), 0, s, attr);
            e = launch_counted(&cfg, simt_gemm_kernel<TIn, TIn, VEC, SIMT_BK, SIMT_MINB, 128, true, TA, TB>, A, B,
                                   C, p.M, p.N, p.K, 0, ex);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename TIn, bool VEC>
cudaError_t launch_ex_ops(const ProblemEx &p, cudaStream_t s) {
    if (p.a_t) return p.b_t ? launch_ex_typed<TIn, VEC, true, true>(p, s) : launch_ex_typed<TIn, VEC, true, false>(p, s);
    return p.b_t ? launch_ex_typed<TIn, VEC, false, true>(p, s) : launch_ex_typed<TIn, VEC, false, false>(p, s);
}

bool aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

// float4 loads and stores: every base 16-byte aligned, every leading dimension
// and used batch stride a multiple of 4, and the contiguous extent of each
// operand a multiple of 4 (a quad is then wholly inside or outside).
bool ex_vec_ok(const ProblemEx &p) {
    if (p.elt != Elt::F32) return false;
    if (!aligned16(p.A) || !aligned16(p.B) || !aligned16(p.C)) return false;
    if (p.lda % 4 || p.ldb % 4 || p.ldc % 4 || p.sa % 4 || p.sb % 4 || p.sc % 4) return false;
    if ((p.a_t ? p.M : p.K) % 4 || (p.b_t ? p.K : p.N) % 4) return false;
    return true;
}

}  // namespace

cudaError_t launch_simt(const Problem &p, bool vec4, int num_sms, cudaStream_t s) {
    switch (p.elt) {
    case Elt::F32:
        return vec4 ? launch_typed<float, float, true>(p, num_sms, s)
                    : launch_typed<float, float, false>(p, num_sms, s);
    case Elt::F16:
        return launch_typed<__half, __half, false>(p, num_sms, s);
    case Elt::BF16:
        return launch_typed<__nv_bfloat16, __nv_bfloat16, false>(p, num_sms, s);
    }
    return cudaErrorInvalidValue;
}

bool simt_ex_vec(const ProblemEx &p) { return ex_vec_ok(p); }

cudaError_t launch_simt_ex(const ProblemEx &p, cudaStream_t s) {
    switch (p.elt) {
    case Elt::F32:
        return ex_vec_ok(p) ? launch_ex_ops<float, true>(p, s) : launch_ex_ops<float, false>(p, s);
    case Elt::F16:
        return launch_ex_ops<__half, false>(p, s);
    case Elt::BF16:
        return launch_ex_ops<__nv_bfloat16, false>(p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
