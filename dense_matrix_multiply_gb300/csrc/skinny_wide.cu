// Skinny 16-bit GEMM (M <= 64, decode batches) on 256-column strips of the
// weights, the K range split over a thread-block cluster.
//
// With few rows of X the product is bound by reading W [K, N] once from HBM
// ("SGEMM measured and the three ledgers", the decode rows of its shape table;
// "Chapter 5 Operators and Runtime", section 5.1.5: bytes in flight =
// bandwidth x latency).  The 128-column skinny kernel (umma_gemm.cu) gives one
// CTA per strip and so cannot run more strips than SMs at once; this kernel
// takes over there: a CTA takes a strip of 256 columns -- 512 contiguous bytes
// of every W row it reads -- and N up to 256 x the SM count runs in one wave
// (N = 28672: 112 CTAs).  When the strips leave SMs idle, the CS CTAs of a
// cluster take K-blocks [r*KB/CS, (r+1)*KB/CS) of a strip (the CS with the
// most CTAs that fit on the SMs at once); all CTAs of one rank start at the
// same K and move through it at the same pace, so the grid reads CS bands of
// whole W rows.  (Where the 128-column kernel fits, it was measured faster:
// N = 12288, 48 strips x 3 here against 96 strips there, 20.4 against 18.7 us
// at M = 1.)
//
// The MMA is the swapped-operand one: each 128-column half of the strip is the
// 128-row operand of its own tcgen05.mma (MN-major in shared memory: two boxes
// of 64 columns x 64 k), the M rows of X the N = nb operand (K-major, one box
// of 64 k x M rows rounded up to 8; nb = M rounded up to 16), accumulating in
// tensor-memory columns [64 h, 64 h + nb) for half h; tensor-memory lane =
// column of C, column = row of C.  A stage is 64 k: 32 KiB of W plus nb * 128
// bytes of X; the 216 KiB ring holds 6 or 5 stages.  With CS = 1 C is stored
// straight from tensor memory; otherwise each CTA writes its FP32 partial
// [nb][256] to its drained ring and the cluster adds the partials through
// distributed shared memory in rank order, each CTA summing and storing an
// equal share of the (row, 4-column) groups.  Deterministic, one launch, no
// workspace; every barrier wait is bounded (about two seconds of
// %globaltimer; on expiry a code goes to the status word, the CTA's abort flag
// is raised, its own loads and MMAs are waited for, and its tensor memory is
// released).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"

namespace gemm_gb300 {
namespace {

constexpr int SW_THREADS = 192;  // warp 0 producer, warp 1 TMEM + MMA issuer, warps 2-5 epilogue
constexpr int SW_KB = 64;        // K per stage
constexpr int SW_MAX_STAGES = 8;
constexpr int SW_W_BOX = 64 * SW_KB * 2;   // 64 columns x 64 k of W: 8 KiB
constexpr int SW_W_STAGE = 4 * SW_W_BOX;   // 256 columns: 32 KiB
constexpr int SW_TILES = 216 * 1024;       // the operand ring
constexpr int SW_SMEM = 1024 + SW_TILES + 256;
constexpr uint32_t SW_TMEM_COLS = 128;     // two accumulators (one per 128-column half) of up to 64 columns
constexpr int SW_LD = 256 + 4;             // floats per row of a partial [nb][256]
constexpr unsigned long long SW_TIMEOUT_NS = 2000000000ull;
constexpr int ST_PRODUCER = 1, ST_MMA = 2, ST_EPILOGUE = 4, ST_DRAIN = 8;
static_assert(64 * SW_LD * 4 <= SW_TILES, "partial fits in the drained ring");

struct SwBars {
    uint64_t full[SW_MAX_STAGES];
    uint64_t empty[SW_MAX_STAGES];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(SwBars) <= 256, "barrier block");

__host__ __device__ constexpr int sw_nb(int M) { return (M + 15) / 16 * 16; }
__host__ __device__ constexpr int sw_x_rows(int M) { return (M + 7) / 8 * 8; }
__host__ __device__ constexpr int sw_x_box(int nb) { return nb * 128; }
__host__ __device__ constexpr int sw_stages(int nb) {
    return SW_TILES / (SW_W_STAGE + sw_x_box(nb)) < SW_MAX_STAGES ? SW_TILES / (SW_W_STAGE + sw_x_box(nb))
                                                                   : SW_MAX_STAGES;
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t sw_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long sw_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void sw_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sw_smem(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void sw_arrive_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sw_smem(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool sw_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(sw_smem(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase of `bar` with this parity; false after SW_TIMEOUT_NS, or
// once `abort` is raised when check_abort.
__device__ __noinline__ bool sw_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort, bool check_abort) {
    const unsigned long long t0 = sw_now();
    for (uint32_t it = 1;; ++it) {
        if (sw_try_wait(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (check_abort && *abort) return false;
            if (sw_now() - t0 > SW_TIMEOUT_NS) return false;
        }
    }
}
__device__ __forceinline__ bool sw_wait(uint64_t *bar, uint32_t parity, volatile int *abort, bool check_abort) {
    if (sw_try_wait(bar, parity)) return true;
    return sw_wait_slow(bar, parity, abort, check_abort);
}
__device__ __forceinline__ void sw_tma_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(sw_smem(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(sw_smem(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void sw_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void sw_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// D[tmem] (+)= A[smem] (128 x 16) . B[smem] (16 x nb), kind::f16, FP32 accumulator.
__device__ __forceinline__ void sw_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void sw_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sw_smem(bar))
                 : "memory");
}
__device__ __forceinline__ void sw_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void sw_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t sw_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t sw_cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void sw_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A float4 of CTA `rank`'s shared memory at the address of `p` in this CTA.
__device__ __forceinline__ float4 sw_ld_peer(const float *p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(sw_smem(p)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}
// Shared-memory matrix descriptor, 128-byte swizzle, descriptor version 1; lbo/sbo in bytes.
__device__ __forceinline__ uint64_t sw_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: FP32 D, A and B of one 16-bit type (0 f16,
// 1 bf16), A MN-major (the W strip), B K-major (the X rows), M = 128, N = nb.
__device__ __forceinline__ uint32_t sw_idesc(uint32_t ab_format, uint32_t nb) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | (1u << 15) | (0u << 16) | ((nb >> 3) << 17) |
           ((128u >> 4) << 24);
}
__device__ __forceinline__ void sw_store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void sw_store(__half *p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ uint32_t sw_pack2(float lo, float hi, __nv_bfloat16 *) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t sw_pack2(float lo, float hi, __half *) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <typename T, uint32_t AB_FORMAT>
__global__ void __launch_bounds__(SW_THREADS, 1)
skinny_wide_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   T *__restrict__ C, int M, int N, int K, int cs, int max_stages, int *status)
{
    extern __shared__ uint8_t sw_raw[];
    const uint32_t raw = sw_smem(sw_raw);
    uint8_t *smem = sw_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int nb = sw_nb(M), x_rows = sw_x_rows(M);
    const int stages = min(sw_stages(nb), max_stages);
    const int x_box = sw_x_box(nb);
    uint8_t *w_tiles = smem;
    uint8_t *x_tiles = smem + stages * SW_W_STAGE;
    float *part = reinterpret_cast<float *>(smem);  // [nb][SW_LD] once the ring is drained
    SwBars *bars = reinterpret_cast<SwBars *>(smem + SW_TILES);
    volatile int *abort_flag = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cs > 1 ? sw_rank() : 0u;
    const int n0 = (int)(cs > 1 ? sw_cluster_id() : blockIdx.x) * 256;
    const int num_kb = (K + SW_KB - 1) / SW_KB;
    const int kb0 = (int)(((long long)num_kb * rank) / cs), kb1 = (int)(((long long)num_kb * (rank + 1)) / cs);
    const bool has_work = kb1 > kb0;
    const int n_left = N - n0;
    const int halves = n_left > 128 ? 2 : 1;  // 128-column halves of the strip inside C

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            sw_init(&bars->full[s], 1);
            sw_init(&bars->empty[s], 1);
        }
        sw_init(&bars->acc_full, 1);
        sw_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sw_smem(&bars->tmem_base)),
                     "r"(SW_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    sw_fence_before();
    __syncthreads();
    sw_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    if (warp == 0 && lane == 0 && g_pdl) {
        // The strip's first ring-full of W is requested into L2 while the
        // previous kernel on the stream finishes (a hint only: no value a later
        // load returns depends on it; X, usually that kernel's output, is left
        // alone).
        const int wboxes = n_left >= 256 ? 4 : (n_left + 63) / 64;
        const int pf = min(kb1 - kb0, stages);
        for (int kb = kb0; kb < kb0 + pf; ++kb)
            for (int j = 0; j < wboxes; ++j)
                asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                                 reinterpret_cast<uint64_t>(&tmW)),
                             "r"(n0 + 64 * j), "r"(kb * SW_KB)
                             : "memory");
    }
    pdl_wait();  // the previous kernel's writes are visible from here on

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        const int wboxes = n_left >= 256 ? 4 : (n_left + 63) / 64;
        const uint32_t tx = (uint32_t)(wboxes * SW_W_BOX + x_rows * 128);
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!sw_wait(&bars->empty[stage], phase ^ 1u, abort_flag, true)) {
                atomicOr(status, ST_PRODUCER);
                *abort_flag = 1;
                break;
            }
            sw_arrive_tx(&bars->full[stage], tx);
            for (int j = 0; j < wboxes; ++j)
                sw_tma_2d(w_tiles + stage * SW_W_STAGE + j * SW_W_BOX, &tmW, &bars->full[stage], n0 + 64 * j,
                          kb * SW_KB);
            sw_tma_2d(x_tiles + stage * x_box, &tmX, &bars->full[stage], kb * SW_KB, 0);
            ++issued;
            if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        // The dependent grid may launch once every CTA has issued its last load:
        // its CTAs take the idle SMs and prefetch while this grid drains
        // (N = 28672 / 20480, K = 4096, M = 1, back to back: 37.0 / 29.8 us
        // against 38.4 / 33.7 with the launch released at the start).
        pdl_launch_dependents();
        // Let every load this thread issued land before the ring is reused.
        for (long long i = (issued > stages ? issued - stages : 0); i < issued; ++i) {
            if (!sw_wait(&bars->full[i % stages], (uint32_t)((i / stages) & 1), abort_flag, false)) {
                atomicOr(status, ST_DRAIN);
                break;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        // A = a 128-column half of the W strip, MN-major: its two 64-column
        // chunks SW_W_BOX bytes apart, a K step of 16 rows 2048 bytes.  B = the
        // X rows, K-major: a K step is 32 bytes inside the 128-byte swizzle row,
        // 8-row groups 1024 bytes apart.
        const uint32_t idesc = sw_idesc(AB_FORMAT, (uint32_t)nb);
        const uint64_t a_desc0 = sw_desc(sw_smem(w_tiles), SW_W_BOX, 1024);
        const uint64_t b_desc0 = sw_desc(sw_smem(x_tiles), 16, 1024);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!sw_wait(&bars->full[stage], phase, abort_flag, true)) { ok = false; break; }
            sw_fence_after();
            const uint64_t bd = b_desc0 + (uint64_t)((stage * x_box) >> 4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h < halves) {
                    const uint64_t ad = a_desc0 + (uint64_t)((stage * SW_W_STAGE + h * 2 * SW_W_BOX) >> 4);
#pragma unroll
                    for (int ks = 0; ks < SW_KB / 16; ++ks)
                        sw_mma(tmem_base + (uint32_t)(64 * h), ad + ks * (2048u >> 4), bd + (uint32_t)(ks * 2),
                               idesc, (kb != kb0 || ks != 0));
                }
            }
            sw_commit(&bars->empty[stage]);
            if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        if (ok) {
            sw_commit(&bars->acc_full);
        } else {
            atomicOr(status, ST_MMA);
            *abort_flag = 1;
        }
        sw_commit(&bars->drain);
        if (!sw_wait(&bars->drain, 0, abort_flag, false)) atomicOr(status, ST_DRAIN);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        // Lane nl of the four warps = column n0 + 128 h + nl of C in half h.
        const int quarter = warp & 3;
        const int nl = quarter * 32 + lane;
        bool ready = true;
        if (has_work && !sw_wait(&bars->acc_full, 0, abort_flag, true)) {
            atomicOr(status, ST_EPILOGUE);
            *abort_flag = 1;
            ready = false;
        }
        sw_fence_after();
        for (int h = 0; h < halves; ++h) {
            const int n = n0 + 128 * h + nl;
#pragma unroll 1
            for (int c = 0; c < nb; c += 32) {
                uint32_t r[32];
                if (has_work && ready) {
                    sw_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(64 * h + c), r);
                    sw_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                if (cs == 1) {
                    if (n < N) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c + j < M) sw_store(C + (size_t)(c + j) * N + n, __uint_as_float(r[j]));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c + j < M) part[(c + j) * SW_LD + 128 * h + nl] = __uint_as_float(r[j]);
                }
            }
        }
    }

    sw_fence_before();
    __syncwarp();
    if (cs > 1) {
        sw_cluster_sync();  // every partial is in its CTA's shared memory, visible cluster-wide
        // (row, four-column group) pairs dealt out to the cs CTAs in equal
        // ranges; the partials of ranks 0 .. cs-1 added in that order.
        const int groups = min(256, n_left) / 4;  // N % 8 == 0: whole groups
        const int total = M * groups;
        const int e0 = (int)(((long long)total * rank) / cs), e1 = (int)(((long long)total * (rank + 1)) / cs);
        for (int e = e0 + threadIdx.x; e < e1; e += SW_THREADS) {
            const int m = e / groups, c4 = (e - m * groups) * 4;
            const float *src = part + m * SW_LD + c4;
            float4 acc = sw_ld_peer(src, 0);
            for (int j = 1; j < cs; ++j) {
                const float4 v = sw_ld_peer(src, (uint32_t)j);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            uint2 w;
            w.x = sw_pack2(acc.x, acc.y, (T *)nullptr);
            w.y = sw_pack2(acc.z, acc.w, (T *)nullptr);
            *reinterpret_cast<uint2 *>(C + (size_t)m * N + n0 + c4) = w;
        }
        __syncwarp();
        sw_cluster_sync();  // every CTA keeps its shared memory until the others have read it
    } else {
        __syncthreads();  // tensor memory read out before it is freed
    }
    if (warp == 1) {
        sw_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(SW_TMEM_COLS)
                     : "memory");
    }
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn sw_encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// 2-D row-major [rows, cols] of 16-bit elements, box [box_rows, box_cols],
// 128-byte swizzle, zero fill out of bounds.
bool sw_map(CUtensorMap *map, const void *base, CUtensorMapDataType dt, int rows, int cols, int box_rows,
            int box_cols) {
    EncodeFn fn = sw_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, uint32_t F>
const void *sw_kernel() {
    return reinterpret_cast<const void *>(skinny_wide_kernel<T, F>);
}

// Largest number of co-resident clusters of cs CTAs (2 <= cs <= 8), per device
// and element type.
int sw_clusters_max(bool bf16, int cs, int dev) {
    static std::atomic<int> cached[64][2][9];
    static std::once_flag once[64][2][9];
    if (cs < 2 || cs > 8) return 0;
    const int t = bf16 ? 1 : 0;
    std::call_once(once[dev & 63][t][cs], [&] {
        const void *kern = t ? sw_kernel<__nv_bfloat16, 1>() : sw_kernel<__half, 0>();
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SW_SMEM) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)cs, 1, 1);
            cfg.blockDim = dim3(SW_THREADS, 1, 1);
            cfg.dynamicSmemBytes = SW_SMEM;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)cs;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        }
        cudaGetLastError();
        cached[dev & 63][t][cs].store(n);
    });
    return cached[dev & 63][t][cs].load();
}

template <typename T, uint32_t F>
cudaError_t launch_wide_typed(const Problem &p, int num_sms, int *status, cudaStream_t s) {
    const CUtensorMapDataType dt = F == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tx, tw;
    if (!sw_map(&tx, p.A, dt, p.M, p.K, sw_x_rows(p.M), 64) || !sw_map(&tw, p.B, dt, p.K, p.N, SW_KB, 64))
        return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // the strips alone, or clusters of cs CTAs splitting K: the cs with the
    // most CTAs that are all resident at once
    const long long tiles = (p.N + 255) / 256;
    const long long num_kb = (p.K + SW_KB - 1) / SW_KB;
    int cs = 1;
    for (int c = 2; c <= 8; ++c)
        if (c <= num_kb && tiles * c <= num_sms && sw_clusters_max(F == 1, c, dev) >= tiles) cs = c;
    if (tiles * cs > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    auto kern = skinny_wide_kernel<T, F>;
    static std::atomic<uint64_t> attr_done{0};  // one bit per device
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SW_SMEM);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * cs), 1, 1);
    cfg.blockDim = dim3(SW_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SW_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cs > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)cs;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (g_pdl) pdl_attr(attr[na++]);
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    return launch_counted(&cfg, kern, tx, tw, static_cast<T *>(p.C), p.M, p.N, p.K, cs, SW_MAX_STAGES, status);
}

}  // namespace

bool skinny_wide_supported(const Problem &p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.A), b = reinterpret_cast<uintptr_t>(p.B),
                    c = reinterpret_cast<uintptr_t>(p.C);
    return p.elt != Elt::F32 && p.M >= 1 && p.M <= 64 && (a & 15) == 0 && (b & 15) == 0 && (c & 7) == 0 &&
           p.K % 8 == 0 && p.N % 8 == 0;
}

cudaError_t launch_skinny_wide(const Problem &p, int num_sms, int *status, cudaStream_t s) {
    if (!skinny_wide_supported(p)) return cudaErrorNotSupported;
    return p.elt == Elt::BF16 ? launch_wide_typed<__nv_bfloat16, 1>(p, num_sms, status, s)
                              : launch_wide_typed<__half, 0>(p, num_sms, status, s);
}

}  // namespace gemm_gb300
