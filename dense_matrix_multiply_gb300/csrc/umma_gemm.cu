// Tensor-core GEMM on sm_103a: tcgen05 MMA, TMEM accumulators, TMA loads,
// warp specialisation, persistent tile loops.  The file holds four kernels:
//   * umma_gemm_kernel -- one CTA per 128 x 256 tile: one row tile (M <= 128)
//     that the skinny kernel does not take, and A rows that only 8-byte
//     cp.async can fetch; described first, below;
//   * umma_pair_kernel -- 256 x 256 tiles on 2-CTA clusters (cta_group::2), the
//     kernel of every larger problem, of the general form (3-D tensor maps,
//     either major-ness, alpha/beta, batches), of the fused FFN gate/up
//     projection (DUAL) and of the row-scaled E4M3 product (F8,
//     kind::f8f6f4);
//   * umma_skinny_kernel -- M <= 64: the weights as the MMA's 128 rows, the
//     M rows of the activations as its N (decode batches);
//   * pair_sk_fixup_kernel -- adds the stream-K partials of the pair kernel.
//
// Problem (row-major): C[M,N] = A[M,K] · B[K,N], A and B both f16 or both bf16
// (or both E4M3 codes), FP32 accumulation in tensor memory, one rounding to
// the output type.  The column-major half entry point reaches these kernels
// through C^T = B^T · A^T.
//
// Prior art and what is kept ("Chapter 5 Operators and Runtime", section 5.1.5
// on asynchronous matrix instructions fed from shared memory, producer and
// consumer handoff through barriers, descriptors and swizzle; section 5.2.2 on
// output tiles and their byte counts; "MTT S4000 FP16 GEMM" on epilogue bank
// conflicts and CTA order):
//   * CTA tile 128 x 256, K step 64.  One tcgen05.mma.cta_group::1.kind::f16
//     instruction is M=128, N=256, K=16; four per K step.
//   * Shared-memory ring of STAGES stages, each holding the A tile (128 rows x
//     128 bytes) and the B tile (64 k-rows x 256 columns, as four 64-column
//     boxes), all in the 128-byte swizzled layout TMA writes and the MMA
//     descriptors describe.  full[s] completes when TMA has landed both tiles
//     (transaction count); empty[s] completes when the MMAs that read stage s
//     are done (tcgen05.commit).
//   * Warp 0: TMA producer.  Warp 1: TMEM allocation and the single MMA-issuing
//     thread.  Warps 2-5: epilogue (TMEM -> registers -> bf16/half -> global).
//   * Two accumulators of 256 FP32 columns each in TMEM (512 columns, the whole
//     tensor memory of the SM), so the epilogue of one tile overlaps the MMAs of
//     the next: acc_full[b] is committed by the MMA thread, acc_empty[b] is
//     arrived on by the 128 epilogue threads.
//   * Persistent grid of one CTA per SM; CTA c takes tiles c, c + grid, ...
//     in an M-grouped order so that concurrently running tiles share operands
//     in L2.
//   * Ragged edges: TMA zero-fills rows/columns/k beyond the matrix; boxes that
//     lie wholly beyond N are not fetched; stores are predicated.
//   * Every barrier wait is bounded (about two seconds of %globaltimer); on
//     expiry the thread records a code in the status word, raises a CTA-wide
//     abort flag, waits (bounded) for its own asynchronous work and leaves; the
//     tensor memory is always released.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"

namespace gemm_gb300 {
namespace {

namespace cg = cooperative_groups;

constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;            // 16 KiB
constexpr int B_BOX = 64 * BK * 2;              // one 64-column box: 8 KiB
constexpr int B_STAGE = BN * BK * 2;            // 32 KiB
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int GROUP_M = 8;
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;

constexpr int SMEM_TILES = STAGES * (A_STAGE + B_STAGE);

// Whether the CTA-pair kernel evens out a part-full last wave with a stream-K
// tail (needs stream-ordered scratch).
#ifndef PAIR_SK
#define PAIR_SK 1
#endif
constexpr bool g_pair_sk = PAIR_SK != 0;
// Whether problems with M <= 64 run on the swapped-operand skinny kernel.
#ifndef UMMA_SKINNY
#define UMMA_SKINNY 1
#endif
constexpr bool g_umma_skinny = UMMA_SKINNY != 0;
constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + SMEM_TILES + 256 /*barriers*/;

// Status codes ORed into the device status word.
constexpr int ST_PRODUCER = 1, ST_MMA = 2, ST_EPILOGUE = 4, ST_DRAIN = 8;

template <int NSTAGES>
struct BarsT {
    uint64_t full[NSTAGES];
    uint64_t empty[NSTAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t peer_done;        // CTA pairs (leader's copy): the peer's producer has finished
    long long peer_issued;     // CTA pairs (leader's copy): stages the peer's producer loaded
    uint32_t tmem_base;
    int abort;
};
using Bars = BarsT<STAGES>;
static_assert(sizeof(Bars) <= 256, "barrier block");

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// Counts `bytes` of the current phase's expected transactions as done.
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Slow path of mbar_wait: spins with a time limit.
__device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort, bool check_abort) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (check_abort && *abort) return false;
            if (globaltimer() - t0 > TIMEOUT_NS) return false;
        }
    }
}
// Waits for the phase of `bar` with the given parity to complete.  Returns false
// after TIMEOUT_NS, or early when `abort` is raised (if check_abort).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort, bool check_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort, check_abort);
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
// Asks for the tile at (x, y) of a 2-D tensor map to be brought into L2 (a
// hint: no shared memory, no barrier, no effect on what later loads return).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
// D[tmem] (+)= A[smem] · B[smem], one M=128 N=256 K=16 step.
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when all previously issued MMAs of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
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
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- CTA-pair (cta_group::2) forms.  A kernel uses one cta_group throughout.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// All threads of both CTAs of the cluster (warp-converged).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// Raises the abort flag of this CTA and of its peer in the pair, so that the
// peer's waits give up at once instead of timing out on their own.
__device__ __forceinline__ void raise_abort_pair(volatile int *abort_flag, uint32_t rank) {
    *abort_flag = 1;
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(map_to_rank((const void *)abort_flag, rank ^ 1u)), "r"(1)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __noinline__ bool mbar_wait_cluster_slow(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                    bool check_abort) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (check_abort && *abort) return false;
            if (globaltimer() - t0 > TIMEOUT_NS) return false;
        }
    }
}
// Bounded wait with cluster-scope acquire (barriers that CTAs of the pair signal).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                  bool check_abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    return mbar_wait_cluster_slow(bar, parity, abort, check_abort);
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both CTAs] · B[smem of both CTAs]: one
// M=256 (128 rows per CTA) N=256 (128 columns of B per CTA) K=16 step.
__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at this shared offset in every CTA of `mask` when
// the pair's previously issued MMAs complete.
__device__ __forceinline__ void umma_commit_pair_multicast(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), descriptor
// version 1.  lbo/sbo in bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor for kind::f16: FP32 accumulator, A and B of the same
// 16-bit type (0 = f16, 1 = bf16); by default A K-major, B MN-major, M = 128,
// N = 256.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, uint32_t m = BM, uint32_t n = BN,
                                                  bool a_mn = false, bool b_mn = true) {
    return (1u << 4)                      // D: FP32
           | (ab_format << 7)             // A type
           | (ab_format << 10)            // B type
           | ((a_mn ? 1u : 0u) << 15)     // A major: 0 = K, 1 = MN
           | ((b_mn ? 1u : 0u) << 16)     // B major
           | ((n >> 3) << 17)     // N / 8
           | ((m >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &tm, int &tn) {
    const int per_group = GROUP_M * tiles_n;
    const int group = t / per_group;
    const int first_m = group * GROUP_M;
    const int gsize = min(tiles_m - first_m, GROUP_M);
    const int r = t - group * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, __nv_bfloat16 *) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __half *) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
// Two FP32 values to E4M3FN codes (nearest, ties to even, saturating to
// +-448), the first in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ void store1(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store1(__half *p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }

// One element of Z = SiLU(G) * U with the unfused chain's rounding points: G and
// U rounded to the storage type, T = round(SiLU(G)) with SiLU(g) = g / (1 + e^-g)
// evaluated in FP32 with the fast exponential and division intrinsics (their
// error, ~1e-6 relative, is far below the 2^-9 of T's rounding), then T * U
// (exact in FP32 for 16-bit factors), returned in FP32 for the final rounding.
// For g -> -inf the denominator overflows to +inf and T -> 0, SiLU's limit.
__device__ __forceinline__ float silu_f32(float gb) { return __fdividef(gb, 1.0f + __expf(-gb)); }
__device__ __forceinline__ float silu_mul(float g, float u, __nv_bfloat16 *) {
    const float gb = __bfloat162float(__float2bfloat16_rn(g));
    const float ub = __bfloat162float(__float2bfloat16_rn(u));
    const float t = __bfloat162float(__float2bfloat16_rn(silu_f32(gb)));
    return t * ub;
}

// A_CPASYNC: A's rows cannot be described by a TMA map (row stride or base not
// 16-byte aligned).  Then four extra warps (6-9) copy the A tile with 8-byte
// cp.async into the same 128-byte-swizzled layout TMA would write, and also
// issue B's TMA loads; full[s] counts their 128 arrivals plus B's bytes.
template <typename T, uint32_t AB_FORMAT, bool A_CPASYNC>
__global__ void __launch_bounds__(A_CPASYNC ? THREADS + 128 : THREADS, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const T *__restrict__ A, T *__restrict__ C, int M, int N, int K, int *status, int stall)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *a_tiles = smem;
    uint8_t *b_tiles = smem + STAGES * A_STAGE;
    Bars *bars = reinterpret_cast<Bars *>(smem + SMEM_TILES);
    volatile int *abort_flag = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_kb = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->full[s], A_CPASYNC ? 128 : 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 128);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!A_CPASYNC) tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel's writes are visible from here on

    if (A_CPASYNC && warp >= 6) {
        // ------------------------------------------------ producer: cp.async A + TMA B
        const int ptid = threadIdx.x - 6 * 32;  // 0..127
        constexpr int LAG = 2;                  // stages of copies in flight per thread
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        auto publish = [&](long long j) {       // this thread's copies of load j have landed
            const int sj = (int)(j % STAGES);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (ptid == 0) mbar_arrive_expect_tx(&bars->full[sj], (uint32_t)B_STAGE);
            else mbar_arrive(&bars->full[sj]);
        };
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, true)) { ok = false; break; }
                if (ptid == 0) {
                    for (int j = 0; j < 4; ++j)
                        tma_load_2d(b_tiles + stage * B_STAGE + j * B_BOX, &tmB, &bars->full[stage],
                                    tn * BN + j * 64, kb * BK);
                }
                uint8_t *a_dst = a_tiles + stage * A_STAGE;
#pragma unroll 4
                for (int j = 0; j < 16; ++j) {
                    const int idx = j * 128 + ptid;
                    const int row = idx >> 4, c8 = idx & 15;  // 8-byte piece c8 of the row's 128 bytes
                    const int gm = tm * BM + row, gk = kb * BK + c8 * 4;
                    const bool in = gm < M && gk < K;      // K % 4 == 0: a piece is all in or all out
                    const T *src = in ? A + (size_t)gm * K + gk : A;
                    const uint32_t dst = smem_u32(a_dst + row * 128 + (((c8 >> 1) ^ (row & 7)) << 4) + ((c8 & 1) << 3));
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(in ? 8 : 0)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                if (issued >= LAG) {
                    static_assert(LAG == 2, "wait_group immediate below");
                    asm volatile("cp.async.wait_group 2;" ::: "memory");
                    publish(issued - LAG);
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (ok) {
            for (long long j = (issued > LAG ? issued - LAG : 0); j < issued; ++j) publish(j);
        } else {
            atomicOr(status, ST_PRODUCER);
            *abort_flag = 1;
        }
    } else if (!A_CPASYNC && warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        // stall != 0 (a test of the bounded waits): issue no load at all, so the
        // MMA thread's first wait runs out and the CTA takes its timeout path.
        for (int t = blockIdx.x; t < num_tiles && ok && !stall; t += gridDim.x) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            const int n_left = N - tn * BN;
            const int boxes = n_left >= BN ? 4 : (n_left + 63) / 64;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, true)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bars->full[stage], (uint32_t)(A_STAGE + boxes * B_BOX));
                tma_load_2d(a_tiles + stage * A_STAGE, &tmA, &bars->full[stage], kb * BK, tm * BM);
                for (int j = 0; j < boxes; ++j)
                    tma_load_2d(b_tiles + stage * B_STAGE + j * B_BOX, &tmB, &bars->full[stage],
                                tn * BN + j * 64, kb * BK);
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) {
            atomicOr(status, ST_PRODUCER);
            *abort_flag = 1;
        }
        // Let every load this thread issued land before the CTA can exit.
        for (long long i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i) {
            const int s = (int)(i % STAGES);
            const uint32_t par = (uint32_t)((i / STAGES) & 1);
            if (!mbar_wait(&bars->full[s], par, abort_flag, false)) {
                atomicOr(status, ST_DRAIN);
                break;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = make_idesc(AB_FORMAT);
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        const uint32_t a_base = smem_u32(a_tiles), b_base = smem_u32(b_tiles);
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++it) {
            const int buf = it & 1;
            const uint32_t acc_par = (uint32_t)((it >> 1) & 1);
            if (!mbar_wait(&bars->acc_empty[buf], acc_par ^ 1u, abort_flag, true)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(&bars->full[stage], phase, abort_flag, true)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a_addr = a_base + stage * A_STAGE;
                const uint32_t b_addr = b_base + stage * B_STAGE;
#pragma unroll
                for (int ks = 0; ks < BK / UMMA_K; ++ks) {
                    // A: K-major; a K step of 16 elements is 32 bytes inside the
                    // 128-byte swizzle row.  8-row groups are 1024 bytes apart.
                    const uint64_t ad = smem_desc_sw128(a_addr + ks * 32, 16, 1024);
                    // B: MN-major; a K step of 16 rows is two 1024-byte atoms.
                    // 64-column boxes are B_BOX bytes apart (leading offset),
                    // 8-row groups 1024 bytes apart (stride offset).
                    const uint64_t bd = smem_desc_sw128(b_addr + ks * 2048, B_BOX, 1024);
                    umma(d_tmem, ad, bd, idesc, (kb | ks) != 0);
                }
                umma_commit(&bars->empty[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            umma_commit(&bars->acc_full[buf]);
        }
        if (!ok) {
            atomicOr(status, ST_MMA);
            *abort_flag = 1;
        }
        // All MMAs of this thread complete before the CTA can release TMEM.
        umma_commit(&bars->drain);
        if (!mbar_wait(&bars->drain, 0, abort_flag, false)) atomicOr(status, ST_DRAIN);
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
        const int row_in_tile = quarter * 32 + lane;
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
            int tm, tn;
            tile_coords(t, tiles_m, tiles_n, tm, tn);
            const int buf = it & 1;
            const uint32_t acc_par = (uint32_t)((it >> 1) & 1);
            if (!mbar_wait(&bars->acc_full[buf], acc_par, abort_flag, true)) { ok = false; break; }
            tc_fence_after();
            __syncwarp();
            const int row = tm * BM + row_in_tile;
            const int n0 = tn * BN;
            T *crow = C + (size_t)row * N;
#pragma unroll 1
            for (int chunk = 0; chunk < BN / 32; ++chunk) {
                const int c0 = n0 + chunk * 32;
                if (c0 >= N) break;  // warp-uniform
                uint32_t r[32];
                tmem_ld_32cols(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN + chunk * 32), r);
                tmem_ld_wait();
                if (row < M) {
                    if (c0 + 32 <= N) {
                        uint4 *dst = reinterpret_cast<uint4 *>(crow + c0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v;
                            v.x = pack2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]), (T *)nullptr);
                            v.y = pack2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]), (T *)nullptr);
                            v.z = pack2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]), (T *)nullptr);
                            v.w = pack2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]), (T *)nullptr);
                            dst[q] = v;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j < N) store1(crow + c0 + j, __uint_as_float(r[j]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bars->acc_empty[buf]);
        }
        if (!ok) {
            atomicOr(status, ST_EPILOGUE);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA pairs
// The product on 256 x 256 tiles computed by a cluster of two CTAs on two SMs
// (tcgen05 cta_group::2).  CTA r of the pair holds rows r*128..+127 of the A
// tile and columns r*128..+127 of the B tile in its own shared memory; the
// leader's (rank 0) single MMA thread issues M=256, N=256, K=16 steps that
// read both CTAs' shared memory and write each CTA's 128 accumulator rows into
// that CTA's tensor memory.  Per CTA a stage is 32 KiB (half the B bytes of
// the single-CTA tile), so six stages fit beside the epilogue's staging boxes.
//   * Both producers load their halves; every load completes on the LEADER's
//     full[s] (the leader arms it with the bytes of both CTAs).
//   * The leader's commit after a stage arrives on empty[s] of both CTAs
//     (multicast), freeing the stage in both.
//   * acc_full[b] of both CTAs is committed the same way; each CTA's 128
//     epilogue threads read their own tensor memory and arrive on the
//     leader's acc_empty[b] (256 arrivals).
//   * The epilogue stages each warp's 32 x 64 output boxes in 128-byte-
//     swizzled shared memory and writes them with TMA stores (full-line writes,
//     clipped at the matrix edge by the tensor map).
// No TMA multicast is used: each CTA fetches only its own operand halves.
//
// The kernel also computes the general form ("SGEMM measured and the three
// ledgers", section 2, the library call with operation flags and leading
// dimensions; section 3, kernel K1, alpha * acc + beta * C):
//     C_b = alpha * op(A_b) * op(B_b) + beta * C_b,   b < batch,
// row-major, with any leading dimensions and batch strides that TMA can
// describe.  All tensor maps are 3-D (inner, outer, batch).  op(A) = A^T (A
// stored [K, M]) makes the A tile MN-major: two 64 x 64 boxes per CTA and
// stage, described like the MN-major B tile.  op(B) = B^T (B stored [N, K])
// makes the B tile K-major: one 64 x 128 box per CTA and stage, described like
// the K-major A tile.  The instruction descriptor's major bits follow.
namespace pairk {
constexpr int PBM = 256, PBN = 256;
constexpr int P_A_STAGE = 128 * BK * 2;                        // 16 KiB per CTA
constexpr int P_B_STAGE = 128 * BK * 2;                        // 16 KiB per CTA
constexpr int P_BOX64 = 64 * BK * 2;                           // one 64 x 64 box: 8 KiB
constexpr uint32_t P_STAGE_TX = 2u * (P_A_STAGE + P_B_STAGE);  // bytes per stage, both CTAs
constexpr int P_STG_BOX = 32 * 64 * 2;                         // one 32-row x 64-column output box
constexpr int P_GROUP_M = 8;                                   // pair tiles per raster group
constexpr int P_STAGES = 6;
// Shared memory: the operand stages, two staging boxes per epilogue warp, the
// barriers.
__host__ __device__ constexpr int smem_tiles(int nst) { return nst * (P_A_STAGE + P_B_STAGE); }
constexpr int SMEM_STAGING = 4 * 2 * P_STG_BOX;
__host__ __device__ constexpr int smem_bytes(int nst) { return 1024 + smem_tiles(nst) + SMEM_STAGING + 256; }
static_assert(smem_bytes(P_STAGES) <= 232448, "shared memory budget");
}  // namespace pairk

// Scalar arguments of the pair kernel.
struct PairArgs {
    void *C;                  // C (read only when beta != 0; written through tmC)
    long long ldc, stride_c;  // elements
    int M, N, K, batch;
    int bn;                   // the tile's N extent (128, 192 or 256)
    int a_t;                  // A stored [K, M] (M contiguous) instead of [M, K]
    int b_t;                  // B stored [N, K] (K contiguous) instead of [K, N]
    int a_bcast, b_bcast;     // batch stride 0: every b reads matrix 0
    float alpha, beta;
    const float *row_scale;   // FP8 products: per-row scale of the output (F8Q: the row's amax)
    const void *a_src;        // F8Q: A [M,K] row-major half, quantised as it is loaded
    int *status;
    // Stream-K tail (sk_tiles > 0): the last sk_tiles tiles are cut into
    // K-block ranges of sk_w spread over clusters sk_first .. G-1, whose FP32
    // partials go to sk_ws (two slots per stream-K cluster, one 32-row x
    // 256-column slab per epilogue warp and CTA, column-major) instead of C.
    float *sk_ws;
    int sk_tiles, sk_w, sk_first;
    int stall;  // test of the bounded waits: 1 = the producers load nothing, 2 = the peer stops after one stage
};

// Tile t -> (batch index, row tile, column tile); M-grouped raster inside a batch.
__device__ __forceinline__ void pair_coords(int t, int tiles_m, int tiles_n, int &bt, int &tm, int &tn) {
    const int tiles_per_batch = tiles_m * tiles_n;
    bt = t / tiles_per_batch;
    const int r0 = t - bt * tiles_per_batch;
    const int per_group = pairk::P_GROUP_M * tiles_n;
    const int group = r0 / per_group;
    const int first_m = group * pairk::P_GROUP_M;
    const int gsize = min(tiles_m - first_m, pairk::P_GROUP_M);
    const int r = r0 - group * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

// Work unit u of cluster c: tile t, K-block range [kb0, kb1) and the index sk
// of the stream-K tile (-1 for a whole tile).  Whole tiles c, c + G, ... below
// num_tiles - sk_tiles come first; then, for c >= sk_first, the cluster's share
// [c'*W, (c'+1)*W) (c' = c - sk_first) of the stream-K iterations (tile-major,
// K-block minor), cut at tile boundaries.  W <= num_kb, so a share touches at
// most two tiles.  Producer, MMA issuer and epilogue walk the same sequence.
__device__ __forceinline__ bool pair_unit(int u, int c, int G, int num_tiles, const PairArgs &a, int num_kb, int &t,
                                          int &kb0, int &kb1, int &sk) {
    const int t_dp = num_tiles - a.sk_tiles;
    const int n_dp = c < t_dp ? (t_dp - 1 - c) / G + 1 : 0;
    if (u < n_dp) {
        t = c + u * G;
        kb0 = 0;
        kb1 = num_kb;
        sk = -1;
        return true;
    }
    if (a.sk_tiles == 0 || c < a.sk_first) return false;
    const long long cc = c - a.sk_first;
    const long long total = (long long)a.sk_tiles * num_kb;
    const long long end = min((cc + 1) * a.sk_w, total);
    long long it = cc * a.sk_w;
    for (int q = u - n_dp; q > 0; --q) {
        if (it >= end) return false;
        it = min((it / num_kb + 1) * num_kb, end);
    }
    if (it >= end) return false;
    sk = (int)(it / num_kb);
    t = t_dp + sk;
    kb0 = (int)(it - (long long)sk * num_kb);
    kb1 = (int)min((long long)num_kb, kb0 + (end - it));
    return true;
}

__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int x,
                                                 int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void unpack8(const uint4 &u, float (&o)[8], const __nv_bfloat16 *) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void unpack8(const uint4 &u, float (&o)[8], const __half *) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
// One M=256 N=bn K=32 step on 8-bit E4M3 operands (kind::f8f6f4), FP32 accumulator.
__device__ __forceinline__ void umma_pair_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// bn: the tile's N extent, a multiple of 64 in [128, 256], chosen per problem
// to fill the last wave (each CTA loads 128 columns of B per stage -- 64 when
// bn = 128 and B is MN-major -- and the MMA reads bn/2 of them; accumulator
// buffers stay 256 columns apart).
// DUAL (the FFN gate/up projection, "Chapter 5 Operators and Runtime",
// section 5.3.1): two weight matrices, tmB = W_g and tmB2 = W_u, both stored
// [K, N].  A tile is 256 x 128 of Z.  Per K step CTA r loads columns
// [64r, 64r + 64) of the tile from W_g into its first B box and the same
// columns of W_u into its second, so ONE N = 256 MMA (each CTA supplying 128 B
// columns) yields G and U side by side: accumulator columns 128r + [0, 64)
// hold G and 128r + [64, 128) hold U for Z columns 64r + [0, 64).  The
// epilogue keeps the unfused chain's rounding points: G and U rounded to the
// output type, T = round(SiLU(G)), Z = round(T * U).  G, U and T never leave
// the SM.
// F8 (the row-scaled FP8 projection, "Chapter 5 Operators and Runtime",
// example 5-8): A = Q [M,K] and B = Wt [N,K], E4M3 codes, both K-major; a K
// block is 128 codes (one 128-byte swizzle row, the same bytes as 64 16-bit
// elements) and one kind::f8f6f4 MMA consumes K = 32 (32 bytes, as a 16-bit
// K = 16 step).  The epilogue multiplies row i by row_scale[i] and rounds to
// T (half).
// F8Q (F8 with the quantisation fused into the load path, example 5-8's second
// scheme): A is the half matrix itself.  Four more warps per CTA (6-9) read
// its tile from global memory, 128 rows x 128 k per stage, multiply each value
// by 448 / amax_i of its row (amax from a pass over the whole rows before the
// product, row_scale[i] = amax_i), convert to E4M3 (nearest, saturating: the
// codes gemm_quantize_rows_e4m3 writes) and store the codes into the stage in
// the swizzled layout TMA would have written; full[s] then counts their eight
// warp arrivals besides the B bytes.  The epilogue scales row i by
// amax_i / 448.
// STALL: the instance the bounded-wait tests launch (args.stall); the
// production instances carry no test code on the producer's path.
template <typename T, uint32_t AB_FORMAT, int PSTAGES, bool DUAL = false, bool F8 = false, bool F8Q = false,
          bool STALL = false>
__global__ void __launch_bounds__(F8Q ? THREADS + 128 : THREADS, 1)
umma_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB2,
                 const PairArgs args)
{
    using namespace pairk;
    using PBars = BarsT<PSTAGES>;
    static_assert(sizeof(PBars) <= 256, "barrier block");
    static_assert(!F8Q || (F8 && !DUAL), "fused quantisation is an FP8 product");
    // bytes the leader's full[s] expects per stage: both CTAs' A and B tiles, or
    // (F8Q) only their B tiles -- the A codes are written by threads.  A plain
    // MN-major B tile 128 wide (64 columns per CTA) is one box: bf16 1000^3 on
    // 32 such tiles 10.2 against 11.4 us when each CTA loaded two.
    const bool b_one_box = !DUAL && !F8 && !args.b_t && args.bn == 128;
    const uint32_t STAGE_TX = F8Q ? 2u * P_B_STAGE : (b_one_box ? 2u * (P_A_STAGE + P_BOX64) : P_STAGE_TX);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *a_tiles = smem;
    uint8_t *b_tiles = smem + PSTAGES * P_A_STAGE;
    uint8_t *staging = smem + smem_tiles(PSTAGES);
    PBars *bars = reinterpret_cast<PBars *>(smem + smem_tiles(PSTAGES) + SMEM_STAGING);
    volatile int *abort_flag = &bars->abort;

    const int M = args.M, N = args.N, K = args.K, bn = args.bn;
    int *status = args.status;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = (int)cluster_id_x(), nclusters = (int)cluster_count_x();
    const int tiles_m = (M + PBM - 1) / PBM, tiles_n = (N + bn - 1) / bn;
    const int tiles_per_batch = tiles_m * tiles_n;
    const int num_tiles = tiles_per_batch * args.batch;
    constexpr int KB = F8 ? 128 : BK;  // K elements per stage (128 bytes per row)
    const int num_kb = (K + KB - 1) / KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&bars->full[s], F8Q ? 1 + 8 : 1);  // F8Q: + 4 converter warps of each CTA
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->peer_done, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 256);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
        if (DUAL) tma_prefetch_desc(&tmB2);
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised before any cross-CTA use
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel's writes are visible from here on

    auto coords = [&](int t, int &bt, int &tm, int &tn) { pair_coords(t, tiles_m, tiles_n, bt, tm, tn); };

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        // Every load of either CTA completes on the LEADER's full[s], which the
        // leader arms with both halves' bytes; both producers wait for the MMAs
        // to free a stage (empty[s], committed to both CTAs).  At the end the
        // peer tells the leader how many stages it loaded (peer_issued, then an
        // arrival on peer_done), and the leader waits until every stage either
        // CTA loaded has landed -- counting, on a path that gave up early, the
        // half of a stage that one side never loaded as done and arming a stage
        // that only the peer loaded -- before the pair passes its final cluster
        // barrier: no load is left in flight into either CTA's shared memory.
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        // stall (STALL instances, a test of the bounded waits): 1 -- neither
        // producer loads anything; 2 -- the peer loads only its first stage and
        // then gives up, as on a failed wait, while the leader goes on.
        const long long stop_after = STALL && args.stall == 2 && !leader ? 1 : (STALL && args.stall == 1 ? 0 : -1);
        for (int u = 0; ok; ++u) {
            int t, kb0, kb1, sk;
            if (STALL && stop_after == 0) break;
            if (!pair_unit(u, cluster, nclusters, num_tiles, args, num_kb, t, kb0, kb1, sk)) break;
            int bt, tm, tn;
            coords(t, bt, tm, tn);
            const int za = args.a_bcast ? 0 : bt, zb = args.b_bcast ? 0 : bt;
            const int row0 = tm * PBM + (int)rank * 128;
            const int col0 = tn * bn + (int)rank * (bn >> 1);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (STALL && issued == stop_after) { ok = false; break; }
                if (!mbar_wait_cluster(&bars->empty[stage], phase ^ 1u, abort_flag, true)) { ok = false; break; }
                const uint32_t full_leader = map_to_rank(&bars->full[stage], 0);
                if (leader) mbar_arrive_expect_tx(&bars->full[stage], STAGE_TX);
                uint8_t *a_dst = a_tiles + stage * P_A_STAGE;
                uint8_t *b_dst = b_tiles + stage * P_B_STAGE;
                const int k0 = kb * KB;
                if (F8Q) {
                    // A comes from the converter warps
                } else if (!args.a_t) {
                    tma_load_3d_pair(a_dst, &tmA, full_leader, k0, row0, za);
                } else {
                    tma_load_3d_pair(a_dst, &tmA, full_leader, row0, k0, za);
                    tma_load_3d_pair(a_dst + P_BOX64, &tmA, full_leader, row0 + 64, k0, za);
                }
                if (DUAL) {
                    // same 64 columns of W_g and of W_u
                    tma_load_3d_pair(b_dst, &tmB, full_leader, col0, k0, 0);
                    tma_load_3d_pair(b_dst + P_BOX64, &tmB2, full_leader, col0, k0, 0);
                } else if (!args.b_t) {
                    tma_load_3d_pair(b_dst, &tmB, full_leader, col0, k0, zb);
                    if (!b_one_box) tma_load_3d_pair(b_dst + P_BOX64, &tmB, full_leader, col0 + 64, k0, zb);
                } else {
                    tma_load_3d_pair(b_dst, &tmB, full_leader, k0, col0, zb);
                }
                ++issued;
                if (++stage == PSTAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) {
            atomicOr(status, ST_PRODUCER);
            raise_abort_pair(abort_flag, rank);
        }
        if (!leader) {
            asm volatile("st.shared::cluster.b64 [%0], %1;" ::"r"(map_to_rank(&bars->peer_issued, 0)), "l"(issued)
                         : "memory");
            mbar_arrive_cluster(map_to_rank(&bars->peer_done, 0));  // release: the count is visible first
        } else {
            long long ip = issued;
            if (mbar_wait_cluster(&bars->peer_done, 0, abort_flag, false)) {
                ip = *reinterpret_cast<volatile long long *>(&bars->peer_issued);
            } else {
                atomicOr(status, ST_DRAIN);
            }
            // Uses of a stage complete in order, and neither side runs more than
            // PSTAGES uses ahead of the MMAs, so only the last PSTAGES can be open.
            // The two counts differ only after one side gave up (and recorded
            // it in the status word): the MMAs may then have read a stage that
            // is completed below without the other half, which is why such a
            // call's C is undefined.
            const long long hi = issued > ip ? issued : ip;
            for (long long i = (hi > PSTAGES ? hi - PSTAGES : 0); i < hi; ++i) {
                const int s = (int)(i % PSTAGES);
                const uint32_t par = (uint32_t)((i / PSTAGES) & 1);
                if (i >= issued) {
                    mbar_arrive_expect_tx(&bars->full[s], STAGE_TX / 2);  // only the peer's half was loaded
                } else if (i >= ip) {
                    mbar_complete_tx(&bars->full[s], STAGE_TX / 2);       // the peer's half never will be
                }
                if (!mbar_wait_cluster(&bars->full[s], par, abort_flag, false)) {
                    atomicOr(status, ST_DRAIN);
                    break;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------------ MMA issuer (leader)
        const bool a_mn = args.a_t != 0, b_mn = DUAL || args.b_t == 0;
        const uint32_t idesc = make_idesc(AB_FORMAT, PBM, DUAL ? 256u : (uint32_t)bn, a_mn, b_mn);
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        // Descriptors of stage 0, K step 0; a stage or K step only moves the
        // start address (bits 0-13, in 16-byte units).  K-major tile: a K step
        // of 16 elements is 32 bytes inside the 128-byte swizzle row, 8-row
        // groups are 1024 bytes apart.  MN-major tile: a K step is 16 rows of
        // 128 bytes (2048 bytes), 64-element MN chunks (boxes) are P_BOX64
        // bytes apart.
        const uint64_t a_desc0 = smem_desc_sw128(smem_u32(a_tiles), a_mn ? P_BOX64 : 16, 1024);
        const uint64_t b_desc0 = smem_desc_sw128(smem_u32(b_tiles), b_mn ? P_BOX64 : 16, 1024);
        const uint32_t a_kstep = (a_mn ? 2048u : 32u) >> 4, b_kstep = (b_mn ? 2048u : 32u) >> 4;
        for (int u = 0; ok; ++u, ++it) {
            int t, kb0, kb1, sk;
            if (!pair_unit(u, cluster, nclusters, num_tiles, args, num_kb, t, kb0, kb1, sk)) break;
            const int buf = it & 1;
            const uint32_t acc_par = (uint32_t)((it >> 1) & 1);
            if (!mbar_wait_cluster(&bars->acc_empty[buf], acc_par ^ 1u, abort_flag, true)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * PBN);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_cluster(&bars->full[stage], phase, abort_flag, true)) { ok = false; break; }
                tc_fence_after();
                const uint64_t ad = a_desc0 + (uint64_t)((stage * P_A_STAGE) >> 4);
                const uint64_t bd = b_desc0 + (uint64_t)((stage * P_B_STAGE) >> 4);
#pragma unroll
                for (int ks = 0; ks < BK / UMMA_K; ++ks) {
                    const uint32_t acc = (kb != kb0) | (ks != 0);
                    if constexpr (F8)
                        umma_pair_f8(d_tmem, ad + ks * a_kstep, bd + ks * b_kstep, idesc, acc);
                    else
                        umma_pair(d_tmem, ad + ks * a_kstep, bd + ks * b_kstep, idesc, acc);
                }
                umma_commit_pair_multicast(&bars->empty[stage], 0x3);
                if (++stage == PSTAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            umma_commit_pair_multicast(&bars->acc_full[buf], 0x3);
        }
        if (!ok) {
            atomicOr(status, ST_MMA);
            raise_abort_pair(abort_flag, rank);
        }
        umma_commit_pair(&bars->drain);
        if (!mbar_wait_cluster(&bars->drain, 0, abort_flag, false)) atomicOr(status, ST_DRAIN);
    } else if (F8Q && warp >= 6) {
        // ------------------------------------------------------------ A converters (F8Q, both CTAs)
        // Warp w (0-3) makes rows 32w .. 32w + 31 of this CTA's 128 rows of the
        // A tile: per pass two rows, lanes 0-15 and 16-31, each lane 8
        // consecutive k of its row (one 16-byte load, 8 codes).
        const int cw = warp - 6;
        const __half *Ah = static_cast<const __half *>(args.a_src);
        const uint32_t full0 = map_to_rank(&bars->full[0], 0);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = 0; ok; ++u) {
            int t, kb0, kb1, sk;
            if (!pair_unit(u, cluster, nclusters, num_tiles, args, num_kb, t, kb0, kb1, sk)) break;
            int bt, tm, tn;
            coords(t, bt, tm, tn);
            const int row_w = tm * PBM + (int)rank * 128 + cw * 32;  // this warp's first row
            // lane l: 448 / amax of row row_w + l (0 for a row of zeros or past M:
            // its codes are 0, as the separate quantiser writes them)
            const float amax = row_w + lane < M ? args.row_scale[row_w + lane] : 0.0f;
            const float inv_l = amax > 0.0f ? 448.0f / amax : 0.0f;
            const int j = lane & 15;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait_cluster(&bars->empty[stage], phase ^ 1u, abort_flag, true))) {
                    ok = false;
                    break;
                }
                const int gk = kb * KB + 8 * j;
                uint4 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int gr = row_w + 2 * i + (lane >> 4);
                    v[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (gr < M && gk < K)  // K % 16 == 0: the 8 values are all in or all out
                        v[i] = __ldg(reinterpret_cast<const uint4 *>(Ah + (size_t)gr * K + gk));
                }
                uint8_t *a_dst = a_tiles + stage * P_A_STAGE;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 2 * i + (lane >> 4);  // row within the warp's 32
                    const float inv = __shfl_sync(0xffffffffu, inv_l, r);
                    const __half2 *h = reinterpret_cast<const __half2 *>(&v[i]);
                    uint32_t w[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const float2 f0 = __half22float2(h[2 * q]);
                        const float2 f1 = __half22float2(h[2 * q + 1]);
                        w[q] = (uint32_t)e4m3x2(f0.x * inv, f0.y * inv) | ((uint32_t)e4m3x2(f1.x * inv, f1.y * inv) << 16);
                    }
                    const int rr = cw * 32 + r;  // row within the CTA's 128
                    const uint32_t dst = smem_u32(a_dst + rr * 128 + ((((j >> 1) ^ (rr & 7))) << 4) + ((j & 1) << 3));
                    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(dst), "r"(w[0]), "r"(w[1]) : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the codes, to the MMAs
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(full0 + (uint32_t)(stage * sizeof(uint64_t)));
                if (++stage == PSTAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            atomicOr(status, ST_PRODUCER);
            raise_abort_pair(abort_flag, rank);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp & 3;
        uint8_t *my_stg = staging + quarter * 2 * P_STG_BOX;  // this warp's two staging boxes
        const float alpha = args.alpha, beta = args.beta;
        const bool use_beta = !DUAL && !F8 && beta != 0.0f;
        int sb = 0;
        int it = 0;
        bool ok = true;
        for (int u = 0;; ++u, ++it) {
            int t, kb0, kb1, sk;
            if (!pair_unit(u, cluster, nclusters, num_tiles, args, num_kb, t, kb0, kb1, sk)) break;
            int bt, tm, tn;
            coords(t, bt, tm, tn);
            const int buf = it & 1;
            const uint32_t acc_par = (uint32_t)((it >> 1) & 1);
            // every lane waits; the warp leaves together if any lane gave up
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(&bars->acc_full[buf], acc_par, abort_flag, true))) {
                ok = false;
                break;
            }
            tc_fence_after();
            __syncwarp();
            const int n0 = tn * bn;
            const int box_row0 = tm * PBM + (int)rank * 128 + quarter * 32;  // warp-uniform
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * PBN);
            // Stream-K segment: write this warp's FP32 partial of the tile
            // (column-major slab: 128-byte rows across the lanes) and free the
            // accumulator; pair_sk_fixup_kernel adds the partials in K order.
            if (sk >= 0) {
                const int ord = ((long long)(cluster - args.sk_first) * args.sk_w) / num_kb == sk ? 0 : 1;
                float *mine = args.sk_ws +
                              ((size_t)(2 * (cluster - args.sk_first) + ord) * 8 + rank * 4 + quarter) * (256 * 32);
                const int ncols = DUAL ? 256 : bn;
#pragma unroll 1
                for (int cc = 0; cc < ncols / 32; ++cc) {
                    uint32_t r[32];
                    tmem_ld_32cols(t_row + (uint32_t)(cc * 32), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) __stcg(mine + (cc * 32 + c) * 32 + lane, __uint_as_float(r[c]));
                }
                tc_fence_before();
                mbar_arrive_cluster(map_to_rank(&bars->acc_empty[buf], 0));
                continue;
            }
            if constexpr (DUAL) {
#pragma unroll 1
                for (int g = 0; g < 2; ++g) {
                    const int c0 = n0 + g * 64;
                    if (c0 >= N) break;  // warp-uniform
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    __syncwarp();
                    uint8_t *rowp = my_stg + sb * P_STG_BOX + lane * 128;
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        uint32_t rg[32], ru[32];
                        tmem_ld_32cols(t_row + (uint32_t)(g * 128 + h * 32), rg);
                        tmem_ld_32cols(t_row + (uint32_t)(g * 128 + 64 + h * 32), ru);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            float z[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                z[e] = silu_mul(__uint_as_float(rg[8 * c + e]), __uint_as_float(ru[8 * c + e]),
                                                (T *)nullptr);
                            uint4 v;
                            v.x = pack2(z[0], z[1], (T *)nullptr);
                            v.y = pack2(z[2], z[3], (T *)nullptr);
                            v.z = pack2(z[4], z[5], (T *)nullptr);
                            v.w = pack2(z[6], z[7], (T *)nullptr);
                            *reinterpret_cast<uint4 *>(rowp + (((h * 4 + c) ^ (lane & 7)) << 4)) = v;
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0 && box_row0 < M) tma_store_3d(&tmC, my_stg + sb * P_STG_BOX, c0, box_row0, 0);
                    sb ^= 1;
                }
            } else {
                const int row = box_row0 + lane;
                const float scale_v =
                    F8 ? (row < M ? (F8Q ? args.row_scale[row] / 448.0f : args.row_scale[row]) : 0.0f) : alpha;
                // This thread's row of C in batch bt, read only when beta != 0.
                const T *c_old = (use_beta && row < M)
                                     ? static_cast<const T *>(args.C) + (long long)bt * args.stride_c +
                                           (long long)row * args.ldc
                                     : nullptr;
#pragma unroll 1
                for (int g = 0; g < (bn >> 6); ++g) {
                    const int c0 = n0 + g * 64;
                    if (c0 >= N) break;  // warp-uniform
                    uint32_t r0[32], r1[32];
                    tmem_ld_32cols(t_row + (uint32_t)(g * 64), r0);
                    tmem_ld_32cols(t_row + (uint32_t)(g * 64 + 32), r1);
                    uint4 old[8];
                    if (use_beta) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int cc = c0 + 8 * c;
                            old[c] = make_uint4(0u, 0u, 0u, 0u);
                            if (c_old != nullptr && cc + 8 <= N) {
                                old[c] = *reinterpret_cast<const uint4 *>(c_old + cc);
                            } else if (c_old != nullptr) {
                                T tmp[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) tmp[e] = cc + e < N ? c_old[cc + e] : T(0.0f);
                                memcpy(&old[c], tmp, 16);
                            }
                        }
                    }
                    tmem_ld_wait();
                    // The store issued two boxes ago read this staging box.
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    __syncwarp();
                    uint8_t *rowp = my_stg + sb * P_STG_BOX + lane * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t *src = c < 4 ? &r0[8 * c] : &r1[8 * (c - 4)];
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = scale_v * __uint_as_float(src[e]);
                        if (use_beta) {
                            float o[8];
                            unpack8(old[c], o, (const T *)nullptr);
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = fmaf(beta, o[e], v[e]);
                        }
                        uint4 w;
                        w.x = pack2(v[0], v[1], (T *)nullptr);
                        w.y = pack2(v[2], v[3], (T *)nullptr);
                        w.z = pack2(v[4], v[5], (T *)nullptr);
                        w.w = pack2(v[6], v[7], (T *)nullptr);
                        *reinterpret_cast<uint4 *>(rowp + ((c ^ (lane & 7)) << 4)) = w;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0 && box_row0 < M) tma_store_3d(&tmC, my_stg + sb * P_STG_BOX, c0, box_row0, bt);
                    sb ^= 1;
                }
            }
            tc_fence_before();
            mbar_arrive_cluster(map_to_rank(&bars->acc_empty[buf], 0));
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        if (!ok && lane == 0) {
            atomicOr(status, ST_EPILOGUE);
            raise_abort_pair(abort_flag, rank);
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();  // no CTA leaves while its peer may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// Stream-K fix-up: each stream-K tile of the CTA-pair kernel is the sum, in K
// order, of the FP32 partials of the clusters whose K ranges cover it; this
// kernel adds them and applies the pair kernel's epilogue (alpha, beta * old
// C, the fused SiLU * U chain, the FP8 row scale; one rounding to T).  Launched
// after the pair kernel on the same stream.  Block (2 sk + r, y): rows
// [128 r, 128 r + 128) of stream-K tile sk, one per thread, output columns
// [8y, 8y + 8) of the tile.
template <typename T, bool DUAL, bool F8>
__global__ void __launch_bounds__(128)
pair_sk_fixup_kernel(const PairArgs args, int num_kb)
{
    pdl_launch_dependents();
    pdl_wait();
    const int sk = (int)(blockIdx.x >> 1), rank = (int)(blockIdx.x & 1);
    const int quarter = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
    const int bn = args.bn, M = args.M, N = args.N;
    const int tiles_m = (M + pairk::PBM - 1) / pairk::PBM, tiles_n = (N + bn - 1) / bn;
    const int num_tiles = tiles_m * tiles_n * args.batch;
    const int zc = (int)blockIdx.y * 8;  // first output column of this thread, in the tile
    if (zc >= bn) return;
    int bt, tm, tn;
    pair_coords(num_tiles - args.sk_tiles + sk, tiles_m, tiles_n, bt, tm, tn);
    const int row = tm * pairk::PBM + rank * 128 + (int)threadIdx.x, col = tn * bn + zc;
    if (row >= M || col >= N) return;
    const long long it0 = (long long)sk * num_kb;
    const int cf = (int)(it0 / args.sk_w), cl = (int)((it0 + num_kb - 1) / args.sk_w);
    // accumulator columns: DUAL -- G at 128 g + j, U at 128 g + 64 + j for
    // output column 64 g + j; otherwise the output column itself.
    constexpr int NACC = DUAL ? 16 : 8;
    int acol[NACC];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if constexpr (DUAL) {
            const int g = (zc + e) >> 6, j = (zc + e) & 63;
            acol[e] = 128 * g + j;
            acol[8 + e] = 128 * g + 64 + j;
        } else {
            acol[e] = zc + e;
        }
    }
    float acc[NACC];
#pragma unroll 1
    for (int c = cf; c <= cl; ++c) {
        const int ord = ((long long)c * args.sk_w) / num_kb == sk ? 0 : 1;
        const float *slab = args.sk_ws + ((size_t)(2 * c + ord) * 8 + rank * 4 + quarter) * (256 * 32) + lane;
        float v[NACC];
#pragma unroll
        for (int e = 0; e < NACC; ++e) v[e] = __ldcg(slab + acol[e] * 32);
#pragma unroll
        for (int e = 0; e < NACC; ++e) acc[e] = c == cf ? v[e] : acc[e] + v[e];
    }
    float z[8];
    if constexpr (DUAL) {
#pragma unroll
        for (int e = 0; e < 8; ++e) z[e] = silu_mul(acc[e], acc[8 + e], (T *)nullptr);
    } else {
        const float sc = F8 ? args.row_scale[row] : args.alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) z[e] = sc * acc[e];
    }
    T *dst = static_cast<T *>(args.C) + (long long)bt * args.stride_c + (long long)row * args.ldc + col;
    if (!DUAL && !F8 && args.beta != 0.0f) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (col + e < N) z[e] = fmaf(args.beta, to_float(dst[e]), z[e]);
    }
    if (col + 8 <= N) {
        uint4 w;
        w.x = pack2(z[0], z[1], (T *)nullptr);
        w.y = pack2(z[2], z[3], (T *)nullptr);
        w.z = pack2(z[4], z[5], (T *)nullptr);
        w.w = pack2(z[6], z[7], (T *)nullptr);
        *reinterpret_cast<uint4 *>(dst) = w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (col + e < N) store1(dst + e, z[e]);
    }
}

// ------------------------------------------- skinny M: weights as the MMA's rows
// For M <= 64 the roles of the operands swap: D = W^T X^T, i.e. C^T, with the
// weights W [K, N] as the MMA's 128-row operand (a 128-column strip of W, MN-
// major in shared memory: two boxes of 64 columns x 128 k per stage) and the M
// rows of X as its N = nb operand (K-major, two boxes of 64 k x M rows rounded
// up to 8; nb = M rounded up to 16, the stale rows past the box only reaching
// accumulator columns that are never stored).  Every MMA row is a useful
// output column; a stage is 32 KiB of W + two X boxes of nb rows, and the
// 216 KiB ring holds 6, 5 or 4 stages for M <= 16, 32 or 64 (used in full when
// the grid leaves a third of the SMs idle, else four), keeping up to 192 KiB
// of W in flight per SM in few, large TMA requests (a 100 MB stream in 64 x
// 128 boxes measured 17.4 against 18.6 us in 64 x 64 boxes); the accumulator
// is nb <= 64 tensor-memory columns.  Tile t = 128
// columns of C; the CS CTAs of a cluster take K-blocks [r*KB/CS, (r+1)*KB/CS)
// of it and add their partials through distributed shared memory in rank
// order (CS = 1: no cluster, C is stored straight from tensor memory).
// Deterministic, one launch, no workspace; every barrier wait is bounded.
constexpr int SKB = 128;                     // K per stage
constexpr int SKS = 8;                       // stages, at most (barrier arrays)
constexpr int SK_W_BOX = 64 * SKB * 2;       // 64 columns x 128 k of W: 16 KiB
constexpr int SK_W_STAGE = 2 * SK_W_BOX;     // 128 columns: 32 KiB
constexpr int SK_SMEM_TILES = 216 * 1024;   // the ring: as many stages as fit
constexpr int SK_SMEM_BYTES = 1024 + SK_SMEM_TILES + 256;
// X's box per 64 k: nb rows of 128 bytes (the MMA reads nb rows; TMA fills the
// first M rounded up to 8); a stage holds two.  W 32 KiB + X 4 / 8 / 12 / 16
// KiB for M <= 16 / 32 / 48 / 64: 6, 5, 4, 4 stages.
__host__ __device__ constexpr int skinny_x_box(int nb) { return nb * 128; }
__host__ __device__ constexpr int skinny_stages(int nb) {
    return SK_SMEM_TILES / (SK_W_STAGE + 2 * skinny_x_box(nb)) < SKS
               ? SK_SMEM_TILES / (SK_W_STAGE + 2 * skinny_x_box(nb))
               : SKS;
}
constexpr uint32_t SK2_TMEM_COLS = 64;
constexpr int SK2_LD = 128 + 4;              // floats per m-row of a partial [nb][128]
using SkBars = BarsT<SKS>;
static_assert(sizeof(SkBars) <= 256, "barrier block");
static_assert(64 * SK2_LD * 4 <= SK_SMEM_TILES, "partial fits in the drained stages");

__host__ __device__ constexpr int skinny_x_rows(int M) { return (M + 7) / 8 * 8; }
__host__ __device__ constexpr int skinny_nb(int M) { return (M + 15) / 16 * 16; }

template <typename T, uint32_t AB_FORMAT>
__global__ void __launch_bounds__(THREADS, 1)
umma_skinny_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   T *__restrict__ C, int M, int N, int K, int cs, int max_stages, int *status)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *w_tiles = smem;
    const int stages = min(skinny_stages(skinny_nb(M)), max_stages);
    const int x_box = skinny_x_box(skinny_nb(M)), x_stage = 2 * x_box;
    uint8_t *x_tiles = smem + stages * SK_W_STAGE;
    float *part = reinterpret_cast<float *>(smem);  // [nb][SK2_LD] once the stages are drained
    SkBars *bars = reinterpret_cast<SkBars *>(smem + SK_SMEM_TILES);
    volatile int *abort_flag = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cs > 1 ? cluster_ctarank() : 0u;
    const int n0 = (int)(cs > 1 ? cluster_id_x() : blockIdx.x) * 128;
    const int num_kb = (K + SKB - 1) / SKB;
    const int kb0 = (int)(((long long)num_kb * rank) / cs), kb1 = (int)(((long long)num_kb * (rank + 1)) / cs);
    const bool has_work = kb1 > kb0;
    const int x_rows = skinny_x_rows(M), nb = skinny_nb(M);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->acc_full[0], 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, SK2_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    if (warp == 0 && lane == 0 && g_pdl) {
        // While the previous kernel on the stream finishes, the strip's first
        // ring-full of W is requested into L2, so that the weight stream does
        // not start from cold DRAM latency after this grid's wait.  A prefetch
        // is only a hint -- it changes no value that a later load returns --
        // so it is correct whatever that kernel writes; X is left alone, since
        // it is usually that kernel's output.
        const int n_left = N - n0;
        const int wboxes = n_left >= 128 ? 2 : (n_left + 63) / 64;
        const int pf = min(kb1 - kb0, stages);
        for (int kb = kb0; kb < kb0 + pf; ++kb)
            for (int j = 0; j < wboxes; ++j) tma_prefetch_l2_2d(&tmW, n0 + 64 * j, kb * SKB);
    }
    pdl_wait();  // the previous kernel's writes are visible from here on

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ producer
        const int n_left = N - n0;
        const int wboxes = n_left >= 128 ? 2 : (n_left + 63) / 64;
        const uint32_t tx = (uint32_t)(wboxes * SK_W_BOX + 2 * x_rows * 64 * 2);
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, true)) {
                atomicOr(status, ST_PRODUCER);
                *abort_flag = 1;
                break;
            }
            mbar_arrive_expect_tx(&bars->full[stage], tx);
            for (int j = 0; j < wboxes; ++j)
                tma_load_2d(w_tiles + stage * SK_W_STAGE + j * SK_W_BOX, &tmW, &bars->full[stage], n0 + 64 * j,
                            kb * SKB);
            tma_load_2d(x_tiles + stage * x_stage, &tmX, &bars->full[stage], kb * SKB, 0);
            tma_load_2d(x_tiles + stage * x_stage + x_box, &tmX, &bars->full[stage], kb * SKB + 64, 0);
            ++issued;
            if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        // The dependent grid may launch once every CTA has issued its last load:
        // its CTAs then take the idle SMs and prefetch their first W stages
        // while this grid's last stages drain, rather than competing with its
        // full-rate stream (N = 12288, K = 4096, back to back, W from DRAM,
        // M = 1 / 8 / 32 / 64: 17.7 / 17.9 / 18.9 / 21.3 us, against 18.7 /
        // 19.0 / 20.0 / 22.5 with the launch released at the start and no
        // prefetch, and 20.0 / 20.1 / 20.3 / 22.4 with the prefetch but the
        // launch released at the start).
        pdl_launch_dependents();
        // Let every load this thread issued land before the stages are reused.
        for (long long i = (issued > stages ? issued - stages : 0); i < issued; ++i) {
            const int s = (int)(i % stages);
            const uint32_t par = (uint32_t)((i / stages) & 1);
            if (!mbar_wait(&bars->full[s], par, abort_flag, false)) {
                atomicOr(status, ST_DRAIN);
                break;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        // A = the W strip, MN-major: 64-column chunks SK_W_BOX bytes apart, a K
        // step of 16 rows is 2048 bytes.  B = the X rows, K-major: a K step is
        // 32 bytes inside the 128-byte swizzle row, 8-row groups 1024 bytes
        // apart, the second 64 k in the next box.
        const uint32_t idesc = make_idesc(AB_FORMAT, 128, (uint32_t)nb, true, false);
        const uint64_t a_desc0 = smem_desc_sw128(smem_u32(w_tiles), SK_W_BOX, 1024);
        const uint64_t b_desc0 = smem_desc_sw128(smem_u32(x_tiles), 16, 1024);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&bars->full[stage], phase, abort_flag, true)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = a_desc0 + (uint64_t)((stage * SK_W_STAGE) >> 4);
            const uint64_t bd = b_desc0 + (uint64_t)((stage * x_stage) >> 4);
#pragma unroll
            for (int ks = 0; ks < SKB / UMMA_K; ++ks)
                umma(tmem_base, ad + ks * (2048u >> 4),
                     bd + (uint32_t)(((ks >> 2) * x_box + (ks & 3) * 32) >> 4), idesc, (kb != kb0 || ks != 0));
            umma_commit(&bars->empty[stage]);
            if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        if (ok) {
            umma_commit(&bars->acc_full[0]);
        } else {
            atomicOr(status, ST_MMA);
            *abort_flag = 1;
        }
        umma_commit(&bars->drain);
        if (!mbar_wait(&bars->drain, 0, abort_flag, false)) atomicOr(status, ST_DRAIN);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        // TMEM lane = column n0 + nl of C, TMEM column = row m.
        const int quarter = warp & 3;
        const int nl = quarter * 32 + lane, n = n0 + nl;
        bool ready = true;
        if (has_work && !mbar_wait(&bars->acc_full[0], 0, abort_flag, true)) {
            atomicOr(status, ST_EPILOGUE);
            *abort_flag = 1;
            ready = false;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < nb; c += 32) {
            uint32_t r[32];
            if (has_work && ready) {
                tmem_ld_32cols(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, r);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = 0u;
            }
            if (cs == 1) {
                if (n < N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c + j < M) store1(C + (size_t)(c + j) * N + n, __uint_as_float(r[j]));
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c + j < M) part[(c + j) * SK2_LD + nl] = __uint_as_float(r[j]);
            }
        }
    }

    tc_fence_before();
    __syncwarp();
    if (cs > 1) {
        cluster_sync();  // every partial is in its CTA's shared memory, visible cluster-wide
        // (row, four-column group) pairs dealt out to the cs CTAs in equal
        // ranges; the partials of ranks 0 .. cs-1 added in that order.
        cg::cluster_group cluster = cg::this_cluster();
        const int groups = min(128, N - n0) / 4;  // N % 8 == 0: whole groups
        const int total = M * groups;
        const int e0 = (int)(((long long)total * rank) / cs), e1 = (int)(((long long)total * (rank + 1)) / cs);
        for (int e = e0 + threadIdx.x; e < e1; e += THREADS) {
            const int m = e / groups, c4 = (e - m * groups) * 4;
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < cs) v[j] = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(part + m * SK2_LD + c4, j));
            float4 acc = v[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) {
                if (j < cs) {
                    acc.x += v[j].x; acc.y += v[j].y; acc.z += v[j].z; acc.w += v[j].w;
                }
            }
            uint2 w;
            w.x = pack2(acc.x, acc.y, (T *)nullptr);
            w.y = pack2(acc.z, acc.w, (T *)nullptr);
            *reinterpret_cast<uint2 *>(C + (size_t)m * N + n0 + c4) = w;
        }
        __syncwarp();
        cluster_sync();  // every CTA keeps its shared memory until the others have read it
    } else {
        __syncthreads();  // tensor memory read out before it is freed
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, SK2_TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D row-major matrix [rows, cols] of 16-bit elements, box [box_rows, box_cols],
// 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap *map, const void *base, CUtensorMapDataType dt, int rows, int cols, int box_rows,
              int box_cols, long long row_elems = 0) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(row_elems > 0 ? row_elems : cols) * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, uint32_t F, bool A_CPASYNC>
cudaError_t launch_typed(const Problem &p, int num_sms, int *status, cudaStream_t s, int stall = 0) {
    const CUtensorMapDataType dt = F == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap ta, tb;
    if (!make_map(&tb, p.B, dt, p.K, p.N, BK, 64)) return cudaErrorInvalidValue;
    if (A_CPASYNC) {
        ta = tb;  // unused by the kernel
    } else if (!make_map(&ta, p.A, dt, p.M, p.K, BM, BK)) {
        return cudaErrorInvalidValue;
    }
    auto kern = umma_gemm_kernel<T, F, A_CPASYNC>;
    static std::atomic<uint64_t> attr_done{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const long long tiles = (long long)((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(A_CPASYNC ? THREADS + 128 : THREADS), SMEM_BYTES, s, attr);
    return launch_counted(&cfg, kern, ta, tb, static_cast<const T *>(p.A), static_cast<T *>(p.C), p.M, p.N, p.K,
                              status, stall);
}

// Largest number of co-resident clusters of cs CTAs (2 <= cs <= 8) of the
// swapped-operand skinny kernel, per device and element type.
int skinny_clusters_max(Elt elt, int cs, int dev) {
    static std::atomic<int> cached[64][2][9];
    static std::once_flag once[64][2][9];
    if (cs < 2 || cs > 8) return 0;
    const int t = elt == Elt::BF16 ? 1 : 0;
    std::call_once(once[dev & 63][t][cs], [&] {
        const void *kern = t ? reinterpret_cast<const void *>(umma_skinny_kernel<__nv_bfloat16, 1>)
                             : reinterpret_cast<const void *>(umma_skinny_kernel<__half, 0>);
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM_BYTES) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)cs, 1, 1);
            cfg.blockDim = dim3(THREADS, 1, 1);
            cfg.dynamicSmemBytes = SK_SMEM_BYTES;
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

// Swapped-operand skinny launch: ceil(N / 128) column strips, each on one CTA
// (cs = 1) or on a cluster of cs CTAs splitting K.
template <typename T, uint32_t F>
cudaError_t launch_skinny_typed(const Problem &p, int cs, int num_sms, int *status, cudaStream_t s) {
    const CUtensorMapDataType dt = F == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (p.M < 1 || p.M > 64 || cs < 1 || cs > 8) return cudaErrorInvalidValue;
    CUtensorMap tx, tw;
    if (!make_map(&tx, p.A, dt, p.M, p.K, skinny_x_rows(p.M), 64) || !make_map(&tw, p.B, dt, p.K, p.N, SKB, 64))
        return cudaErrorInvalidValue;
    auto kern = umma_skinny_kernel<T, F>;
    static std::atomic<uint64_t> attr_done{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const long long tiles_n = (p.N + 127) / 128;
    if (tiles_n * cs > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    // The whole ring (up to six stages) when the grid leaves a third of the SMs
    // idle, else four stages: measured back to back at N = 12288 (96 CTAs),
    // M = 1 / 8 / 32, 18.8 / 18.9 / 19.9 us against 19.9 / 20.4 / 21.2 with
    // four; with 128-148 CTAs the deeper ring was 3 % slower.
    const int max_stages = 3 * tiles_n * cs <= 2LL * num_sms ? SKS : 4;
    if (cs == 1) {
        cudaLaunchAttribute a1[1];
        const cudaLaunchConfig_t c1 = pdl_config(dim3((unsigned)tiles_n), dim3(THREADS), SK_SMEM_BYTES, s, a1);
        return launch_counted(&c1, kern, tx, tw, static_cast<T *>(p.C), p.M, p.N, p.K, 1, max_stages, status);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles_n * cs), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SK_SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    pdl_attr(attr[1]);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 2 : 1;
    return launch_counted(&cfg, kern, tx, tw, static_cast<T *>(p.C), p.M, p.N, p.K, cs, max_stages, status);
}

// 3-D tensor map of `batch` matrices of [outer, inner] 16-bit elements: row
// stride ld elements, matrix stride `stride` elements; box [box_outer,
// box_inner], 128-byte swizzle, zero fill out of bounds.  batch == 1 ignores
// stride.
bool make_map3(CUtensorMap *map, const void *base, CUtensorMapDataType dt, long long inner, long long outer,
               long long batch, long long ld, long long stride, int box_inner, int box_outer, int esize = 2) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    if (batch <= 1) stride = ld * outer;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)(batch > 1 ? batch : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(stride * esize)};
    const cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest number of co-resident two-CTA clusters of the pair kernel, per device
// (0: the pair kernel cannot be launched).
template <typename T, uint32_t F, bool DUAL = false, bool F8 = false, bool F8Q = false, bool STALL = false>
int pair_clusters_max(int dev) {
    static std::atomic<int> cached[64];
    static std::once_flag once[64];
    std::call_once(once[dev & 63], [&] {
        auto kern = umma_pair_kernel<T, F, pairk::P_STAGES, DUAL, F8, F8Q, STALL>;
        const int smem = pairk::smem_bytes(pairk::P_STAGES);
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2, 1, 1);
            cfg.blockDim = dim3(F8Q ? THREADS + 128 : THREADS, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        }
        cudaGetLastError();
        cached[dev & 63].store(n);
    });
    return cached[dev & 63].load();
}

template <typename T, uint32_t F, bool DUAL, bool F8 = false, bool F8Q = false, bool STALL = false>
cudaError_t launch_pair_cfg(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                            const CUtensorMap &tb2, const PairArgs &args, int clusters, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(F8Q ? THREADS + 128 : THREADS, 1, 1);
    cfg.dynamicSmemBytes = pairk::smem_bytes(pairk::P_STAGES);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    pdl_attr(attr[1]);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 2 : 1;
    return launch_counted(&cfg, umma_pair_kernel<T, F, pairk::P_STAGES, DUAL, F8, F8Q, STALL>, ta, tb, tc, tb2,
                          args);
}

// Whether T tiles of KB K-blocks on G clusters take a stream-K tail: the last
// wave holds rem = T mod G <= G / 4 tiles (a nearly empty wave still costs
// most of a tile time: with half the clusters busy it measured 85 % of a full
// wave, so spreading a fuller one gains too little) and a tile is long
// enough (KB >= 48) for the saving to exceed the fix-up's cost (scratch, a
// second kernel, ~8 us back to back).  Measured on GB300: FP16 3072 x 5120 x
// 6144 (240 tiles, rem 12) 142 -> 126 us; the BF16 FFN 1024 x 12288 x 4096
// (rem 40) 66 -> 77 us, so it keeps whole tiles.
bool sk_worth(long long tiles, int clusters, long long num_kb) {
    if (!g_pair_sk || clusters <= 0 || tiles <= clusters) return false;
    const long long rem = tiles % clusters;
    return rem > 0 && rem * 4 <= clusters && num_kb >= 48;
}

// Whether a problem of T tiles (256 wide) of KB K-blocks runs as stream-K over
// all of its tiles, four clusters per tile: the tiles would occupy at most a
// quarter of the G co-resident clusters and K is long (KB >= 64), so that the
// spread pays for the partials and the fix-up kernel.  Measured back to back on
// GB300, bf16, against whole tiles: 512 x 512 x 8192 and 256 x 1024 x 8192
// 21.4 against 40.5 us, 768 x 768 x 4096 18.8 against 22.9, 1024 x 1024 x 4096
// 22.4 against 23.1; where it is not taken it lost: 1024 x 2048 x 6144 (32
// tiles) 34.7 against 32.4, 1000 x 1000 x 3072 (48 K-blocks) 20.8 against
// 19.3, 1000^3 (16 K-blocks) 18.3 against 11.4.
bool sk_small(long long tiles, int clusters_max, long long num_kb) {
    return g_pair_sk && g_pdl && tiles > 0 && tiles * 4 <= clusters_max && num_kb >= 64;
}

// Launch with a stream-K tail when sk_worth: the last rem tiles' K iterations
// are spread over the G_sk = min(G, 4 rem) highest clusters,
// W = ceil(rem * KB / G_sk) each, instead of leaving G - rem clusters idle for
// a whole tile time; a tile then has at most ceil(KB / W) + 1 <= 5
// contributors.  Their partial slabs live in stream-ordered scratch, and
// pair_sk_fixup_kernel, next on the stream, adds them.  Without scratch (or
// allow_sk false) the tail runs as whole tiles.
template <typename T, uint32_t F, bool DUAL = false, bool F8 = false>
cudaError_t launch_pair_planned(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                                const CUtensorMap &tb2, PairArgs args, int clusters, long long tiles, bool allow_sk,
                                cudaStream_t s, int small_clusters = 0) {
    const long long num_kb = (args.K + (F8 ? 128 : BK) - 1) / (F8 ? 128 : BK);
    if (allow_sk && small_clusters > 0) {
        // every tile's K iterations in equal shares over 4 clusters per tile;
        // the fix-up kernel adds the partials
        const long long g_sk = std::min<long long>(small_clusters, 4 * tiles);
        const long long w = (tiles * num_kb + g_sk - 1) / g_sk;
        const size_t ws_bytes = (size_t)g_sk * 2 * 8 * 256 * 32 * sizeof(float);
        void *buf = nullptr;
        if (cudaMallocAsync(&buf, ws_bytes, s) == cudaSuccess) {
            args.sk_ws = static_cast<float *>(buf);
            args.sk_tiles = (int)tiles;
            args.sk_w = (int)w;
            args.sk_first = 0;
            cudaError_t e = launch_pair_cfg<T, F, DUAL, F8>(ta, tb, tc, tb2, args, (int)g_sk, s);
            if (e == cudaSuccess) {
                cudaLaunchAttribute fa[1];
                const cudaLaunchConfig_t fc =
                    pdl_config(dim3((unsigned)(2 * tiles), (unsigned)(args.bn / 8), 1), dim3(128), 0, s, fa);
                e = launch_counted(&fc, pair_sk_fixup_kernel<T, DUAL, F8>, static_cast<const PairArgs>(args),
                                   (int)num_kb);
            }
            const cudaError_t f = cudaFreeAsync(buf, s);
            return e != cudaSuccess ? e : f;
        }
        cudaGetLastError();
    }
    const long long rem = clusters > 0 ? tiles % clusters : 0;
    if (allow_sk && sk_worth(tiles, clusters, num_kb)) {
        const long long g_sk = std::min<long long>(clusters, 4 * rem);
        const long long w = (rem * num_kb + g_sk - 1) / g_sk;
        const size_t ws_bytes = (size_t)g_sk * 2 * 8 * 256 * 32 * sizeof(float);
        void *buf = nullptr;
        if (cudaMallocAsync(&buf, ws_bytes, s) == cudaSuccess) {
            args.sk_ws = static_cast<float *>(buf);
            args.sk_tiles = (int)rem;
            args.sk_w = (int)w;
            args.sk_first = clusters - (int)g_sk;
            cudaError_t e = launch_pair_cfg<T, F, DUAL, F8>(ta, tb, tc, tb2, args, clusters, s);
            if (e == cudaSuccess) {
                cudaLaunchAttribute fa[1];
                const cudaLaunchConfig_t fc =
                    pdl_config(dim3((unsigned)(2 * rem), (unsigned)(args.bn / 8), 1), dim3(128), 0, s, fa);
                e = launch_counted(&fc, pair_sk_fixup_kernel<T, DUAL, F8>, static_cast<const PairArgs>(args),
                                       (int)num_kb);
            }
            const cudaError_t f = cudaFreeAsync(buf, s);
            return e != cudaSuccess ? e : f;
        }
        cudaGetLastError();
    }
    return launch_pair_cfg<T, F, DUAL, F8>(ta, tb, tc, tb2, args, clusters, s);
}

// The general problem on CTA pairs.  Returns cudaErrorNotSupported, before any
// launch, when a tensor map cannot describe an operand.
template <typename T, uint32_t F>
cudaError_t launch_pair_typed(const ProblemEx &p, int clusters_max, int *status, cudaStream_t s,
                              bool allow_sk = true, int stall = 0) {
    const CUtensorMapDataType dt = F == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const long long ba = p.sa == 0 ? 1 : p.batch, bb = p.sb == 0 ? 1 : p.batch;
    CUtensorMap ta, tb, tc;
    const bool ok_a = p.a_t ? make_map3(&ta, p.A, dt, p.M, p.K, ba, p.lda, p.sa, 64, BK)
                            : make_map3(&ta, p.A, dt, p.K, p.M, ba, p.lda, p.sa, BK, 128);
    const bool ok_b = p.b_t ? make_map3(&tb, p.B, dt, p.K, p.N, bb, p.ldb, p.sb, BK, 128)
                            : make_map3(&tb, p.B, dt, p.N, p.K, bb, p.ldb, p.sb, 64, BK);
    const bool ok_c = make_map3(&tc, p.C, dt, p.N, p.M, p.batch, p.ldc, p.sc, 64, 32);
    if (!ok_a || !ok_b || !ok_c) return cudaErrorNotSupported;
    // N extent of a tile: 256 when a stream-K tail evens out the last wave;
    // otherwise the one of 256, 192, 128 (TMA-store boxes are 64 columns wide)
    // with the fewest waves of tiles over the clusters, widest on ties:
    // per-tile time is set mostly by the operand feed, which does not shrink
    // with the tile's N.
    const long long tiles_mb = (long long)((p.M + pairk::PBM - 1) / pairk::PBM) * p.batch;
    int bn = 256;
    const bool small = allow_sk && sk_small(tiles_mb * ((p.N + 255) / 256), clusters_max, (p.K + BK - 1) / BK);
    const bool sk_ok = small || (allow_sk && sk_worth(tiles_mb * ((p.N + 255) / 256), clusters_max,
                                                      (p.K + BK - 1) / BK));
    long long best = -1;
    for (int cand = 256; cand >= 128 && !sk_ok; cand -= 64) {
        const long long t = tiles_mb * ((p.N + cand - 1) / cand);
        const long long waves = (t + clusters_max - 1) / clusters_max;
        const long long cost = waves * (cand > 224 ? cand : 224);
        if (best < 0 || cost < best) { best = cost; bn = cand; }
    }
    // Under one wave even at 128 columns: the narrowest tiles, the most SMs
    // busy (measured back to back: bf16 1024^3 9.9 vs 10.2 us with 192-wide
    // tiles, 2048 x 1024 x 512 7.8 vs 8.2, 1000 x 1536 x 1000 10.0 vs 10.7).
    if (!sk_ok && tiles_mb * ((p.N + 127) / 128) <= clusters_max) bn = 128;
    const long long tiles = tiles_mb * ((p.N + bn - 1) / bn);
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const int clusters = (int)(tiles < clusters_max ? tiles : clusters_max);
    PairArgs args = {};
    args.C = p.C;
    args.ldc = p.ldc;
    args.stride_c = p.sc;
    args.M = p.M;
    args.N = p.N;
    args.K = p.K;
    args.batch = p.batch;
    args.bn = bn;
    args.a_t = p.a_t;
    args.b_t = p.b_t;
    args.a_bcast = p.sa == 0;
    args.b_bcast = p.sb == 0;
    args.alpha = p.alpha;
    args.beta = p.beta;
    args.status = status;
    args.stall = stall;
    if (stall) return launch_pair_cfg<T, F, false, false, false, true>(ta, tb, tc, tb, args, clusters, s);
    return launch_pair_planned<T, F>(ta, tb, tc, tb, args, clusters, tiles, allow_sk, s, small ? clusters_max : 0);
}

// Z = SiLU(X W_g) * (X W_u): p.A = X [M,K], p.B = W_g [K,N], p.C = Z [M,N];
// w_u = W_u [K,N].  256 x 128 tiles of Z on CTA pairs.
template <typename T, uint32_t F>
cudaError_t launch_pair_silu_mul_typed(const Problem &p, const void *w_u, int clusters_max, int *status,
                                       cudaStream_t s) {
    const CUtensorMapDataType dt = F == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap ta, tg, tu, tc;
    if (!make_map3(&ta, p.A, dt, p.K, p.M, 1, p.K, 0, BK, 128)) return cudaErrorInvalidValue;
    if (!make_map3(&tg, p.B, dt, p.N, p.K, 1, p.N, 0, 64, BK)) return cudaErrorInvalidValue;
    if (!make_map3(&tu, w_u, dt, p.N, p.K, 1, p.N, 0, 64, BK)) return cudaErrorInvalidValue;
    if (!make_map3(&tc, p.C, dt, p.N, p.M, 1, p.N, 0, 64, 32)) return cudaErrorInvalidValue;
    const int bn = 128;
    const long long tiles = (long long)((p.M + pairk::PBM - 1) / pairk::PBM) * ((p.N + bn - 1) / bn);
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const int clusters = (int)(tiles < clusters_max ? tiles : clusters_max);
    PairArgs args = {};
    args.C = p.C;
    args.ldc = p.N;
    args.M = p.M;
    args.N = p.N;
    args.K = p.K;
    args.batch = 1;
    args.bn = bn;
    args.alpha = 1.0f;
    args.status = status;
    return launch_pair_planned<T, F, true>(ta, tg, tc, tu, args, clusters, tiles, true, s);
}

// C [M,N] half = diag(scale) Q Wt^T on CTA pairs, Q [M,K] and Wt [N,K] E4M3.
cudaError_t launch_pair_e4m3(const void *Q, const float *scale, const void *Wt, void *C, int M, int N, int K,
                             int clusters_max, int *status, cudaStream_t s) {
    CUtensorMap ta, tb, tc;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_map3(&ta, Q, u8, K, M, 1, K, 0, 128, 128, 1) || !make_map3(&tb, Wt, u8, K, N, 1, K, 0, 128, 128, 1) ||
        !make_map3(&tc, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, N, M, 1, N, 0, 64, 32))
        return cudaErrorNotSupported;
    const long long tiles_m = (M + pairk::PBM - 1) / pairk::PBM;
    int bn = 256;
    const bool sk_ok = sk_worth(tiles_m * ((N + 255) / 256), clusters_max, (K + 127) / 128);
    long long best = -1;
    for (int cand = 256; cand >= 128 && !sk_ok; cand -= 64) {
        const long long t = tiles_m * ((N + cand - 1) / cand);
        const long long waves = (t + clusters_max - 1) / clusters_max;
        const long long cost = waves * (cand > 224 ? cand : 224);
        if (best < 0 || cost < best) { best = cost; bn = cand; }
    }
    const long long tiles = tiles_m * ((N + bn - 1) / bn);
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const int clusters = (int)(tiles < clusters_max ? tiles : clusters_max);
    PairArgs args = {};
    args.C = C;
    args.ldc = N;
    args.M = M;
    args.N = N;
    args.K = K;
    args.batch = 1;
    args.bn = bn;
    args.b_t = 1;
    args.alpha = 1.0f;
    args.row_scale = scale;
    args.status = status;
    return launch_pair_planned<__half, 0, false, true>(ta, tb, tc, tb, args, clusters, tiles, true, s);
}

// C [M,N] half = diag(amax / 448) E4M3(diag(448 / amax) A) Wt^T on CTA pairs,
// the quantisation of A [M,K] (half) done by the kernel's converter warps as
// each tile is loaded; amax [M] from launch_row_amax_f16.  Same tile plan as
// launch_pair_e4m3 without the stream-K tail.
cudaError_t launch_pair_e4m3_fused(const void *A, const float *amax, const void *Wt, void *C, int M, int N, int K,
                                   int clusters_max, int *status, cudaStream_t s) {
    CUtensorMap tb, tc;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_map3(&tb, Wt, u8, K, N, 1, K, 0, 128, 128, 1) ||
        !make_map3(&tc, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, N, M, 1, N, 0, 64, 32))
        return cudaErrorNotSupported;
    const long long tiles_m = (M + pairk::PBM - 1) / pairk::PBM;
    int bn = 256;
    long long best = -1;
    for (int cand = 256; cand >= 128; cand -= 64) {
        const long long t = tiles_m * ((N + cand - 1) / cand);
        const long long waves = (t + clusters_max - 1) / clusters_max;
        const long long cost = waves * (cand > 224 ? cand : 224);
        if (best < 0 || cost < best) { best = cost; bn = cand; }
    }
    const long long tiles = tiles_m * ((N + bn - 1) / bn);
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const int clusters = (int)(tiles < clusters_max ? tiles : clusters_max);
    PairArgs args = {};
    args.C = C;
    args.ldc = N;
    args.M = M;
    args.N = N;
    args.K = K;
    args.batch = 1;
    args.bn = bn;
    args.b_t = 1;
    args.alpha = 1.0f;
    args.row_scale = amax;
    args.a_src = A;
    args.status = status;
    return launch_pair_cfg<__half, 0, false, true, true>(tb, tb, tc, tb, args, clusters, s);
}

// The tight problem of the plain entry points as a general one; lda: row
// stride of A in elements (0: K).
ProblemEx plain_ex(const Problem &p, long long lda = 0) {
    ProblemEx q = {};
    q.A = p.A;
    q.B = p.B;
    q.C = p.C;
    q.M = p.M;
    q.N = p.N;
    q.K = p.K;
    q.batch = 1;
    q.lda = lda > 0 ? lda : p.K;
    q.ldb = p.N;
    q.ldc = p.N;
    q.alpha = 1.0f;
    q.beta = 0.0f;
    q.elt = p.elt;
    return q;
}

}  // namespace

namespace {
bool aligned(const void *q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; }
// TMA can describe A: 16-byte aligned base and row stride.
bool a_tma_ok(const Problem &p) { return aligned(p.A, 16) && (p.K % 8) == 0; }
// 8-byte cp.async can fetch A: 8-byte aligned base and row stride.
bool a_cpasync_ok(const Problem &p) { return aligned(p.A, 8) && (p.K % 4) == 0; }
}  // namespace

// Copies A [M, K] (rows 8-byte aligned, K % 4 == 0) into rows of lda elements
// (16-byte aligned), so that TMA can describe it.  Elements K..lda-1 of a row
// are left as they are: the tensor map declares K columns, so TMA never reads
// them.
__global__ void pad_rows_kernel(const uint2 *__restrict__ A, uint2 *__restrict__ Ap, long long rows,
                                long long chunks_per_row, long long lda_chunks) {
    const long long total = rows * chunks_per_row;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const long long r = i / chunks_per_row, c = i - r * chunks_per_row;
        Ap[r * lda_chunks + c] = __ldg(A + i);
    }
}

bool umma_supported(const Problem &p) {
    if (p.elt == Elt::F32) return false;
    // B through TMA (16-byte aligned base and row stride); C rows 16-byte
    // aligned for the vector epilogue stores; A through TMA or cp.async.
    return aligned(p.B, 16) && aligned(p.C, 16) && (p.N % 8) == 0 && (a_tma_ok(p) || a_cpasync_ok(p));
}

cudaError_t launch_umma(const Problem &p, int num_sms, int *status, cudaStream_t s, bool may_allocate) {
    if (!umma_supported(p)) return cudaErrorInvalidValue;
    if (!a_tma_ok(p)) {
        // Large problems: stage A once into 16-byte-aligned rows (stream-ordered
        // scratch from the device's default pool) and run the CTA-pair kernel;
        // the copy costs 4*M*K bytes of traffic against 2*M*N*K FLOPs.  If that
        // scratch is not available, or for small problems, A is fetched with
        // cp.async by the single-CTA kernel instead.
        if (may_allocate && p.M > BM && p.N >= 1024) {
            int dev = 0;
            cudaError_t e = cudaGetDevice(&dev);
            if (e != cudaSuccess) return e;
            const int cmax = p.elt == Elt::BF16 ? pair_clusters_max<__nv_bfloat16, 1>(dev)
                                                : pair_clusters_max<__half, 0>(dev);
            const long long lda = ((long long)p.K + 7) / 8 * 8;
            void *ap = nullptr;
            if (cmax > 0 && cudaMallocAsync(&ap, (size_t)p.M * lda * 2, s) == cudaSuccess) {
                const long long chunks = (long long)p.M * (p.K / 4);
                const int grid = (int)std::min<long long>((chunks + 255) / 256, (long long)num_sms * 16);
                note_launch();
                pad_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const uint2 *>(p.A), static_cast<uint2 *>(ap),
                                                     p.M, p.K / 4, lda / 4);
                e = cudaGetLastError();
                if (e == cudaSuccess) {
                    Problem q = p;
                    q.A = ap;
                    const ProblemEx qe = plain_ex(q, lda);
                    e = p.elt == Elt::BF16 ? launch_pair_typed<__nv_bfloat16, 1>(qe, cmax, status, s)
                                           : launch_pair_typed<__half, 0>(qe, cmax, status, s);
                }
                const cudaError_t f = cudaFreeAsync(ap, s);
                return e != cudaSuccess ? e : f;
            }
            cudaGetLastError();  // fall through to cp.async
        }
        return p.elt == Elt::BF16 ? launch_typed<__nv_bfloat16, 1, true>(p, num_sms, status, s)
                                  : launch_typed<__half, 0, true>(p, num_sms, status, s);
    }
    // Weights as the MMA's rows (umma_skinny_kernel): 128-column strips of C,
    // one CTA each, or clusters of cs CTAs splitting K when the strips alone
    // leave SMs idle -- the cs with the most CTAs, all of them resident at once.
    if (p.M <= 64 && g_umma_skinny) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const long long tiles_n = (p.N + 127) / 128;
        const long long num_kb = (p.K + SKB - 1) / SKB;
        if (tiles_n <= num_sms) {
            int cs = 1;
            for (int c = 2; c <= 8; ++c)
                if (c <= num_kb && tiles_n * c <= num_sms && skinny_clusters_max(p.elt, c, dev) >= tiles_n) cs = c;
            return p.elt == Elt::BF16 ? launch_skinny_typed<__nv_bfloat16, 1>(p, cs, num_sms, status, s)
                                      : launch_skinny_typed<__half, 0>(p, cs, num_sms, status, s);
        }
        // More 128-column strips than SMs: 256-column strips (skinny_wide.cu),
        // one CTA each while they fit on the SMs at once.  N = 28672, K = 4096,
        // back to back, W from DRAM: M = 1 / 8 / 32 / 64 at 37.9 / 38.6 / 39.6 /
        // 41.0 us, against 48.9 (the GEMV) / 57.4 / 38.7 / 39.7 for the
        // single-CTA 128 x 256 tiles.
        if ((p.N + 255) / 256 <= num_sms && skinny_wide_supported(p))
            return launch_skinny_wide(p, num_sms, status, s);
    }
    // 256-row tiles on CTA pairs once M fills more than one 128-row tile.
    if (p.M > BM) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const int cmax = p.elt == Elt::BF16 ? pair_clusters_max<__nv_bfloat16, 1>(dev)
                                            : pair_clusters_max<__half, 0>(dev);
        if (cmax > 0) {
            const ProblemEx q = plain_ex(p);
            return p.elt == Elt::BF16 ? launch_pair_typed<__nv_bfloat16, 1>(q, cmax, status, s, may_allocate)
                                      : launch_pair_typed<__half, 0>(q, cmax, status, s, may_allocate);
        }
    }
    if (p.elt == Elt::BF16) return launch_typed<__nv_bfloat16, 1, false>(p, num_sms, status, s);
    return launch_typed<__half, 0, false>(p, num_sms, status, s);
}

// ------------------------------------------------------- allocation-free variant
// Scratch of the allocation-free entry point (gemm_bf16_rm_noalloc).  The
// tensor-core kernel's only scratch is its 4-byte status word, in which a CTA
// records a pipeline timeout.  The regular entry points keep that word in
// memory the library cudaMallocs on first use of a device; this variant keeps
// it in the file-scope array below instead, so it never allocates.  Every GPU
// that loads the library holds these kNoallocScratchBytes until the process
// exits.  The word is zeroed once, at set-up; a timeout ORs a code into it,
// and it stays set until gemm_synchronize reads and clears it (so a timeout
// is reported even when further calls were queued after it).  All calls share
// the array: calls that overlap on the GPU share the word, and a timeout of
// either is reported to whichever thread synchronises first.
static __device__ __align__(256) int g_noalloc_scratch[kNoallocScratchBytes / sizeof(int)];

namespace {
struct NoallocScratch {
    std::once_flag once;
    std::atomic<bool> ready{false};
    int *ptr = nullptr;  // device address of g_noalloc_scratch on this device
    cudaError_t err = cudaSuccess;
};
NoallocScratch g_noalloc[kMaxDevices];
}  // namespace

size_t umma_noalloc_scratch_need(const Problem &) { return sizeof(int); }

cudaError_t launch_umma_noalloc(const Problem &p, int num_sms, cudaStream_t s, bool stall) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    NoallocScratch &d = g_noalloc[dev];
    // Set-up, once per device, with that device current: in host code the
    // array's name is only a host-side stand-in, so its device address is
    // looked up here and passed to the kernel; the status word is zeroed.
    std::call_once(d.once, [&] {
        d.err = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.ptr), g_noalloc_scratch);
        if (d.err == cudaSuccess) d.err = cudaMemset(d.ptr, 0, sizeof(int));
        if (d.err == cudaSuccess) d.ready.store(true, std::memory_order_release);
    });
    if (d.err != cudaSuccess) return d.err;
    if (umma_noalloc_scratch_need(p) > kNoallocScratchBytes) return cudaErrorInvalidValue;
    if (stall) return launch_umma_stall_test(p, num_sms, d.ptr, s);
    return launch_umma(p, num_sms, d.ptr, s, /*may_allocate=*/false);
}

cudaError_t take_noalloc_status(int dev, int *code) {
    *code = 0;
    if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
    NoallocScratch &d = g_noalloc[dev];
    if (!d.ready.load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaMemcpy(code, d.ptr, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && *code != 0) e = cudaMemset(d.ptr, 0, sizeof(int));
    return e;
}

bool umma_silu_mul_supported(const Problem &p, const void *w_u) {
    if (p.elt != Elt::BF16) return false;
    return aligned(p.A, 16) && aligned(p.B, 16) && aligned(w_u, 16) && aligned(p.C, 16) && (p.K % 8) == 0 &&
           (p.N % 8) == 0;
}

cudaError_t launch_umma_silu_mul(const Problem &p, const void *w_u, int *status, cudaStream_t s) {
    if (!umma_silu_mul_supported(p, w_u)) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int cmax = pair_clusters_max<__nv_bfloat16, 1, true>(dev);
    if (cmax <= 0) return cudaErrorNotSupported;
    return launch_pair_silu_mul_typed<__nv_bfloat16, 1>(p, w_u, cmax, status, s);
}

bool umma_ex_supported(const ProblemEx &p) {
    if (p.elt == Elt::F32) return false;
    if (!aligned(p.A, 16) || !aligned(p.B, 16) || !aligned(p.C, 16)) return false;
    if (p.lda % 8 || p.ldb % 8 || p.ldc % 8) return false;
    if (p.batch > 1 && (p.sa % 8 || p.sb % 8 || p.sc % 8)) return false;
    // TMA moves the contiguous dimension in 16-byte pieces: each stored
    // matrix's contiguous extent must be a whole number of them, or a store
    // would touch elements past the end of a row of C.
    if ((p.a_t ? p.M : p.K) % 8 || (p.b_t ? p.K : p.N) % 8 || p.N % 8) return false;
    return true;
}

cudaError_t launch_umma_ex(const ProblemEx &p, int *status, cudaStream_t s) {
    if (!umma_ex_supported(p)) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int cmax = p.elt == Elt::BF16 ? pair_clusters_max<__nv_bfloat16, 1>(dev)
                                        : pair_clusters_max<__half, 0>(dev);
    if (cmax <= 0) return cudaErrorNotSupported;
    return p.elt == Elt::BF16 ? launch_pair_typed<__nv_bfloat16, 1>(p, cmax, status, s)
                              : launch_pair_typed<__half, 0>(p, cmax, status, s);
}

bool umma_e4m3_supported(const void *Q, const void *Wt, const void *C, int N, int K) {
    return aligned(Q, 16) && aligned(Wt, 16) && aligned(C, 16) && (K % 16) == 0 && (N % 8) == 0;
}

cudaError_t launch_umma_e4m3_rowscale(const void *Q, const float *scale, const void *Wt, void *C, int M, int N,
                                      int K, int *status, cudaStream_t s) {
    if (!umma_e4m3_supported(Q, Wt, C, N, K)) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int cmax = pair_clusters_max<__half, 0, false, true>(dev);
    if (cmax <= 0) return cudaErrorNotSupported;
    return launch_pair_e4m3(Q, scale, Wt, C, M, N, K, cmax, status, s);
}

cudaError_t launch_umma_pair_stall_test(const Problem &p, int mode, int *status, cudaStream_t s) {
    if (mode != 1 && mode != 2) return cudaErrorInvalidValue;
    if (!umma_supported(p) || !a_tma_ok(p) || p.M <= BM) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // (the test instance: its shared-memory attribute is set by this query)
    const int cmax = p.elt == Elt::BF16 ? pair_clusters_max<__nv_bfloat16, 1, false, false, false, true>(dev)
                                        : pair_clusters_max<__half, 0, false, false, false, true>(dev);
    if (cmax <= 0) return cudaErrorNotSupported;
    const ProblemEx q = plain_ex(p);
    return p.elt == Elt::BF16 ? launch_pair_typed<__nv_bfloat16, 1>(q, cmax, status, s, false, mode)
                              : launch_pair_typed<__half, 0>(q, cmax, status, s, false, mode);
}

bool umma_e4m3_fused_supported(const void *A, const void *Wt, const void *C, int N, int K) {
    return aligned(A, 16) && umma_e4m3_supported(A, Wt, C, N, K);
}

cudaError_t launch_umma_e4m3_fused(const void *A, const void *Wt, void *C, int M, int N, int K, int *status,
                                   cudaStream_t s) {
    if (!umma_e4m3_fused_supported(A, Wt, C, N, K)) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int cmax = pair_clusters_max<__half, 0, false, true, true>(dev);
    if (cmax <= 0) return cudaErrorNotSupported;
    // the rows' amax, in stream-ordered scratch for the duration of the call
    void *amax = nullptr;
    e = cudaMallocAsync(&amax, (size_t)M * sizeof(float), s);
    if (e != cudaSuccess) return e;
    e = launch_row_amax_f16(A, static_cast<float *>(amax), M, K, s);
    if (e == cudaSuccess)
        e = launch_pair_e4m3_fused(A, static_cast<const float *>(amax), Wt, C, M, N, K, cmax, status, s);
    const cudaError_t f = cudaFreeAsync(amax, s);
    return e != cudaSuccess ? e : f;
}

cudaError_t launch_umma_stall_test(const Problem &p, int num_sms, int *status, cudaStream_t s) {
    if (!umma_supported(p) || !a_tma_ok(p)) return cudaErrorInvalidValue;
    if (p.elt == Elt::BF16) return launch_typed<__nv_bfloat16, 1, false>(p, num_sms, status, s, 1);
    return launch_typed<__half, 0, false>(p, num_sms, status, s, 1);
}

}  // namespace gemm_gb300
