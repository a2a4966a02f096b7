"""Parity of the general form C_b = alpha op(A_b) op(B_b) + beta C_b (gemm_ex)
with the oracle, through the C ABI, on the tensor-core CTA pairs (16-bit,
TMA-describable strides) and the SIMT kernel (FP32, and 16-bit with strides TMA
cannot describe).

Every matrix lives in a larger buffer with padded leading dimensions and batch
strides; the padding holds NaN, so a kernel that reads outside a matrix makes a
NaN result, and one that writes outside C changes padding bytes that the tests
check are untouched."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu

NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}
SEED = 0xE0  # seed block of these problems


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def padded(dtype, outer, inner, ld, stride, batch, seed, fill=True):
    """Flat buffer of `batch` stored matrices [outer, inner] (leading dimension
    ld, matrix stride `stride`) with seeded uniform[-1,1] values; NaN elsewhere."""
    size = max(1, (batch - 1) * stride + outer * ld)
    if dtype == "f32":
        buf = np.full(size, np.nan, dtype=np.float32)
    else:
        buf = np.full(size, NAN_BITS[dtype], dtype=np.uint16)
    if fill:
        for b in range(batch if stride > 0 else 1):
            buf[b * stride: b * stride + outer * ld].reshape(outer, ld)[:, :inner] = \
                synthetic.matrix(dtype, outer, inner, seed + b).reshape(outer, inner)
    return buf


def widen(dtype, bits):
    if dtype == "f32":
        return bits.astype(np.float64)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dev(buf):
    return torch.from_numpy(buf if buf.dtype == np.float32 else buf.view(np.int16)).cuda()


def host(t, dtype):
    h = t.cpu().numpy()
    return h if dtype == "f32" else h.view(np.uint16)


def run_ex(dtype, layout, op_a, op_b, M, N, K, alpha, beta, batch=1, pad=8, sa=None, sb=None,
           force=None, c_fill=True, seed=0):
    """Builds padded operands, runs gemm_ex and the oracle; returns (C_gpu
    [batch,M,N] float64, oracle dict, kernel name, C buffer before/after)."""
    a_r, a_c = (M, K) if op_a == "N" else (K, M)
    b_r, b_c = (K, N) if op_b == "N" else (N, K)
    # (outer, inner) of each stored matrix in memory order
    oi = (lambda r, c: (r, c)) if layout == "rm" else (lambda r, c: (c, r))
    (ao, ai), (bo, bi), (co, ci) = oi(a_r, a_c), oi(b_r, b_c), oi(M, N)
    # pad a multiple of 8: leading dimensions rounded up to multiples of 8 (16
    # bytes for 16-bit elements), as the tensor-core path needs
    up = (lambda x: (x + 7) // 8 * 8) if pad % 8 == 0 else (lambda x: x)
    lda, ldb, ldc = up(ai) + pad, up(bi) + pad, up(ci) + pad
    sa = ao * lda + 16 if sa is None else sa
    sb = bo * ldb + 24 if sb is None else sb
    sc = co * ldc + 8
    s0 = synthetic.seed_for(SEED, 0) + 1000 * seed
    A = padded(dtype, ao, ai, lda, sa, batch, s0 + 100)
    B = padded(dtype, bo, bi, ldb, sb, batch, s0 + 200)
    C0 = padded(dtype, co, ci, ldc, sc, batch, s0 + 300, fill=c_fill)
    dA, dB, dC = dev(A), dev(B), dev(C0.copy())
    g.gemm_force_kernel(force)
    try:
        g.gemm_ex(dtype, layout, op_a, op_b, M, N, K, alpha, dA, lda, sa, dB, ldb, sb, beta, dC, ldc, sc,
                  batch)
        name = g.gemm_last_kernel()
    finally:
        g.gemm_force_kernel(None)
    g.gemm_synchronize()
    torch.cuda.synchronize()
    C1 = host(dC, dtype)
    ref = oracle.gemm_ex(dtype, layout, op_a, op_b, M, N, K, alpha, A, lda, sa, B, ldb, sb, beta, C0, ldc,
                         sc, batch)
    out = np.empty((batch, M, N))
    for b in range(batch):
        m = widen(dtype, C1[b * sc: b * sc + co * ldc].reshape(co, ldc)[:, :ci])
        out[b] = m if layout == "rm" else m.T
    # padding of C untouched: every element outside the matrices keeps its bits
    mask = np.ones(C1.size, dtype=bool)
    for b in range(batch):
        mask[b * sc: b * sc + co * ldc].reshape(co, ldc)[:, :ci] = False
    assert np.array_equal(C1[mask].view(np.uint8) if dtype != "f32" else C1[mask].view(np.uint32),
                          C0[mask].view(np.uint8) if dtype != "f32" else C0[mask].view(np.uint32))
    return out, ref, name


def check(dtype, out, ref, K, alpha):
    res = compare.check_ex(dtype + "_rm", out, ref, K, alpha)
    assert res["ok"], res


COMBOS = [(d, l, oa, ob) for d in ("f32", "f16", "bf16") for l in ("rm", "cm")
          for oa in "NT" for ob in "NT"]


@pytest.mark.parametrize("dtype,layout,op_a,op_b", COMBOS)
def test_every_layout_and_operation(dtype, layout, op_a, op_b):
    """Several tiles and a ragged edge in M and N (multiples of 8, so that the
    16-bit problems qualify for the tensor cores)."""
    M, N, K = 296, 200, 136
    out, ref, name = run_ex(dtype, layout, op_a, op_b, M, N, K, 0.75, -0.5, batch=2,
                            seed=COMBOS.index((dtype, layout, op_a, op_b)))
    assert name == ("simt_ex_f32_vec4" if dtype == "f32" else f"umma_ex_{dtype}")
    check(dtype, out, ref, K, 0.75)


@pytest.mark.parametrize("dtype,layout,op_a,op_b", [(d, l, oa, ob) for d in ("f16", "bf16")
                                                    for l in ("rm", "cm") for oa in "NT" for ob in "NT"])
def test_extents_not_multiple_of_8_use_the_simt_kernel(dtype, layout, op_a, op_b):
    """M = 300 and N = 203: some stored matrix's contiguous extent is not a
    whole number of 16-byte pieces, which the tensor-core path refuses."""
    M, N, K = 300, 203, 136
    out, ref, name = run_ex(dtype, layout, op_a, op_b, M, N, K, 0.75, -0.5, batch=2)
    assert name == f"simt_ex_{dtype}"
    check(dtype, out, ref, K, 0.75)


@pytest.mark.parametrize("dtype,layout,op_a,op_b", [("f16", "rm", "T", "N"), ("bf16", "cm", "N", "T"),
                                                    ("f32", "rm", "T", "T"), ("bf16", "rm", "N", "N")])
def test_unaligned_leading_dimensions_use_the_simt_kernel(dtype, layout, op_a, op_b):
    M, N, K = 150, 130, 70
    out, ref, name = run_ex(dtype, layout, op_a, op_b, M, N, K, 1.25, 0.5, batch=2, pad=3)
    assert name.startswith("simt_ex_")
    check(dtype, out, ref, K, 1.25)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op_a,op_b", [("N", "T"), ("T", "N")])
def test_forced_simt_on_tensor_core_shapes(dtype, op_a, op_b):
    M, N, K = 260, 136, 72
    out, ref, name = run_ex(dtype, "rm", op_a, op_b, M, N, K, -1.0, 2.0, batch=2, force="simt")
    assert name == f"simt_ex_{dtype}"
    check(dtype, out, ref, K, -1.0)


@pytest.mark.parametrize("dtype,force", [("f32", None), ("bf16", None), ("bf16", "simt")])
def test_beta_zero_never_reads_C(dtype, force):
    """C holds NaN everywhere; with beta == 0 none of it may reach the result."""
    M, N, K = 200, 136, 64
    out, ref, name = run_ex(dtype, "rm", "N", "T", M, N, K, 1.0, 0.0, batch=2, force=force, c_fill=False)
    assert np.isfinite(out).all()
    check(dtype, out, ref, K, 1.0)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("alpha,K", [(0.0, 64), (1.0, 0)])
def test_no_product_term_scales_C(dtype, alpha, K):
    M, N = 70, 90
    out, ref, name = run_ex(dtype, "cm", "T", "N", M, N, K, alpha, -2.0, batch=3)
    assert name == "scale_c"
    check(dtype, out, ref, K, alpha)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_batch_stride_zero_shares_one_operand(dtype):
    """One weight matrix B for every batch entry (stride 0), as in a shared
    projection X_b W^T."""
    M, N, K = 192, 256, 128
    out, ref, name = run_ex(dtype, "rm", "N", "T", M, N, K, 1.0, 0.0, batch=3, sb=0)
    check(dtype, out, ref, K, 1.0)
    assert name == ("simt_ex_f32_vec4" if dtype == "f32" else "umma_ex_bf16")


def test_many_small_batch_entries():
    M, N, K = 64, 64, 64
    out, ref, name = run_ex("bf16", "rm", "T", "T", M, N, K, 0.5, 1.0, batch=40)
    assert name == "umma_ex_bf16"
    check("bf16", out, ref, K, 0.5)


def test_batch_count_beyond_one_grid_dimension():
    """More batch entries than one launch's grid.y holds (65535)."""
    M, N, K, batch = 2, 3, 4, 70000
    out, ref, name = run_ex("f32", "rm", "N", "N", M, N, K, 1.0, 1.0, batch=batch, pad=0)
    assert name.startswith("simt_ex_f32")
    check("f32", out, ref, K, 1.0)


@pytest.mark.parametrize("M", [1, 100, 128])
def test_short_M_on_the_pairs(M):
    N, K = 264, 72
    out, ref, name = run_ex("f16", "rm", "N", "N", M, N, K, 1.0, 0.25)
    assert name == "umma_ex_f16"
    check("f16", out, ref, K, 1.0)


def test_linear_layer_shape_X_times_W_transposed():
    """X [M,K] times W^T with W stored [N,K] (a linear layer's weight layout),
    several tiles in each direction and a ragged N."""
    M, N, K = 1024, 1544, 1024
    out, ref, name = run_ex("bf16", "rm", "N", "T", M, N, K, 1.0, 0.0, pad=0)
    assert name == "umma_ex_bf16"
    check("bf16", out, ref, K, 1.0)


def test_plain_case_matches_the_plain_entry_point():
    """alpha = 1, beta = 0, no transposes, tight strides: gemm_ex and
    gemm_bf16_rm run the same kernel and give the same bits."""
    M, N, K = 512, 768, 256
    A, B = synthetic.problem_inputs("bf16_rm", M, N, K, SEED)
    dA, dB = dev(A), dev(B)
    c1 = torch.empty(M * N, dtype=torch.int16, device="cuda")
    c2 = torch.empty(M * N, dtype=torch.int16, device="cuda")
    g.gemm_bf16_rm(dA, dB, c1, M, N, K)
    g.gemm_ex("bf16", "rm", "N", "N", M, N, K, 1.0, dA, K, 0, dB, N, 0, 0.0, c2, N, 0, 1)
    g.gemm_synchronize()
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_overlapping_batches_of_A(dtype):
    """Batch strides smaller than a matrix (a sliding window over A's rows) are
    legal for the operands that are only read."""
    M, N, K, batch = 136, 200, 64, 3
    lda = K
    sa = 8 * lda                     # each A_b starts 8 rows after A_{b-1}
    A = synthetic.matrix(dtype, M + 8 * (batch - 1), K, synthetic.seed_for(SEED, 40))
    B = synthetic.matrix(dtype, batch * K, N, synthetic.seed_for(SEED, 41))
    C0 = np.zeros(batch * M * N, dtype=np.float32 if dtype == "f32" else np.uint16)
    dA, dB, dC = dev(A), dev(B), dev(C0)
    g.gemm_ex(dtype, "rm", "N", "N", M, N, K, 1.0, dA, lda, sa, dB, N, K * N, 0.0, dC, N, M * N, batch)
    g.gemm_synchronize()
    out = widen(dtype, host(dC, dtype)).reshape(batch, M, N)
    ref = oracle.gemm_ex(dtype, "rm", "N", "N", M, N, K, 1.0, A, lda, sa, B, N, K * N, 0.0, None, N, M * N, batch)
    check(dtype, out, ref, K, 1.0)


def test_column_major_batched_half_sampled():
    """Column-major f16, A transposed, 16 batch entries of 512 x 768 x 1024 on
    the tensor cores; every output of entries 0 and 15 against the oracle."""
    M, N, K, batch = 512, 768, 1024, 16
    A = synthetic.matrix("f16", batch * M, K, synthetic.seed_for(SEED, 42))    # A_b^T stored [K, M] col-major
    B = synthetic.matrix("f16", batch * K, N, synthetic.seed_for(SEED, 43))
    C0 = np.zeros(batch * M * N, dtype=np.uint16)
    dA, dB, dC = dev(A), dev(B), dev(C0)
    # column-major: A stored K x M (op T) with lda = K, B stored K x N with ldb = K, C M x N with ldc = M
    g.gemm_ex("f16", "cm", "T", "N", M, N, K, 1.0, dA, K, M * K, dB, K, K * N, 0.0, dC, M, M * N, batch)
    assert g.gemm_last_kernel() == "umma_ex_f16"
    g.gemm_synchronize()
    out = widen("f16", host(dC, "f16"))
    for b in (0, batch - 1):
        ref = oracle.gemm_ex("f16", "cm", "T", "N", M, N, K, 1.0, A[b * M * K:(b + 1) * M * K], K, 0,
                             B[b * K * N:(b + 1) * K * N], K, 0, 0.0, None, M, 0, 1)
        got = out[b * M * N:(b + 1) * M * N].reshape(N, M).T[None]
        check("f16", got, ref, K, 1.0)


@pytest.mark.parametrize("dtype,op_a,op_b", [("bf16", "N", "T"), ("f16", "T", "N")])
def test_stream_k_tail_batched_alpha_beta(dtype, op_a, op_b):
    """Five batches of 256 x 4096 x 3072 make 80 pair tiles: the 4-6 tiles past
    a full wave (all in the last batch) are summed from stream-K partials, and
    alpha and beta * old C are applied once, after the sum.  The last batch is
    checked whole against the oracle."""
    M, N, K, batch, alpha, beta = 256, 4096, 3072, 5, 0.5, -1.25
    a_r, a_c = (M, K) if op_a == "N" else (K, M)
    b_r, b_c = (K, N) if op_b == "N" else (N, K)
    lda, ldb, ldc = a_c + 8, b_c + 16, N + 8
    sa, sb, sc = a_r * lda + 64, b_r * ldb + 32, M * ldc + 8
    s0 = synthetic.seed_for(SEED, 0) + 7000
    A = padded(dtype, a_r, a_c, lda, sa, batch, s0 + 100)
    B = padded(dtype, b_r, b_c, ldb, sb, batch, s0 + 200)
    C0 = padded(dtype, M, N, ldc, sc, batch, s0 + 300)
    dA, dB, dC = dev(A), dev(B), dev(C0.copy())
    g.gemm_ex(dtype, "rm", op_a, op_b, M, N, K, alpha, dA, lda, sa, dB, ldb, sb, beta, dC, ldc, sc, batch)
    assert g.gemm_last_kernel() == f"umma_ex_{dtype}"
    g.gemm_synchronize()
    C1 = host(dC, dtype)
    for b in (batch - 1,):
        ref = oracle.gemm_ex(dtype, "rm", op_a, op_b, M, N, K, alpha, A[b * sa:], lda, 0, B[b * sb:], ldb, 0,
                             beta, C0[b * sc:], ldc, 0, 1)
        out = widen(dtype, C1[b * sc: b * sc + M * ldc].reshape(M, ldc)[:, :N])[None]
        check(dtype, out, ref, K, alpha)

@pytest.mark.parametrize("dtype,op_a,op_b", [("bf16", "N", "N"), ("f16", "T", "T")])
def test_small_long_k_split_batched_alpha_beta(dtype, op_a, op_b):
    """Two batches of 304 x 264 x 4160 make 8 pair tiles of 65 K-blocks: every
    tile runs as stream-K over four clusters, and alpha and beta * old C are
    applied once, after the partials are added.  Both batches and the padding
    are checked."""
    M, N, K, batch, alpha, beta = 304, 264, 4160, 2, 0.5, -1.25
    a_r, a_c = (M, K) if op_a == "N" else (K, M)
    b_r, b_c = (K, N) if op_b == "N" else (N, K)
    lda, ldb, ldc = a_c + 8, b_c + 16, N + 8
    sa, sb, sc = a_r * lda + 64, b_r * ldb + 32, M * ldc + 8
    s0 = synthetic.seed_for(SEED, 0) + 8000
    A = padded(dtype, a_r, a_c, lda, sa, batch, s0 + 100)
    B = padded(dtype, b_r, b_c, ldb, sb, batch, s0 + 200)
    C0 = padded(dtype, M, N, ldc, sc, batch, s0 + 300)
    dA, dB, dC = dev(A), dev(B), dev(C0.copy())
    launches = g.gemm_kernel_launches()
    g.gemm_ex(dtype, "rm", op_a, op_b, M, N, K, alpha, dA, lda, sa, dB, ldb, sb, beta, dC, ldc, sc, batch)
    assert g.gemm_last_kernel() == f"umma_ex_{dtype}"
    assert g.gemm_kernel_launches() - launches == 2  # the pair kernel and the fix-up
    g.gemm_synchronize()
    C1 = host(dC, dtype)
    for b in range(batch):
        ref = oracle.gemm_ex(dtype, "rm", op_a, op_b, M, N, K, alpha, A[b * sa:], lda, 0, B[b * sb:], ldb, 0,
                             beta, C0[b * sc:], ldc, 0, 1)
        out = widen(dtype, C1[b * sc: b * sc + M * ldc].reshape(M, ldc)[:, :N])[None]
        check(dtype, out, ref, K, alpha)
        # the padding columns of C are left as they were
        pad = C1[b * sc: b * sc + M * ldc].reshape(M, ldc)[:, N:]
        assert np.array_equal(pad, C0[b * sc: b * sc + M * ldc].reshape(M, ldc)[:, N:])
