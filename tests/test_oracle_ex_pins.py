"""Pins of the oracle's general form C_b <- alpha op(A_b) op(B_b) + beta C_b
("SGEMM measured and the three ledgers", section 2: operation flags, leading
dimensions and the row-/column-major reading of the same bytes; section 3,
kernel K1: alpha * acc + beta * C).

The storage buffers here are built from logical matrices by numpy slicing
(placing op(X)'s stored form inside a padded buffer), and the expected values
are exact integer products of the logical matrices -- neither goes through the
oracle's index arithmetic.  Padding holds NaN, so an index that strays into it
shows up."""

import numpy as np
import pytest

import oracle
from oracle import compare

NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}


def encode(dtype, values):
    v = np.asarray(values, dtype=np.float32)
    if dtype == "f32":
        return v
    if dtype == "f16":
        out = v.astype(np.float16)
        assert np.array_equal(out.astype(np.float32), v)
        return out.view(np.uint16)
    b = v.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def build(dtype, layout, op, mats, ld, stride):
    """Flat buffer holding, for each b, the stored form of mats[b] (mats[b] itself
    for op 'N', its transpose for 'T') at offset b*stride with leading dimension
    ld; every other element is NaN."""
    stored = [m if op == "N" else m.T for m in mats]
    R, Cc = stored[0].shape
    inner, outer = (Cc, R) if layout == "rm" else (R, Cc)
    size = max(1, (len(mats) - 1) * stride + outer * ld)
    if dtype == "f32":
        buf = np.full(size, np.nan, dtype=np.float32)
    else:
        buf = np.full(size, NAN_BITS[dtype], dtype=np.uint16)
    for b, s in enumerate(stored):
        view = buf[b * stride: b * stride + outer * ld].reshape(outer, ld)[:, :inner]
        view[...] = encode(dtype, s if layout == "rm" else s.T)
    return buf


COMBOS = [(d, l, oa, ob) for d in ("f32", "f16", "bf16") for l in ("rm", "cm")
          for oa in "NT" for ob in "NT"]


@pytest.mark.parametrize("dtype,layout,op_a,op_b", COMBOS)
def test_ex_bruteforce_integers(dtype, layout, op_a, op_b):
    rng = np.random.default_rng(COMBOS.index((dtype, layout, op_a, op_b)))
    M, N, K, batch = 5, 4, 6, 3
    alpha, beta = 2.0, -3.0
    A = [rng.integers(-4, 5, (M, K)).astype(np.float64) for _ in range(batch)]
    B = [rng.integers(-4, 5, (K, N)).astype(np.float64) for _ in range(batch)]
    C = [rng.integers(-4, 5, (M, N)).astype(np.float64) for _ in range(batch)]
    ra, rb = (M, K) if op_a == "N" else (K, M), (K, N) if op_b == "N" else (N, K)
    lda = (ra[1] if layout == "rm" else ra[0]) + 3
    ldb = (rb[1] if layout == "rm" else rb[0]) + 2
    ldc = (N if layout == "rm" else M) + 1
    outer = lambda r, ld, lay: (r[0] if lay == "rm" else r[1]) * ld
    sa, sb, sc = outer(ra, lda, layout) + 5, outer(rb, ldb, layout) + 7, outer((M, N), ldc, layout) + 2
    bufA = build(dtype, layout, op_a, A, lda, sa)
    bufB = build(dtype, layout, op_b, B, ldb, sb)
    bufC = build(dtype, layout, "N", C, ldc, sc)
    r = oracle.gemm_ex(dtype, layout, op_a, op_b, M, N, K, alpha, bufA, lda, sa, bufB, ldb, sb,
                       beta, bufC, ldc, sc, batch)
    for b in range(batch):
        P = A[b] @ B[b]
        assert np.array_equal(r["P"][b], P)
        assert np.array_equal(r["S"][b], np.abs(A[b]) @ np.abs(B[b]))
        assert np.array_equal(r["BC"][b], beta * C[b])
        assert np.array_equal(r["C"][b], alpha * P + beta * C[b])


@pytest.mark.parametrize("variant", ["f32_rm", "f16_cm", "bf16_rm", "bf16_cm"])
def test_ex_plain_case_is_the_plain_product(variant):
    dtype, layout = variant.split("_")
    rng = np.random.default_rng(7)
    M, N, K = 9, 7, 33
    A = encode(dtype, rng.integers(-64, 65, M * K) / 32.0)
    B = encode(dtype, rng.integers(-64, 65, K * N) / 16.0)
    C_ref, S = oracle.gemm(variant, A, B, M, N, K)
    ld_a = K if layout == "rm" else M
    ld_b = N if layout == "rm" else K
    ld_c = N if layout == "rm" else M
    r = oracle.gemm_ex(dtype, layout, "N", "N", M, N, K, 1.0, A, ld_a, 0, B, ld_b, 0, 0.0, None, ld_c, 0)
    assert np.array_equal(r["C"][0], C_ref)
    assert np.array_equal(r["S"][0], S)


@pytest.mark.parametrize("op_a,op_b", [("N", "N"), ("T", "N"), ("N", "T"), ("T", "T")])
def test_ex_column_major_is_row_major_of_the_transpose(op_a, op_b):
    """The page's identity: the column-major C = op(A) op(B) written into a buffer
    is the row-major C^T = op(B)^T op(A)^T, with the operands' roles swapped."""
    rng = np.random.default_rng(11)
    M, N, K = 6, 5, 7
    lda = (M if op_a == "N" else K) + 2
    ldb = (K if op_b == "N" else N) + 1
    A = rng.standard_normal(lda * (K if op_a == "N" else M)).astype(np.float32)
    B = rng.standard_normal(ldb * (N if op_b == "N" else K)).astype(np.float32)
    cm = oracle.gemm_ex("f32", "cm", op_a, op_b, M, N, K, 1.5, A, lda, 0, B, ldb, 0, 0.0, None, M, 0)
    rm = oracle.gemm_ex("f32", "rm", op_b, op_a, N, M, K, 1.5, B, ldb, 0, A, lda, 0, 0.0, None, N, 0)
    assert np.array_equal(cm["C"][0], rm["C"][0].T)


def test_ex_beta_zero_and_alpha_zero_read_nothing():
    M, N, K = 3, 4, 5
    nanA = np.full(M * K, np.nan, dtype=np.float32)
    nanB = np.full(K * N, np.nan, dtype=np.float32)
    nanC = np.full(M * N, np.nan, dtype=np.float32)
    ones_a = np.ones(M * K, dtype=np.float32)
    ones_b = np.ones(K * N, dtype=np.float32)
    r = oracle.gemm_ex("f32", "rm", "N", "N", M, N, K, 1.0, ones_a, K, 0, ones_b, N, 0, 0.0, nanC, N, 0)
    assert np.array_equal(r["C"][0], np.full((M, N), float(K)))
    C = np.arange(M * N, dtype=np.float32)
    r = oracle.gemm_ex("f32", "rm", "N", "N", M, N, K, 0.0, nanA, K, 0, nanB, N, 0, 2.0, C, N, 0)
    assert np.array_equal(r["C"][0], 2.0 * C.reshape(M, N))
    r = oracle.gemm_ex("f32", "rm", "N", "N", M, N, 0, 1.0, nanA, 1, 0, nanB, N, 0, -1.0, C, N, 0)
    assert np.array_equal(r["C"][0], -C.reshape(M, N))


def test_ex_stride_zero_reuses_one_matrix():
    rng = np.random.default_rng(3)
    M, N, K, batch = 4, 3, 5, 4
    A = rng.integers(-3, 4, M * K).astype(np.float32)
    B = rng.integers(-3, 4, batch * K * N).astype(np.float32)
    r = oracle.gemm_ex("f32", "rm", "N", "N", M, N, K, 1.0, A, K, 0, B, N, K * N, 0.0, None, N, M * N, batch)
    for b in range(batch):
        assert np.array_equal(r["C"][b], A.reshape(M, K).astype(np.float64)
                              @ B[b * K * N:(b + 1) * K * N].reshape(K, N))


def test_ex_rejects_out_of_range_storage():
    A = np.zeros(12, dtype=np.float32)
    with pytest.raises(ValueError):   # lda below the row length
        oracle.gemm_ex("f32", "rm", "N", "N", 3, 4, 4, 1.0, A, 3, 0, A, 4, 0, 0.0, None, 4, 0)
    with pytest.raises(ValueError):   # the second batch matrix runs past the buffer
        oracle.gemm_ex("f32", "rm", "N", "N", 3, 4, 4, 1.0, A, 4, 12, A, 4, 0, 0.0, None, 4, 0, 2)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_ex_tolerance_admits_exact_rounding_and_rejects_a_step(dtype):
    """The exactly rounded result passes; a result moved by a few output steps
    (or by far more than the FP32 allowance) fails."""
    rng = np.random.default_rng(5)
    M, N, K = 16, 16, 1024
    mk = lambda n: encode(dtype, (rng.integers(-128, 129, n) / 128.0).astype(np.float32))
    A, B, C = mk(M * K), mk(K * N), mk(M * N)
    variant = dtype + "_rm"
    r = oracle.gemm_ex(dtype, "rm", "N", "N", M, N, K, 0.75, A, K, 0, B, N, 0, -0.5, C, N, 0)
    exact = compare.round_to(variant, r["C"])
    assert compare.check_ex(variant, exact, r, K, 0.75)["ok"]
    if dtype == "f32":
        moved = r["C"] + 1e-4 * r["S"] + 1.0
    else:
        moved = r["C"] + 8 * compare.ulp_out(dtype, r["C"]) + 0.1 * np.sqrt(K / 512.0) * np.maximum(1, np.abs(r["C"]))
    assert not compare.check_ex(variant, moved, r, K, 0.75)["ok"]
