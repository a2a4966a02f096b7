"""Pins of the CPU oracle against facts other than itself (no GPU needed).

Each check would fail for a plausible mistake in the oracle: brute force on
small integers and dyadic fractions (exact rational arithmetic in Python) catches
a dropped term, a wrong sign, a swapped index or a transposed operand; the
closed forms ones*ones = K and I*B = B pin the accumulation and the indexing of
B; the transpose identity ties the column-major indexing to the row-major one
("SGEMM measured and the three ledgers", section 2); the decoders are checked
exhaustively against IEEE conversions done by numpy; a float64 library matmul on
the decoded inputs checks random problems of moderate size.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import compare

VARIANTS = [f"{d}_{l}" for d in ("f32", "f16", "bf16") for l in ("rm", "cm")]


def encode(dtype, values):
    """Exact encoding of small dyadic values (representable in every type used)."""
    v = np.asarray(values, dtype=np.float32).reshape(-1)
    if dtype == "f32":
        return v
    if dtype == "f16":
        out = v.astype(np.float16)
        assert np.array_equal(out.astype(np.float32), v), "value not exact in half"
        return out.view(np.uint16)
    b = v.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def store(layout, mat):
    """Flat storage buffer of a logical 2-D matrix in the given layout."""
    mat = np.asarray(mat)
    return mat.reshape(-1) if layout == "rm" else mat.T.reshape(-1)


def exact_product(a, b):
    """Brute force in exact rationals: returns (C, S) as nested lists of Fractions."""
    M, K = len(a), len(a[0]) if a else 0
    N = len(b[0]) if b else 0
    C = [[sum((Fraction(a[i][k]) * Fraction(b[k][j]) for k in range(K)), Fraction(0))
          for j in range(N)] for i in range(M)]
    S = [[sum((abs(Fraction(a[i][k]) * Fraction(b[k][j])) for k in range(K)), Fraction(0))
          for j in range(N)] for i in range(M)]
    return C, S


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 4), (7, 5, 3), (5, 9, 16), (3, 1, 64), (1, 6, 2)])
def test_bruteforce_small_integers(variant, shape):
    dtype, layout = variant.split("_")
    M, N, K = shape
    rng = np.random.default_rng(1000 + M * 100 + N * 10 + K)
    a = rng.integers(-8, 9, size=(M, K))
    b = rng.integers(-8, 9, size=(K, N))
    C, S = oracle.gemm(variant, encode(dtype, store(layout, a)), encode(dtype, store(layout, b)), M, N, K)
    Ce, Se = exact_product(a.tolist(), b.tolist())
    assert C.shape == (M, N)
    for i in range(M):
        for j in range(N):
            assert C[i, j] == float(Ce[i][j]), (i, j)
            assert S[i, j] == float(Se[i][j]), (i, j)


@pytest.mark.parametrize("variant", VARIANTS)
def test_bruteforce_dyadic_fractions(variant):
    """Non-integer values with few significant bits: every partial sum is exact in
    double, so the oracle must equal the rational result exactly."""
    dtype, layout = variant.split("_")
    M, N, K = 6, 7, 11
    rng = np.random.default_rng(7)
    a = rng.integers(-64, 65, size=(M, K)) / 32.0
    b = rng.integers(-64, 65, size=(K, N)) / 16.0
    C, S = oracle.gemm(variant, encode(dtype, store(layout, a)), encode(dtype, store(layout, b)), M, N, K)
    Ce, Se = exact_product([[Fraction(x) for x in r] for r in a.tolist()],
                           [[Fraction(x) for x in r] for r in b.tolist()])
    assert np.array_equal(C, np.array([[float(x) for x in r] for r in Ce]))
    assert np.array_equal(S, np.array([[float(x) for x in r] for r in Se]))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(37, 29, 41), (1, 64, 256), (64, 1, 100)])
def test_closed_form_ones(variant, shape):
    dtype, layout = variant.split("_")
    M, N, K = shape
    A = encode(dtype, np.ones(M * K))
    B = encode(dtype, np.ones(K * N))
    C, S = oracle.gemm(variant, A, B, M, N, K)
    assert np.all(C == K) and np.all(S == K)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(37, 29, 41), (41, 29, 37), (16, 16, 16)])
def test_closed_form_identity(variant, shape):
    """I·B = B with the rectangular identity delta_ik: row i of C is row i of B for
    i < min(M, K), zero below."""
    dtype, layout = variant.split("_")
    M, N, K = shape
    eye = np.eye(M, K)
    rng = np.random.default_rng(3)
    b = rng.integers(-100, 101, size=(K, N)) / 8.0
    C, _ = oracle.gemm(variant, encode(dtype, store(layout, eye)), encode(dtype, store(layout, b)), M, N, K)
    want = np.zeros((M, N))
    r = min(M, K)
    want[:r] = b[:r]
    assert np.array_equal(C, want)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_transpose_identity(dtype):
    """Column-major C = A·B and row-major C^T = B^T·A^T on the same buffers are the
    same numbers: the buffers read row-major are the transposes."""
    M, N, K = 23, 17, 31
    rng = np.random.default_rng(11)
    a = rng.uniform(-1, 1, size=M * K).astype(np.float32)
    b = rng.uniform(-1, 1, size=K * N).astype(np.float32)
    if dtype == "f16":
        a, b = a.astype(np.float16).view(np.uint16), b.astype(np.float16).view(np.uint16)
    elif dtype == "bf16":
        a, b = (a.view(np.uint32) >> 16).astype(np.uint16), (b.view(np.uint32) >> 16).astype(np.uint16)
    C_cm, S_cm = oracle.gemm(f"{dtype}_cm", a, b, M, N, K)
    C_rm, S_rm = oracle.gemm(f"{dtype}_rm", b, a, N, M, K)
    assert np.array_equal(C_cm, C_rm.T)
    assert np.array_equal(S_cm, S_rm.T)
    # and a non-square row-major product differs from its transpose-swapped misuse
    C_wrong, _ = oracle.gemm(f"{dtype}_rm", a, b, M, N, K)
    assert not np.array_equal(C_wrong, C_cm)


def test_decode_f16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode("f16", bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_bf16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32)
    got = oracle.decode("bf16", bits.astype(np.uint16))
    with np.errstate(invalid="ignore"):
        want = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


@pytest.mark.parametrize("variant", VARIANTS)
def test_random_against_float64_library_matmul(variant):
    dtype, layout = variant.split("_")
    M, N, K = 45, 70, 133
    rng = np.random.default_rng(5)
    a = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    b = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    if dtype == "f16":
        a, b = a.astype(np.float16).astype(np.float32), b.astype(np.float16).astype(np.float32)
    elif dtype == "bf16":
        a = ((a.view(np.uint32) >> 16) << 16).view(np.float32)
        b = ((b.view(np.uint32) >> 16) << 16).view(np.float32)
    C, S = oracle.gemm(variant, encode(dtype, store(layout, a)), encode(dtype, store(layout, b)), M, N, K)
    ref = a.astype(np.float64) @ b.astype(np.float64)
    sref = np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64))
    assert np.all(np.abs(C - ref) <= 1e-13 * sref)
    assert np.allclose(S, sref, rtol=1e-13, atol=0)


@pytest.mark.parametrize("variant", ["f32_rm", "f16_cm", "bf16_rm", "bf16_cm"])
def test_rows_and_entries_match_full(variant):
    dtype, layout = variant.split("_")
    M, N, K = 19, 23, 57
    rng = np.random.default_rng(9)
    a = rng.integers(-50, 51, size=(M, K)) / 16.0
    b = rng.integers(-50, 51, size=(K, N)) / 16.0
    A, B = encode(dtype, store(layout, a)), encode(dtype, store(layout, b))
    C, S = oracle.gemm(variant, A, B, M, N, K)
    rows = [18, 0, 7, 7]
    Cr, Sr = oracle.gemm_rows(variant, A, B, M, N, K, rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows])
    ii = rng.integers(0, M, size=40)
    jj = rng.integers(0, N, size=40)
    Ce, Se = oracle.gemm_entries(variant, A, B, M, N, K, ii, jj)
    assert np.array_equal(Ce, C[ii, jj]) and np.array_equal(Se, S[ii, jj])


def test_empty_and_degenerate():
    C, S = oracle.gemm("f32_rm", np.zeros(0, np.float32), np.zeros(0, np.float32), 0, 5, 0)
    assert C.shape == (0, 5)
    # K = 0: the empty sum is zero
    C, S = oracle.gemm("f32_rm", np.zeros(0, np.float32), np.zeros(0, np.float32), 3, 4, 0)
    assert np.array_equal(C, np.zeros((3, 4))) and np.array_equal(S, np.zeros((3, 4)))
    # NaN in row 1 of A propagates to row 1 of C only
    a = np.ones((3, 4), np.float32)
    a[1, 2] = np.nan
    C, _ = oracle.gemm("f32_rm", a.reshape(-1), np.ones(4 * 5, np.float32), 3, 5, 4)
    assert np.all(np.isnan(C[1])) and np.all(C[[0, 2]] == 4.0)


def test_bad_arguments_rejected():
    with pytest.raises(ValueError):
        oracle.gemm("f32_rm", np.zeros(5, np.float32), np.zeros(6, np.float32), 2, 3, 3)
    with pytest.raises(RuntimeError):
        oracle.gemm_entries("f32_rm", np.zeros(6, np.float32), np.zeros(9, np.float32), 2, 3, 3, [2], [0])


def test_half_tolerance_worked_value():
    """The contest's tolerance 0.01*sqrt(K/512) printed as 0.057 at K = 16384."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tolerance_half.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    for K, printed, digits in rows:
        tol = compare.tol_half(np.array([0.0]), int(K))[0]
        assert round(tol, int(digits)) == float(printed)
    # relative factor: at |C_ref| = 30 the tolerance is 30x the absolute one
    assert compare.tol_half(np.array([30.0]), 512)[0] == pytest.approx(0.3)


def test_compare_flags_violations():
    ref = np.array([[1.0, 2.0], [3.0, 4.0]])
    S = np.array([[10.0, 10.0], [10.0, 10.0]])
    ok = compare.check("f32_rm", ref + 5e-5, ref, S, 64)
    assert ok["ok"] and ok["n_bad"] == 0
    bad = compare.check("f32_rm", ref + np.array([[0, 2e-4], [0, 0]]), ref, S, 64)
    assert not bad["ok"] and bad["n_bad"] == 1
    nan = compare.check("bf16_rm", np.array([[np.nan, 2.0], [3.0, 4.0]]), ref, S, 64)
    assert not nan["ok"]


def test_round_to_output_type():
    assert compare.round_to("bf16_rm", np.array([4100.0]))[0] == 4096.0
    assert compare.round_to("f16_cm", np.array([4100.0]))[0] == 4100.0
    assert compare.round_to("f32_rm", np.array([16777217.0]))[0] == 16777216.0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("K", [16, 64, 512, 4096])
def test_half_tolerance_admits_the_exact_rounding(dtype, K):
    """The correctly rounded value of C_ref always passes; for bf16 at small K, where
    the ulp floor is what binds, a value two ulps off fails."""
    rng = np.random.default_rng(K)
    c = np.concatenate([rng.uniform(-20, 20, 20000), 2.0 ** np.arange(-5, 5) * (1 + 2.0 ** -9)])
    if dtype == "f16":
        r = c.astype(np.float16).astype(np.float64)
    else:
        r = compare.round_to("bf16_rm", c.astype(np.float32).astype(np.float64))
    tol = compare.tol_half(c, K, dtype)
    assert np.all(np.abs(r - c) <= tol)
    off = r + 2.0 * compare.ulp_out(dtype, c) * np.sign(c)
    if dtype == "bf16" and K <= 64:
        big = np.abs(c) >= 1.0
        assert np.all(np.abs(off - c)[big] > tol[big])


def test_output_ulp_values():
    assert compare.ulp_out("bf16", np.array([1.0]))[0] == 2.0 ** -7
    assert compare.ulp_out("bf16", np.array([7.9]))[0] == 2.0 ** -5
    assert compare.ulp_out("f16", np.array([1.0]))[0] == 2.0 ** -10
    assert compare.ulp_out("f16", np.array([0.0]))[0] == 2.0 ** -24
    assert compare.ulp_out("f16", np.array([1e-6]))[0] == 2.0 ** -24  # subnormal spacing


def test_round_bf16_matches_float32_path_and_ties():
    """Rounding float64 to bf16 once equals the float32 route wherever the value is
    already a float32 (no double rounding there), and ties go to even."""
    rng = np.random.default_rng(21)
    x = rng.uniform(-50, 50, 5000).astype(np.float32).astype(np.float64)
    assert np.array_equal(oracle.round_bf16(x), compare.round_to("bf16_rm", x))
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert oracle.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert oracle.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2 * 2.0 ** -7
    assert oracle.round_bf16(np.array([-3.0]))[0] == -3.0


def test_silu_identities():
    """SiLU(0) = 0; SiLU(x) - SiLU(-x) = x; SiLU -> x for large x, -> 0 for very
    negative x; SiLU(x) = x * sigmoid(x) with the library logistic function."""
    from scipy.special import expit
    x = np.linspace(-30, 30, 2001)
    s = oracle.silu(x)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(s - oracle.silu(-x), x, rtol=0, atol=1e-12)
    assert np.allclose(s, x * expit(x), rtol=1e-14, atol=1e-300)
    assert abs(oracle.silu(np.array([40.0]))[0] - 40.0) < 1e-15 * 40
    assert abs(oracle.silu(np.array([-40.0]))[0]) < 1e-15


def test_silu_mul_brute_force_small():
    """The gate/up chain on tiny integer inputs against a pure-Python evaluation of
    the same definition (exact integer sums, math.exp, the same rounding points)."""
    import math
    M, N, K = 3, 5, 4
    rng = np.random.default_rng(17)
    x = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    wg = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    wu = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    enc = lambda a: (a.reshape(-1).view(np.uint32) >> 16).astype(np.uint16)
    r = oracle.silu_mul(enc(x), enc(wg), enc(wu), M, N, K)
    Z, G, U, T = r["Z"], r["G"], r["U"], r["T"]
    rb = lambda v: float(oracle.round_bf16(np.array([v]))[0])
    for i in range(M):
        for j in range(N):
            g = rb(sum(int(x[i, k]) * int(wg[k, j]) for k in range(K)))
            u = rb(sum(int(x[i, k]) * int(wu[k, j]) for k in range(K)))
            t = rb(g / (1.0 + math.exp(-g)))
            assert (G[i, j], U[i, j], T[i, j]) == (g, u, t)
            assert Z[i, j] == rb(t * u)


def test_silu_mul_tolerance_admits_one_step_moves():
    """Moving G or U by one bf16 step (a rounding-boundary flip) stays within the
    tolerance, and so does an FP32-level error in a cancelling U; a 5% error in
    Z does not."""
    rng = np.random.default_rng(3)
    g = oracle.round_bf16(rng.normal(0, 2, 4000))
    u = oracle.round_bf16(rng.normal(0, 2, 4000))
    s_g = np.abs(g) + 1.0
    s_u = np.abs(u) + 1.0
    t = oracle.round_bf16(oracle.silu(g))
    z = oracle.round_bf16(t * u)
    tol = compare.tol_silu_mul(g, u, t, z, s_g, s_u)
    g2 = g + compare.ulp_out("bf16", g)
    t2 = oracle.round_bf16(oracle.silu(g2))
    z2 = oracle.round_bf16(t2 * u)
    assert np.all(np.abs(z2 - z) <= tol)
    u2 = u + compare.ulp_out("bf16", u)
    z3 = oracle.round_bf16(t * u2)
    assert np.all(np.abs(z3 - z) <= tol)
    u4 = oracle.round_bf16(u + 0.9e-5 * s_u)
    z4 = oracle.round_bf16(t * u4)
    assert np.all(np.abs(z4 - z) <= tol)
    big = (np.abs(z) > 0.5) & (g > 0)
    assert np.all((np.abs(1.05 * z - z) > tol)[big])
