"""Pins of the oracle's FP8 functions ("Chapter 5 Operators and Runtime",
section 5.4.3, example 5-7: row-wise E4M3FN quantisation with the scale taken
from the whole row; section 5.4.4, example 5-8: FP8 input times FP8 weights).

The E4M3FN decoder and encoder are checked against torch's float8_e4m3fn
conversions (an independent library routine): every code, and every midpoint
between neighbouring values with its two FP32 neighbours (ties, round-down and
round-up cases) across the subnormal and normal ranges.  The worked example
5-7 (tests/golden/fp8_rowscale_example.txt) pins the scale convention, and
small problems are brute-forced in exact rationals."""

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
if not hasattr(torch, "float8_e4m3fn"):
    pytest.skip("torch without float8_e4m3fn", allow_module_level=True)


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "fp8_rowscale_example.txt")
    out = {}
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


def test_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.decode_e4m3(codes), torch_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    assert oracle.decode_e4m3([0x7E])[0] == 448.0 and np.isnan(oracle.decode_e4m3([0x7F])[0])
    assert oracle.decode_e4m3([0x01])[0] == 2.0 ** -9 and oracle.decode_e4m3([0x08])[0] == 2.0 ** -6


def test_encode_midpoints_and_neighbours():
    vals = np.unique(oracle.decode_e4m3(np.arange(0, 0x7F, dtype=np.uint8)))  # 0 .. 448
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    down = np.nextafter(mids, np.float32(0))
    xs = np.concatenate([vals.astype(np.float32), mids, up, down])
    xs = np.concatenate([xs, -xs])
    assert np.array_equal(oracle.encode_e4m3(xs), torch_encode(xs))


def test_encode_random_and_saturation():
    rng = np.random.default_rng(0)
    x = np.clip(rng.standard_normal(20000) * 100, -448, 448).astype(np.float32)
    assert np.array_equal(oracle.encode_e4m3(x), torch_encode(x))
    sat = oracle.encode_e4m3(np.array([449.0, 1e6, -500.0, 464.0], dtype=np.float32))
    assert list(sat) == [0x7E, 0x7E, 0xFE, 0x7E]


def test_worked_example_5_7():
    g = golden()
    n, b = int(g["row_length"]), int(g["block_length"])
    row = np.zeros(n, dtype=np.float16)
    row[0], row[b] = g["first_block_value"], g["second_block_value"]
    Q, scale = oracle.quantize_rows_e4m3(row.view(np.uint16), 1, n)
    amax = g["second_block_value"]
    assert abs(float(np.float32(1.0) * (np.float32(448.0) / np.float32(amax))) - g["scaled_first_element"]) < 1e-5
    assert oracle.decode_e4m3(Q[0, :1])[0] == g["quantised_first_element"]
    assert scale[0] == np.float32(amax) / np.float32(448.0)
    w = np.zeros((1, n), dtype=np.uint8)
    w[0, 0] = oracle.encode_e4m3([1.0])[0]
    C, _ = oracle.gemm_e4m3_rowscale(Q, scale, w, 1, 1, n)
    exact = g["dequantised_first_element_num"] / g["dequantised_first_element_den"]
    assert abs(C[0, 0] - exact) <= 2.0 ** -23 * exact          # 55/56 up to the FP32 scale
    # quantising the first block alone (its own maximum 1) would give exactly 1:
    Qb, sb = oracle.quantize_rows_e4m3(row[:b].view(np.uint16), 1, b)
    Cb, _ = oracle.gemm_e4m3_rowscale(Qb, sb, w[:, :b], 1, 1, b)
    one = g["blockwise_dequantised_first_element"]
    assert abs(Cb[0, 0] - one) <= 2.0 ** -23 * one              # 448 * fl32(1/448)
    rel = (Cb[0, 0] - C[0, 0]) / Cb[0, 0]
    assert abs(rel - g["relative_difference_num"] / g["relative_difference_den"]) < 1e-6


def test_quantize_rows_against_float32_steps():
    """Each code equals torch's E4M3 conversion of the FP32 product a * (448/amax)
    computed with numpy float32 arithmetic; rows of zeros give zeros."""
    rng = np.random.default_rng(1)
    M, K = 37, 300
    a = (rng.standard_normal((M, K)) * rng.uniform(0.01, 100, (M, 1))).astype(np.float16)
    a[5] = 0
    a[6, :] = 0
    a[6, 299] = -3.0                       # the maximum at the very end of a row
    Q, scale = oracle.quantize_rows_e4m3(a.view(np.uint16), M, K)
    af = a.astype(np.float32)
    amax = np.abs(af).max(axis=1)
    for i in range(M):
        if amax[i] == 0:
            assert not Q[i].any() and scale[i] == 0
            continue
        inv = np.float32(448.0) / amax[i]
        assert np.array_equal(Q[i], torch_encode(af[i] * inv))
        assert scale[i] == amax[i] / np.float32(448.0)
    assert np.abs(oracle.decode_e4m3(Q.reshape(-1))).max() == 448.0  # each row's maximum maps to 448


def test_rowscale_gemm_brute_force():
    rng = np.random.default_rng(2)
    M, N, K = 5, 4, 24
    Q = rng.integers(0, 256, (M, K), dtype=np.uint8)
    Q[(Q & 0x7F) == 0x7F] = 0x11                   # no NaN codes
    W = rng.integers(0, 256, (N, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x22
    scale = rng.uniform(0.001, 2, M).astype(np.float32)
    C, S = oracle.gemm_e4m3_rowscale(Q, scale, W, M, N, K)
    dq = torch_decode(Q.reshape(-1)).reshape(M, K)
    dw = torch_decode(W.reshape(-1)).reshape(N, K)
    for i in range(M):
        for j in range(N):
            acc = sum(Fraction(dq[i, k]) * Fraction(dw[j, k]) for k in range(K))
            sab = sum(abs(Fraction(dq[i, k]) * Fraction(dw[j, k])) for k in range(K))
            assert C[i, j] == float(Fraction(float(scale[i])) * acc)
            assert S[i, j] == float(Fraction(float(scale[i])) * sab)
    rows = np.array([3, 0])
    Cr, _ = oracle.gemm_e4m3_rowscale(Q, scale, W, M, N, K, rows=rows)
    assert np.array_equal(Cr, C[rows])


def test_e4m3_code_generator_stays_finite_and_in_range():
    import synthetic
    c = synthetic.e4m3_codes(64, 64, 123, 4, 10)
    v = np.abs(oracle.decode_e4m3(c))
    assert np.isfinite(v).all()
    assert v.min() >= 2.0 ** -3 and v.max() <= 1.875 * 2.0 ** 3
    assert np.array_equal(c, synthetic.e4m3_codes(64, 64, 123, 4, 10))


def test_e4m3_tolerance_admits_rounding_and_rejects_a_step():
    from oracle import compare
    C_ref = np.array([1.0, 100.0, -3.5, 1000.0])
    S = np.abs(C_ref) * 10
    exact = C_ref.astype(np.float16).astype(np.float64)
    assert compare.check_e4m3(exact, C_ref, S)["ok"]
    moved = C_ref + 4 * compare.ulp_out("f16", C_ref) + 1e-4 * S
    assert not compare.check_e4m3(moved, C_ref, S)["ok"]


def test_e4m3_tolerance_is_half_an_ulp_without_cancellation():
    """Positive codes at K = 4096: nothing cancels (S = |C|), so the FP32
    allowance is ~1e-5 of |C| and the tolerance is about half an ulp.  The
    exactly rounded value passes; a result one or two half-precision steps away
    from it fails."""
    from oracle import compare
    import synthetic
    M, N, K = 8, 16, 4096
    Q = synthetic.e4m3_codes(M, K, 31, 4, 10) & np.uint8(0x7F)   # clear the sign bits
    W = synthetic.e4m3_codes(N, K, 32, 4, 10) & np.uint8(0x7F)
    scale = np.full(M, 2.0 ** -12, dtype=np.float32)
    C_ref, S = oracle.gemm_e4m3_rowscale(Q, scale, W, M, N, K)
    assert np.array_equal(S, C_ref)
    exact = C_ref.astype(np.float16).astype(np.float64)
    assert compare.check_e4m3(exact, C_ref, S)["ok"]
    step = compare.ulp_out("f16", exact)
    for n_steps in (1, 2):
        for sign in (1.0, -1.0):
            assert not compare.check_e4m3(exact + sign * n_steps * step, C_ref, S)["ok"], (n_steps, sign)
    tol = compare.tol_e4m3(C_ref, S)
    assert np.all(tol < compare.ulp_out("f16", C_ref))


def test_e4m3_tolerance_half_ulp_taken_in_the_wider_binade():
    """A sum just below a power of two whose FP32 value may cross it is allowed
    half an ulp of the wider binade (where the rounding then happens)."""
    from oracle import compare
    C_ref = np.array([2048.0 - 2.0 ** -6])
    S = np.array([2048.0])
    tol = compare.tol_e4m3(C_ref, S)
    d = 1e-5 * 2048.0 + 2.0 ** -23 * C_ref[0]
    assert tol[0] == d + 0.5 * 2.0  # half of the ulp 2.0 of [2048, 4096)
