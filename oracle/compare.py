"""Acceptance tolerances for a GEMM result against the oracle -- TEST INFRASTRUCTURE ONLY.

FP32 output: |C - C_ref| <= 1e-5 * sum_k |a_ik * b_kj|, per element.
Half / bf16 output: |C - C_ref| <= 1e-2 * sqrt(K/512) * max(1, |C_ref|), per element.

The half form is the contest's correctness rule ("MTT S4000 FP16 GEMM",
section 1: tolerance 0.01*sqrt(K/512), 0.057 at K = 16384), widened by the
relative factor max(1, |C_ref|) so that outputs much larger than one are judged
against their own half/bf16 spacing. The FP32 form scales with the sum of
absolute products, the natural bound for any summation order.

Floor for 16-bit outputs: the contest stated its rule for half output at
K >= 512.  For bf16 output and K below about 78, 0.01*sqrt(K/512) is smaller
than bf16's own relative rounding step (2^-8 at the bottom of a binade), so even
the exactly rounded value of C_ref can fail it.  The tolerance is therefore
never smaller than one unit in the last place of the output type at |C_ref|:
half an ulp for the single rounding of the FP32 sum, the other half for an FP32
accumulation error that moves the sum across a rounding boundary.
"""

from __future__ import annotations

import math

import numpy as np


def tol_f32(S: np.ndarray) -> np.ndarray:
    return 1e-5 * np.asarray(S, dtype=np.float64)


_MANT_BITS = {"f16": 10, "bf16": 7}
_MIN_EXP = {"f16": -14, "bf16": -126}


def ulp_out(dtype: str, x: np.ndarray) -> np.ndarray:
    """Spacing of the 16-bit output type ('f16' or 'bf16') in the binade of |x|."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(np.where(a > 0, e, _MIN_EXP[dtype]), _MIN_EXP[dtype])
    return np.exp2(e - _MANT_BITS[dtype])


def tol_half(C_ref: np.ndarray, K: int, dtype: str | None = None) -> np.ndarray:
    """0.01*sqrt(K/512)*max(1,|C_ref|); with dtype given, floored at one output ulp."""
    c = np.asarray(C_ref, dtype=np.float64)
    t = 1e-2 * math.sqrt(K / 512.0) * np.maximum(1.0, np.abs(c))
    if dtype is not None and K > 0:
        t = np.maximum(t, ulp_out(dtype, c))
    return t


def tolerance(variant: str, C_ref: np.ndarray, S: np.ndarray, K: int) -> np.ndarray:
    if variant.startswith("f32"):
        return tol_f32(S)
    return tol_half(C_ref, K, variant.split("_")[0])


def check(variant: str, C: np.ndarray, C_ref: np.ndarray, S: np.ndarray, K: int) -> dict:
    """Element-wise comparison; C is the result widened to float64, same shape as C_ref."""
    C = np.asarray(C, dtype=np.float64)
    C_ref = np.asarray(C_ref, dtype=np.float64)
    if C.shape != C_ref.shape:
        raise ValueError(f"shape {C.shape} != reference shape {C_ref.shape}")
    tol = tolerance(variant, C_ref, S, K)
    err = np.abs(C - C_ref)
    bad = ~(err <= tol)  # NaN in C counts as a violation
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0), np.where(err > 0, np.inf, 0.0))
    return {
        "n": int(C.size),
        "n_bad": int(bad.sum()),
        "max_abs_err": float(np.nanmax(err)) if C.size else 0.0,
        "max_err_over_tol": float(np.nanmax(ratio)) if C.size else 0.0,
        "ok": bool(not bad.any()),
    }


def round_to(variant: str, x: np.ndarray) -> np.ndarray:
    """Round exact float64 values once to the output type (nearest, ties to even) and
    return them as float64 again. Used only for closed forms whose exact value is
    known, e.g. ones*ones = K or I*B = B."""
    x = np.asarray(x, dtype=np.float64)
    if variant.startswith("f32"):
        return x.astype(np.float32).astype(np.float64)
    if variant.startswith("f16"):
        return x.astype(np.float16).astype(np.float64)
    # bf16: the values used here are exact in float32, so round float32 -> bf16.
    f = x.astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def tol_silu_mul(G: np.ndarray, U: np.ndarray, T: np.ndarray, Z: np.ndarray,
                 S_G: np.ndarray, S_U: np.ndarray) -> np.ndarray:
    """Tolerance of Z = bf16(bf16(SiLU(G)) * U) against the oracle's rounded G, U, T, Z.

    The GPU's FP32 sums may differ from the exact ones by the FP32 accumulation
    allowance 1e-5 * sum_k |a_ik b_kj| (S_G, S_U) -- large relative to G or U when
    their terms nearly cancel -- and then round to the neighbouring bf16 value;
    SiLU is evaluated in FP32.  So:
      dG = 2^-7 |G| + 1e-5 S_G,   dU = 2^-7 |U| + 1e-5 S_U   (one bf16 step each;
                                                             2^-7 bounds a step)
      dT = |SiLU'(G)| dG + 2^-7 |T|,  SiLU'(g) = s (1 + g (1 - s)), s = 1/(1+e^-g)
      dZ = dT |U| + |T| dU + ulp(Z).
    """
    G, U, T, Z, S_G, S_U = (np.asarray(a, dtype=np.float64) for a in (G, U, T, Z, S_G, S_U))
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-G))
    slope = np.abs(s * (1.0 + G * (1.0 - s)))
    dG = 2.0 ** -7 * np.abs(G) + 1e-5 * S_G
    dU = 2.0 ** -7 * np.abs(U) + 1e-5 * S_U
    dT = slope * dG + 2.0 ** -7 * np.abs(T)
    return dT * np.abs(U) + np.abs(T) * dU + ulp_out("bf16", Z)


def tol_ex(variant: str, ref: dict, K: int, alpha: float) -> np.ndarray:
    """Tolerance of the general form alpha op(A) op(B) + beta C against
    ``oracle.gemm_ex``'s outputs (P, S, BC, C).

    The device sums the products in FP32 (acc), forms alpha * acc + beta * c in
    FP32 and rounds once to the output type.  So the allowance is the variant's
    own rule applied to the scaled product -- 1e-5 |alpha| S for FP32, the
    half/bf16 rule at |alpha P| -- plus 2^-22 (|alpha P| + |beta c|) for the two
    FP32 roundings of the combination (each at most 2^-24 relative), plus, for
    16-bit outputs, one output ulp at |C| for the final rounding of the combined
    value.  With alpha = 1 and beta = 0 this is the plain rule plus the
    2^-22 |P| term."""
    dtype = variant.split("_")[0]
    P, S, BC, C = (np.asarray(ref[k], dtype=np.float64) for k in ("P", "S", "BC", "C"))
    prod = alpha * P
    if alpha == 0 or K == 0:
        base = np.zeros_like(P)
    elif dtype == "f32":
        base = tol_f32(abs(alpha) * S)
    else:
        base = tol_half(prod, K, dtype)
    t = base + 2.0 ** -22 * (np.abs(prod) + np.abs(BC))
    if dtype != "f32":
        t = t + ulp_out(dtype, C)
    return t


def check_ex(variant: str, C: np.ndarray, ref: dict, K: int, alpha: float) -> dict:
    """Element-wise comparison of a general-form result (float64, shape of ref['C'])."""
    C = np.asarray(C, dtype=np.float64)
    C_ref = np.asarray(ref["C"], dtype=np.float64)
    if C.shape != C_ref.shape:
        raise ValueError(f"shape {C.shape} != reference shape {C_ref.shape}")
    tol = tol_ex(variant, ref, K, alpha)
    err = np.abs(C - C_ref)
    bad = ~(err <= tol)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0), np.where(err > 0, np.inf, 0.0))
    return {
        "n": int(C.size),
        "n_bad": int(bad.sum()),
        "max_abs_err": float(np.nanmax(err)) if C.size else 0.0,
        "max_err_over_tol": float(np.nanmax(ratio)) if C.size else 0.0,
        "ok": bool(not bad.any()),
    }


def tol_e4m3(C_ref: np.ndarray, S: np.ndarray) -> np.ndarray:
    """Tolerance of the row-scaled FP8 product (half output) against
    ``oracle.gemm_e4m3_rowscale``.  No page states one; it follows from the
    arithmetic.  The codes and the FP32 row scale are the same on both sides and
    every E4M3 x E4M3 product is exact in FP32, so the FP32 value v that is
    finally rounded to half differs from C_ref by at most
        d = 1e-5 * S              (FP32 accumulation, S = |scale| sum_k |q w|)
          + 2^-23 * |C_ref|       (the FP32 rounding of scale * acc, with slack),
    and the one rounding of v to half adds at most half an ulp at |v|, taken
    here at the largest magnitude v can have, |C_ref| + d (a v pushed across a
    power of two is rounded in the wider binade).  So |C - C_ref| <= d +
    ulp(|C_ref| + d) / 2: less than one ulp when the terms do not cancel (S close
    to |C_ref|)."""
    C_ref = np.asarray(C_ref, dtype=np.float64)
    d = 1e-5 * np.asarray(S, dtype=np.float64) + 2.0 ** -23 * np.abs(C_ref)
    return d + 0.5 * ulp_out("f16", np.abs(C_ref) + d)


def check_e4m3(C: np.ndarray, C_ref: np.ndarray, S: np.ndarray) -> dict:
    C = np.asarray(C, dtype=np.float64)
    C_ref = np.asarray(C_ref, dtype=np.float64)
    if C.shape != C_ref.shape:
        raise ValueError(f"shape {C.shape} != reference shape {C_ref.shape}")
    tol = tol_e4m3(C_ref, S)
    err = np.abs(C - C_ref)
    bad = ~(err <= tol)
    return {"n": int(C.size), "n_bad": int(bad.sum()),
            "max_abs_err": float(np.nanmax(err)) if C.size else 0.0,
            "max_err_over_tol": float(np.nanmax(err / tol)) if C.size else 0.0,
            "ok": bool(not bad.any())}
