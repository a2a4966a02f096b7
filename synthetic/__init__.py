"""Seeded synthetic matrices for the GEMM workloads.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark. It holds no part of the product's arithmetic: it only draws
random numbers and rounds them once to the storage type, so that both sides
receive the very same bits.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), in its published 64-bit form. The i-th output
(i = 1, 2, ...) of a stream with seed s is mix(s + i*0x9E3779B97F4A7C15), so a
whole matrix is drawn with one vectorised pass.

Distributions, as the workloads state them:
  * uniform[-1, 1]: u = (x >> 40) * 2^-24 in [0, 1), value 2u - 1. Every value is
    a multiple of 2^-23 and exact in float32.
  * N(0, sigma^2): Box-Muller in float64 from two outputs per element, rounded
    once to float32 (round to nearest even), then scaled by sigma. For the FFN
    weight sigma^2 = 1/4096, so sigma = 2^-6 and the scaling is exact.
Half and bf16 inputs are the float32 values rounded once, to nearest even.

Values are generated in the buffer's storage order: element t of the returned
flat buffer is draw t of the stream, whatever the layout the caller reads it in.
"""

from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

SEED_BASE = 0xD5E10000


def seed_for(config_id: int, matrix_id: int) -> int:
    """Seed of one matrix of one workload: base + 16*config + matrix (A/X=1, B/W=2)."""
    return SEED_BASE + 16 * int(config_id) + int(matrix_id)


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start+1 .. start+n of the SplitMix64 stream with the given seed."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = i * GOLDEN + np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform_pm1(seed: int, n: int) -> np.ndarray:
    """n float32 values, uniform on [-1, 1) with 24-bit resolution (exact in float32)."""
    x = splitmix64(seed, n)
    u = (x >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    return (2.0 * u - 1.0).astype(np.float32)


def normal(seed: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n float32 values ~ N(0, sigma^2) by Box-Muller (cosine branch only)."""
    x = splitmix64(seed, 2 * n)
    u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return z.astype(np.float32) * np.float32(sigma)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((b[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return r


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to IEEE half (nearest, ties to even); returns uint16 bit patterns."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen half bit patterns to float32 (exact)."""
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


def draw(dist: str, seed: int, n: int, sigma: float = 1.0) -> np.ndarray:
    if dist == "uniform":
        return uniform_pm1(seed, n)
    if dist == "normal":
        return normal(seed, n, sigma)
    raise ValueError(f"unknown distribution {dist!r}")


def matrix(dtype: str, rows: int, cols: int, seed: int, dist: str = "uniform",
           sigma: float = 1.0) -> np.ndarray:
    """A flat storage buffer of rows*cols elements.

    dtype 'f32' returns float32; 'f16' and 'bf16' return the uint16 bit patterns
    of the float32 draws rounded once to that type.
    """
    v = draw(dist, seed, rows * cols, sigma)
    if dtype == "f32":
        return v
    if dtype == "f16":
        return f32_to_f16_bits(v)
    if dtype == "bf16":
        return f32_to_bf16_bits(v)
    raise ValueError(f"unknown dtype {dtype!r}")


# The five workloads, by what they are. Each entry: (config id, list of
# problems); a problem is (variant, M, N, K, distribution of A, sigma A,
# distribution of B, sigma B).
def e4m3_codes(rows: int, cols: int, seed: int, exp_lo: int = 4, exp_hi: int = 10) -> np.ndarray:
    """Random FP8 E4M3FN codes built bit by bit (no rounding involved): a random
    sign, an exponent field uniform in [exp_lo, exp_hi] and a random 3-bit
    fraction, i.e. values of magnitude 2^(exp_lo-7) .. 1.875 * 2^(exp_hi-7).
    exp_hi <= 14 keeps every code finite (field 15 holds 448 and NaN)."""
    if not (1 <= exp_lo <= exp_hi <= 14):
        raise ValueError("exponent fields must lie in 1..14")
    x = splitmix64(seed, rows * cols)
    sign = (x >> np.uint64(63)).astype(np.uint8)
    frac = ((x >> np.uint64(32)) & np.uint64(7)).astype(np.uint8)
    span = np.uint64(exp_hi - exp_lo + 1)
    expo = (((x & np.uint64(0xFFFFFFFF)) % span) + np.uint64(exp_lo)).astype(np.uint8)
    return ((sign << 7) | (expo << 3) | frac).astype(np.uint8)


WORKLOADS = {
    "sgemm_f32_rm_256": (0, [("f32_rm", 256, 256, 256, "uniform", 1.0, "uniform", 1.0)]),
    "sgemm_f32_rm_4096": (1, [("f32_rm", 4096, 4096, 4096, "uniform", 1.0, "uniform", 1.0)]),
    "hgemm_f16_cm_8192": (2, [("f16_cm", 8192, 8192, 8192, "uniform", 1.0, "uniform", 1.0)]),
    "hgemm_f16_cm_3072x5120x6144": (2, [("f16_cm", 3072, 5120, 6144, "uniform", 1.0, "uniform", 1.0)]),
    "ffn_bf16_rm_1024x12288x4096": (3, [("bf16_rm", 1024, 12288, 4096, "normal", 1.0, "normal", 1.0 / 64.0)]),
}

EDGE_SHAPES = [  # (M, N, K) of the ragged/edge sweep, run on the f32 and bf16 paths
    (1000, 1000, 1000),
    (1, 12288, 4096),
    (32, 12288, 4096),
    (64, 64, 64),
    (8192, 4096, 4100),
    (8192, 4096, 4096),
]
EDGE_CONFIG_ID = 4


def problem_inputs(variant: str, M: int, N: int, K: int, config_id: int,
                   dist_a: str = "uniform", sigma_a: float = 1.0,
                   dist_b: str = "uniform", sigma_b: float = 1.0):
    """Storage buffers (A, B) of one problem. Layout follows the variant:
    *_rm stores A as [M,K] and B as [K,N] row-major; *_cm stores them column-major."""
    dtype = variant.split("_")[0]
    a = matrix(dtype, M, K, seed_for(config_id, 1), dist_a, sigma_a)
    b = matrix(dtype, K, N, seed_for(config_id, 2), dist_b, sigma_b)
    return a, b
