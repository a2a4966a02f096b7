"""Helpers of the GPU parity tests: move seeded host buffers to the device, call
an entry point of the library through its C ABI, bring the result back as
float64 in logical [M, N] order."""

from __future__ import annotations

import numpy as np
import torch

import dense_matrix_multiply_gb300 as g
import oracle
from oracle import compare

ENTRY = {"f32_rm": "gemm_f32_rm", "f16_cm": "gemm_f16_cm", "bf16_rm": "gemm_bf16_rm"}


def to_device(buf: np.ndarray, offset_elems: int = 0) -> torch.Tensor:
    """A CUDA tensor holding buf; with offset_elems > 0 the data starts that many
    elements into a larger allocation (to exercise unaligned pointers)."""
    if buf.dtype == np.float32:
        t = torch.from_numpy(np.ascontiguousarray(buf))
    else:
        t = torch.from_numpy(np.ascontiguousarray(buf).view(np.int16))
    if offset_elems:
        big = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device="cuda")
        view = big[offset_elems:]
        view.copy_(t.to("cuda"))
        return view
    return t.to("cuda")


def empty_out(variant: str, M: int, N: int, offset_elems: int = 0, fill=None) -> torch.Tensor:
    dt = torch.float32 if variant.startswith("f32") else torch.int16
    big = torch.empty(M * N + offset_elems, dtype=dt, device="cuda")
    if fill is not None:
        big.fill_(fill)
    return big[offset_elems:]


def widen(variant: str, t: torch.Tensor, M: int, N: int) -> np.ndarray:
    """Device result -> float64 numpy [M, N] (logical order)."""
    h = t.cpu().numpy()
    if variant.startswith("f32"):
        v = h.astype(np.float64)
    elif variant.startswith("f16"):
        v = h.view(np.uint16).view(np.float16).astype(np.float64)
    else:
        v = (h.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if variant.endswith("_cm"):
        return v.reshape(N, M).T
    return v.reshape(M, N)


def run(variant: str, A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, force=None,
        a_off: int = 0, b_off: int = 0, c_off: int = 0, stream=None):
    """Runs one entry point on host buffers; returns (C float64 [M,N], kernel name, C tensor)."""
    dA = to_device(A, a_off)
    dB = to_device(B, b_off)
    dC = empty_out(variant, M, N, c_off, fill=-1)
    g.gemm_force_kernel(force)
    try:
        if stream is not None:
            with torch.cuda.stream(stream):
                getattr(g, ENTRY[variant])(dA, dB, dC, M, N, K)
        else:
            getattr(g, ENTRY[variant])(dA, dB, dC, M, N, K)
        name = g.gemm_last_kernel()
    finally:
        g.gemm_force_kernel(None)
    g.gemm_synchronize()
    torch.cuda.synchronize()
    return widen(variant, dC, M, N), name, dC


def kernel_view(variant, A, B, M, N, K):
    """The row-major problem the kernels run: a column-major C = A·B is the
    row-major C^T = B^T·A^T on the same buffers ("SGEMM measured and the three
    ledgers", section 2).  Returns (row-major variant, A', B', M', N', transposed)."""
    if variant.endswith("_cm"):
        return variant.replace("_cm", "_rm"), B, A, N, M, True
    return variant, A, B, M, N, False


def band_rows(M, band=256):
    """Two rows of every `band`-row band of the kernel's output, one in each half
    (the two CTAs of a pair tile), moving through the 32-row quarters (epilogue
    warps) from band to band; plus the last row."""
    rows = set()
    for b in range((M + band - 1) // band):
        for h in range(2):
            r = b * band + h * (band // 2) + ((b + h) % 4) * 32 + (7 * b + 3 * h) % 32
            if r < M:
                rows.add(r)
    rows.add(M - 1)
    return np.array(sorted(rows), dtype=np.int64)


def band_cols(N, band=256):
    """One column of every `band`-column band, at a varying offset; plus the last."""
    cols = {min(N - 1, b * band + (67 * b + 13) % band) for b in range((N + band - 1) // band)}
    cols.add(N - 1)
    return np.array(sorted(cols), dtype=np.int64)


def check_bands(variant, C, A, B, M, N, K):
    """C (float64, logical [M, N]) against the oracle on whole rows -- two from
    every 256-row band of the kernel's output -- and whole columns -- one from
    every 256-column band.  Returns (rows result, columns result) of
    compare.check."""
    kv, kA, kB, kM, kN, tr = kernel_view(variant, A, B, M, N, K)
    Ck = C.T if tr else C  # the kernel's [kM, kN] output
    rows = band_rows(kM)
    R_ref, R_S = oracle.gemm_rows(kv, kA, kB, kM, kN, K, rows)
    res_r = compare.check(kv, Ck[rows], R_ref, R_S, K)
    cols = band_cols(kN)
    ii = np.repeat(np.arange(kM, dtype=np.int64), cols.size)
    jj = np.tile(cols, kM)
    E_ref, E_S = oracle.gemm_entries(kv, kA, kB, kM, kN, K, ii, jj)
    res_c = compare.check(kv, Ck[ii, jj], E_ref, E_S, K)
    return res_r, res_c
