"""Helpers of the GPU parity tests: move seeded host buffers to the device, call
an entry point of the library through its C ABI, bring the result back as
float64 in logical [M, N] order."""

from __future__ import annotations

import numpy as np
import torch

import dense_matrix_multiply_gb300 as g

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


def sample_indices(M: int, N: int, n: int, seed: int = 0):
    """Random (i, j) pairs plus the four corners and the last row/column edges."""
    rng = np.random.default_rng(seed)
    ii = list(rng.integers(0, M, size=n))
    jj = list(rng.integers(0, N, size=n))
    for i, j in [(0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)]:
        ii.append(i)
        jj.append(j)
    for t in range(min(64, N)):
        ii.append(M - 1)
        jj.append(N - 1 - t)
    for t in range(min(64, M)):
        ii.append(M - 1 - t)
        jj.append(N - 1)
    return np.array(ii, dtype=np.int64), np.array(jj, dtype=np.int64)
