"""Closed forms at the full size of every workload, compared bit for bit.

ones(M,K)·ones(K,N) = K and I·B = B (I the rectangular identity δ_ik) have
exactly representable results: every partial sum of ones·ones is an integer
below 2^24, and each output of I·B has a single nonzero product.  So the GPU
result must equal the exact value rounded once to the output type, whatever
the summation order -- including the paths that only the full-size shapes
take: the SGEMM whose last round is split into two K halves that are added
(4096^3: two grids), the tensor-core stream-K tail whose partials a second
kernel adds (FP16 column-major 3072x5120x6144), A rows that TMA cannot
describe, staged into aligned rows (bf16 K = 4100), and the allocation-free
entry point, which runs the same shapes without stream-K or staging.

For bf16 at K = 4100 the exact 4100 is not a bf16 value: the expected result
is its nearest-even rounding, 4096.  Inputs are made on the device (ones, the
identity) or drawn by the seeded generator (B of I·B).
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu

ENTRY = {"f32_rm": "gemm_f32_rm", "f16_cm": "gemm_f16_cm", "bf16_rm": "gemm_bf16_rm",
         "bf16_rm_noalloc": "gemm_bf16_rm_noalloc"}

# (variant, M, N, K, expected kernel, expected launches per call)
FULL = [
    ("f32_rm", 256, 256, 256, "simt_f32_vec4", 1),
    ("f32_rm", 4096, 4096, 4096, "simt_f32_vec4", 2),            # split last round: whole rounds + half-K pairs
    ("f32_rm", 8192, 4096, 4100, "simt_f32_vec4", None),
    ("f32_rm", 8192, 4096, 4096, "simt_f32_vec4", None),
    ("f16_cm", 8192, 8192, 8192, "umma_f16", 1),
    ("f16_cm", 3072, 5120, 6144, "umma_f16", 2),                  # stream-K tail + fix-up kernel
    ("bf16_rm", 1024, 12288, 4096, "umma_bf16", 1),
    ("bf16_rm", 8192, 4096, 4100, "umma_bf16", 2),                # A staged into aligned rows + CTA pairs
    ("bf16_rm", 8192, 4096, 4096, "umma_bf16", 1),
    ("bf16_rm_noalloc", 1024, 12288, 4096, "umma_bf16_noalloc", 1),
    ("bf16_rm_noalloc", 8192, 4096, 4100, "umma_bf16_noalloc", 1),  # A by cp.async, single-CTA tiles
    ("bf16_rm_noalloc", 8192, 4096, 4096, "umma_bf16_noalloc", 1),
    ("bf16_rm_noalloc", 3072, 5120, 6144, "umma_bf16_noalloc", 1),  # whole tiles where bf16_rm takes stream-K
]


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def _dtype(variant):
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[variant.split("_")[0]]


def _call(variant, dA, dB, M, N, K):
    """One call through the C ABI; returns (C tensor in storage order, kernel, launches)."""
    dC = torch.full((M * N,), -1.0, dtype=_dtype(variant), device="cuda")
    before = g.gemm_kernel_launches()
    getattr(g, ENTRY[variant])(dA, dB, dC, M, N, K)
    launches = g.gemm_kernel_launches() - before
    name = g.gemm_last_kernel()
    g.gemm_synchronize()
    torch.cuda.synchronize()
    return dC, name, launches


def _storage_identity(variant, M, K):
    """The rectangular identity δ_ik of M x K, as the variant stores A."""
    eye = torch.eye(M, K, dtype=_dtype(variant), device="cuda")
    return (eye.t() if variant.startswith("f16_cm") else eye).contiguous().reshape(-1)


@pytest.mark.parametrize("case", FULL, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_ones_times_ones_full_size(case):
    variant, M, N, K, kernel, launches = case
    dt = _dtype(variant)
    dA = torch.ones(M * K, dtype=dt, device="cuda")
    dB = torch.ones(K * N, dtype=dt, device="cuda")
    dC, name, n = _call(variant, dA, dB, M, N, K)
    assert name == kernel
    if launches is not None:
        assert n == launches, (name, n)
    want = compare.round_to(variant.replace("_noalloc", ""), np.array([float(K)]))[0]
    got = dC.float()
    bad = int((got != float(want)).sum().item())
    assert bad == 0, (name, bad, torch.unique(got)[:8].tolist())


@pytest.mark.parametrize("case", FULL, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_identity_times_B_full_size(case):
    variant, M, N, K, kernel, _ = case
    base = variant.replace("_noalloc", "")
    b = synthetic.matrix(base.split("_")[0], K, N, synthetic.seed_for(9, 7))  # storage order of the variant
    if b.dtype == np.float32:
        dB = torch.from_numpy(b).cuda()
    else:
        dB = torch.from_numpy(b.view(np.int16)).cuda().view(_dtype(variant))
    dA = _storage_identity(variant, M, K)
    dC, name, _ = _call(variant, dA, dB, M, N, K)
    assert name == kernel
    r = min(M, K)
    if variant.startswith("f16_cm"):
        # column-major: column j of C holds rows 0..M-1 of column j of B
        got = dC.reshape(N, M)
        want = torch.zeros(N, M, dtype=dB.dtype, device="cuda")
        want[:, :r] = dB.reshape(N, K)[:, :r]
    else:
        got = dC.reshape(M, N)
        want = torch.zeros(M, N, dtype=dB.dtype, device="cuda")
        want[:r] = dB.reshape(K, N)[:r]
    # values compared (a zero product may leave -0 where +0 is stored)
    bad = int((got.float() != want.float()).sum().item())
    assert bad == 0, (name, bad)
