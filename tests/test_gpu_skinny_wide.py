"""The wide skinny tensor-core kernel ("umma_skinny_wide"), through the C ABI.

It gives each 256-column strip of B to a cluster of CS CTAs (CS = 1 .. 8) that
split K and add their partials through distributed shared memory in rank order.
The cases cover every CS the dispatch picks (1: a single K block or more strips
than SMs; 3: N = 12288; 8: narrow problems), strips cut by the right edge of C
(8, 136, 184 and 200 columns: one or two 128-column halves, a W box partly or
wholly outside B), ragged K (K % 64 != 0), M from 1 to 64 (X boxes of 8 to 64
rows), more strips than SMs (two waves), and FP16 through the column-major entry
point (the swap makes the row-major M the column-major N).  Random inputs
against the oracle element by element; closed forms bit for bit at the decode
size; a second call bit-identical.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

from gpu_util import run

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu

TEST_CONFIG = 9
FORCE = "umma_skinny_wide"

# (variant, M, N, K): M, N, K of the entry point's own problem
CASES = [
    ("bf16_rm", 1, 4096, 4096),     # 16 strips x CS 8
    ("bf16_rm", 5, 1032, 1000),     # last strip 8 columns (one half, one W box); K = 1000
    ("bf16_rm", 17, 2056, 2056),    # 9 strips x 8
    ("bf16_rm", 33, 520, 12296),    # 3 strips x 8, 193 K blocks
    ("bf16_rm", 64, 12288, 512),    # 48 strips x 3, M = 64
    ("bf16_rm", 48, 136, 25600),    # one strip of 136 columns: two halves, three W boxes
    ("bf16_rm", 8, 12288, 1024),    # 48 x 3
    ("bf16_rm", 64, 200, 64),       # one K block: CS 1; the fourth W box partly outside B
    ("bf16_rm", 2, 40000, 128),     # 157 strips: more than the SMs, CS 1
    ("f16_cm", 3000, 24, 1000),     # row-major M = 24, N = 3000 (last strip 184 columns)
    ("f16_cm", 2048, 1, 768),       # row-major M = 1
]


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def _kernel(variant):
    return "umma_skinny_wide_f16" if variant.startswith("f16") else "umma_skinny_wide_bf16"


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_matches_oracle_and_is_deterministic(case):
    variant, M, N, K = case
    A, B = synthetic.problem_inputs(variant, M, N, K, TEST_CONFIG)
    C, name, _ = run(variant, A, B, M, N, K, force=FORCE)
    assert name == _kernel(variant)
    C_ref, S = oracle.gemm(variant, A, B, M, N, K)
    res = compare.check(variant, C, C_ref, S, K)
    assert res["ok"], res
    C2, _, _ = run(variant, A, B, M, N, K, force=FORCE)
    assert np.array_equal(C, C2), "not run-to-run deterministic"


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_closed_forms_at_decode_size(M):
    """ones·ones = K = 4096 (exact in bf16) and I·B = B's first M rows, at the
    decode projection N = 12288, K = 4096 (48 strips on clusters of 3)."""
    N, K = 12288, 4096
    ones_a = torch.ones(M * K, dtype=torch.bfloat16, device="cuda")
    ones_b = torch.ones(K * N, dtype=torch.bfloat16, device="cuda")
    out = torch.full((M * N,), -1.0, dtype=torch.bfloat16, device="cuda")
    g.gemm_force_kernel(FORCE)
    try:
        g.gemm_bf16_rm(ones_a, ones_b, out, M, N, K)
        assert g.gemm_last_kernel() == "umma_skinny_wide_bf16"
    finally:
        g.gemm_force_kernel(None)
    g.gemm_synchronize()
    assert int((out.float() != 4096.0).sum().item()) == 0

    b = synthetic.matrix("bf16", K, N, synthetic.seed_for(9, 8))
    dB = torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
    eye = torch.eye(M, K, dtype=torch.bfloat16, device="cuda").reshape(-1)
    g.gemm_force_kernel(FORCE)
    try:
        g.gemm_bf16_rm(eye, dB, out, M, N, K)
    finally:
        g.gemm_force_kernel(None)
    g.gemm_synchronize()
    want = dB.reshape(K, N)[:M].float()
    assert int((out.reshape(M, N).float() != want).sum().item()) == 0


def test_rejects_what_it_cannot_run():
    buf = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
    g.gemm_force_kernel(FORCE)
    try:
        for (M, N, K) in [(65, 64, 64), (8, 64, 100), (8, 60, 64)]:  # M > 64, K % 8, N % 8
            with pytest.raises(g.GemmError):
                g.gemm_bf16_rm(buf, buf[8192:], buf[32768:], M, N, K)
    finally:
        g.gemm_force_kernel(None)
