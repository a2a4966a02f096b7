"""Failure detection without a GPU fault: the tensor-core kernel's pipeline waits
are bounded, so a kernel whose producer never issues a load gives up after about
two seconds, records a timeout that gemm_synchronize reports, and leaves the
context usable for the next call."""

import time

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(lib):
    M, N, K = 256, 256, 256
    A, B = synthetic.problem_inputs("bf16_rm", M, N, K, 9)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.zeros(M * N, dtype=torch.int16, device="cuda")
    g.gemm_synchronize()                      # no stale timeout record
    g.gemm_force_kernel("umma_stall")
    try:
        g.gemm_bf16_rm(dA, dB, dC, M, N, K)   # the launch itself succeeds
        assert g.gemm_last_kernel() == "umma_stall"
    finally:
        g.gemm_force_kernel(None)
    t0 = time.time()
    with pytest.raises(g.GemmError) as err:
        g.gemm_synchronize()
    elapsed = time.time() - t0
    assert err.value.status == 5              # GEMM_ERR_TIMEOUT
    assert 1.0 < elapsed < 30.0
    g.gemm_synchronize()                      # the record was cleared
    # the same context computes correctly afterwards
    g.gemm_bf16_rm(dA, dB, dC, M, N, K)
    g.gemm_synchronize()
    h = dC.cpu().numpy().view(np.uint16)
    C = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(M, N)
    C_ref, S = oracle.gemm("bf16_rm", A, B, M, N, K)
    assert compare.check("bf16_rm", C, C_ref, S, K)["ok"]
