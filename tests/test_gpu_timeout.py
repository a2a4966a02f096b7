"""Failure detection without a GPU fault: the tensor-core kernels' pipeline waits
are bounded, so a kernel whose producers never issue a load gives up after about
two seconds, records a timeout that gemm_synchronize reports, and leaves the
context usable for the next call.  Both the single-CTA kernel ("umma_stall") and
the CTA-pair kernel ("umma_stall_pair": the leader's MMA thread gives up and
raises the abort flag of both CTAs of the pair; "umma_stall_peer": the pair's
second CTA gives up after one stage while the first has loaded further, and
the first waits for its own outstanding loads before the pair ends) are
exercised."""

import time

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("family,M", [("umma_stall", 256), ("umma_stall_pair", 512), ("umma_stall_peer", 512)])
def test_bounded_wait_reports_timeout_and_context_survives(lib, family, M):
    N, K = 256, 256
    A, B = synthetic.problem_inputs("bf16_rm", M, N, K, 9)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.zeros(M * N, dtype=torch.int16, device="cuda")
    g.gemm_synchronize()                      # no stale timeout record
    g.gemm_force_kernel(family)
    try:
        g.gemm_bf16_rm(dA, dB, dC, M, N, K)   # the launch itself succeeds
        assert g.gemm_last_kernel() == family
    finally:
        g.gemm_force_kernel(None)
    t0 = time.time()
    with pytest.raises(g.GemmError) as err:
        g.gemm_synchronize()
    elapsed = time.time() - t0
    assert err.value.status == 5              # GEMM_ERR_TIMEOUT
    # a wait that runs out takes about two seconds; a CTA that gives up at once
    # (umma_stall_peer) ends the pair without one
    assert elapsed < 30.0 and (family == "umma_stall_peer" or elapsed > 1.0)
    g.gemm_synchronize()                      # the record was cleared
    # the same context computes correctly afterwards
    g.gemm_bf16_rm(dA, dB, dC, M, N, K)
    g.gemm_synchronize()
    h = dC.cpu().numpy().view(np.uint16)
    C = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(M, N)
    C_ref, S = oracle.gemm("bf16_rm", A, B, M, N, K)
    assert compare.check("bf16_rm", C, C_ref, S, K)["ok"]
