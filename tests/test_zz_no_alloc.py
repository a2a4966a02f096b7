"""The allocation-free bf16 entry point, through the C ABI.

It serves callers that cannot call cudaMalloc -- applications whose device
memory is owned by their own allocator, or latency-critical paths that cannot
afford cudaMalloc's implicit synchronisation.  Its result must match the
regular allocating entry point gemm_bf16_rm within the tolerance the parity
tests use, on two calls in a row (the second reuses the static scratch the
first one left behind).  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu


def _bits_to_f64(t: torch.Tensor) -> np.ndarray:
    h = t.cpu().numpy().view(np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("shape", [(1024, 12288, 4096), (1000, 1000, 1000), (300, 520, 264), (256, 512, 100),
                                   (1024, 2048, 1028), (32, 4096, 4096)])
def test_noalloc_matches_allocating_entry_point(lib, shape):
    M, N, K = shape
    clib = g.load()
    A, B = synthetic.problem_inputs("bf16_rm", M, N, K, 3, "normal", 1.0, "normal", 1.0 / 64.0)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    ref = torch.empty(M * N, dtype=torch.int16, device="cuda")
    out = torch.full((M * N,), -1, dtype=torch.int16, device="cuda")
    clib.gemm_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))

    assert clib.gemm_bf16_rm(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), M, N, K) == 0
    torch.cuda.synchronize()
    want = _bits_to_f64(ref)
    tol = compare.tol_half(want, K, "bf16")

    for call in range(2):
        out.fill_(-1)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = clib.gemm_bf16_rm_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K)
        assert st == 0, clib.gemm_last_error()
        assert clib.gemm_last_kernel() == b"umma_bf16_noalloc"
        torch.cuda.synchronize()
        if call == 1:
            # the second call (set-up done) leaves device memory untouched
            assert torch.cuda.mem_get_info()[0] == free_before
        got = _bits_to_f64(out)
        assert np.all(np.abs(got - want) <= tol), f"call {call}: max err {np.max(np.abs(got - want))}"


def test_noalloc_rejects_what_the_tensor_core_kernel_cannot_run(lib):
    clib = g.load()
    buf = torch.zeros(1 << 20, dtype=torch.int16, device="cuda")
    p = buf.data_ptr()
    # K = 102: A's rows are only 4-byte aligned, neither TMA nor 8-byte cp.async
    st = clib.gemm_bf16_rm_noalloc(p, p + 2 * 200 * 102, p + 2 * 400 * 102, 200, 128, 102)
    assert st == 1 and b"aligned" in clib.gemm_last_error()
    # unaligned A
    st = clib.gemm_bf16_rm_noalloc(p + 2, p + 2 * 300 * 128, p + 2 * 600 * 128, 256, 128, 128)
    assert st == 1
    # host-side checks as in gemm_bf16_rm
    assert clib.gemm_bf16_rm_noalloc(p, p, p, -1, 8, 8) == 1
    assert clib.gemm_bf16_rm_noalloc(p, p + 1024, p + 2048, 64, 64, 64) == 2
    assert clib.gemm_bf16_rm_noalloc(p, p, p, 0, 8, 8) == 0
