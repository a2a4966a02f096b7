"""The allocation-free bf16 entry point, through the C ABI.

gemm_bf16_rm_noalloc serves callers that cannot call cudaMalloc: programs
whose device memory is owned by their own allocator (a framework's caching
pool that has already reserved the GPU, an embedding program with a fixed
memory budget) and latency-critical paths that cannot take cudaMalloc's
implicit synchronisation.  Its scratch -- the kernel's 4-byte timeout status
word -- lives in a static device array instead.

Each case runs it twice in a row (the second call finds the static array as the
first one left it) and checks every call against the CPU oracle with the
parity tests' bf16 tolerance, and against the regular entry point
gemm_bf16_rm within the same tolerance.  The library's own launch count must be
exactly one kernel per call: the regular entry point's allocating branches (A
staged into aligned rows, the stream-K tail with its fix-up kernel) each add a
kernel, so a call that took one of them would show.  This file is collected
last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

from gpu_util import check_bands

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu


def _bits_to_f64(t: torch.Tensor) -> np.ndarray:
    h = t.cpu().numpy().view(np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# (M, N, K, what gemm_bf16_rm does differently for this shape)
SHAPES = [
    (1000, 1000, 1000, "same kernel"),
    (300, 520, 264, "same kernel"),
    (256, 512, 100, "same kernel"),
    (32, 4096, 4096, "skinny kernel"),
    (8, 20480, 1024, "256-column skinny kernel (strips past the SM count)"),
    (1024, 2048, 1028, "stages A into aligned rows (K % 8 = 4)"),
    (1024, 12288, 4096, "same kernel (the FFN projection)"),
    (3072, 5120, 6144, "adds a stream-K tail and its fix-up kernel"),
    (8192, 4096, 4100, "stages A into aligned rows"),
]
FULL_ORACLE_FMAS = 3e9  # above this, whole rows and columns from every tile band


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}")
def test_noalloc_matches_oracle_and_allocating_entry_point(lib, shape):
    M, N, K, _ = shape
    clib = g.load()
    A, B = synthetic.problem_inputs("bf16_rm", M, N, K, 3, "normal", 1.0, "normal", 1.0 / 64.0)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    ref = torch.empty(M * N, dtype=torch.int16, device="cuda")
    out = torch.full((M * N,), -1, dtype=torch.int16, device="cuda")
    clib.gemm_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))

    # the regular (allocating) entry point on the same inputs
    assert clib.gemm_bf16_rm(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), M, N, K) == 0
    assert clib.gemm_synchronize() == 0
    regular = _bits_to_f64(ref).reshape(M, N)

    full = M * N * K <= FULL_ORACLE_FMAS
    if full:
        C_ref, S = oracle.gemm("bf16_rm", A, B, M, N, K)

    for call in range(2):
        out.fill_(-1)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        launches = clib.gemm_kernel_launches()
        st = clib.gemm_bf16_rm_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K)
        assert st == 0, clib.gemm_last_error()
        assert clib.gemm_kernel_launches() - launches == 1, "a kernel besides the GEMM was launched"
        assert clib.gemm_last_kernel() == b"umma_bf16_noalloc"
        assert clib.gemm_synchronize() == 0
        if call == 1:
            # the second call (set-up done) leaves device memory untouched
            assert torch.cuda.mem_get_info()[0] == free_before
        got = _bits_to_f64(out).reshape(M, N)
        if full:
            res = compare.check("bf16_rm", got, C_ref, S, K)
            assert res["ok"], (call, res)
        else:
            res_r, res_c = check_bands("bf16_rm", got, A, B, M, N, K)
            assert res_r["ok"] and res_c["ok"], (call, res_r, res_c)
        # against the regular entry point, within the same bf16 tolerance
        tol = compare.tol_half(regular, K, "bf16")
        err = np.abs(got - regular)
        assert np.all(err <= tol), f"call {call}: max err vs gemm_bf16_rm {err.max()}"


def test_noalloc_timeout_is_reported(lib):
    """A call whose pipeline waits run out (the "umma_stall" test hook: a
    producer that issues no loads) leaves its code in the static status word;
    gemm_synchronize reports it once, and the next call is correct."""
    clib = g.load()
    M, N, K = 256, 256, 128
    A, B = synthetic.problem_inputs("bf16_rm", M, N, K, 3)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    out = torch.full((M * N,), -1, dtype=torch.int16, device="cuda")
    clib.gemm_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert clib.gemm_force_kernel(b"umma_stall") == 0
    try:
        st = clib.gemm_bf16_rm_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K)
    finally:
        clib.gemm_force_kernel(None)
    assert st == 0 and clib.gemm_last_kernel() == b"umma_stall"
    assert clib.gemm_synchronize() == 5  # GEMM_ERR_TIMEOUT
    assert clib.gemm_synchronize() == 0  # reported once
    st = clib.gemm_bf16_rm_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K)
    assert st == 0 and clib.gemm_synchronize() == 0
    C_ref, S = oracle.gemm("bf16_rm", A, B, M, N, K)
    res = compare.check("bf16_rm", _bits_to_f64(out).reshape(M, N), C_ref, S, K)
    assert res["ok"], res


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
