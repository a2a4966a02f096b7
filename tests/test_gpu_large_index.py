"""Largest-size cases: operands of more than 2^31 elements, so that every
element offset past the first 2^31 needs 64-bit index arithmetic in the
kernels (row * K, k * N).  To keep host memory small, a large operand is a
seeded block repeated along its long dimension (row r of A is row r mod R of
the block); the oracle checks sampled outputs on the same repeated values,
including the last rows and columns, computed from the plain definition on the
sampled rows or columns."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu
CFG = 0xB16
BLOCK = 1024


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield lib
    torch.cuda.empty_cache()


def tiled_rows(block, rows, cols, dtype):
    """Device tensor of `rows` x `cols` whose row r is block[r % len(block)]."""
    tdt = torch.float32 if dtype == "f32" else torch.int16
    hb = torch.from_numpy(block.reshape(-1, cols) if dtype == "f32" else block.reshape(-1, cols).view(np.int16))
    db = hb.cuda()
    out = torch.empty((rows, cols), dtype=tdt, device="cuda")
    nb = db.shape[0]
    for r0 in range(0, rows, nb):
        n = min(nb, rows - r0)
        out[r0:r0 + n].copy_(db[:n])
    return out.reshape(-1)


def widen(dtype, t):
    h = t.cpu().numpy()
    if dtype == "f32":
        return h.astype(np.float64)
    if dtype == "f16":
        return h.view(np.float16).astype(np.float64)
    return (h.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype,M,N,K,expect", [
    ("bf16", 65600, 256, 32768, "umma_bf16"),      # A: 2.15e9 elements, 4.3 GB
    ("f32", 65600, 128, 32768, "simt_f32_vec4"),   # A: 2.15e9 elements, 8.6 GB
])
def test_A_beyond_2_31_elements(dtype, M, N, K, expect):
    assert M * K > 2 ** 31
    blk = synthetic.matrix(dtype, BLOCK, K, synthetic.seed_for(CFG, 1))
    B = synthetic.matrix(dtype, K, N, synthetic.seed_for(CFG, 2))
    dA = tiled_rows(blk, M, K, dtype)
    dB = torch.from_numpy(B if dtype == "f32" else B.view(np.int16)).cuda()
    dC = torch.empty(M * N, dtype=dA.dtype, device="cuda")
    getattr(g, f"gemm_{dtype}_rm")(dA, dB, dC, M, N, K)
    assert g.gemm_last_kernel() == expect
    g.gemm_synchronize()
    C = widen(dtype, dC).reshape(M, N)
    rows = np.array([0, 1, BLOCK - 1, 2 ** 31 // K - 1, 2 ** 31 // K, 2 ** 31 // K + 1, M - 2, M - 1])
    A_rows = blk.reshape(BLOCK, K)[rows % BLOCK]
    C_ref, S = oracle.gemm(f"{dtype}_rm", A_rows.reshape(-1), B, len(rows), N, K)
    res = compare.check(f"{dtype}_rm", C[rows], C_ref, S, K)
    assert res["ok"], res
    del dA, dB, dC


@pytest.mark.parametrize("force,expect", [(None, "umma_bf16"), ("gemv", "gemv_bf16")])
def test_decode_weights_beyond_2_31_elements(force, expect):
    """M = 1 with W [65536, 32800] bf16 (2.15e9 elements): the 256-column skinny
    tensor-core kernel (129 strips) and the GEMV."""
    M, N, K = 1, 32800, 65536
    assert K * N > 2 ** 31
    x = synthetic.matrix("bf16", 1, K, synthetic.seed_for(CFG, 3))
    wblk = synthetic.matrix("bf16", BLOCK, N, synthetic.seed_for(CFG, 4))
    dW = tiled_rows(wblk, K, N, "bf16")
    dx = torch.from_numpy(x.view(np.int16)).cuda()
    dc = torch.empty(N, dtype=torch.int16, device="cuda")
    g.gemm_force_kernel(force)
    try:
        g.gemm_bf16_rm(dx, dW, dc, M, N, K)
        assert g.gemm_last_kernel().startswith(expect)
    finally:
        g.gemm_force_kernel(None)
    g.gemm_synchronize()
    c = widen("bf16", dc)
    cols = np.array([0, 1, 1023, 16384, N - 2, N - 1])
    W_cols = wblk.reshape(BLOCK, N)[:, cols][np.arange(K) % BLOCK]   # [K, len(cols)]
    c_ref, S = oracle.gemm("bf16_rm", x, np.ascontiguousarray(W_cols).reshape(-1), 1, len(cols), K)
    res = compare.check("bf16_rm", c[cols][None, :], c_ref, S, K)
    assert res["ok"], res
    del dW
