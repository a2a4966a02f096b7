"""Parity of the FP8 path with the oracle, through the C ABI ("Chapter 5
Operators and Runtime", examples 5-7 and 5-8).

The row-wise quantisation decides integer codes with floating point, so both
sides take those decisions in FP32 and the codes and scales must match bit for
bit.  The row-scaled E4M3 product is compared element by element within
``compare.tol_e4m3`` on the oracle's own codes, on small shapes in full and on
the pages' workload (A [4096,4096], W [4096,1536]) on sampled rows."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu
CFG = 0xF8


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def half_rows(M, K, seed, spread=True):
    """Half bits of a seeded [M,K] matrix whose rows span very different scales."""
    x = synthetic.normal(synthetic.seed_for(CFG, seed), M * K).reshape(M, K)
    if spread:
        x = x * np.exp2(np.arange(M) % 24 - 12)[:, None]   # 2^-12 .. 2^11
    return synthetic.f32_to_f16_bits(x.astype(np.float32).reshape(-1)).reshape(M, K)


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1)).cuda()


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.int16)).cuda()


def quantize_gpu(A, M, K, a_off=0, q_off=0):
    big = torch.zeros(M * K + a_off, dtype=torch.int16, device="cuda")
    dA = big[a_off:]
    dA.copy_(dev_u16(A))
    qbig = torch.full((M * K + q_off,), 0x5A, dtype=torch.uint8, device="cuda")
    dQ = qbig[q_off:]
    dS = torch.full((M,), -1.0, dtype=torch.float32, device="cuda")
    g.gemm_quantize_rows_e4m3(dA, dQ, dS, M, K)
    name = g.gemm_last_kernel()
    g.gemm_synchronize()
    return dQ.cpu().numpy().reshape(M, K), dS.cpu().numpy(), name


@pytest.mark.parametrize("M,K,a_off,q_off,expect", [
    (64, 4096, 0, 0, "quantize_e4m3_vec"), (37, 304, 0, 0, "quantize_e4m3_vec"),
    (37, 300, 0, 0, "quantize_e4m3_scalar"), (5, 4096, 1, 0, "quantize_e4m3_scalar"),
    (9, 64, 0, 3, "quantize_e4m3_scalar"), (1, 8, 0, 0, "quantize_e4m3_vec"), (300, 1000, 0, 0, "quantize_e4m3_vec"),
    (12, 8200, 0, 0, "quantize_e4m3_vec"), (20, 2056, 0, 0, "quantize_e4m3_vec"),
    (7, 5000, 0, 0, "quantize_e4m3_vec"), (33, 8192, 0, 0, "quantize_e4m3_vec")])
# K > 8192: two passes over A; K > 4096: a row held by two warps (M = 7: a CTA
# with one row past M); else a row held by one warp
def test_quantize_rows_bit_exact(M, K, a_off, q_off, expect):
    A = half_rows(M, K, 1)
    if M > 6:
        A[3] = 0                              # a row of zeros
        A[4, :] = 0
        A[4, K - 1] = synthetic.f32_to_f16_bits(np.array([-3.0], dtype=np.float32))[0]  # max at the end
        A[6] = synthetic.f32_to_f16_bits(np.full(K, 2.0 ** -20, dtype=np.float32))     # subnormal halves
    Q, S, name = quantize_gpu(A, M, K, a_off, q_off)
    assert name == expect
    Qr, Sr = oracle.quantize_rows_e4m3(A, M, K)
    assert np.array_equal(Q, Qr)
    assert np.array_equal(S.view(np.uint32), Sr.view(np.uint32))


def test_quantize_worked_example_5_7():
    """One row of 256: 1 at position 0 and 10 at position 128 -> code of 44."""
    row = np.zeros((1, 256), dtype=np.float16)
    row[0, 0], row[0, 128] = 1, 10
    Q, S, _ = quantize_gpu(row.view(np.uint16), 1, 256)
    assert oracle.decode_e4m3(Q[0, :1])[0] == 44.0
    assert oracle.decode_e4m3(Q[0, 128:129])[0] == 448.0
    assert S[0] == np.float32(10) / np.float32(448)


def rowscale_case(M, N, K, seed):
    # rows of N(0,1) halves (a spread of row scales would overflow the half output)
    A = half_rows(M, K, seed, spread=False)
    Q, S = oracle.quantize_rows_e4m3(A, M, K)
    W = synthetic.e4m3_codes(N, K, synthetic.seed_for(CFG, seed + 50))
    return Q, S, W


def run_rowscale(Q, S, W, M, N, K):
    dQ, dS, dW = dev_u8(Q), torch.from_numpy(S).cuda(), dev_u8(W)
    dC = torch.full((M * N,), 0x7E00, dtype=torch.int16, device="cuda")
    g.gemm_e4m3_rowscale(dQ, dS, dW, dC, M, N, K)
    name = g.gemm_last_kernel()
    g.gemm_synchronize()
    C = dC.cpu().numpy().view(np.float16).astype(np.float64).reshape(M, N)
    return C, name


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 200, 272), (512, 1536, 4096), (1, 8, 16),
                                   (130, 264, 4112), (1024, 392, 640)])
def test_rowscale_product(M, N, K):
    Q, S, W = rowscale_case(M, N, K, 2)
    C, name = run_rowscale(Q, S, W, M, N, K)
    assert name == "umma_e4m3_rowscale"
    C_ref, Sab = oracle.gemm_e4m3_rowscale(Q, S, W, M, N, K)
    assert np.isfinite(C_ref).all() and np.abs(C_ref).max() < 60000
    res = compare.check_e4m3(C, C_ref, Sab)
    assert res["ok"], res


def test_rowscale_pages_workload_sampled_rows():
    """Example 5-8's shapes: A [4096,4096] half quantised on the GPU, W [4096,1536]
    E4M3 (given as Wt [1536,4096]); codes checked in full, the product on rows."""
    M, K, N = 4096, 4096, 1536
    A = half_rows(M, K, 3, spread=False)
    Qg, Sg, _ = quantize_gpu(A, M, K)
    Q, S = oracle.quantize_rows_e4m3(A, M, K)
    assert np.array_equal(Qg, Q) and np.array_equal(Sg.view(np.uint32), S.view(np.uint32))
    W = synthetic.e4m3_codes(N, K, synthetic.seed_for(CFG, 60))
    C, _ = run_rowscale(Q, S, W, M, N, K)
    rows = np.concatenate([np.random.default_rng(0).integers(0, M, 48), [0, 255, 256, M - 1]])
    C_ref, Sab = oracle.gemm_e4m3_rowscale(Q, S, W, M, N, K, rows=rows)
    res = compare.check_e4m3(C[rows], C_ref, Sab)
    assert res["ok"], res


def test_rowscale_k_zero_and_rejections():
    M, N = 64, 64
    dC = torch.full((M * N,), 0x3C00, dtype=torch.int16, device="cuda")
    q = torch.zeros(16, dtype=torch.uint8, device="cuda")
    s = torch.ones(M, dtype=torch.float32, device="cuda")
    g.gemm_e4m3_rowscale(q, s, q, dC, M, N, 0)
    g.gemm_synchronize()
    assert not dC.any()
    Q = torch.zeros(M * 24, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GemmError, match="INVALID"):
        g.gemm_e4m3_rowscale(Q, s, Q, dC, M, N, 24)     # K % 16 != 0
    assert "K % 16" in g.gemm_last_error()


# ---------------------------------------------------------- quantisation fused into the product
def run_fused(A, W, M, N, K):
    dA, dW = dev_u16(A), dev_u8(W)
    dC = torch.full((M * N,), 0x7E00, dtype=torch.int16, device="cuda")
    g.gemm_e4m3_rowscale_fused(dA, dW, dC, M, N, K)
    name = g.gemm_last_kernel()
    g.gemm_synchronize()
    return dC.cpu().numpy().view(np.float16).astype(np.float64).reshape(M, N), name


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 200, 272), (512, 1536, 4096), (1, 8, 16),
                                   (130, 264, 4112), (1024, 392, 640), (600, 1000, 1008)])
def test_fused_quantisation_product(M, N, K):
    """The fused scheme against the oracle (quantise the rows, then the row-scaled
    product), and bit for bit against the separate scheme on the same tiles:
    the converter warps must write the quantiser's very codes."""
    A = half_rows(M, K, 4, spread=False)
    if M > 6:
        A[3] = 0                               # a row of zeros: codes 0, scale 0
        A[5, :] = 0
        A[5, K - 1] = synthetic.f32_to_f16_bits(np.array([-3.0], dtype=np.float32))[0]
    W = synthetic.e4m3_codes(N, K, synthetic.seed_for(CFG, 70))
    C, name = run_fused(A, W, M, N, K)
    assert name == "umma_e4m3_rowscale_fused"
    Q, S = oracle.quantize_rows_e4m3(A, M, K)
    C_ref, Sab = oracle.gemm_e4m3_rowscale(Q, S, W, M, N, K)
    res = compare.check_e4m3(C, C_ref, Sab)
    assert res["ok"], res
    # the separate scheme (no stream-K tail below K = 48 blocks of 128): same bits
    Qg, Sg, _ = quantize_gpu(A, M, K)
    C_sep, _ = run_rowscale(Qg, Sg, W, M, N, K)
    assert np.array_equal(C.view(np.uint64), C_sep.view(np.uint64))


def test_fused_quantisation_pages_workload_sampled_rows():
    """Example 5-8's shapes (A [4096,4096] half, W [4096,1536] E4M3): the fused
    product equals the separate one bit for bit and the oracle on sampled rows."""
    M, K, N = 4096, 4096, 1536
    A = half_rows(M, K, 3, spread=False)
    W = synthetic.e4m3_codes(N, K, synthetic.seed_for(CFG, 60))
    C, _ = run_fused(A, W, M, N, K)
    Qg, Sg, _ = quantize_gpu(A, M, K)
    C_sep, _ = run_rowscale(Qg, Sg, W, M, N, K)
    assert np.array_equal(C.view(np.uint64), C_sep.view(np.uint64))
    rows = np.concatenate([np.random.default_rng(1).integers(0, M, 48), [0, 255, 256, M - 1]])
    Q, S = oracle.quantize_rows_e4m3(A[rows], rows.size, K)
    C_ref, Sab = oracle.gemm_e4m3_rowscale(Q, S, W, rows.size, N, K)
    res = compare.check_e4m3(C[rows], C_ref, Sab)
    assert res["ok"], res


def test_fused_quantisation_k_zero_and_rejections():
    M, N = 64, 64
    dC = torch.full((M * N,), 0x3C00, dtype=torch.int16, device="cuda")
    a = torch.zeros(M * 32 + 8, dtype=torch.int16, device="cuda")
    w = torch.zeros(N * 32, dtype=torch.uint8, device="cuda")
    g.gemm_e4m3_rowscale_fused(a, w, dC, M, N, 0)
    g.gemm_synchronize()
    assert not dC.any()
    with pytest.raises(g.GemmError, match="INVALID"):
        g.gemm_e4m3_rowscale_fused(a, w, dC, M, N, 24)    # K % 16 != 0
    with pytest.raises(g.GemmError, match="INVALID"):
        g.gemm_e4m3_rowscale_fused(a[1:], w, dC, M, N, 32)  # A not 16-byte aligned
    assert "aligned" in g.gemm_last_error()
