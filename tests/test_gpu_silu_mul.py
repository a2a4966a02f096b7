"""The fused FFN gate/up projection Z = SiLU(X W_g) * (X W_u) ("Chapter 5
Operators and Runtime", section 5.3.1) against the oracle's chain with the same
rounding points, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu

FFN_CONFIG = 3


def inputs(M, N, K, cfg=FFN_CONFIG):
    X = synthetic.matrix("bf16", M, K, synthetic.seed_for(cfg, 1), "normal", 1.0)
    Wg = synthetic.matrix("bf16", K, N, synthetic.seed_for(cfg, 2), "normal", 1.0 / 64.0)
    Wu = synthetic.matrix("bf16", K, N, synthetic.seed_for(cfg, 3), "normal", 1.0 / 64.0)
    return X, Wg, Wu


def dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda()


def run(X, Wg, Wu, M, N, K):
    Z = torch.full((M * N,), -1, dtype=torch.int16, device="cuda")
    g.gemm_bf16_rm_silu_mul(dev(X), dev(Wg), dev(Wu), Z, M, N, K)
    name = g.gemm_last_kernel()
    g.gemm_synchronize()
    h = Z.cpu().numpy().view(np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(M, N), name


def check(Zg, r):
    Zr = r["Z"]
    tol = compare.tol_silu_mul(r["G"], r["U"], r["T"], Zr, r["S_G"], r["S_U"])
    err = np.abs(Zg - Zr)
    assert np.all(err <= tol), f"max err/tol {np.max(err / np.maximum(tol, 1e-300))}"
    exact = np.mean(Zg == Zr)
    assert exact >= 0.99, f"only {exact:.4f} of Z bit-exact with the oracle"


@pytest.mark.parametrize("shape", [(300, 520, 264), (256, 384, 128), (64, 256, 64), (520, 1032, 512),
                                   (1024, 2048, 4096)])
def test_silu_mul_matches_oracle(lib, shape):
    M, N, K = shape
    X, Wg, Wu = inputs(M, N, K)
    Zg, name = run(X, Wg, Wu, M, N, K)
    assert name == "umma_bf16_silu_mul"
    check(Zg, oracle.silu_mul(X, Wg, Wu, M, N, K))


def test_silu_mul_ffn_workload_sampled_rows(lib):
    """The FFN shape X[1024,4096], W[4096,12288]: every column of 48 sampled rows
    (first, last and random), and bit-identical on a second run."""
    M, N, K = 1024, 12288, 4096
    X, Wg, Wu = inputs(M, N, K)
    Zg, _ = run(X, Wg, Wu, M, N, K)
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(5).integers(0, M, 46)]))
    check(Zg[rows], oracle.silu_mul(X, Wg, Wu, M, N, K, rows=rows))
    Zg2, _ = run(X, Wg, Wu, M, N, K)
    assert np.array_equal(Zg, Zg2)


def test_silu_mul_edges(lib):
    M, N = 40, 64
    X, Wg, Wu = inputs(M, N, 8)
    Z = torch.full((M * N,), 7, dtype=torch.int16, device="cuda")
    g.gemm_bf16_rm_silu_mul(dev(X), dev(Wg), dev(Wu), Z, M, N, 0)   # K = 0: Z = 0
    torch.cuda.synchronize()
    assert torch.all(Z == 0)
    clib = g.load()
    buf = torch.zeros(1 << 20, dtype=torch.int16, device="cuda")
    p = buf.data_ptr()
    # unaligned X
    assert clib.gemm_bf16_rm_silu_mul(p + 2, p + 65536, p + 131072, p + 262144, 64, 64, 64) == 1
    # Z overlapping W_u
    assert clib.gemm_bf16_rm_silu_mul(p, p + 65536, p + 131072, p + 131072, 64, 64, 64) == 2
