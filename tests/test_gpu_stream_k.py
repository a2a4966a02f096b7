"""The stream-K tail of the CTA-pair tensor-core kernel, against the oracle.

When the 256 x 256 tiles leave the last wave nearly empty (at most a quarter
of the clusters) and K is long (at least 48 K-blocks), the K iterations of the
remainder tiles are spread over the clusters and each such tile is the sum, in
K order, of two to five FP32 partials.  The shapes below make 80 or 81 tiles,
4 to 7 tiles past a full wave of the 74-76 CTA pairs of a GB300; two more make
192 tiles, 40 past two waves, which run as whole tiles; four more are under a
quarter of a wave with at least 64 K-blocks, and every one of their tiles is
split.  Checked: whole rows
from every quarter of both CTA halves of every 256-row band (so every tile,
stream-K or not, is hit), and bit-identical results on a second run."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

from gpu_util import run

pytestmark = pytest.mark.gpu

SEED = 23  # seed block of these problems


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def band_rows(M):
    rows = set()
    for b0 in range(0, M, 256):
        for off in (0, 37, 70, 101, 133, 168, 200, 255):
            if b0 + off < M:
                rows.add(b0 + off)
    return np.array(sorted(rows), dtype=np.int64)


CASES = [
    ("bf16_rm", 2048, 2560, 3072),  # 8 x 10 tiles
    ("bf16_rm", 2304, 2296, 3080),  # 9 x 9 tiles, ragged N and K
    ("f16_cm", 2560, 2048, 3072),   # C^T = B^T A^T: 8 x 10 tiles
    ("bf16_rm", 1024, 12288, 2048), # 4 x 48 tiles: 40 in the last wave
    ("bf16_rm", 1000, 12040, 1032), # 4 x 48 tiles, ragged M, N and K
    # problems under a quarter of a wave with long K: stream-K over every tile, 4 shares each
    ("bf16_rm", 768, 768, 4096),    # 9 tiles on 36 clusters, 16 K-blocks per share
    ("bf16_rm", 520, 776, 4104),    # 12 tiles of 65 K-blocks, ragged M, N and K: shares cross tiles
    ("f16_cm", 1000, 520, 4104),    # C^T: 12 tiles of 65 K-blocks, shares of 17
    ("bf16_rm", 256, 256, 4160),    # one tile, four shares
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_stream_k_tail_rows(case):
    variant, M, N, K = case
    A, B = synthetic.problem_inputs(variant, M, N, K, SEED)
    C, name, _ = run(variant, A, B, M, N, K)
    assert name.startswith("umma"), name
    if variant == "f16_cm":
        # the tiles are those of C^T: check whole columns of C as well
        cols = band_rows(N)
        ii = np.repeat(np.arange(M), len(cols))
        jj = np.tile(cols, M)
        ref, S = oracle.gemm_entries(variant, A, B, M, N, K, ii, jj)
        res = compare.check(variant, C[ii, jj], ref, S, K)
        assert res["ok"], res
    rows = band_rows(M)
    ref, S = oracle.gemm_rows(variant, A, B, M, N, K, rows)
    res = compare.check(variant, C[rows], ref, S, K)
    assert res["ok"], res
    assert np.all(np.isfinite(C))
    C2, _, _ = run(variant, A, B, M, N, K)
    assert np.array_equal(C, C2), "not run-to-run deterministic"
