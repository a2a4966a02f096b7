"""The packed-FMA SGEMM's split last round, against the oracle.

A plain FP32 problem of at least one full round of resident CTAs (three
128 x 64 tiles per SM) whose last round is part full, with at least 32 K
blocks of 16, runs as two grids: the whole rounds, then the remaining tiles
as clusters of two CTAs that each sum half of the K blocks and exchange their
halves through distributed shared memory.  The shapes below leave 12 to 405
tiles past full rounds on a 152-SM GB300 (of 456 slots).  Checked: whole rows from each
32-row quarter of every 128-row tile (the two CTAs of a cluster store
alternate quarters), the ragged last tiles in M, N and K, bit-identical
results on a second run, and back-to-back calls that read each other's C."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g
from gpu_util import run

pytestmark = pytest.mark.gpu

SEED = 37  # seed block of these problems


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def quarter_rows(M):
    rows = set()
    for b0 in range(0, M, 128):
        for off in (0, 31, 37, 63, 70, 95, 101, 127):
            if b0 + off < M:
                rows.add(b0 + off)
    rows.add(M - 1)
    return np.array(sorted(rows), dtype=np.int64)


def split_tail(M, N, K):
    """Tiles the library runs as K halves on this GPU (0: one grid)."""
    slots = 3 * torch.cuda.get_device_properties(0).multi_processor_count
    tiles = -(-M // 128) * -(-N // 64)
    rem = tiles % slots
    if tiles < slots or rem == 0 or -(-K // 16) < 32:
        return 0
    return rem


CASES = [
    (2300, 1660, 1000),   # 18 x 26 tiles: 12 past a round; ragged M, N and K (63 K blocks: 31 + 32)
    (2304, 2432, 2048),   # 18 x 38 tiles: 228 past a round, exactly half of it
    (2048, 2560, 512),    # 16 x 40 tiles: 184 past a round, the shortest K (16 + 16 blocks)
    (2560, 2560, 4096),   # 20 x 40 tiles: 344 past a round, more than half of it
    (2600, 2600, 1000),   # 21 x 41 tiles: 405 past a round; ragged M, N and K
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_split_tail_rows(case):
    M, N, K = case
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert split_tail(M, N, K) > 0
    A, B = synthetic.problem_inputs("f32_rm", M, N, K, SEED)
    C, name, _ = run("f32_rm", A, B, M, N, K)
    assert name == "simt_f32_vec4", name
    rows = quarter_rows(M)
    ref, S = oracle.gemm_rows("f32_rm", A, B, M, N, K, rows)
    res = compare.check("f32_rm", C[rows], ref, S, K)
    assert res["ok"], res
    assert np.all(np.isfinite(C))
    C2, _, _ = run("f32_rm", A, B, M, N, K)
    assert np.array_equal(C, C2), "not run-to-run deterministic"


def test_split_tail_back_to_back():
    """Three split problems queued with no synchronisation, each reading the
    previous one's C as its A: each stage agrees with the oracle applied to the
    C that stage read."""
    M, dims = 2304, [1024, 1664, 2432, 1664]
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert all(split_tail(M, dims[s + 1], dims[s]) > 0 for s in range(3))
    x = synthetic.matrix("f32", M, dims[0], synthetic.seed_for(SEED, 1), "normal", 1.0)
    ws = [synthetic.matrix("f32", dims[s], dims[s + 1], synthetic.seed_for(SEED, 2 + s), "normal",
                           1.0 / np.sqrt(dims[s])) for s in range(3)]
    a = torch.from_numpy(x).cuda()
    outs = []
    for s in range(3):
        c = torch.full((M * dims[s + 1],), -1.0, dtype=torch.float32, device="cuda")
        g.gemm_f32_rm(a, torch.from_numpy(ws[s]).cuda(), c, M, dims[s + 1], dims[s])
        outs.append(c)
        a = c
    g.gemm_synchronize()
    torch.cuda.synchronize()
    prev = x
    rows = quarter_rows(M)
    for s in range(3):
        K, N = dims[s], dims[s + 1]
        c = outs[s].cpu().numpy()
        ref, S = oracle.gemm_rows("f32_rm", prev, ws[s], M, N, K, rows)
        res = compare.check("f32_rm", c.reshape(M, N)[rows].astype(np.float64), ref, S, K)
        assert res["ok"], (s, res)
        prev = c


def test_launch_count():
    """The library counts its launches: two grids for a split problem, one
    otherwise."""
    for (M, N, K), want in (((2304, 2432, 2048), 2 if split_tail(2304, 2432, 2048) else 1),
                            ((256, 256, 256), 1)):
        a = torch.zeros(M * K, dtype=torch.float32, device="cuda")
        b = torch.zeros(K * N, dtype=torch.float32, device="cuda")
        c = torch.empty(M * N, dtype=torch.float32, device="cuda")
        n0 = g.gemm_kernel_launches()
        g.gemm_f32_rm(a, b, c, M, N, K)
        assert g.gemm_kernel_launches() - n0 == want
        g.gemm_synchronize()
        assert torch.count_nonzero(c).item() == 0
