"""bench.py's CPU-baseline leg (no GPU): the oracle's timed sample of output
rows is spread over all of M, and the same rows of the timed output buffer are
checked against it; a wrong element or a transposed layout is caught."""

import numpy as np
import pytest

import bench
import oracle
import synthetic


def test_sample_rows_spread_over_m():
    assert list(bench.sample_rows(10, 1)) == [0]
    assert list(bench.sample_rows(10, 4)) == [0, 3, 6, 9]
    r = bench.sample_rows(4096, 700)
    assert r[0] == 0 and r[-1] == 4095 and len(np.unique(r)) == 700
    assert len(bench.sample_rows(5, 50)) == 5


def _library_like_output(variant, A, B, M, N, K):
    """The oracle's full product rounded to the output type and laid out as the
    library stores it (what a correct GPU run leaves in C)."""
    C, _ = oracle.gemm(variant, A, B, M, N, K)
    if variant == "f32_rm":
        return C.astype(np.float32).reshape(-1)
    if variant == "bf16_rm":
        return synthetic.f32_to_bf16_bits(C.astype(np.float32)).reshape(-1).view(np.int16)
    return synthetic.f32_to_f16_bits(C.astype(np.float32)).T.reshape(-1).view(np.int16)  # column-major


@pytest.mark.parametrize("variant", ["f32_rm", "bf16_rm", "f16_cm"])
def test_parity_of_the_sampled_rows(variant):
    M, N, K = 70, 48, 40
    A, B = synthetic.problem_inputs(variant, M, N, K, 1)
    fps, nrows, dt, threads, rows, ref = bench.cpu_sample(variant, A, B, M, N, K, 0.01)
    assert fps > 0 and ref is not None and len(rows) == nrows
    host_c = _library_like_output(variant, A, B, M, N, K)
    good = bench.sample_parity(variant, host_c, M, N, K, rows, ref)
    assert good["ok"] and good["rows"] == len(rows) and good["elements"] == len(rows) * N
    # one wrong element in a sampled row
    bad = host_c.copy()
    i = int(rows[len(rows) // 2])
    if variant == "f16_cm":
        bad[i + 5 * M] = bad[i + 5 * M] ^ 0x4000
    elif variant == "bf16_rm":
        bad[i * N + 5] = bad[i * N + 5] ^ 0x4000
    else:
        bad[i * N + 5] += 1.0
    assert not bench.sample_parity(variant, bad, M, N, K, rows, ref)["ok"]


def test_a_transposed_layout_is_caught():
    M, N, K = 64, 64, 32
    A, B = synthetic.problem_inputs("f32_rm", M, N, K, 2)
    _, _, _, _, rows, ref = bench.cpu_sample("f32_rm", A, B, M, N, K, 0.01)
    C = _library_like_output("f32_rm", A, B, M, N, K).reshape(M, N).T.reshape(-1).copy()
    assert not bench.sample_parity("f32_rm", C, M, N, K, rows, ref)["ok"]


def test_other_variants_give_no_reference():
    M, N, K = 8, 16, 32
    A = synthetic.matrix("bf16", M, K, synthetic.seed_for(3, 1))
    B = synthetic.matrix("bf16", K, N, synthetic.seed_for(3, 2))
    W = synthetic.matrix("bf16", K, N, synthetic.seed_for(3, 3))
    flops, ref = bench.oracle_rows("bf16_silu_mul", A, B, M, N, K, np.arange(M), (W,))
    assert ref is None and flops == 4.0 * M * N * K
