"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Closed forms are compared bit for bit; random inputs element by element within
the tolerances (FP32: 1e-5 * sum_k |a_ik b_kj|; half/bf16: 1e-2 * sqrt(K/512) *
max(1, |C_ref|)); the full-size workloads on sampled outputs that the oracle
computes one by one.  Every kernel family the dispatcher can choose is hit.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

from gpu_util import run, to_device, empty_out, widen, check_bands

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu

VARIANTS = ["f32_rm", "f16_cm", "bf16_rm"]
TEST_CONFIG = 9  # seed block of the test-only problems


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def encode(variant, values):
    v = np.ascontiguousarray(values, dtype=np.float32).reshape(-1)
    if variant.startswith("f32"):
        return v
    if variant.startswith("f16"):
        return synthetic.f32_to_f16_bits(v)
    return synthetic.f32_to_bf16_bits(v)


def store(variant, mat):
    mat = np.asarray(mat)
    return mat.reshape(-1) if variant.endswith("_rm") else mat.T.reshape(-1)


def assert_parity(variant, C, A, B, M, N, K):
    C_ref, S = oracle.gemm(variant, A, B, M, N, K)
    res = compare.check(variant, C, C_ref, S, K)
    assert res["ok"], res


# ------------------------------------------------------------------ closed forms
CLOSED_SHAPES = [(256, 256, 256), (1000, 1000, 1000), (64, 64, 64), (1, 12288, 4096),
                 (300, 520, 264), (130, 200, 100), (8, 64, 4100)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", CLOSED_SHAPES)
def test_ones_times_ones_is_K(variant, shape):
    M, N, K = shape
    A = encode(variant, np.ones(M * K))
    B = encode(variant, np.ones(K * N))
    C, name, _ = run(variant, A, B, M, N, K)
    want = compare.round_to(variant, np.array([float(K)]))[0]
    assert np.all(C == want), (name, np.unique(C)[:8])


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(256, 256, 256), (300, 520, 264), (264, 136, 300), (1000, 1000, 1000),
                                   (5, 96, 40), (130, 200, 100)])
def test_identity_times_B_is_B(variant, shape):
    M, N, K = shape
    eye = np.eye(M, K, dtype=np.float32)
    b = synthetic.uniform_pm1(synthetic.seed_for(TEST_CONFIG, 2), K * N).reshape(K, N)
    A = encode(variant, store(variant, eye))
    B = encode(variant, store(variant, b))
    C, name, _ = run(variant, A, B, M, N, K)
    # the expected rows are B's stored values (already rounded to the type)
    if variant.startswith("f32"):
        b_val = b.astype(np.float64)
    elif variant.startswith("f16"):
        b_val = synthetic.f16_bits_to_f32(B).reshape(N, K).T.astype(np.float64)
    else:
        b_val = synthetic.bf16_bits_to_f32(B).reshape(K, N).astype(np.float64)
    want = np.zeros((M, N))
    r = min(M, K)
    want[:r] = b_val[:r]
    assert np.array_equal(C, want), name


# ------------------------------------------------------------------ random, mid size
# (variant, M, N, K, forced family or None, expected kernel or None)
MID_CASES = [
    ("f32_rm", 256, 256, 256, None, "simt_f32_vec4"),
    ("f32_rm", 300, 520, 272, None, "simt_f32_vec4"),
    ("f32_rm", 129, 68, 1000, None, "simt_f32_vec4"),
    ("f32_rm", 257, 131, 77, None, "simt_f32_scalar"),
    ("f32_rm", 1030, 700, 600, None, "simt_f32_vec4"),        # 99 tiles: every tile as two half-K CTAs
    ("f32_rm", 512, 520, 264, None, "simt_f32_vec4"),         # 36 tiles: the small-tile kernel
    ("f32_rm", 200, 300, 96, "simt_scalar", "simt_f32_scalar"),
    ("f32_rm", 5, 300, 999, None, "gemv_f32_vec"),
    ("f32_rm", 3, 301, 257, None, "gemv_f32_scalar"),
    ("f32_rm", 8, 1000, 520, "gemv_scalar", "gemv_f32_scalar"),
    ("bf16_rm", 300, 520, 264, None, "umma_bf16"),
    ("bf16_rm", 129, 264, 520, None, "umma_bf16"),
    ("bf16_rm", 640, 1024, 1024, None, "umma_bf16"),
    ("bf16_rm", 130, 200, 100, None, "umma_bf16"),          # K % 8 = 4: A through cp.async
    ("bf16_rm", 300, 264, 4100 - 3840, None, "umma_bf16"),  # K = 260
    ("bf16_rm", 130, 200, 102, None, "simt_bf16_scalar"),   # K % 4 = 2: no tensor-core path
    ("bf16_rm", 520, 1032, 260, None, "umma_bf16"),         # unaligned A staged, CTA pairs
    ("f16_cm", 1032, 520, 260, None, "umma_f16"),
    ("bf16_rm", 256, 256, 256, "simt_scalar", "simt_bf16_scalar"),
    ("bf16_rm", 4, 520, 1000, "gemv", "gemv_bf16_vec"),
    ("bf16_rm", 4, 520, 1000, None, "umma_bf16"),            # skinny M: 5 strips, K split over clusters
    ("bf16_rm", 7, 130, 77, None, "gemv_bf16_scalar"),
    ("bf16_rm", 16, 256, 64, "umma", "umma_bf16"),
    ("f16_cm", 512, 256, 512, None, "umma_f16"),
    ("f16_cm", 264, 300, 520, None, "umma_f16"),
    ("f16_cm", 300, 264, 520, None, "simt_f16_scalar"),
    ("f16_cm", 250, 3, 128, None, "gemv_f16_scalar"),
    ("f16_cm", 1000, 8, 1000, "gemv", "gemv_f16_vec"),
    ("f16_cm", 1000, 8, 1000, None, "umma_f16"),
    ("bf16_rm", 1, 1024, 512, "umma", "umma_bf16"),          # skinny M = 1: 8 strips x 4 ranks
    ("bf16_rm", 1, 4096, 1024, None, "umma_bf16"),           # M = 1, 32 strips x 4: the skinny kernel
    ("bf16_rm", 1, 12288, 512, None, "umma_bf16"),           # M = 1, 96 strips: the skinny kernel
    ("bf16_rm", 1, 12288, 512, "gemv", "gemv_bf16_vec"),     # the same on the GEMV
    ("bf16_rm", 1, 20480, 520, None, "umma_bf16"),           # 160 strips > SMs: 80 strips of 256 columns
    ("f16_cm", 2048, 1, 768, None, "umma_f16"),              # row-major M = 1 through the swap
    ("bf16_rm", 2, 264, 128, None, "umma_bf16"),             # 3 strips (the last one 8 columns)
    ("bf16_rm", 64, 2048, 4096, None, "umma_bf16"),          # 16 strips on clusters, M = 64
    ("bf16_rm", 60, 520, 1000, None, "umma_bf16"),           # ragged N and K
    ("bf16_rm", 40, 5000, 520, None, "umma_bf16"),           # 40 strips, ragged N
    ("bf16_rm", 33, 10240, 256, None, "umma_bf16"),          # 80 strips, one CTA each, M = 33
    ("f16_cm", 2000, 128, 2056, None, "umma_f16"),           # row-major M = 128, N = 2000
    ("bf16_rm", 8, 12288, 1024, None, "umma_bf16"),          # 96 strips, one CTA each
    ("bf16_rm", 16, 4096, 12288, None, "umma_bf16"),         # long K, 32 strips on clusters
    ("bf16_rm", 3, 1032, 2000, None, "umma_bf16"),           # 8-row X box, 3 rows used; ragged K
    ("f16_cm", 1000, 24, 3000, None, "umma_f16"),            # row-major M = 24 through the swap
    ("bf16_rm", 2600, 4104, 520, None, "umma_bf16"),         # CTA pairs over 2.5 waves, ragged M and N
    ("bf16_rm", 1000, 12296, 264, None, "umma_bf16"),        # ragged M and N, 3 waves
]


@pytest.mark.parametrize("case", MID_CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}-{c[4]}")
def test_random_mid_size(case):
    variant, M, N, K, force, expect = case
    A, B = synthetic.problem_inputs(variant, M, N, K, TEST_CONFIG)
    C, name, _ = run(variant, A, B, M, N, K, force=force)
    if expect:
        assert name == expect
    assert_parity(variant, C, A, B, M, N, K)


# ------------------------------------------------------------------ the workloads
def _workload_cases():
    out = []
    for wl, (cfg, probs) in synthetic.WORKLOADS.items():
        for (variant, M, N, K, da, sa, db, sb) in probs:
            out.append((wl, variant, M, N, K, cfg, da, sa, db, sb))
    for (M, N, K) in synthetic.EDGE_SHAPES:
        for variant in ("f32_rm", "bf16_rm"):
            out.append((f"edge_{variant}_{M}x{N}x{K}", variant, M, N, K, synthetic.EDGE_CONFIG_ID,
                        "uniform", 1.0, "uniform", 1.0))
    return out


@pytest.mark.parametrize("case", _workload_cases(), ids=lambda c: c[0])
def test_workload_sampled(case):
    """Full-size workload in the launch configuration the bench times: whole rows
    of C, two from every 256-row band of the kernel's tiles, and whole columns,
    one from every 256-column band, against the oracle; then a second run must be
    bit-identical."""
    wl, variant, M, N, K, cfg, da, sa, db, sb = case
    A, B = synthetic.problem_inputs(variant, M, N, K, cfg, da, sa, db, sb)
    C, name, dC = run(variant, A, B, M, N, K)
    res_r, res_c = check_bands(variant, C, A, B, M, N, K)
    assert res_r["ok"], (name, "rows", res_r)
    assert res_c["ok"], (name, "columns", res_c)
    assert np.all(np.isfinite(C)), name
    C2, name2, _ = run(variant, A, B, M, N, K)
    assert name2 == name and np.array_equal(C, C2), "not run-to-run deterministic"


def test_sgemm_256_full_oracle():
    """The small SGEMM workload against the full oracle, every element."""
    (variant, M, N, K, *_), = synthetic.WORKLOADS["sgemm_f32_rm_256"][1]
    A, B = synthetic.problem_inputs(variant, M, N, K, 0)
    C, name, _ = run(variant, A, B, M, N, K)
    assert name == "simt_f32_vec4"
    assert_parity(variant, C, A, B, M, N, K)


# ------------------------------------------------------------------ edges and hygiene
@pytest.mark.parametrize("variant", VARIANTS)
def test_k_zero_gives_zeros(variant):
    M, N = 37, 45
    dA = to_device(encode(variant, np.ones(1)))
    dC = empty_out(variant, M, N, fill=7)
    getattr(g, {"f32_rm": "gemm_f32_rm", "f16_cm": "gemm_f16_cm", "bf16_rm": "gemm_bf16_rm"}[variant])(
        dA, dA, dC, M, N, 0)
    assert g.gemm_last_kernel() == "zero_fill"
    torch.cuda.synchronize()
    assert np.all(widen(variant, dC, M, N) == 0.0)


@pytest.mark.parametrize("variant,shape", [("f32_rm", (300, 260, 128)), ("bf16_rm", (300, 264, 128)),
                                           ("f32_rm", (4, 256, 64)), ("bf16_rm", (4, 256, 64))])
def test_nan_row_propagates(variant, shape):
    M, N, K = shape
    a = synthetic.uniform_pm1(3, M * K).reshape(M, K)
    a[M // 2, K // 3] = np.nan
    b = synthetic.uniform_pm1(4, K * N)
    C, name, _ = run(variant, encode(variant, a), encode(variant, b), M, N, K)
    assert np.all(np.isnan(C[M // 2]))
    assert np.all(np.isfinite(np.delete(C, M // 2, axis=0)))


@pytest.mark.parametrize("variant,shape,force", [
    ("f32_rm", (300, 260, 272), None), ("f32_rm", (300, 261, 77), None), ("f32_rm", (3, 300, 100), None),
    ("bf16_rm", (300, 264, 520), None), ("bf16_rm", (130, 200, 100), None), ("bf16_rm", (3, 300, 100), None),
    ("f16_cm", (264, 300, 520), None)])
def test_no_write_outside_C(variant, shape, force):
    """Canary values around C stay untouched (out-of-bounds stores would change them)."""
    M, N, K = shape
    A, B = synthetic.problem_inputs(variant, M, N, K, TEST_CONFIG)
    pad = 4096
    dt = torch.float32 if variant.startswith("f32") else torch.int16
    big = torch.full((M * N + 2 * pad,), 12345 if dt == torch.int16 else 1.2345e6, dtype=dt, device="cuda")
    dC = big[pad:pad + M * N]
    g.gemm_force_kernel(force)
    try:
        getattr(g, {"f32_rm": "gemm_f32_rm", "f16_cm": "gemm_f16_cm", "bf16_rm": "gemm_bf16_rm"}[variant])(
            to_device(A), to_device(B), dC, M, N, K)
    finally:
        g.gemm_force_kernel(None)
    torch.cuda.synchronize()
    h = big.cpu()
    assert torch.all(h[:pad] == h[0]) and torch.all(h[pad + M * N:] == h[0])
    assert_parity(variant, widen(variant, dC, M, N), A, B, M, N, K)


@pytest.mark.parametrize("variant,shape,expect", [
    ("f32_rm", (260, 264, 128), "simt_f32_scalar"),
    ("bf16_rm", (260, 264, 128), "simt_bf16_scalar"),
    ("bf16_rm", (2, 264, 128), "gemv_bf16_scalar")])
def test_unaligned_pointers(variant, shape, expect):
    M, N, K = shape
    A, B = synthetic.problem_inputs(variant, M, N, K, TEST_CONFIG)
    C, name, _ = run(variant, A, B, M, N, K, a_off=1, b_off=1, c_off=1)
    assert name == expect
    assert_parity(variant, C, A, B, M, N, K)


def test_runs_on_the_callers_stream():
    M, N, K = 512, 512, 512
    A, B = synthetic.problem_inputs("bf16_rm", M, N, K, TEST_CONFIG)
    s = torch.cuda.Stream()
    C, name, _ = run("bf16_rm", A, B, M, N, K, stream=s)
    assert name == "umma_bf16"
    assert_parity("bf16_rm", C, A, B, M, N, K)


def test_forced_family_that_cannot_run_is_rejected():
    dA = to_device(np.zeros(64 * 64, np.float32))
    dC = empty_out("f32_rm", 64, 64)
    g.gemm_force_kernel("umma")
    try:
        with pytest.raises(g.GemmError):
            g.gemm_f32_rm(dA, dA.clone(), dC, 64, 64, 64)
    finally:
        g.gemm_force_kernel(None)
    g.gemm_force_kernel("gemv")
    try:
        with pytest.raises(g.GemmError):
            g.gemm_f32_rm(dA, dA.clone(), dC, 64, 64, 64)  # M > 8
    finally:
        g.gemm_force_kernel(None)


def test_matmul_convenience_matches_oracle():
    M, N, K = 200, 264, 136
    for dt, variant in ((torch.float32, "f32_rm"), (torch.bfloat16, "bf16_rm"), (torch.float16, "f16_rm")):
        a = synthetic.uniform_pm1(21, M * K)
        b = synthetic.uniform_pm1(22, K * N)
        ta = torch.from_numpy(a).reshape(M, K).to(dt).cuda()
        tb = torch.from_numpy(b).reshape(K, N).to(dt).cuda()
        out = g.matmul(ta, tb)
        torch.cuda.synchronize()
        A = ta.cpu().reshape(-1)
        B = tb.cpu().reshape(-1)
        if dt != torch.float32:
            A = A.view(torch.int16).numpy().view(np.uint16)
            B = B.view(torch.int16).numpy().view(np.uint16)
        else:
            A, B = A.numpy(), B.numpy()
        C_ref, S = oracle.gemm(variant, A, B, M, N, K)
        res = compare.check(variant, out.float().cpu().numpy(), C_ref, S, K)
        assert res["ok"], (dt, res)
