"""The Python binding's host-side checks of tensor arguments (no GPU): a tensor
with the wrong element size, too few elements for the M, N, K it is called
with, or a non-contiguous layout where the entry point takes a tight matrix is
refused before its address reaches the library, so no kernel is launched on
memory the call does not own.  CPU tensors reach the device check last, which
refuses them too.  The span of a gemm_ex operand is pinned against the set of
element offsets the storage rule addresses, enumerated by brute force."""

import itertools

import numpy as np
import pytest
import torch

import dense_matrix_multiply_gb300 as g


@pytest.fixture(scope="module", autouse=True)
def built(lib):
    return lib.load()


def launches():
    return g.gemm_kernel_launches()


def refused(fn, *args, match):
    before = launches()
    with pytest.raises(ValueError, match=match):
        fn(*args)
    assert launches() == before


def test_tight_entry_points_refuse_short_tensors():
    M, N, K = 8, 16, 32
    for name, dt in (("gemm_f32_rm", torch.float32), ("gemm_bf16_rm", torch.bfloat16),
                     ("gemm_f16_cm", torch.float16), ("gemm_bf16_rm_noalloc", torch.int16)):
        fn = getattr(g, name)
        A, B, C = (torch.zeros(n, dtype=dt) for n in (M * K, K * N, M * N))
        refused(fn, A[:-1], B, C, M, N, K, match=r"A holds 255 elements, the call needs 256")
        refused(fn, A, B[:-1], C, M, N, K, match=r"B holds 511 elements, the call needs 512")
        refused(fn, A, B, C[:-1], M, N, K, match=r"C holds 127 elements, the call needs 128")
        # sized right, the tensors are still refused for living on the host
        refused(fn, A, B, C, M, N, K, match="CUDA device")


def test_wrong_element_size_is_refused():
    M, N, K = 4, 8, 8
    A = torch.zeros(M * K, dtype=torch.float16)
    B = torch.zeros(K * N, dtype=torch.float16)
    C = torch.zeros(M * N, dtype=torch.float16)
    refused(g.gemm_f32_rm, A, B, C, M, N, K, match="4-byte elements")
    Af = torch.zeros(M * K, dtype=torch.float32)
    refused(g.gemm_bf16_rm, Af, B, C, M, N, K, match="2-byte elements")


def test_non_contiguous_tight_operand_is_refused():
    M, N, K = 4, 8, 8
    A = torch.zeros(K, M, dtype=torch.float32).t()   # [M, K] view, column-major in memory
    B = torch.zeros(K * N, dtype=torch.float32)
    C = torch.zeros(M * N, dtype=torch.float32)
    refused(g.gemm_f32_rm, A, B, C, M, N, K, match="contiguous")


def test_empty_dimensions_need_no_room():
    # M = 0: nothing is read or written, so empty tensors pass the size checks
    e = torch.zeros(0, dtype=torch.float32)
    refused(g.gemm_f32_rm, e, e, e, 0, 16, 16, match="CUDA device")
    # K = 0: A and B are not read, C (M x N) is written
    C = torch.zeros(4 * 4, dtype=torch.float32)
    refused(g.gemm_f32_rm, e, e, C, 4, 4, 0, match="CUDA device")
    refused(g.gemm_f32_rm, e, e, C[:-1], 4, 4, 0, match="C holds 15 elements")


def test_other_entry_points_check_every_operand():
    M, N, K = 4, 8, 16
    h = lambda n: torch.zeros(n, dtype=torch.int16)
    u8 = lambda n: torch.zeros(n, dtype=torch.uint8)
    f = lambda n: torch.zeros(n, dtype=torch.float32)
    refused(g.gemm_bf16_rm_silu_mul, h(M * K), h(K * N), h(K * N - 1), h(M * N), M, N, K,
            match="W_u holds")
    refused(g.gemm_quantize_rows_e4m3, h(M * K), u8(M * K), f(M - 1), M, K, match="scale holds 3")
    refused(g.gemm_quantize_rows_e4m3, h(M * K), h(M * K), f(M), M, K, match="1-byte elements")
    refused(g.gemm_e4m3_rowscale, u8(M * K), f(M), u8(N * K - 1), h(M * N), M, N, K, match="Wt holds")
    refused(g.gemm_e4m3_rowscale, u8(M * K), f(M), u8(N * K), h(M * N), M, N, K, match="CUDA device")
    refused(g.gemm_e4m3_rowscale_fused, h(M * K), u8(N * K), h(M * N - 1), M, N, K, match="C holds")


def brute_span(outer, inner, ld, stride, batch):
    """One past the largest element offset the storage rule addresses."""
    offs = [b * stride + o * ld + i for b, o, i in itertools.product(range(batch), range(outer), range(inner))]
    return max(offs) + 1 if offs else 0


def test_span_matches_brute_force():
    from dense_matrix_multiply_gb300 import _span
    for outer, inner, ld, stride, batch in itertools.product((0, 1, 3), (0, 1, 5), (5, 7), (0, 20, 40), (1, 2, 3)):
        assert _span(outer, inner, ld, stride, batch) == brute_span(outer, inner, ld, stride, batch), \
            (outer, inner, ld, stride, batch)
    assert _span(3, 5, -1, 0, 1) == 0   # negative leading dimension: left to the library


def test_gemm_ex_checks_the_span_of_each_operand():
    M, N, K, pad, batch = 6, 10, 12, 3, 2
    # row-major, op(A) = A^T: A stored [K, M] with lda = M + pad
    lda, ldb, ldc = M + pad, N + pad, N + pad
    sa, sb, sc = K * lda, K * ldb, M * ldc
    need_a = (batch - 1) * sa + (K - 1) * lda + M
    big = torch.zeros(need_a + 100, dtype=torch.float32)
    A = big[100:]                                    # exactly need_a elements from its first one
    B = torch.zeros((batch - 1) * sb + (K - 1) * ldb + N, dtype=torch.float32)
    C = torch.zeros((batch - 1) * sc + (M - 1) * ldc + N, dtype=torch.float32)
    args = lambda a, b, c: ("f32", "rm", "T", "N", M, N, K, 1.0, a, lda, sa, b, ldb, sb, 0.0, c, ldc, sc, batch)
    refused(g.gemm_ex, *args(A, B, C), match="CUDA device")
    refused(g.gemm_ex, *args(big[101:], B, C), match=f"A holds {need_a - 1} elements")
    # a slice keeps the storage behind it (a strided call may use it), so the
    # short operands are fresh tensors
    refused(g.gemm_ex, *args(A, B[:-1].clone(), C), match="B holds")
    refused(g.gemm_ex, *args(A, B, C[:-1].clone()), match="C holds")
    # a strided view over a wider buffer is fine: its storage covers the span
    wide = torch.zeros(K, lda, dtype=torch.float32)
    view = wide[:, :M]
    assert not view.is_contiguous()
    refused(g.gemm_ex, "f32", "rm", "T", "N", M, N, K, 1.0, view, lda, 0, B, ldb, sb, 0.0, C, ldc, sc, 1,
            match="CUDA device")
    # alpha = 0: A and B are not read, so they may be empty
    e = torch.zeros(0, dtype=torch.float32)
    refused(g.gemm_ex, *args(e, e, C)[:7], 0.0, *args(e, e, C)[8:], match="CUDA device")


def test_column_major_span_uses_columns_as_lines():
    from dense_matrix_multiply_gb300 import _span
    # column-major C [M, N] with ldc: N columns of M elements
    M, N, ldc = 5, 3, 7
    stored = np.zeros(_span(N, M, ldc), dtype=np.int8)
    for r, c in itertools.product(range(M), range(N)):
        stored[r + c * ldc] = 1     # every (r, c) of the column-major storage rule is inside the span
    assert stored.sum() == M * N and stored[-1] == 1
