"""The C-ABI library builds, loads and exports every symbol include/gemm.h
declares; host-side argument checks that return before any device work.
No GPU is needed: nothing here launches a kernel."""

import ctypes
import os
import re
import subprocess

import pytest

import dense_matrix_multiply_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def built():
    g.ensure_built()
    return g.load()


def test_header_declares_the_three_entry_points():
    syms = declared_symbols()
    for name in ("gemm_f32_rm", "gemm_f16_cm", "gemm_bf16_rm"):
        assert name in syms
    assert len(syms) == len(set(syms))


def test_library_exports_every_declared_symbol(built):
    for name in declared_symbols():
        assert hasattr(built, name), name
    # and the binding wraps each of them
    assert set(declared_symbols()) == set(g.SIGNATURES)


def test_only_the_api_is_exported(built):
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(declared_symbols()) <= exported
    assert not [s for s in exported if s.startswith("_ZN") and "gemm_gb300" in s]


def test_library_is_built_for_sm_103a_only():
    from dense_matrix_multiply_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_launch_counter_reads_without_a_gpu(built):
    # calls rejected on the host launch nothing
    n0 = g.gemm_kernel_launches()
    assert isinstance(n0, int) and n0 >= 0
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.addressof(buf)
    assert built.gemm_f32_rm(p, p + 1024, p + 2048, -1, 4, 4) == 1
    assert g.gemm_kernel_launches() == n0


def test_status_strings(built):
    for code, name in g.STATUS_NAMES.items():
        assert g.gemm_status_string(code) == name
    assert g.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


def test_force_kernel_names(built):
    for fam in ("simt", "simt_scalar", "gemv", "gemv_scalar", "umma", "umma_skinny_wide", "umma_stall", "umma_stall_pair", "umma_stall_peer", None, ""):
        g.gemm_force_kernel(fam)
    with pytest.raises(g.GemmError):
        g.gemm_force_kernel("cpu")
    g.gemm_force_kernel(None)


def test_host_side_argument_errors(built):
    lib = built
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.addressof(buf)
    for fn in (lib.gemm_f32_rm, lib.gemm_f16_cm, lib.gemm_bf16_rm):
        assert fn(p, p + 1024, p + 2048, -1, 4, 4) == 1          # negative dimension
        assert fn(p, p + 1024, p + 2048, 4, 4, -4) == 1
        assert fn(p, p + 1024, p + 2048, 0, 4, 4) == 0           # empty output: no-op
        assert lib.gemm_last_kernel() == b"noop"
        assert fn(p, p + 1024, p + 2048, 4, 0, 4) == 0
        assert fn(p, p + 1024, None, 4, 4, 4) == 1                # null C
        assert fn(None, p + 1024, p + 2048, 4, 4, 4) == 1         # null A with K > 0
        assert fn(p, p + 16, p + 8, 4, 4, 4) == 2                 # C overlaps A and B
        assert fn(p, p + 1024, p + 1024, 4, 4, 4) == 2            # C is B


def test_stream_is_per_thread(built):
    import threading
    g.gemm_set_stream(1234)
    seen = []
    t = threading.Thread(target=lambda: seen.append(g.gemm_get_stream()))
    t.start()
    t.join()
    assert g.gemm_get_stream() == 1234 and seen == [0]
    g.gemm_set_stream(None)
    assert g.gemm_get_stream() == 0


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(g, "_lib", None)
    with pytest.raises(RuntimeError, match="CUDA extension missing"):
        g.load()


def test_general_form_host_side_errors(built):
    """gemm_ex rejects bad arguments before touching a device."""
    lib = built
    buf = ctypes.create_string_buffer(1 << 16)
    p = ctypes.addressof(buf)
    A, B, C = p, p + 16384, p + 32768

    def ex(dtype=0, layout=0, oa=0, ob=0, M=4, N=4, K=4, alpha=1.0, a=A, lda=4, sa=0, b=B, ldb=4, sb=0,
           beta=0.0, c=C, ldc=4, sc=16, batch=1):
        return lib.gemm_ex(dtype, layout, oa, ob, M, N, K, alpha, a, lda, sa, b, ldb, sb, beta, c, ldc, sc, batch)

    assert ex(dtype=3) == 1 and ex(layout=2) == 1 and ex(oa=2) == 1 and ex(ob=-1) == 1
    assert ex(M=-1) == 1 and ex(K=-1) == 1 and ex(batch=-1) == 1 and ex(sa=-4) == 1
    assert ex(lda=3) == 1                     # row-major A [4,4] needs lda >= 4
    assert ex(M=6, oa=1, lda=5) == 1          # A stored [K,M] = [4,6] needs lda >= 6
    assert ex(N=6, ob=1, ldb=3) == 1          # B stored [N,K] = [6,4] needs ldb >= 4
    assert ex(ldc=3) == 1
    assert ex(layout=1, M=6, lda=4) == 1      # column-major A [6,4] needs lda >= 6
    assert ex(batch=2, sc=8) == 1             # the two C matrices would overlap
    assert ex(c=None) == 1 and ex(a=None) == 1
    assert ex(M=0) == 0 and lib.gemm_last_kernel() == b"noop"
    assert ex(batch=0) == 0 and ex(N=0) == 0
    assert ex(c=A + 8) == 2                   # C overlaps A
    assert ex(b=C + 32, ldb=4) == 2           # C overlaps B
    # B's third matrix (stride 4096 floats = 16384 bytes) starts exactly at C
    assert ex(batch=3, sc=16, sb=4096, b=C - 2 * 16384) == 2
    assert ex(lda=1 << 61, batch=1) == 1      # span overflows


def test_fp8_host_side_errors(built):
    lib = built
    buf = ctypes.create_string_buffer(1 << 16)
    p = ctypes.addressof(buf)
    A, Q, S, W, C = p, p + 8192, p + 16384, p + 24576, p + 32768
    q = lib.gemm_quantize_rows_e4m3
    assert q(A, Q, S, -1, 4) == 1 and q(A, Q, S, 4, -1) == 1
    assert q(A, Q, S, 0, 4) == 0 and lib.gemm_last_kernel() == b"noop"
    assert q(None, Q, S, 4, 4) == 1 and q(A, Q, None, 4, 4) == 1
    assert q(A, A + 8, S, 4, 4) == 2          # Q overlaps A
    assert q(A, Q, Q + 4, 4, 4) == 2          # scale overlaps Q
    r = lib.gemm_e4m3_rowscale
    assert r(Q, S, W, C, -1, 4, 16) == 1 and r(Q, S, W, C, 4, 4, -16) == 1
    assert r(Q, S, W, C, 0, 4, 16) == 0 and r(Q, S, W, C, 4, 0, 16) == 0
    assert r(Q, S, W, None, 4, 4, 16) == 1 and r(None, S, W, C, 4, 4, 16) == 1
    assert r(Q, S, W, Q + 8, 4, 4, 16) == 2   # C overlaps Q
    assert r(Q, S, W, S, 4, 4, 16) == 2       # C overlaps scale
