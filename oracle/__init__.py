"""CPU oracle for dense C = A·B -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never loads it, and the
two share no code. The arithmetic lives in ``oracle.c`` (plain C, FP64
accumulation, ascending k); this module only builds and loads it and marshals
numpy arrays.

Every function here is pinned by ``tests/test_oracle_pins.py`` against brute
force on small integer inputs (exact rational arithmetic), closed forms
(ones·ones = K, I·B = B), the row-major/column-major transpose identity,
bit-exhaustive checks of the half and bf16 decoders, and a float64 library
matmul on the decoded values.  ``gemm_ex`` (the general form with alpha,
beta, operation flags, leading dimensions and batches) is pinned by
``tests/test_oracle_ex_pins.py``: exact integer results for every layout and
operation pair with NaN-filled padding, reduction to ``gemm`` in the plain
case, and the row-/column-major transpose identity.  ``silu_mul`` is pinned by
brute force and by SiLU's identities in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
LAYOUTS = {"rm": 0, "cm": 1}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            lib.oracle_gemm.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, i64, dp, dp]
            lib.oracle_gemm_rows.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, i64,
                                             vp, i64, dp, dp]
            lib.oracle_gemm_entries.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, i64,
                                                vp, vp, i64, dp, dp]
            d = ctypes.c_double
            lib.oracle_gemm_ex.argtypes = [ctypes.c_int] * 4 + [i64, i64, i64, d,
                                           vp, i64, i64, vp, i64, i64, d, vp, i64, i64, i64,
                                           dp, dp, dp, dp]
            lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
            lib.oracle_decode_e4m3.restype = ctypes.c_double
            lib.oracle_encode_e4m3.argtypes = [ctypes.c_float]
            lib.oracle_encode_e4m3.restype = ctypes.c_uint8
            lib.oracle_quantize_rows_e4m3.argtypes = [vp, i64, i64, vp, vp]
            lib.oracle_gemm_e4m3_rowscale.argtypes = [vp, vp, vp, i64, i64, i64, vp, i64, dp, dp]
            lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_f16.restype = ctypes.c_double
            lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_bf16.restype = ctypes.c_double
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _buf(x: np.ndarray, dtype: str, n: int) -> np.ndarray:
    want = np.float32 if dtype == "f32" else np.uint16
    x = np.ascontiguousarray(x).reshape(-1)
    if x.dtype != want:
        raise TypeError(f"{dtype} buffer must be {np.dtype(want).name}, got {x.dtype}")
    if x.size != n:
        raise ValueError(f"buffer holds {x.size} elements, expected {n}")
    return x


def _ptr(x: np.ndarray):
    return x.ctypes.data_as(ctypes.c_void_p)


def _variant(variant: str):
    dtype, layout = variant.split("_")
    return dtype, layout


def gemm(variant: str, A: np.ndarray, B: np.ndarray, M: int, N: int, K: int):
    """Full product of a problem, e.g. variant 'f32_rm', 'f16_cm', 'bf16_rm' (any
    dtype/layout pair is accepted). A and B are flat storage buffers.

    Returns (C, S): float64 arrays of logical shape [M, N] holding the exact-order
    FP64 sums and sum_k |a_ik b_kj|.
    """
    dtype, layout = _variant(variant)
    lib = _load()
    a = _buf(A, dtype, M * K)
    b = _buf(B, dtype, K * N)
    C = np.empty(M * N, dtype=np.float64)
    S = np.empty(M * N, dtype=np.float64)
    rc = lib.oracle_gemm(DTYPES[dtype], LAYOUTS[layout], _ptr(a), _ptr(b), M, N, K, _ptr(C), _ptr(S))
    if rc:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    if layout == "rm":
        return C.reshape(M, N), S.reshape(M, N)
    return C.reshape(N, M).T, S.reshape(N, M).T


def gemm_rows(variant: str, A, B, M: int, N: int, K: int, rows):
    """Output rows ``rows`` only: returns (C, S) of shape [len(rows), N]."""
    dtype, layout = _variant(variant)
    lib = _load()
    a = _buf(A, dtype, M * K)
    b = _buf(B, dtype, K * N)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    C = np.empty(r.size * N, dtype=np.float64)
    S = np.empty(r.size * N, dtype=np.float64)
    rc = lib.oracle_gemm_rows(DTYPES[dtype], LAYOUTS[layout], _ptr(a), _ptr(b), M, N, K,
                              _ptr(r), r.size, _ptr(C), _ptr(S))
    if rc:
        raise RuntimeError(f"oracle_gemm_rows failed ({rc})")
    return C.reshape(r.size, N), S.reshape(r.size, N)


def gemm_entries(variant: str, A, B, M: int, N: int, K: int, ii, jj):
    """Single entries C[ii[t], jj[t]]: returns (C, S) of shape [len(ii)]."""
    dtype, layout = _variant(variant)
    lib = _load()
    a = _buf(A, dtype, M * K)
    b = _buf(B, dtype, K * N)
    i = np.ascontiguousarray(ii, dtype=np.int64)
    j = np.ascontiguousarray(jj, dtype=np.int64)
    if i.shape != j.shape:
        raise ValueError("ii and jj differ in length")
    C = np.empty(i.size, dtype=np.float64)
    S = np.empty(i.size, dtype=np.float64)
    rc = lib.oracle_gemm_entries(DTYPES[dtype], LAYOUTS[layout], _ptr(a), _ptr(b), M, N, K,
                                 _ptr(i), _ptr(j), i.size, _ptr(C), _ptr(S))
    if rc:
        raise RuntimeError(f"oracle_gemm_entries failed ({rc})")
    return C, S


OPS = {"N": 0, "T": 1}


def gemm_ex(dtype: str, layout: str, op_a: str, op_b: str, M: int, N: int, K: int,
            alpha: float, A, lda: int, stride_a: int, B, ldb: int, stride_b: int,
            beta: float, C, ldc: int, stride_c: int, batch: int = 1) -> dict:
    """General form C_b <- alpha op(A_b) op(B_b) + beta C_b, b < batch ("SGEMM
    measured and the three ledgers", sections 2 and 3).  dtype 'f32' | 'f16' |
    'bf16', layout 'rm' | 'cm', op_a / op_b 'N' | 'T'; A, B, C are flat storage
    buffers (C may be None when beta == 0).  Returns a dict of float64 arrays
    of shape [batch, M, N]: C (the result), P (the product sum), S (the sum of
    absolute products) and BC (beta * C_in)."""
    lib = _load()
    want = np.float32 if dtype == "f32" else np.uint16

    def flat(x):
        if x is None:
            return np.zeros(1, dtype=want)
        x = np.ascontiguousarray(x).reshape(-1)
        if x.dtype != want:
            raise TypeError(f"{dtype} buffer must be {np.dtype(want).name}, got {x.dtype}")
        return x

    a, b, c = flat(A), flat(B), flat(C)
    # The storage each matrix spans must lie inside its buffer.
    a_rows, a_cols = (M, K) if op_a == "N" else (K, M)
    b_rows, b_cols = (K, N) if op_b == "N" else (N, K)
    for name, buf, r, cc, ld, st, used in (
            ("A", a, a_rows, a_cols, lda, stride_a, alpha != 0 and K > 0),
            ("B", b, b_rows, b_cols, ldb, stride_b, alpha != 0 and K > 0),
            ("C", c, M, N, ldc, stride_c, beta != 0)):
        if not used or batch == 0 or r == 0 or cc == 0:
            continue
        inner, outer = (cc, r) if layout == "rm" else (r, cc)
        if ld < inner:
            raise ValueError(f"ld{name.lower()} {ld} < {inner}")
        span = (batch - 1) * st + (outer - 1) * ld + inner
        if span > buf.size:
            raise ValueError(f"{name} spans {span} elements, buffer holds {buf.size}")
    out = {k: np.empty(batch * M * N, dtype=np.float64) for k in ("C", "P", "S", "BC")}
    rc = lib.oracle_gemm_ex(DTYPES[dtype], LAYOUTS[layout], OPS[op_a], OPS[op_b], M, N, K, float(alpha),
                            _ptr(a), lda, stride_a, _ptr(b), ldb, stride_b, float(beta), _ptr(c), ldc,
                            stride_c, batch, _ptr(out["C"]), _ptr(out["P"]), _ptr(out["S"]),
                            _ptr(out["BC"]))
    if rc:
        raise RuntimeError(f"oracle_gemm_ex failed ({rc})")
    return {k: v.reshape(batch, M, N) for k, v in out.items()}


def decode_e4m3(codes) -> np.ndarray:
    """The oracle's decoder of E4M3FN codes, as float64."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib.oracle_decode_e4m3(int(v)) for v in c], dtype=np.float64)


def encode_e4m3(x) -> np.ndarray:
    """Nearest E4M3FN codes (ties to even, clamped to +-448) of float32 values."""
    lib = _load()
    v = np.asarray(x, dtype=np.float32).reshape(-1)
    return np.array([lib.oracle_encode_e4m3(float(t)) for t in v], dtype=np.uint8)


def quantize_rows_e4m3(A, M: int, K: int):
    """Row-wise E4M3 quantisation of a half [M,K] row-major matrix ("Chapter 5
    Operators and Runtime", example 5-7): returns (Q uint8 [M,K], scale float32
    [M]) with q_ik = E4M3(a_ik * 448/amax_i) and scale_i = amax_i / 448."""
    lib = _load()
    a = _buf(A, "f16", M * K)
    Q = np.empty(M * K, dtype=np.uint8)
    sc = np.empty(M, dtype=np.float32)
    if lib.oracle_quantize_rows_e4m3(_ptr(a), M, K, _ptr(Q), _ptr(sc)):
        raise RuntimeError("oracle_quantize_rows_e4m3 failed")
    return Q.reshape(M, K), sc


def gemm_e4m3_rowscale(Q, scale, Wt, M: int, N: int, K: int, rows=None):
    """C[i,j] = scale_i * sum_k q_ik w_kj with Q [M,K] and the weights given as
    Wt [N,K] (example 5-8).  Returns (C, S) float64 of shape [M or len(rows), N]."""
    lib = _load()
    q = np.ascontiguousarray(Q, dtype=np.uint8).reshape(-1)
    w = np.ascontiguousarray(Wt, dtype=np.uint8).reshape(-1)
    sc = np.ascontiguousarray(scale, dtype=np.float32).reshape(-1)
    if q.size != M * K or w.size != N * K or sc.size != M:
        raise ValueError("buffer sizes do not match M, N, K")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = M if r is None else r.size
    C = np.empty(n * N, dtype=np.float64)
    S = np.empty(n * N, dtype=np.float64)
    rc = lib.oracle_gemm_e4m3_rowscale(_ptr(q), _ptr(sc), _ptr(w), M, N, K,
                                       None if r is None else _ptr(r), n, _ptr(C), _ptr(S))
    if rc:
        raise RuntimeError("oracle_gemm_e4m3_rowscale failed")
    return C.reshape(n, N), S.reshape(n, N)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 values rounded once to the nearest bf16 value (ties to even),
    returned as float64: the significand is scaled to 8 bits and rounded with
    numpy's round-half-to-even.  Normal range only (no overflow or subnormal
    handling, which the callers' values never reach)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x / (1 + e^-x) in float64 ("Chapter 5 Operators and Runtime",
    section 5.3.1)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def silu_mul(X, W_g, W_u, M: int, N: int, K: int, rows=None):
    """The FFN gate/up chain of section 5.3.1 with its rounding points:
    G = X W_g and U = X W_u (FP64 sums of the stored bf16 inputs), each rounded
    to bf16; T = bf16(SiLU(G)); Z = bf16(T * U).  Returns a dict of float64
    arrays of shape [M, N] (or [len(rows), N] when rows is given): Z, the rounded
    intermediates G, U, T, and S_G, S_U = sum_k |x_ik w_kj| of the two products."""
    if rows is None:
        G, S_G = gemm("bf16_rm", X, W_g, M, N, K)
        U, S_U = gemm("bf16_rm", X, W_u, M, N, K)
    else:
        G, S_G = gemm_rows("bf16_rm", X, W_g, M, N, K, rows)
        U, S_U = gemm_rows("bf16_rm", X, W_u, M, N, K, rows)
    G = round_bf16(G)
    U = round_bf16(U)
    T = round_bf16(silu(G))
    Z = round_bf16(T * U)
    return {"Z": Z, "G": G, "U": U, "T": T, "S_G": S_G, "S_U": S_U}


def decode(dtype: str, bits) -> np.ndarray:
    """The oracle's own decoder of half/bf16 bit patterns, as float64."""
    lib = _load()
    fn = lib.oracle_decode_f16 if dtype == "f16" else lib.oracle_decode_bf16
    b = np.asarray(bits, dtype=np.uint16).reshape(-1)
    return np.array([fn(int(v)) for v in b], dtype=np.float64)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's later calls (its results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))
