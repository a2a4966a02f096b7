"""Python binding of the GB300 dense GEMM library (libgemm_gb300.so).

Argument marshalling only: every step of C = A·B runs in the library's CUDA
kernels.  The C entry points are exposed under the same names and take either
torch CUDA tensors (their data pointers are passed, and the library is pointed
at torch's current stream first) or raw device addresses as integers.

There is no CPU path.  If the shared library has not been built, or the device
is not a GB300, calls raise instead of computing anything elsewhere.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB

GEMM_OK = 0
STATUS_NAMES = {
    0: "GEMM_OK",
    1: "GEMM_ERR_INVALID_VALUE",
    2: "GEMM_ERR_ALIAS",
    3: "GEMM_ERR_UNSUPPORTED_DEVICE",
    4: "GEMM_ERR_CUDA",
    5: "GEMM_ERR_TIMEOUT",
}

# Every symbol include/gemm.h declares, with its ctypes signature.
_VP, _I = ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "gemm_f32_rm": ([_VP, _VP, _VP, _I, _I, _I], _I),
    "gemm_f16_cm": ([_VP, _VP, _VP, _I, _I, _I], _I),
    "gemm_bf16_rm": ([_VP, _VP, _VP, _I, _I, _I], _I),
    "gemm_bf16_rm_noalloc": ([_VP, _VP, _VP, _I, _I, _I], _I),
    "gemm_bf16_rm_silu_mul": ([_VP, _VP, _VP, _VP, _I, _I, _I], _I),
    "gemm_ex": ([_I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _VP, ctypes.c_int64, ctypes.c_int64,
                 _VP, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, _VP, ctypes.c_int64, ctypes.c_int64,
                 _I], _I),
    "gemm_quantize_rows_e4m3": ([_VP, _VP, _VP, _I, _I], _I),
    "gemm_e4m3_rowscale": ([_VP, _VP, _VP, _VP, _I, _I, _I], _I),
    "gemm_e4m3_rowscale_fused": ([_VP, _VP, _VP, _I, _I, _I], _I),
    "gemm_set_stream": ([_VP], _I),
    "gemm_get_stream": ([], _VP),
    "gemm_synchronize": ([], _I),
    "gemm_status_string": ([_I], ctypes.c_char_p),
    "gemm_last_kernel": ([], ctypes.c_char_p),
    "gemm_kernel_launches": ([], ctypes.c_ulonglong),
    "gemm_last_error": ([], ctypes.c_char_p),
    "gemm_force_kernel": ([ctypes.c_char_p], _I),
}

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def ensure_built() -> str:
    """Compiles the library if it is missing or older than its sources."""
    return _build.build()


def load():
    """The loaded shared library (ctypes.CDLL).  Raises if it was never built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA extension missing: {LIB_PATH} has not been built "
                    "(run dense_matrix_multiply_gb300.ensure_built() or __graft_entry__.build())")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _addr(x) -> int:
    if isinstance(x, int):
        return x
    if x is None:
        return 0
    return x.data_ptr()


def _bind_torch_stream(*tensors) -> None:
    """Points the library at torch's current stream of the tensors' device.
    Every tensor argument must live on one CUDA device: a kernel given another
    device's address would read memory it cannot reach."""
    dev = None
    for t in tensors:
        if hasattr(t, "is_cuda"):
            if not t.is_cuda:
                raise ValueError("tensors must live on a CUDA device")
            if dev is None:
                dev = t.device
            elif t.device != dev:
                raise ValueError(f"tensors on two devices: {dev} and {t.device}")
    if dev is not None:
        import torch
        load().gemm_set_stream(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))


def _span(outer: int, inner: int, ld: int, stride: int = 0, batch: int = 1) -> int:
    """Elements from a stored matrix's first element to one past its last:
    `batch` matrices of `outer` lines of `inner` elements, lines `ld` apart and
    matrices `stride` apart.  0 for an empty matrix or a negative argument,
    which the library itself rejects."""
    if min(outer, inner, ld, stride, batch) < 0 or outer == 0 or inner == 0 or batch == 0:
        return 0
    return (batch - 1) * stride + (outer - 1) * ld + inner


def _check(name: str, t, elt_size: int, need: int, tight: bool = True) -> None:
    """Host-side check of one tensor argument before its address is passed on:
    the element size of the entry point, and room for the `need` elements the
    call reads or writes from the tensor's first element (the tensor's own
    elements for the tight layouts of the named entry points, which also need
    a contiguous tensor; the rest of its storage for gemm_ex, whose leading
    dimensions may step over a wider buffer).  A raw address (an int) or None
    is passed as it is."""
    if t is None or isinstance(t, int):
        return
    if t.element_size() != elt_size:
        raise ValueError(f"{name}: the entry point takes {elt_size}-byte elements, got {t.dtype}")
    if tight:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        room = t.numel()
    else:
        room = t.untyped_storage().nbytes() // elt_size - t.storage_offset()
    if room < need:
        raise ValueError(f"{name} holds {room} elements, the call needs {need}")


def _dims(M: int, N: int, K: int):
    """Elements of the tight A [M,K], B [K,N] and C [M,N] a call touches: none
    when M or N is 0 (a no-op) or a dimension is negative (the library rejects
    the call); C alone when K is 0 (zeros are written)."""
    M, N, K = int(M), int(N), int(K)
    if min(M, N, K) < 0 or M == 0 or N == 0:
        return 0, 0, 0
    return M * K, K * N, M * N


_ELT = {"gemm_f32_rm": 4, "gemm_f16_cm": 2, "gemm_bf16_rm": 2, "gemm_bf16_rm_noalloc": 2}


def _call(name: str, A, B, C, M: int, N: int, K: int) -> None:
    lib = load()
    na, nb, nc = _dims(M, N, K)
    for arg, t, need in (("A", A, na), ("B", B, nb), ("C", C, nc)):
        _check(f"{name}: {arg}", t, _ELT[name], need)
    _bind_torch_stream(A, B, C)
    st = getattr(lib, name)(_addr(A), _addr(B), _addr(C), int(M), int(N), int(K))
    if st != GEMM_OK:
        raise GemmError(st, name, lib.gemm_last_error().decode())


def gemm_f32_rm(A, B, C, M: int, N: int, K: int) -> None:
    """C[M,N] = A[M,K]·B[K,N], row-major float32, FP32 FFMA only."""
    _call("gemm_f32_rm", A, B, C, M, N, K)


def gemm_f16_cm(A, B, C, M: int, N: int, K: int) -> None:
    """C = A·B, column-major half (lda = M, ldb = K, ldc = M), FP32 accumulation."""
    _call("gemm_f16_cm", A, B, C, M, N, K)


def gemm_bf16_rm(A, B, C, M: int, N: int, K: int) -> None:
    """C[M,N] = A[M,K]·B[K,N], row-major bf16, FP32 accumulation."""
    _call("gemm_bf16_rm", A, B, C, M, N, K)


def gemm_bf16_rm_noalloc(A, B, C, M: int, N: int, K: int) -> None:
    """As gemm_bf16_rm, on the tensor-core kernel with its scratch in a static
    device array: the call allocates no device memory."""
    _call("gemm_bf16_rm_noalloc", A, B, C, M, N, K)


def gemm_bf16_rm_silu_mul(X, W_g, W_u, Z, M: int, N: int, K: int) -> None:
    """Z[M,N] = SiLU(X W_g) * (X W_u), bf16 row-major, the FFN gate/up projection."""
    lib = load()
    nx, nw, nz = _dims(M, N, K)
    for arg, t, need in (("X", X, nx), ("W_g", W_g, nw), ("W_u", W_u, nw), ("Z", Z, nz)):
        _check(f"gemm_bf16_rm_silu_mul: {arg}", t, 2, need)
    _bind_torch_stream(X, W_g, W_u, Z)
    st = lib.gemm_bf16_rm_silu_mul(_addr(X), _addr(W_g), _addr(W_u), _addr(Z), int(M), int(N), int(K))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_bf16_rm_silu_mul", lib.gemm_last_error().decode())


def gemm_quantize_rows_e4m3(A, Q, scale, M: int, K: int) -> None:
    """Row-wise E4M3 quantisation of a half [M,K] matrix: Q [M,K] codes (uint8),
    scale [M] float32, a_ik ~ Q[i,k] * scale_i."""
    lib = load()
    na = _dims(M, 1, K)[0]
    rows = max(int(M), 0)  # the scales are written even for K = 0 (scale 0)
    for arg, t, size, need in (("A", A, 2, na), ("Q", Q, 1, na), ("scale", scale, 4, rows)):
        _check(f"gemm_quantize_rows_e4m3: {arg}", t, size, need)
    _bind_torch_stream(A, Q, scale)
    st = lib.gemm_quantize_rows_e4m3(_addr(A), _addr(Q), _addr(scale), int(M), int(K))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_quantize_rows_e4m3", lib.gemm_last_error().decode())


def gemm_e4m3_rowscale(Q, scale, Wt, C, M: int, N: int, K: int) -> None:
    """C[M,N] (half) = diag(scale) Q[M,K] W[K,N], with the E4M3 weights given as Wt [N,K]."""
    lib = load()
    nq, nw, nc = _dims(M, N, K)
    rows = int(M) if nq else 0  # the scales are read only when the product has terms
    for arg, t, size, need in (("Q", Q, 1, nq), ("scale", scale, 4, rows), ("Wt", Wt, 1, nw), ("C", C, 2, nc)):
        _check(f"gemm_e4m3_rowscale: {arg}", t, size, need)
    _bind_torch_stream(Q, scale, Wt, C)
    st = lib.gemm_e4m3_rowscale(_addr(Q), _addr(scale), _addr(Wt), _addr(C), int(M), int(N), int(K))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_e4m3_rowscale", lib.gemm_last_error().decode())


def gemm_e4m3_rowscale_fused(A, Wt, C, M: int, N: int, K: int) -> None:
    """C[M,N] (half) = diag(amax/448) E4M3(diag(448/amax) A) W, the row-wise
    quantisation of the half A [M,K] fused into the product's load path; the
    E4M3 weights given as Wt [N,K]."""
    lib = load()
    na, nw, nc = _dims(M, N, K)
    for arg, t, size, need in (("A", A, 2, na), ("Wt", Wt, 1, nw), ("C", C, 2, nc)):
        _check(f"gemm_e4m3_rowscale_fused: {arg}", t, size, need)
    _bind_torch_stream(A, Wt, C)
    st = lib.gemm_e4m3_rowscale_fused(_addr(A), _addr(Wt), _addr(C), int(M), int(N), int(K))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_e4m3_rowscale_fused", lib.gemm_last_error().decode())


DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
LAYOUTS = {"rm": 0, "cm": 1}
OPS = {"N": 0, "T": 1}


def gemm_ex(dtype: str, layout: str, op_a: str, op_b: str, M: int, N: int, K: int, alpha: float,
            A, lda: int, stride_a: int, B, ldb: int, stride_b: int, beta: float, C, ldc: int,
            stride_c: int, batch: int = 1) -> None:
    """C_b = alpha op(A_b) op(B_b) + beta C_b for b < batch.  dtype 'f32' | 'f16' |
    'bf16', layout 'rm' | 'cm', op_a / op_b 'N' | 'T'; leading dimensions and
    strides in elements (see include/gemm.h for the storage rules)."""
    lib = load()
    M, N, K, batch = int(M), int(N), int(K), int(batch)
    cm = layout == "cm"
    a_r, a_c = (M, K) if op_a == "N" else (K, M)
    b_r, b_c = (K, N) if op_b == "N" else (N, K)
    # (lines, elements per line) of each stored matrix in memory order
    (ao, ai), (bo, bi), (co, ci) = ((c, r) if cm else (r, c) for r, c in ((a_r, a_c), (b_r, b_c), (M, N)))
    # A and B are read only when the product has terms; C is written whenever
    # it has elements (and read when beta != 0)
    reads_ab = K > 0 and float(alpha) != 0.0 and M > 0 and N > 0
    size = {"f32": 4, "f16": 2, "bf16": 2}.get(dtype, 0)
    if size:
        _check("gemm_ex: A", A, size, _span(ao, ai, int(lda), int(stride_a), batch) if reads_ab else 0, tight=False)
        _check("gemm_ex: B", B, size, _span(bo, bi, int(ldb), int(stride_b), batch) if reads_ab else 0, tight=False)
        _check("gemm_ex: C", C, size, _span(co, ci, int(ldc), int(stride_c), batch), tight=False)
    _bind_torch_stream(A, B, C)
    st = lib.gemm_ex(DTYPES[dtype], LAYOUTS[layout], OPS[op_a], OPS[op_b], int(M), int(N), int(K),
                     float(alpha), _addr(A), int(lda), int(stride_a), _addr(B), int(ldb), int(stride_b),
                     float(beta), _addr(C), int(ldc), int(stride_c), int(batch))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_ex", lib.gemm_last_error().decode())


def gemm_set_stream(stream) -> None:
    """Stream for this thread's later calls: a torch.cuda.Stream, a raw handle or None."""
    handle = getattr(stream, "cuda_stream", stream)
    st = load().gemm_set_stream(ctypes.c_void_p(handle or 0))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_set_stream")


def gemm_get_stream() -> int:
    return load().gemm_get_stream() or 0


def gemm_synchronize() -> None:
    lib = load()
    st = lib.gemm_synchronize()
    if st != GEMM_OK:
        raise GemmError(st, "gemm_synchronize", lib.gemm_last_error().decode())


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def gemm_last_kernel() -> str:
    return load().gemm_last_kernel().decode()


def gemm_kernel_launches() -> int:
    return int(load().gemm_kernel_launches())


def gemm_last_error() -> str:
    return load().gemm_last_error().decode()


def gemm_force_kernel(family) -> None:
    st = load().gemm_force_kernel(family.encode() if family else None)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_force_kernel", str(family))


def matmul(a, b, out=None):
    """C = a @ b for 2-D row-major torch CUDA tensors of one dtype (float32,
    bfloat16 or float16).  float16 goes through the column-major entry point on
    the same buffers (row-major C = A·B is column-major C^T = B^T·A^T)."""
    import torch
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"bad shapes {tuple(a.shape)} @ {tuple(b.shape)}")
    if a.dtype != b.dtype:
        raise ValueError("a and b must share a dtype")
    a = a.contiguous()
    b = b.contiguous()
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=a.dtype, device=a.device)
    elif out.shape != (M, N) or out.dtype != a.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] tensor of the input dtype")
    if a.dtype == torch.float32:
        gemm_f32_rm(a, b, out, M, N, K)
    elif a.dtype == torch.bfloat16:
        gemm_bf16_rm(a, b, out, M, N, K)
    elif a.dtype == torch.float16:
        gemm_f16_cm(b, a, out, N, M, K)
    else:
        raise ValueError(f"unsupported dtype {a.dtype}")
    return out
