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
    """Points the library at torch's current stream of the tensors' device."""
    for t in tensors:
        if hasattr(t, "is_cuda"):
            import torch
            if not t.is_cuda:
                raise ValueError("tensors must live on a CUDA device")
            load().gemm_set_stream(ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream))
            return


def _call(name: str, A, B, C, M: int, N: int, K: int) -> None:
    lib = load()
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
    _bind_torch_stream(X, W_g, W_u, Z)
    st = lib.gemm_bf16_rm_silu_mul(_addr(X), _addr(W_g), _addr(W_u), _addr(Z), int(M), int(N), int(K))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_bf16_rm_silu_mul", lib.gemm_last_error().decode())


def gemm_quantize_rows_e4m3(A, Q, scale, M: int, K: int) -> None:
    """Row-wise E4M3 quantisation of a half [M,K] matrix: Q [M,K] codes (uint8),
    scale [M] float32, a_ik ~ Q[i,k] * scale_i."""
    lib = load()
    _bind_torch_stream(A, Q, scale)
    st = lib.gemm_quantize_rows_e4m3(_addr(A), _addr(Q), _addr(scale), int(M), int(K))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_quantize_rows_e4m3", lib.gemm_last_error().decode())


def gemm_e4m3_rowscale(Q, scale, Wt, C, M: int, N: int, K: int) -> None:
    """C[M,N] (half) = diag(scale) Q[M,K] W[K,N], with the E4M3 weights given as Wt [N,K]."""
    lib = load()
    _bind_torch_stream(Q, scale, Wt, C)
    st = lib.gemm_e4m3_rowscale(_addr(Q), _addr(scale), _addr(Wt), _addr(C), int(M), int(N), int(K))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_e4m3_rowscale", lib.gemm_last_error().decode())


def gemm_e4m3_rowscale_fused(A, Wt, C, M: int, N: int, K: int) -> None:
    """C[M,N] (half) = diag(amax/448) E4M3(diag(448/amax) A) W, the row-wise
    quantisation of the half A [M,K] fused into the product's load path; the
    E4M3 weights given as Wt [N,K]."""
    lib = load()
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
