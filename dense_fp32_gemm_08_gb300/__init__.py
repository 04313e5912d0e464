"""GB300 single-precision GEMM: Python binding of the C ABI declared in ``include/sgemm.h``.

This module only marshals arguments: every step of C = alpha * (A . B) + beta * C runs in
the CUDA kernels of ``libsgemm_gb300.so`` (built in-tree by ``_build.build()``). There is no
CPU fallback: if the library is missing, every call raises ``RuntimeError``.

Pointer arguments accept either an integer device address or a torch CUDA tensor (its
``data_ptr()`` is passed). ``stream`` is an integer ``cudaStream_t``, a ``torch.cuda.Stream``
or None (torch's current stream when torch has CUDA, else the legacy default stream).
Non-OK statuses raise ``SgemmError`` carrying the status code and the library's message.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

__all__ = [
    "SgemmError", "library_path", "lib", "sgemm", "sgemm_strided_batched", "sgemm_3xtf32",
    "sgemm_3xtf32_strided_batched", "sgemm_tf32", "sgemm_tf32_strided_batched", "sgemm_ex",
    "sgemm_ex_strided_batched", "sgemm_fused", "sgemm_fused_strided_batched", "sgemm_host",
    "sgemm_noalloc", "sgemm_status_string", "sgemm_last_error",
    "sgemm_device_status", "sgemm_release_workspace", "sgemm_num_configs",
    "sgemm_config_name", "sgemm_select_config", "sgemm_force_config",
    "sgemm_selftest_bounded_wait", "matmul",
    "SGEMM_OK", "SGEMM_ERR_INVALID_VALUE", "SGEMM_ERR_LAUNCH", "SGEMM_ERR_TIMEOUT",
    "SGEMM_ERR_UNSUPPORTED",
]

SGEMM_OK = 0
SGEMM_ERR_INVALID_VALUE = 1
SGEMM_ERR_LAUNCH = 2
SGEMM_ERR_TIMEOUT = 3
SGEMM_ERR_UNSUPPORTED = 4

SGEMM_OP_N, SGEMM_OP_T = 0, 1
SGEMM_PATH_SIMT, SGEMM_PATH_3XTF32, SGEMM_PATH_TF32 = 0, 1, 2
_PATHS = {"simt": SGEMM_PATH_SIMT, "3xtf32": SGEMM_PATH_3XTF32, "tf32": SGEMM_PATH_TF32}
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2, "gelu_tanh": 3, "silu": 4}

_LIBRARY = Path(__file__).resolve().with_name("libsgemm_gb300.so")
_lib = None


class SgemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def library_path() -> Path:
    return _LIBRARY


def lib() -> ctypes.CDLL:
    """The loaded C library (raises RuntimeError when it has not been built)."""
    global _lib
    if _lib is None:
        if not _LIBRARY.exists():
            raise RuntimeError(f"{_LIBRARY.name} is not built; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = _bind(ctypes.CDLL(str(_LIBRARY)))
    return _lib


def _bind(L):
    i64, f32, p, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
    gemm = [i64, i64, i64, f32, p, i64, p, i64, f32, p, i64, p]
    batched = [i64, i64, i64, f32, p, i64, i64, p, i64, i64, f32, p, i64, i64, i64, p]
    for name, args in (("sgemm", gemm), ("sgemm_3xtf32", gemm), ("sgemm_noalloc", gemm),
                       ("sgemm_host", gemm),
                       ("sgemm_tf32", gemm), ("sgemm_strided_batched", batched),
                       ("sgemm_3xtf32_strided_batched", batched),
                       ("sgemm_tf32_strided_batched", batched)):
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = i32
    L.sgemm_ex.argtypes = [i32, i32, i32] + gemm
    L.sgemm_ex.restype = i32
    L.sgemm_ex_strided_batched.argtypes = [i32, i32, i32] + batched
    L.sgemm_ex_strided_batched.restype = i32
    L.sgemm_fused.argtypes = [i32, i32, i32] + gemm[:-1] + [p, i32, p]
    L.sgemm_fused.restype = i32
    L.sgemm_fused_strided_batched.argtypes = [i32, i32, i32] + batched[:-1] + [p, i32, p]
    L.sgemm_fused_strided_batched.restype = i32
    L.sgemm_status_string.argtypes = [i32]
    L.sgemm_status_string.restype = ctypes.c_char_p
    L.sgemm_last_error.argtypes = []
    L.sgemm_last_error.restype = ctypes.c_char_p
    L.sgemm_device_status.argtypes = [p]
    L.sgemm_device_status.restype = i32
    L.sgemm_release_workspace.argtypes = []
    L.sgemm_release_workspace.restype = i32
    L.sgemm_num_configs.argtypes = []
    L.sgemm_num_configs.restype = i32
    L.sgemm_config_name.argtypes = [i32]
    L.sgemm_config_name.restype = ctypes.c_char_p
    L.sgemm_select_config.argtypes = [i64, i64, i64, f32, p, i64, p, i64, p, i64, i64]
    L.sgemm_select_config.restype = i32
    L.sgemm_force_config.argtypes = [i32]
    L.sgemm_force_config.restype = i32
    L.sgemm_selftest_bounded_wait.argtypes = [i32, p]
    L.sgemm_selftest_bounded_wait.restype = i32
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    data_ptr = getattr(x, "data_ptr", None)
    if data_ptr is None:
        raise TypeError(f"expected a device address or a CUDA tensor, got {type(x).__name__}")
    if not x.is_cuda:
        raise TypeError("tensor arguments must live on a CUDA device")
    if str(x.dtype) != "torch.float32":
        raise TypeError("tensor arguments must be float32")
    return data_ptr()


def _stream(s):
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int) -> None:
    if status != SGEMM_OK:
        L = lib()
        msg = (L.sgemm_last_error() or b"").decode() or L.sgemm_status_string(status).decode()
        raise SgemmError(status, msg)


def sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """C = alpha * (A . B) + beta * C on the FP32 SIMT path (asynchronous on ``stream``)."""
    _check(lib().sgemm(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                       _stream(stream)))


def sgemm_strided_batched(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                          strideC, batch, stream=None) -> None:
    """``batch`` products; problem b uses A + b*strideA, B + b*strideB, C + b*strideC."""
    _check(lib().sgemm_strided_batched(M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb,
                                       strideB, beta, _ptr(C), ldc, strideC, batch,
                                       _stream(stream)))


def sgemm_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """The same operation on the tcgen05 tensor cores with the 3xTF32 split."""
    _check(lib().sgemm_3xtf32(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                              _stream(stream)))


def sgemm_3xtf32_strided_batched(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C,
                                 ldc, strideC, batch, stream=None) -> None:
    _check(lib().sgemm_3xtf32_strided_batched(M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B),
                                              ldb, strideB, beta, _ptr(C), ldc, strideC, batch,
                                              _stream(stream)))


def sgemm_tf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """One TF32 product per multiply-add: faster, TF32 accuracy (see include/sgemm.h)."""
    _check(lib().sgemm_tf32(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                            _stream(stream)))


def sgemm_tf32_strided_batched(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                               strideC, batch, stream=None) -> None:
    _check(lib().sgemm_tf32_strided_batched(M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb,
                                            strideB, beta, _ptr(C), ldc, strideC, batch,
                                            _stream(stream)))


def _op(t) -> int:
    if t in (0, 1):
        return int(t)
    if isinstance(t, str) and t.upper() in ("N", "T"):
        return SGEMM_OP_T if t.upper() == "T" else SGEMM_OP_N
    return int(bool(t))


def sgemm_ex(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, path="simt",
             stream=None) -> None:
    """C = alpha * op(A) op(B) + beta * C; transa / transb are 'N' / 'T' (or 0 / 1),
    path is 'simt', '3xtf32' or 'tf32' (or its enum value)."""
    pth = _PATHS.get(path, path) if isinstance(path, str) else int(path)
    _check(lib().sgemm_ex(_op(transa), _op(transb), pth, M, N, K, alpha, _ptr(A), lda, _ptr(B),
                          ldb, beta, _ptr(C), ldc, _stream(stream)))


def sgemm_ex_strided_batched(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                             beta, C, ldc, strideC, batch, path="simt", stream=None) -> None:
    pth = _PATHS.get(path, path) if isinstance(path, str) else int(path)
    _check(lib().sgemm_ex_strided_batched(_op(transa), _op(transb), pth, M, N, K, alpha, _ptr(A),
                                          lda, strideA, _ptr(B), ldb, strideB, beta, _ptr(C), ldc,
                                          strideC, batch, _stream(stream)))


def sgemm_fused(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias=None,
                act="none", path="simt", stream=None) -> None:
    """C = act(alpha * op(A) op(B) + bias) + beta * C; act is 'none', 'relu', 'gelu',
    'gelu_tanh' or 'silu' (or its enum value); bias is an N-vector or None."""
    pth = _PATHS.get(path, path) if isinstance(path, str) else int(path)
    code = ACTIVATIONS[act] if isinstance(act, str) else int(act)
    _check(lib().sgemm_fused(_op(transa), _op(transb), pth, M, N, K, alpha, _ptr(A), lda,
                             _ptr(B), ldb, beta, _ptr(C), ldc, _ptr(bias), code, _stream(stream)))


def sgemm_fused_strided_batched(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                                beta, C, ldc, strideC, batch, bias=None, act="none", path="simt",
                                stream=None) -> None:
    pth = _PATHS.get(path, path) if isinstance(path, str) else int(path)
    code = ACTIVATIONS[act] if isinstance(act, str) else int(act)
    _check(lib().sgemm_fused_strided_batched(_op(transa), _op(transb), pth, M, N, K, alpha,
                                             _ptr(A), lda, strideA, _ptr(B), ldb, strideB, beta,
                                             _ptr(C), ldc, strideC, batch, _ptr(bias), code,
                                             _stream(stream)))


def _host_ptr(x):
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):  # a CPU torch tensor (pinned or not)
        if x.is_cuda:
            raise TypeError("sgemm_host takes host tensors")
        if str(x.dtype) != "torch.float32":
            raise TypeError("tensor arguments must be float32")
        return x.data_ptr()
    import numpy as np
    a = x if isinstance(x, np.ndarray) else np.asarray(x)
    if a.dtype != np.float32:
        raise TypeError("arrays must be float32")
    return a.ctypes.data


def sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """C = alpha * A.B + beta * C with host-memory operands (numpy arrays, CPU tensors or
    addresses); returns when C holds the result. Pinned memory lets copies overlap compute."""
    _check(lib().sgemm_host(M, N, K, alpha, _host_ptr(A), lda, _host_ptr(B), ldb, beta,
                            _host_ptr(C), ldc, _stream(stream)))


def sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """sgemm() that allocates no device memory (its scratch is a static array in the library)."""
    _check(lib().sgemm_noalloc(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                               _stream(stream)))


def sgemm_status_string(status: int) -> str:
    return lib().sgemm_status_string(status).decode()


def sgemm_last_error() -> str:
    return (lib().sgemm_last_error() or b"").decode()


def sgemm_device_status(stream=None) -> int:
    """Synchronises ``stream``; returns the status code (does not raise)."""
    return lib().sgemm_device_status(_stream(stream))


def sgemm_release_workspace() -> None:
    _check(lib().sgemm_release_workspace())


def sgemm_num_configs() -> int:
    return lib().sgemm_num_configs()


def sgemm_config_name(i: int) -> str | None:
    name = lib().sgemm_config_name(i)
    return None if name is None else name.decode()


def sgemm_select_config(M, N, K, alpha, A, lda, B, ldb, C, ldc, batch=1) -> int:
    return lib().sgemm_select_config(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                                     batch)


def sgemm_force_config(i: int) -> None:
    _check(lib().sgemm_force_config(i))


def sgemm_selftest_bounded_wait(which: int, stream=None) -> None:
    """Queue a kernel whose bounded wait expires (failure-path test); see include/sgemm.h."""
    _check(lib().sgemm_selftest_bounded_wait(which, _stream(stream)))


def matmul(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, tensor_cores: bool = False,
           stream=None):
    """torch convenience: row-major 2-D CUDA float32 tensors, returns C (allocated if None).

    Rows must be contiguous (stride(1) == 1); the row stride is the leading dimension.
    """
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("matmul expects A (M x K) and B (K x N)")
    M, K = A.shape
    N = B.shape[1]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
        beta = 0.0
    for t in (A, B, C):
        if t.stride(1) != 1 and t.shape[1] > 1:
            raise ValueError("rows must be contiguous")
    fn = sgemm_3xtf32 if tensor_cores else sgemm
    fn(M, N, K, alpha, A, max(A.stride(0), 1), B, max(B.stride(0), 1), beta, C,
       max(C.stride(0), 1), stream)
    return C
