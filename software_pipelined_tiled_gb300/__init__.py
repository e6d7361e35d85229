"""Python binding of the software-pipelined tiled GEMM library (libsptgemm.so).

Argument marshalling only: every step of the product runs in the library's
CUDA kernels.  PyTorch is used for device memory and streams.  There is no
fallback: if the library is missing or no sm_103 device is present, calls
raise.

    import software_pipelined_tiled_gb300 as sptg
    C = sptg.gemm(A, Bcm, out_dtype=torch.float16)   # C = A @ Bcm.T

A is M x K row-major; B is K x N column-major, passed as its storage, the
N x K row-major tensor ``Bcm`` (``Bcm[j, k] = B[k, j]``); C is M x N row-major.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH, build

__all__ = ["DTYPES", "SptgError", "Config", "load", "gemm", "gemm_host", "gemm_raw", "plan_square",
           "gemm_strided_raw",
           "gemm_skinny_noalloc_raw",
           "stream_scale",
           "last_config",
           "last_error", "device_error", "status_string", "LIB_PATH", "build"]

# sptg_dtype values of include/sptgemm.h
DTYPES = {"f16_f32": 0, "f16_f16": 1, "s8_s32": 2, "bf16_bf16": 3, "bf16_f32": 4}
STATUS = {0: "SPTG_OK", -1: "SPTG_ERR_ARG", -2: "SPTG_ERR_ALIGN", -3: "SPTG_ERR_UNSUPPORTED",
          -4: "SPTG_ERR_LAUNCH", -5: "SPTG_ERR_TIMEOUT", -6: "SPTG_ERR_NOMEM",
          -7: "SPTG_ERR_CONFIG"}
KERNELS = {"auto": 0, "square": 1, "skinny": 2, "skinny_cluster": 3, "skinny_rows": 4,
           "skinny_pair": 5}

# the C functions every build must export (checked by the tests)
EXPORTS = ("sptg_gemm", "sptg_gemm_ex", "sptg_gemm_strided", "sptg_gemm_host",
           "sptg_plan_square", "sptg_plan", "sptg_status_string", "sptg_last_error",
           "sptg_last_config", "sptg_device_error", "sptg_version", "sptg_gemm_skinny_noalloc",
           "sptg_stream_scale", "sptg_stream_scale_ex")


class SptgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Config(ctypes.Structure):
    """sptg_config: 0 in a field means "let the library choose"."""
    _fields_ = [("kernel", ctypes.c_int), ("bn", ctypes.c_int), ("stages", ctypes.c_int),
                ("splits", ctypes.c_int), ("timeout_ms", ctypes.c_int),
                ("inject_stall", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("no_overlap", ctypes.c_int), ("trace", ctypes.c_void_p),
                ("stream_k", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libsptgemm.so (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if path is None and not os.path.exists(p):
            build()
        lib = ctypes.CDLL(p)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.sptg_gemm.argtypes = [i64, i64, i64, ctypes.c_int, vp, vp, vp, vp]
        lib.sptg_gemm.restype = ctypes.c_int
        lib.sptg_gemm_ex.argtypes = [i64, i64, i64, ctypes.c_int, vp, vp, vp, vp,
                                     ctypes.POINTER(Config)]
        lib.sptg_gemm_ex.restype = ctypes.c_int
        lib.sptg_gemm_strided.argtypes = [i64, i64, i64, ctypes.c_int, vp, i64, vp, i64, vp, i64,
                                          vp, ctypes.POINTER(Config)]
        lib.sptg_gemm_strided.restype = ctypes.c_int
        lib.sptg_gemm_host.argtypes = [i64, i64, i64, ctypes.c_int, vp, vp, vp, vp,
                                       ctypes.POINTER(Config)]
        lib.sptg_gemm_host.restype = ctypes.c_int
        lib.sptg_status_string.argtypes = [ctypes.c_int]
        lib.sptg_status_string.restype = ctypes.c_char_p
        lib.sptg_last_error.argtypes = []
        lib.sptg_last_error.restype = ctypes.c_char_p
        lib.sptg_last_config.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
        lib.sptg_last_config.restype = ctypes.c_int
        lib.sptg_device_error.argtypes = [vp]
        lib.sptg_device_error.restype = ctypes.c_int
        lib.sptg_gemm_skinny_noalloc.argtypes = [i64, i64, i64, ctypes.c_int, vp, vp, vp, vp]
        lib.sptg_gemm_skinny_noalloc.restype = ctypes.c_int
        lib.sptg_stream_scale.argtypes = [i64, ctypes.c_float, vp, vp, vp]
        lib.sptg_stream_scale.restype = ctypes.c_int
        lib.sptg_stream_scale_ex.argtypes = [i64, ctypes.c_float, vp, vp, vp,
                                             ctypes.POINTER(Config)]
        lib.sptg_stream_scale_ex.restype = ctypes.c_int
        lib.sptg_plan_square.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_int)]
        lib.sptg_plan_square.restype = ctypes.c_int
        lib.sptg_plan.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                  ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_int)]
        lib.sptg_plan.restype = ctypes.c_int
        lib.sptg_version.argtypes = []
        lib.sptg_version.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def plan_square(M: int, N: int, K: int, dtype: str, sm_count: int,
                config: Config | None = None) -> dict:
    """The square kernel's plan for a shape on a GPU of sm_count SMs (host only)."""
    out = (ctypes.c_int * 7)()
    cfg = ctypes.byref(config) if config is not None else None
    rc = int(load().sptg_plan_square(M, N, K, DTYPES[dtype], sm_count, cfg, out))
    if rc != 0:
        raise SptgError(rc, last_error() or status_string(rc))
    keys = ("bn", "pair", "tiles", "workers", "stream_k_tiles", "stream_k_workers", "max_contrib")
    return dict(zip(keys, list(out)))


def plan(M: int, N: int, K: int, dtype: str, sm_count: int,
         config: Config | None = None) -> dict:
    """The kernel sptg_gemm would choose for a shape on a GPU of sm_count SMs (host only)."""
    out = (ctypes.c_int * 6)()
    cfg = ctypes.byref(config) if config is not None else None
    rc = int(load().sptg_plan(M, N, K, DTYPES[dtype], sm_count, cfg, out))
    if rc != 0:
        raise SptgError(rc, last_error() or status_string(rc))
    names = {v: k for k, v in KERNELS.items()}
    keys = ("kernel", "width", "grid", "cluster", "mma_n", "stream_k_tiles")
    d = dict(zip(keys, list(out)))
    d["kernel"] = names[d["kernel"]]
    return d


def status_string(status: int) -> str:
    return load().sptg_status_string(int(status)).decode()


def last_error() -> str:
    return load().sptg_last_error().decode()


def last_config() -> str:
    lib = load()
    buf = ctypes.create_string_buffer(512)
    lib.sptg_last_config(buf, len(buf))
    return buf.value.decode()


def _current_stream(device_index: int) -> int:
    """Raw handle of PyTorch's current stream on a device."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return int(raw(device_index))
    return torch.cuda.current_stream(device_index).cuda_stream


def _stream_handle(stream, device_index: int | None = None) -> int:
    if stream is None:
        import torch
        return _current_stream(torch.cuda.current_device() if device_index is None
                               else device_index)
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gemm_raw(M: int, N: int, K: int, dtype: str | int, A_ptr: int, B_ptr: int, C_ptr: int,
             stream: int = 0, config: Config | None = None) -> int:
    """Calls sptg_gemm_ex with raw device pointers; returns the status code."""
    d = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    cfg = ctypes.byref(config) if config is not None else None
    return int((_lib or load()).sptg_gemm_ex(M, N, K, d, A_ptr, B_ptr, C_ptr, stream, cfg))


def gemm_strided_raw(M: int, N: int, K: int, dtype: str | int, A_ptr: int, lda: int, B_ptr: int,
                     ldb: int, C_ptr: int, ldc: int, stream: int = 0,
                     config: Config | None = None) -> int:
    """Calls sptg_gemm_strided (leading dimensions in elements); returns the status code."""
    d = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    cfg = ctypes.byref(config) if config is not None else None
    return int((_lib or load()).sptg_gemm_strided(M, N, K, d, A_ptr, lda, B_ptr, ldb, C_ptr, ldc,
                                                  stream, cfg))


def gemm_skinny_noalloc_raw(M: int, N: int, K: int, dtype: str | int, A_ptr: int, B_ptr: int,
                            C_ptr: int, stream: int = 0) -> int:
    """Calls sptg_gemm_skinny_noalloc (the skinny kernel with its split-K
    scratch in a fixed array inside the library, so the call allocates
    nothing); returns the status code."""
    d = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    return int(load().sptg_gemm_skinny_noalloc(M, N, K, d, A_ptr, B_ptr, C_ptr, stream))


_KEYS: dict = {}


def _dtype_key(in_dtype, out_dtype) -> str:
    key = _KEYS.get((in_dtype, out_dtype))
    if key is not None:
        return key
    import torch
    names = {torch.float16: "f16", torch.bfloat16: "bf16", torch.int8: "s8",
             torch.float32: "f32", torch.int32: "s32"}
    key = f"{names.get(in_dtype, '?')}_{names.get(out_dtype, '?')}"
    if key not in DTYPES:
        raise ValueError(f"unsupported input/output dtype pair {in_dtype} -> {out_dtype}")
    _KEYS[(in_dtype, out_dtype)] = key
    return key


def _row_pitch(t, name: str) -> int:
    """Elements between rows of a 2-D tensor whose rows are contiguous."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1) or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name} must be a 2-D tensor with contiguous rows (stride(1) == 1)")
    return max(int(t.stride(0)), int(t.shape[1]))


def gemm(A, Bcm, C=None, out_dtype=None, stream=None, config: Config | None = None,
         kernel: str | None = None, stages: int = 0, bn: int = 0, splits: int = 0,
         cta_pair: int = 0, stream_k: int = 0):
    """C = A * B on the GPU, with A (M x K) and Bcm (N x K) CUDA tensors.

    Each of A, Bcm and C may be a row-strided view (contiguous rows, any row
    pitch meeting the library's 16-byte rule), e.g. a column slice of a wider
    matrix; C's elements outside the view are left untouched.  out_dtype
    defaults to the input type for binary16/bfloat16 and int32 for int8.
    Returns C.  Raises SptgError on any failure.
    """
    import torch
    if A.dim() != 2 or Bcm.dim() != 2 or A.shape[1] != Bcm.shape[1]:
        raise ValueError("A must be M x K and Bcm N x K")
    if A.dtype != Bcm.dtype:
        raise ValueError("A and Bcm must have the same dtype")
    if not (A.is_cuda and Bcm.is_cuda):
        raise ValueError("A and Bcm must be CUDA tensors")
    lda, ldb = _row_pitch(A, "A"), _row_pitch(Bcm, "Bcm")
    M, K = A.shape
    N = Bcm.shape[0]
    if out_dtype is None:
        out_dtype = C.dtype if C is not None else (torch.int32 if A.dtype == torch.int8 else A.dtype)
    key = _dtype_key(A.dtype, out_dtype)
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype, device=A.device)
    elif C.shape != (M, N) or C.dtype != out_dtype or not C.is_cuda:
        raise ValueError("C must be an M x N CUDA tensor of the output dtype")
    ldc = _row_pitch(C, "C")
    if config is None and (kernel or stages or bn or splits or cta_pair or stream_k):
        config = Config(KERNELS[kernel or "auto"], bn, stages, splits, 0, 0, cta_pair)
        config.stream_k = stream_k
    dev = A.get_device()
    args = (M, N, K, DTYPES[key], A.data_ptr(), lda, Bcm.data_ptr(), ldb, C.data_ptr(), ldc,
            _stream_handle(stream, dev), ctypes.byref(config) if config is not None else None)
    lib = _lib or load()
    if dev == torch.cuda.current_device():
        rc = lib.sptg_gemm_strided(*args)
    else:
        with torch.cuda.device(dev):
            rc = lib.sptg_gemm_strided(*args)
    if rc != 0:
        raise SptgError(rc, last_error() or status_string(rc))
    return C


def gemm_host(A, Bcm, C=None, out_dtype=None, stream=None, config: Config | None = None):
    """C = A * B with A, Bcm and C in host memory (pinned for asynchronous copies).

    The library copies the operands to its own device buffers, multiplies, and
    copies C back, all enqueued on `stream` (default: the current stream);
    the call returns without waiting.  Returns C (allocated pinned if None).
    """
    import torch
    if A.dim() != 2 or Bcm.dim() != 2 or A.shape[1] != Bcm.shape[1]:
        raise ValueError("A must be M x K and Bcm N x K")
    if A.dtype != Bcm.dtype or A.is_cuda or Bcm.is_cuda:
        raise ValueError("A and Bcm must be host tensors of the same dtype")
    if not (A.is_contiguous() and Bcm.is_contiguous()):
        raise ValueError("A and Bcm must be contiguous")
    M, K = A.shape
    N = Bcm.shape[0]
    if out_dtype is None:
        out_dtype = C.dtype if C is not None else (torch.int32 if A.dtype == torch.int8 else A.dtype)
    key = _dtype_key(A.dtype, out_dtype)
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype).pin_memory()
    elif C.shape != (M, N) or C.dtype != out_dtype or C.is_cuda or not C.is_contiguous():
        raise ValueError("C must be a contiguous M x N host tensor of the output dtype")
    cfg = ctypes.byref(config) if config is not None else None
    rc = int((_lib or load()).sptg_gemm_host(M, N, K, DTYPES[key], A.data_ptr(), Bcm.data_ptr(),
                                             C.data_ptr(), _stream_handle(stream), cfg))
    if rc != 0:
        raise SptgError(rc, last_error() or status_string(rc))
    return C


def stream_scale(x, alpha: float, out=None, stream=None, config: Config | None = None):
    """out = alpha * x for a contiguous binary32 CUDA tensor x (out may be x)."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must match x")
    cfg = ctypes.byref(config) if config is not None else None
    rc = int((_lib or load()).sptg_stream_scale_ex(x.numel(), float(alpha), x.data_ptr(),
                                                   out.data_ptr(), _stream_handle(stream), cfg))
    if rc != 0:
        raise SptgError(rc, last_error() or status_string(rc))
    return out


def device_error(stream=None) -> int:
    """Synchronizes the stream and returns (and clears) the device error status."""
    return int(load().sptg_device_error(_stream_handle(stream)))
