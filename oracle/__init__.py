"""CPU oracle for the software-pipelined tiled GEMM: C = A * B, written plainly.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` may import this package; the library itself never
does, and the two share no code.

The arithmetic lives in ``oracle_gemm.c`` (and, for the streaming pipeline
``out = alpha * in``, ``oracle_stream.c``) (a plain triple loop, fp64 sums for
binary16/bfloat16 inputs, int64 sums for int8 inputs).  This module builds
that file with the host C compiler and marshals numpy arrays to it.

Source of the definition: "Hiding Memory Latency in CUDA: Asynchronous Loads
and Software Pipelines", opening section (a tiled GEMM loads A and B tiles,
multiplies and accumulates, and advances along K) and section 15 (the
pipeline feeds FP32 accumulators of the same product); "Pipeline GPU Kernel",
Step 5 item 4 (pipelining reorders loads and never changes the arithmetic).
The reference result is hence the definition of the matrix product itself.

Layouts: A row-major M x K; B column-major K x N, stored as the N x K array
``Bcm`` with ``Bcm[j, k] = B[k, j]``; C row-major M x N.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

IN_F16 = 0
IN_BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "oracle_gemm.c"), os.path.join(_HERE, "oracle_stream.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles oracle_gemm.c for the host (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm_float.argtypes = [i64, i64, i64, ctypes.c_int, p, p, p, p]
        lib.oracle_gemm_float_at.argtypes = [i64, i64, i64, ctypes.c_int, p, p, i64, p, p, p, p]
        lib.oracle_gemm_s8.argtypes = [i64, i64, i64, p, p, p]
        lib.oracle_gemm_s8_at.argtypes = [i64, i64, i64, p, p, i64, p, p, p]
        lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_f16.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_scale_f32.argtypes = [i64, ctypes.c_float, p, p]
        lib.oracle_scale_f32.restype = None
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        for f in (lib.oracle_gemm_float, lib.oracle_gemm_float_at,
                  lib.oracle_gemm_s8, lib.oracle_gemm_s8_at):
            f.restype = ctypes.c_int
        try:
            lib.oracle_set_threads(len(os.sched_getaffinity(0)))
        except AttributeError:  # pragma: no cover - non-Linux hosts
            pass
        _lib = lib
        return lib


def threads() -> int:
    """Number of OpenMP threads the oracle uses (all cores of the affinity mask)."""
    return int(_load().oracle_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits16(x) -> np.ndarray:
    """Raw 16-bit patterns of a binary16/bfloat16 array (numpy or torch)."""
    if hasattr(x, "detach"):  # torch tensor; bfloat16 has no numpy dtype
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype == np.int16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected 16-bit float patterns, got {x.dtype}")
    return x


def _int8(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.int8:
        raise TypeError(f"expected int8, got {x.dtype}")
    return x


def decode(bits: int, in_type: int) -> float:
    """Exact value of one binary16 (IN_F16) or bfloat16 (IN_BF16) pattern."""
    lib = _load()
    f = lib.oracle_decode_bf16 if in_type == IN_BF16 else lib.oracle_decode_f16
    return float(f(int(bits) & 0xFFFF))


def gemm_float(A, Bcm, in_type: int):
    """C = A * B and S = sum_k |A_ik B_kj|, both float64 M x N.

    A: M x K and Bcm: N x K (B column-major), binary16 or bfloat16 patterns.
    """
    a, b = _bits16(A), _bits16(Bcm)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    if M and N:
        rc = _load().oracle_gemm_float(M, N, K, in_type, _ptr(a), _ptr(b), _ptr(C), _ptr(S))
        if rc != 0:
            raise MemoryError("oracle could not allocate decoded inputs")
    return C, S


def gemm_float_at(A, Bcm, in_type: int, rows, cols):
    """The float product at the positions (rows[t], cols[t]); returns (C, S)."""
    a, b = _bits16(A), _bits16(Bcm)
    M, K = a.shape
    N, _ = b.shape
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be equal-length 1-D")
    if len(r) and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("sample position out of range")
    out = np.empty(len(r), dtype=np.float64)
    sabs = np.empty(len(r), dtype=np.float64)
    _load().oracle_gemm_float_at(M, N, K, in_type, _ptr(a), _ptr(b), len(r),
                                 _ptr(r), _ptr(c), _ptr(out), _ptr(sabs))
    return out, sabs


def gemm_s8(A, Bcm):
    """Exact int8 product C = A * B as int64 M x N (Bcm: N x K)."""
    a, b = _int8(A), _int8(Bcm)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    C = np.empty((M, N), dtype=np.int64)
    if M and N:
        _load().oracle_gemm_s8(M, N, K, _ptr(a), _ptr(b), _ptr(C))
    return C


def gemm_s8_at(A, Bcm, rows, cols):
    """The exact int8 product at the positions (rows[t], cols[t])."""
    a, b = _int8(A), _int8(Bcm)
    M, K = a.shape
    N, _ = b.shape
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if len(r) and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("sample position out of range")
    out = np.empty(len(r), dtype=np.int64)
    _load().oracle_gemm_s8_at(M, N, K, _ptr(a), _ptr(b), len(r), _ptr(r), _ptr(c), _ptr(out))
    return out


def scale_f32(x, alpha: float):
    """out[i] = alpha * in[i] in binary32, one rounding per element."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(a)
    if a.size:
        _load().oracle_scale_f32(a.size, float(alpha), _ptr(a), _ptr(out))
    return out
