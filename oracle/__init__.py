"""CPU oracle for the half-precision GEMM library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``complexity_matmul_gb300``) never imports it and shares no code with it.

Contents
--------
* :func:`gemm` -- O1, the plain definition ``C64 = A @ B`` as a sequential FP64
  triple loop in C (``oracle.c``), optionally on a sample of output rows.
  Every Strassen-family algorithm reaches this same result in exact arithmetic
  (FalconGEMM write-up, section "从 Strassen 出发": Strassen is algebraically
  equivalent to the standard product, only the rounding differs).
* :mod:`oracle.rounding` -- round-to-nearest-even from FP64 to FP16 / BF16,
  used to form the single final cast ``Cref = RNE_dtype(C64)`` (FalconGEMM
  write-up, numerics paragraph: accumulate in FP32 on chip and cast once at
  the end).
* :mod:`oracle.strassen` -- O2, textbook one- and two-level Strassen written as
  (U, V, W) coefficient tables and applied in the three steps the write-up
  names for the basic GPU pipeline: combine A and B blocks, run the block
  products, combine the products into C (section "从 LCMA 到 FalconGEMM").
* :mod:`oracle.epilogue` -- O3, the element-wise epilogue
  ``D = act(C64 + bias) + residual`` in FP64 (DeepGEMM tuning blog, section
  3.3; "Kernel 与性能", section "Fusion").

Pins (``tests/test_oracle_*.py``): hand-computed golden products, A.I = A,
linearity, agreement with numpy's matmul, exhaustive decoder checks, the Brent
equations for the Strassen tables, a brute-force 2x2 check, a recursive
Strassen written independently of the tables, hand-computed epilogues, normal
table values of GELU and the tanh form's known gap to it.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

F16 = 0
BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", f"liboracle.{platform.machine()}.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc/OpenMP for the host (x86_64 or aarch64)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-Wall",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_gemm.argtypes = [ctypes.c_int] + [ctypes.c_int64] * 3 + [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            lib.oracle_decode_f16.restype = ctypes.c_double
            lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_bf16.restype = ctypes.c_double
            lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the C triple loop runs on (OpenMP)."""
    return int(_load().oracle_num_threads())


def decode_c(bits: int, dtype: int) -> float:
    """Decode one 16-bit pattern with the C decoder (exposed for the pins)."""
    lib = _load()
    return lib.oracle_decode_bf16(bits) if dtype == BF16 else lib.oracle_decode_f16(bits)


def _bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are uint16 bit patterns (or float16)")
    return x


def gemm(A_bits: np.ndarray, Bnk_bits: np.ndarray, dtype: int, rows=None) -> np.ndarray:
    """O1: ``C64[r, j] = sum_k A[rows[r], k] * B[k, j]`` in FP64.

    ``A_bits``: M x K uint16 patterns (row-major A).  ``Bnk_bits``: N x K
    uint16 patterns, i.e. the K x N operand B stored column-major.  ``rows``:
    optional sequence of output row indices (default: all M rows).
    Returns an ``len(rows) x N`` float64 array.
    """
    A = _bits(A_bits)
    B = _bits(Bnk_bits)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("A must be M x K and B must be stored N x K")
    M, K = A.shape
    N = B.shape[0]
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    C = np.zeros((nrows, N), dtype=np.float64)
    rc = _load().oracle_gemm(
        int(dtype), M, N, K, A.ctypes.data if A.size else None, K,
        B.ctypes.data if B.size else None, K,
        rows_arr.ctypes.data if rows_arr is not None and nrows else None, nrows,
        C.ctypes.data if C.size else None)
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return C


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Decode FP16/BF16 bit patterns to float64 with numpy (exact)."""
    b = np.asarray(bits)
    if b.dtype == np.float16:
        return b.astype(np.float64)
    b = b.astype(np.uint16)
    with np.errstate(invalid="ignore", over="ignore"):
        if dtype == F16:
            return b.view(np.float16).astype(np.float64)
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


from . import rounding  # noqa: E402  (re-exported submodules)
from . import strassen  # noqa: E402
from . import epilogue  # noqa: E402


def reference_output(C64: np.ndarray, dtype: int) -> np.ndarray:
    """``Cref = RNE_dtype(C64)`` as uint16 bit patterns (one final cast)."""
    return rounding.rne_bits(C64, dtype)
