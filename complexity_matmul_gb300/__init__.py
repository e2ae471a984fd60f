"""Python binding of ``liblcgemm`` (argument marshalling only).

Every step of the GEMM runs in the CUDA kernels of ``liblcgemm``; this module
only loads the library with ctypes, converts arguments and raises on status
codes.  There is no CPU or library fallback: if the library is missing or
was built for another machine, :func:`lib` raises.

The names mirror ``include/lcgemm.h``: ``lcgemm_create`` -> :class:`Handle`,
``lcgemm_run`` -> :meth:`Handle.run`, and so on.  :func:`gemm` is a
convenience wrapper for torch CUDA tensors (device memory and the current
stream come from torch).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

F16, BF16 = 0, 1
PLAIN, STRASSEN1, STRASSEN2, AUTO, STRASSEN1_UNFUSED = 0, 1, 2, 3, 4
ALGOS = {"plain": PLAIN, "strassen1": STRASSEN1, "strassen2": STRASSEN2, "auto": AUTO,
         "strassen1_unfused": STRASSEN1_UNFUSED}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
OK, ERR_ARG, ERR_ALIGN, ERR_UNSUPPORTED, ERR_ALIAS, ERR_CUDA, ERR_TIMEOUT, ERR_NOMEM = 0, -1, -2, -3, -4, -5, -6, -7
ERR_TOO_LARGE, ERR_CAPTURE = -8, -9
OPT_WAIT_TIMEOUT_US, OPT_GROUP_ORDER, OPT_SPLIT, OPT_MAX_CTAS = 1, 2, 3, 4
OPT_PEAK_GFLOPS, OPT_HBM_GBPS, OPT_DEBUG_DROP_SIGNAL, OPT_PLAIN_KERNEL, OPT_LCMA_KERNEL, OPT_PDL = 5, 6, 7, 8, 9, 10
ACT_NONE, ACT_RELU, ACT_GELU, ACT_GELU_TANH = 0, 1, 2, 3
ACTS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU, "gelu_tanh": ACT_GELU_TANH}

EXPORTS = ("lcgemm_create", "lcgemm_destroy", "lcgemm_run", "lcgemm_run_host", "lcgemm_last_algo",
           "lcgemm_select", "lcgemm_estimate", "lcgemm_sync_status", "lcgemm_set_option",
           "lcgemm_strerror", "lcgemm_strassen1_noalloc", "lcgemm_run_epilogue", "lcgemm_noalloc_status",
           "lcgemm_noalloc_debug_fail")

_lock = threading.Lock()
_lib = None


class LcgemmError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})")


class Epilogue(ctypes.Structure):
    """``lcgemm_epilogue``: C = act(A.B + bias) + residual (device pointers or None)."""
    _fields_ = [("bias", ctypes.c_void_p), ("residual", ctypes.c_void_p), ("ldr", ctypes.c_int64),
                ("act", ctypes.c_int)]


def lib_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = False):
    """Load ``liblcgemm`` (built by ``__graft_entry__.build()`` / ``_build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"liblcgemm is not built for this machine ({path}); run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'` first")
            _build.build()
        L = ctypes.CDLL(path)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.lcgemm_create.argtypes = [ctypes.POINTER(vp), i32]
        L.lcgemm_destroy.argtypes = [vp]
        run_args = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, vp]
        L.lcgemm_run.argtypes = run_args
        L.lcgemm_run_host.argtypes = run_args
        L.lcgemm_run_epilogue.argtypes = run_args[:-1] + [ctypes.POINTER(Epilogue), vp]
        L.lcgemm_last_algo.argtypes = [vp]
        L.lcgemm_select.argtypes = [vp, i64, i64, i64, i32]
        L.lcgemm_estimate.argtypes = [vp, i64, i64, i64, i32, i32, ctypes.POINTER(ctypes.c_double)]
        L.lcgemm_sync_status.argtypes = [vp, vp]
        L.lcgemm_set_option.argtypes = [vp, i32, i64]
        L.lcgemm_strassen1_noalloc.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, vp]
        L.lcgemm_noalloc_status.argtypes = [vp]
        L.lcgemm_noalloc_debug_fail.argtypes = []
        L.lcgemm_strerror.argtypes = [i32]
        L.lcgemm_strerror.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name != "lcgemm_strerror":
                getattr(L, name).restype = i32
        _lib = L
        return L


def strerror(code: int) -> str:
    try:
        return lib().lcgemm_strerror(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def _check(code: int, what: str) -> int:
    if code < 0:
        raise LcgemmError(code, what)
    return code


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"lcgemm takes float16 or bfloat16 tensors, got {t.dtype}")


def _ld(t) -> int:
    """Leading dimension to pass for a 2-D tensor (a single row may use any ld >= its length)."""
    if t.shape[0] > 1:
        return t.stride(0)
    return max(8, (t.shape[1] + 7) // 8 * 8)


def _algo_code(algo) -> int:
    return ALGOS[algo] if isinstance(algo, str) else int(algo)


def _act_code(act) -> int:
    return ACTS[act] if isinstance(act, str) else int(act)


PLANNING_DEVICE = -1


class Handle:
    """Owns an ``lcgemm_t`` (workspace, error word, options) for one device.

    ``Handle(PLANNING_DEVICE)`` answers cost-model queries without touching CUDA.
    """

    def __init__(self, device: int = 0):
        self._lib = lib()
        h = ctypes.c_void_p()
        _check(self._lib.lcgemm_create(ctypes.byref(h), int(device)), "lcgemm_create")
        self._h = h
        self.device = int(device)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.lcgemm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def ptr(self):
        return self._h

    # raw ABI calls ---------------------------------------------------------
    def run_raw(self, M, N, K, A, lda, B, ldb, C, ldc, dtype, algo, stream=None) -> int:
        """``lcgemm_run`` with raw integers / pointers; returns the status code."""
        return self._lib.lcgemm_run(self._h, M, N, K, A, lda, B, ldb, C, ldc, dtype, _algo_code(algo), stream)

    def run_epilogue_raw(self, M, N, K, A, lda, B, ldb, C, ldc, dtype, algo, bias=None, residual=None, ldr=0,
                         act=ACT_NONE, stream=None) -> int:
        ep = Epilogue(bias, residual, int(ldr), _act_code(act))
        return self._lib.lcgemm_run_epilogue(self._h, M, N, K, A, lda, B, ldb, C, ldc, dtype, _algo_code(algo),
                                             ctypes.byref(ep), stream)

    def run_host_raw(self, M, N, K, A, lda, B, ldb, C, ldc, dtype, algo, stream=None) -> int:
        return self._lib.lcgemm_run_host(self._h, M, N, K, A, lda, B, ldb, C, ldc, dtype, _algo_code(algo), stream)

    def last_algo(self) -> int:
        return _check(self._lib.lcgemm_last_algo(self._h), "lcgemm_last_algo")

    def select(self, M, N, K, dtype=BF16) -> int:
        return _check(self._lib.lcgemm_select(self._h, M, N, K, dtype), "lcgemm_select")

    def estimate(self, M, N, K, dtype=BF16, algo=PLAIN) -> float:
        s = ctypes.c_double()
        _check(self._lib.lcgemm_estimate(self._h, M, N, K, dtype, _algo_code(algo), ctypes.byref(s)),
               "lcgemm_estimate")
        return s.value

    def sync_status(self, stream=None) -> int:
        return self._lib.lcgemm_sync_status(self._h, stream)

    def set_option(self, option: int, value: int):
        _check(self._lib.lcgemm_set_option(self._h, int(option), int(value)), "lcgemm_set_option")

    # torch convenience -----------------------------------------------------
    def run(self, A, Bnk, C=None, algo="plain", stream=None, bias=None, residual=None, act="none"):
        """C = act(A . B + bias) + residual for torch CUDA tensors.

        ``A``: M x K (row stride >= K, unit column stride); ``Bnk``: the K x N
        operand stored as N x K (the column-major layout of B); ``C``: M x N
        output (allocated if None); ``bias``: N values or None; ``residual``:
        M x N (may be ``C`` itself) or None; ``act``: "none", "relu", "gelu" or
        "gelu_tanh".  Runs on ``stream`` (default: torch's current stream).
        Returns C.
        """
        import torch
        if A.dim() != 2 or Bnk.dim() != 2 or A.shape[1] != Bnk.shape[1]:
            raise ValueError("A must be M x K and Bnk must be N x K")
        if A.dtype != Bnk.dtype:
            raise TypeError("A and B must have the same dtype")
        if A.stride(1) != 1 or Bnk.stride(1) != 1:
            raise ValueError("A and Bnk must be contiguous along K")
        M, K = A.shape
        N = Bnk.shape[0]
        if C is None:
            # rows padded to a multiple of 8 elements: the library needs 16-byte row starts
            C = torch.empty((M, (N + 7) // 8 * 8), dtype=A.dtype, device=A.device)[:, :N]
        if C.dtype != A.dtype or C.stride(1) != 1 or tuple(C.shape) != (M, N):
            raise ValueError("C must be M x N of the input dtype with unit column stride")
        if stream is None:
            stream = torch.cuda.current_stream(A.device)
        sp = ctypes.c_void_p(stream.cuda_stream)
        args = (M, N, K, A.data_ptr(), _ld(A), Bnk.data_ptr(), _ld(Bnk), C.data_ptr(), _ld(C), _dtype_code(A),
                _algo_code(algo))
        if bias is None and residual is None and _act_code(act) == ACT_NONE:
            _check(self.run_raw(*args, sp), "lcgemm_run")
            return C
        if bias is not None and (bias.dtype != A.dtype or bias.dim() != 1 or bias.shape[0] != N
                                 or bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous vector of N values of the input dtype")
        if residual is not None and (residual.dtype != A.dtype or tuple(residual.shape) != (M, N)
                                     or residual.stride(1) != 1):
            raise ValueError("residual must be M x N of the input dtype with unit column stride")
        rc = self.run_epilogue_raw(*args, bias=None if bias is None else bias.data_ptr(),
                                   residual=None if residual is None else residual.data_ptr(),
                                   ldr=0 if residual is None else _ld(residual), act=act, stream=sp)
        _check(rc, "lcgemm_run_epilogue")
        return C


_default = {}


def default_handle(device: int = 0) -> Handle:
    h = _default.get(device)
    if h is None:
        h = _default[device] = Handle(device)
    return h


def gemm(A, Bnk, algo="plain", out=None, bias=None, residual=None, act="none"):
    """C = act(A . B + bias) + residual on A's device with the per-device default handle."""
    return default_handle(A.device.index or 0).run(A, Bnk, out, algo, bias=bias, residual=residual, act=act)
