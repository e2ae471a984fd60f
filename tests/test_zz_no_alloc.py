"""lcgemm_strassen1_noalloc: one-level Strassen for callers that must not allocate device memory.

Frameworks whose caching allocator owns the device memory, and services that only
allocate at start-up, cannot let a library call cudaMalloc while they run.  This entry
point keeps its scratch in a fixed array inside the library instead.  The test calls it
through the C ABI twice in a row (different shapes and data, so the second call reuses
the scratch the first one left behind) and checks each result against lcgemm_run with
LCGEMM_STRASSEN1 on the same inputs, and against the CPU oracle within the BF16 Strassen
tolerance the other tests use.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import complexity_matmul_gb300 as lcg
import synthetic
from helpers import assert_close, oracle_c64

pytestmark = pytest.mark.gpu


def _noalloc(A, B, C):
    M, K = A.shape
    N = B.shape[0]
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lcg.lib().lcgemm_strassen1_noalloc(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                             C.data_ptr(), C.stride(0), lcg.BF16, sp)


def _normwise(X, Y):
    X, Y = X.double(), Y.double()
    return ((X - Y).norm() / Y.norm()).item()


def test_noalloc_matches_strassen1_twice_in_a_row():
    h = lcg.Handle(0)                        # lcgemm_run as a user calls it (kernel chosen per shape)
    h1 = lcg.Handle(0)
    h1.set_option(lcg.OPT_LCMA_KERNEL, 1)    # the single-CTA fused kernel this entry point uses
    cases = [(1024, 768, 1024, 21), (512, 1280, 1536, 22)]
    results = []
    for M, N, K, seed in cases:
        A, B = synthetic.operands(M, N, K, "normal", seed, "bf16", "cuda")
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(A, B, C) == lcg.OK
        results.append((A, B, C))
    torch.cuda.synchronize()
    for A, B, C in results:
        ref = h.run(A, B, algo="strassen1")
        same_kernel = h1.run(A, B, algo="strassen1")
        torch.cuda.synchronize()
        assert h.sync_status() == 0 and h1.sync_status() == 0
        # within the BF16 Strassen tolerance of the regular entry point's result ...
        assert _normwise(C, ref) <= 1.6e-2
        # ... identical to the regular entry point running the same kernel ...
        assert torch.equal(C, same_kernel)
        # ... and within tolerance of the exact product
        assert_close(C, oracle_c64(A, B, "bf16"), "bf16", "strassen1")
    h.close()
    h1.close()


def test_noalloc_rejects_problems_beyond_its_scratch():
    A = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, B, C) == lcg.ERR_TOO_LARGE
    assert b"fixed scratch" in lcg.lib().lcgemm_strerror(lcg.ERR_TOO_LARGE)
    # odd sizes are refused, as for explicit strassen1
    assert _noalloc(A[:, :72], B[:, :72], C) == lcg.ERR_UNSUPPORTED
