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


def test_noalloc_matches_strassen1_twice_in_a_row():
    h = lcg.Handle(0)
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
        torch.cuda.synchronize()
        assert h.sync_status() == 0
        assert torch.equal(C, ref)                                   # same kernels, same rounding
        assert_close(C, oracle_c64(A, B, "bf16"), "bf16", "strassen1")
    h.close()


def test_noalloc_rejects_problems_beyond_its_scratch():
    A = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, B, C) == lcg.ERR_TOO_LARGE
    assert b"fixed scratch" in lcg.lib().lcgemm_strerror(lcg.ERR_TOO_LARGE)
    # odd sizes are refused, as for explicit strassen1
    assert _noalloc(A[:, :72], B[:, :72], C) == lcg.ERR_UNSUPPORTED
