"""lcgemm_strassen1_noalloc: one-level Strassen for callers that must not allocate device memory.

Frameworks whose caching allocator owns the device memory, and services that only
allocate at start-up, cannot let a library call cudaMalloc while they run.  This entry
point keeps its scratch in a fixed array inside the library instead.  The tests call it
through the C ABI, always twice in a row (different shapes and data, so the second call
reuses the scratch the first one left behind), and check each result against lcgemm_run
with LCGEMM_STRASSEN1 on the same inputs and against the CPU oracle, within the Strassen
tolerances the other tests use (bit for bit on integer inputs).  lcgemm_noalloc_status
reports a device-side wait that ran out; the test plants that error from the host.  This
file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import complexity_matmul_gb300 as lcg
import synthetic
from helpers import assert_bit_exact, assert_close, oracle_c64

pytestmark = pytest.mark.gpu


def _noalloc(A, B, C, dtype=lcg.BF16):
    M, K = A.shape
    N = B.shape[0]
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lcg.lib().lcgemm_strassen1_noalloc(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                             C.data_ptr(), C.stride(0), dtype, sp)


def _status():
    return lcg.lib().lcgemm_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _normwise(X, Y):
    X, Y = X.double(), Y.double()
    return ((X - Y).norm() / Y.norm()).item()


def _code(dtype):
    return lcg.BF16 if dtype == "bf16" else lcg.F16


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
    assert _status() == lcg.OK
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


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_noalloc_ragged_half_blocks(dtype):
    """Quadrants that are not multiples of the 128 x 128 Group tile: 500 x 504 (the same block
    split lcgemm_run uses: bit for bit against it) and 499 x 501 (odd quadrant widths, which
    lcgemm_run would pad: against the oracle), each on integer inputs (exact) and N(0,1)."""
    h1 = lcg.Handle(0)
    h1.set_option(lcg.OPT_LCMA_KERNEL, 1)
    dt = torch.float16 if dtype == "f16" else torch.bfloat16
    for dist, seed in (("int3", 31), ("normal", 32)):
        runs = []
        for (M, N, K) in ((1000, 1008, 1040), (998, 1002, 1040)):
            A, B = synthetic.operands(M, N, K, dist, seed, dtype, "cuda")
            C = torch.empty((M, (N + 7) // 8 * 8), dtype=dt, device="cuda")[:, :N]
            assert _noalloc(A, B, C, _code(dtype)) == lcg.OK
            runs.append((A, B, C))
        assert _status() == lcg.OK
        for A, B, C in runs:
            ref64 = oracle_c64(A, B, dtype)
            if dist == "int3":
                assert_bit_exact(C, ref64, dtype)
            else:
                assert_close(C, ref64, dtype, "strassen1")
            if C.shape[1] % 16 == 0:
                same = h1.run(A, B, algo="strassen1")
                torch.cuda.synchronize()
                assert h1.sync_status() == 0
                assert torch.equal(C, same)
    h1.close()


def test_noalloc_fit_boundary_1792():
    """M = N = K = 1792 is the largest cube whose summed operands fit the fixed scratch: it runs
    (twice, the second time on other data) and matches the oracle on sampled rows; a deeper K no
    longer fits."""
    n = 1792
    rows = synthetic.row_sample(n, 64)
    for seed in (41, 42):
        A, B = synthetic.operands(n, n, n, "normal", seed, "bf16", "cuda")
        C = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(A, B, C) == lcg.OK
        assert _status() == lcg.OK
        assert_close(C, oracle_c64(A, B, "bf16", rows=rows), "bf16", "strassen1", rows=rows)
    A = torch.zeros((n, 1936), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((n, 1936), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, B, C) == lcg.ERR_TOO_LARGE


def test_noalloc_rejects_problems_beyond_its_scratch():
    A = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((2048, 2048), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, B, C) == lcg.ERR_TOO_LARGE
    assert b"fixed scratch" in lcg.lib().lcgemm_strerror(lcg.ERR_TOO_LARGE)
    # odd sizes are refused, as for explicit strassen1 without padding
    assert _noalloc(A[:, :72], B[:, :72], C) == lcg.ERR_UNSUPPORTED


def test_noalloc_empty_k_writes_zeros():
    """K = 0: C is the empty product, zeros, as lcgemm_run gives (two calls, C pre-filled)."""
    for M, N in ((64, 48), (130, 66)):
        A = torch.zeros((M, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
        B = torch.zeros((N, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
        C = torch.full((M, (N + 7) // 8 * 8), 5.0, dtype=torch.bfloat16, device="cuda")
        sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lcg.lib().lcgemm_strassen1_noalloc(M, N, 0, A.data_ptr(), 8, B.data_ptr(), 8, C.data_ptr(), C.stride(0),
                                                lcg.BF16, sp)
        assert rc == lcg.OK
        torch.cuda.synchronize()
        assert bool((C[:, :N] == 0).all())
        assert bool((C[:, N:] == 5.0).all())


def test_noalloc_allocates_nothing():
    """After a first call (which looks up the array's device address), further calls leave the
    device's free memory unchanged."""
    A, B = synthetic.operands(1024, 1024, 1024, "normal", 51, "bf16", "cuda")
    C = torch.empty((1024, 1024), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, B, C) == lcg.OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert _noalloc(A, B, C) == lcg.OK
    assert _status() == lcg.OK
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_status_reports_a_failed_wait_once():
    """A wait that ran out leaves the array's error word set; lcgemm_noalloc_status reports
    LCGEMM_ERR_TIMEOUT once and clears it, and later calls work.  The failure is planted from the
    host (lcgemm_noalloc_debug_fail), so no device-side wait has to run out."""
    assert _status() == lcg.OK
    assert lcg.lib().lcgemm_noalloc_debug_fail() == lcg.OK
    A, B = synthetic.operands(512, 512, 512, "int3", 61, "bf16", "cuda")
    C = torch.empty((512, 512), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, B, C) == lcg.OK             # a later call does not hide the earlier failure
    assert _status() == lcg.ERR_TIMEOUT
    assert _status() == lcg.OK
    for _ in range(2):
        assert _noalloc(A, B, C) == lcg.OK
    assert _status() == lcg.OK
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")
