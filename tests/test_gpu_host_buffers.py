"""lcgemm_run_host: host buffers in and out, copies pipelined with the GEMM (GPU, through the C ABI)."""
import ctypes

import numpy as np
import pytest
import torch

import complexity_matmul_gb300 as lcg
import synthetic
from helpers import assert_bit_exact, oracle_c64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    handle = lcg.Handle(0)
    yield handle
    handle.close()


def _run_host(h, A, B, C, algo):
    """lcgemm_run_host on host tensors (A: M x K, B stored N x K, C: M x N; any row strides)."""
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = h.run_host_raw(A.shape[0], B.shape[0], A.shape[1], A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                        C.data_ptr(), C.stride(0), lcg.BF16, lcg.ALGOS[algo], sp)
    torch.cuda.synchronize()
    return rc


@pytest.mark.parametrize("M,N,K", [(8192, 2048, 1024), (4096, 1000, 520), (300, 260, 136), (6000, 512, 256),
                                   (4100, 4200, 512), (8192, 8192, 256), (2048, 10000, 128)])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffers_match_device_path(h, M, N, K, pinned):
    """The block-gridded, pipelined host path (ragged edge blocks included) gives the device path's
    result: bit for bit on integer inputs, and to FP32 summation order on N(0,1) inputs (at most one
    BF16 ulp apart)."""
    for dist in ("int3", "normal"):
        A, B = synthetic.operands(M, N, K, dist, 31, "bf16", "cuda")
        ref = h.run(A, B, algo="plain").cpu()
        Ah, Bh = A.cpu(), B.cpu()
        Ch = torch.full((M, N), 7.0, dtype=torch.bfloat16)
        if pinned:
            Ah, Bh, Ch = Ah.pin_memory(), Bh.pin_memory(), Ch.pin_memory()
        assert _run_host(h, Ah, Bh, Ch, "auto") == 0
        assert h.sync_status() == 0
        if dist == "int3":
            assert torch.equal(Ch, ref)
        else:
            diff = (Ch.float() - ref.float()).abs()
            sigma = ref.float().pow(2).mean().sqrt()
            bound = ref.float().abs() * 2.0 ** -7 + 1e-4 * sigma     # one BF16 ulp, plus FP32 noise near 0
            assert bool((diff <= bound).all())
            assert (Ch == ref).float().mean().item() > 0.99


def test_host_buffers_strided_integer_bit_exact(h):
    M, N, K = 4608, 384, 200
    Abig = synthetic.matrix(M, 264, "int3", 32, "bf16")
    Bbig = synthetic.matrix(N, 216, "int3", 33, "bf16")
    Cbig = torch.full((M, 400), 7.0, dtype=torch.bfloat16).pin_memory()
    A, B, C = Abig[:, :K], Bbig[:, :K], Cbig[:, 8:8 + N]
    assert _run_host(h, A, B, C, "plain") == 0
    assert_bit_exact(C, oracle_c64(A.contiguous(), B.contiguous(), "bf16"), "bf16")
    assert (Cbig[:, :8] == 7).all() and (Cbig[:, 8 + N:] == 7).all()


@pytest.mark.parametrize("algo", ["strassen1", "strassen2"])
def test_host_buffers_strassen(h, algo):
    M, N, K = 2048, 1024, 512
    A, B = synthetic.operands(M, N, K, "int3", 34, "bf16")
    C = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    assert _run_host(h, A.pin_memory(), B.pin_memory(), C, algo) == 0
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")


def test_host_buffers_repeated_calls_do_not_race(h):
    """Back-to-back calls reuse the staging buffers: each call waits for the previous one's copies."""
    M, N, K = 8192, 1024, 512
    data = [synthetic.operands(M, N, K, "int3", 40 + i, "bf16") for i in range(3)]
    outs = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in data]
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    pinned = [(A.pin_memory(), B.pin_memory()) for A, B in data]
    for (Ah, Bh), C in zip(pinned, outs):
        assert h.run_host_raw(M, N, K, Ah.data_ptr(), K, Bh.data_ptr(), K, C.data_ptr(), N, lcg.BF16, lcg.PLAIN,
                              sp) == 0
    torch.cuda.synchronize()
    for (A, B), C in zip(data, outs):
        assert_bit_exact(C, oracle_c64(A, B, "bf16", rows=np.arange(0, M, 97)), "bf16", rows=np.arange(0, M, 97))
