"""lcgemm_run captured into CUDA graphs: every kernel path replays correctly on new input contents,
and a capture that would need a handle buffer to grow is refused without breaking the capture."""
import ctypes

import numpy as np
import pytest
import torch

import complexity_matmul_gb300 as lcg
import oracle
import synthetic
from helpers import assert_bit_exact, oracle_c64, oracle_epilogue

pytestmark = pytest.mark.gpu

# (M, N, K, algo, plain kernel option, epilogue): the CTA-pair tiles, the single-CTA tiles with a
# last-arriver split-K sum (counters reset in the graph) and with the separate reduction, the GEMV,
# the stream-K skinny kernel (epoch-tagged counters, reset in the graph), one- and two-level Strassen
CASES = [(2048, 2048, 1024, "plain", 0, False), (16, 14336, 3072, "plain", 1, False),
         (128, 256, 8192, "plain", 0, True), (1, 4096, 4096, "plain", 0, False),
         (16, 1024, 4096, "plain", 3, False), (1024, 1024, 1024, "strassen1", 0, True),
         (512, 512, 512, "strassen2", 0, False), (130, 66, 72, "strassen1", 0, False)]


@pytest.mark.parametrize("M,N,K,algo,kernel,ep", CASES)
def test_capture_and_replay(M, N, K, algo, kernel, ep):
    h = lcg.Handle(0)
    if kernel:
        h.set_option(lcg.OPT_PLAIN_KERNEL, kernel)
    A, B = synthetic.operands(M, N, K, "int3", 90, "bf16", "cuda")
    C = torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")[:, :N]
    bias = synthetic.matrix(1, N, "int3", 91, "bf16", "cuda")[0] if ep else None
    kw = {"bias": bias, "act": "relu"} if ep else {}
    h.run(A, B, C, algo=algo, **kw)        # outside the capture: buffers get their size
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h.run(A, B, C, algo=algo, **kw)
    for seed in (92, 93):
        A2, B2 = synthetic.operands(M, N, K, "int3", seed, "bf16", "cuda")
        A.copy_(A2)
        B.copy_(B2)
        C.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert h.sync_status() == 0
        if ep:
            D64, _ = oracle_epilogue(A, B, "bf16", bias, None, "relu")
            assert_bit_exact(C, D64, "bf16")
        else:
            assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")
    h.close()


def test_capture_refuses_buffer_growth():
    h = lcg.Handle(0)                      # fresh handle: no workspace yet
    M = N = K = 1024
    A, B = synthetic.operands(M, N, K, "int3", 94, "bf16", "cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Ah = torch.empty((4, 64), dtype=torch.bfloat16).pin_memory()
    Ch = torch.empty((4, 64), dtype=torch.bfloat16).pin_memory()
    g = torch.cuda.CUDAGraph()
    codes = []
    with torch.cuda.graph(g):
        C.fill_(1.0)
        sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        codes.append(h.run_raw(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), N, lcg.BF16,
                               lcg.STRASSEN1, sp))
        codes.append(h.run_host_raw(4, 64, 64, Ah.data_ptr(), 64, Ah.data_ptr(), 64, Ch.data_ptr(), 64, lcg.BF16,
                                    lcg.PLAIN, sp))
    assert codes == [lcg.ERR_CAPTURE, lcg.ERR_CAPTURE]
    g.replay()                             # the capture (the fill alone) is still a valid graph
    torch.cuda.synchronize()
    assert bool((C == 1.0).all())
    # the same run outside the capture works and later captures of it succeed
    h.run(A, B, C, algo="strassen1")
    torch.cuda.synchronize()
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")
    h.close()


def test_capture_claimed_items():
    """The CTA-pair kernel's claimed-item path (8 CTAs, 64 tiles = 16 waves): the counter's reset is
    part of the graph, so every replay runs every tile once."""
    M = N = 2048
    K = 512
    h = lcg.Handle(0)
    h.set_option(lcg.OPT_PLAIN_KERNEL, 2)
    h.set_option(lcg.OPT_MAX_CTAS, 8)
    A, B = synthetic.operands(M, N, K, "int3", 95, "bf16", "cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    h.run(A, B, C, algo="plain")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h.run(A, B, C, algo="plain")
    for seed in (96, 97):
        A2, B2 = synthetic.operands(M, N, K, "int3", seed, "bf16", "cuda")
        A.copy_(A2)
        B.copy_(B2)
        C.fill_(0)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        assert h.sync_status() == 0
        assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")
    h.close()


def test_capture_cluster_k_sums():
    """The single-CTA kernel whose K chunks are summed inside clusters of four (16 x 4096 x 14336),
    captured with a fused epilogue and replayed on new operands: a cluster launch inside a graph."""
    M, N, K = 16, 4096, 14336
    h = lcg.Handle(0)
    A, B = synthetic.operands(M, N, K, "int3", 98, "bf16", "cuda")
    b = synthetic.matrix(1, N, "int3", 99, "bf16", "cuda")[0]
    R = synthetic.matrix(M, N, "int3", 100, "bf16", "cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    h.run(A, B, C, algo="plain", bias=b, residual=R, act="relu")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h.run(A, B, C, algo="plain", bias=b, residual=R, act="relu")
    for seed in (101, 102):
        A2, B2 = synthetic.operands(M, N, K, "int3", seed, "bf16", "cuda")
        A.copy_(A2)
        B.copy_(B2)
        C.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert h.sync_status() == 0
        D64, _ = oracle_epilogue(A, B, "bf16", b, R, "relu")
        assert_bit_exact(C, D64, "bf16")
    h.close()
