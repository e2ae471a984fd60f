"""Parity of the weight-streaming kernels against the CPU oracle: the stream-K tensor-core skinny kernel
(M <= 256) and the CUDA-core GEMV (M <= 4)."""
import numpy as np
import pytest
import torch

import complexity_matmul_gb300 as lcg
import synthetic
from helpers import MAXERR_SIGMA, assert_bit_exact, assert_close, assert_epilogue_close, oracle_c64, oracle_epilogue, \
    padded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    handle = lcg.Handle(0)
    handle.set_option(lcg.OPT_PLAIN_KERNEL, 3)
    yield handle
    handle.close()


def _run(h, A, B, **ep):
    C = h.run(A, B, algo="plain", **ep)
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    return C


# every padded width of A (16 .. 256), ragged M, N (partial 128-row blocks of B) and K (partial slabs)
SHAPES = [(1, 8, 8), (1, 128, 4096), (2, 200, 72), (15, 129, 1000), (16, 1024, 64), (17, 257, 520),
          (31, 384, 136), (33, 640, 4096), (64, 128, 8), (100, 1000, 264), (128, 256, 1024), (129, 130, 200),
          (200, 512, 2048), (256, 384, 96)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_bit_exact(h, M, N, K, dtype):
    A, B = synthetic.operands(M, N, K, "int3", 71, dtype, "cuda")
    assert_bit_exact(_run(h, A, B), oracle_c64(A, B, dtype), dtype)


@pytest.mark.parametrize("M,N,K", [(1, 14336, 4096), (16, 14336, 4096), (128, 4096, 14336), (256, 4096, 4096),
                                   (1, 4096, 14336)])
def test_llm_shapes_normal(h, M, N, K):
    """The skinny LLM workload (activations N(0,1), weights N(0, 0.02^2)) against the oracle."""
    A = synthetic.matrix(M, K, "normal", 1004, "bf16", "cuda")
    B = synthetic.matrix(N, K, "normal", 2004, "bf16", "cuda", scale=0.02)
    assert_close(_run(h, A, B), oracle_c64(A, B, "bf16"), "bf16", "plain")


@pytest.mark.parametrize("M,N,K", [(1, 128, 8192), (3, 256, 65536), (16, 128, 1 << 17)])
def test_many_ctas_per_block(h, M, N, K):
    """Few blocks and long K: every block's slabs spread over many CTAs, summed by the last to arrive."""
    A, B = synthetic.operands(M, N, K, "int3", 72, "bf16", "cuda", scale_a=1.0)
    A = (A.float() / 4).to(A.dtype)      # |C| <= 9K/4 < 2^24: the FP32 sums stay exact
    assert_bit_exact(_run(h, A, B), oracle_c64(A, B, "bf16"), "bf16")


def test_repeated_launches_reuse_counters(h):
    """The per-block arrival counters are never reset: later launches (new epochs) must count afresh."""
    A, B = synthetic.operands(16, 1024, 4096, "int3", 73, "bf16", "cuda")
    ref = oracle_c64(A, B, "bf16")
    for _ in range(5):
        assert_bit_exact(_run(h, A, B), ref, "bf16")
    A2, B2 = synthetic.operands(7, 2048, 2048, "int3", 74, "bf16", "cuda")
    assert_bit_exact(_run(h, A2, B2), oracle_c64(A2, B2, "bf16"), "bf16")
    assert_bit_exact(_run(h, A, B), ref, "bf16")


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "gelu_tanh"])
@pytest.mark.parametrize("M,N,K", [(16, 1024, 4096), (5, 300, 512), (128, 512, 1024)])
def test_epilogue(h, act, M, N, K):
    A, B = synthetic.operands(M, N, K, "int3", 75, "bf16", "cuda")
    A = (A.float() / 8).to(A.dtype)
    B = (B.float() / 8).to(B.dtype)
    b = (synthetic.matrix(1, N, "int3", 76, "bf16", "cuda")[0].float() / 8).to(torch.bfloat16)
    R = padded(M, N, "bf16", (synthetic.matrix(M, N, "int3", 77, "bf16", "cuda").float() / 8).to(torch.bfloat16))
    C = _run(h, A, B, bias=b, residual=R, act=act)
    D64, pre = oracle_epilogue(A, B, "bf16", b, R, act)
    if act in ("none", "relu"):
        assert_bit_exact(C, D64, "bf16")
    else:
        assert_epilogue_close(C, D64, pre, "bf16", act)


def test_in_place_residual(h):
    M, N, K = 16, 512, 4096
    A, B = synthetic.operands(M, N, K, "int3", 78, "bf16", "cuda")
    R = padded(M, N, "bf16", synthetic.matrix(M, N, "int3", 79, "bf16", "cuda"))
    D64, _ = oracle_epilogue(A, B, "bf16", None, R, "relu")
    C = R.clone()
    _run(h, A, B, C=C, residual=C, act="relu")
    assert_bit_exact(C, D64, "bf16")


def test_default_choice_and_fallback():
    """Without an option 64 x 512 x 1024 runs the default (tiled) kernel; the skinny option on M > 256
    falls back to the tiled kernels."""
    hd = lcg.Handle(0)
    try:
        A, B = synthetic.operands(64, 512, 1024, "int3", 80, "bf16", "cuda")
        assert_bit_exact(_run(hd, A, B), oracle_c64(A, B, "bf16"), "bf16")
        hd.set_option(lcg.OPT_PLAIN_KERNEL, 3)
        A, B = synthetic.operands(300, 256, 512, "int3", 81, "bf16", "cuda")
        assert_bit_exact(_run(hd, A, B), oracle_c64(A, B, "bf16"), "bf16")
    finally:
        hd.close()


def test_strided_operands(h):
    M, N, K = 9, 384, 1024
    Abig = synthetic.matrix(M, K + 64, "int3", 82, "bf16", "cuda")
    Bbig = synthetic.matrix(N, K + 128, "int3", 83, "bf16", "cuda")
    A, B = Abig[:, :K], Bbig[:, :K]
    C = _run(h, A, B)
    assert_bit_exact(C, oracle_c64(A.contiguous(), B.contiguous(), "bf16"), "bf16")


# ---------------------------------------------------------------- CUDA-core GEMV (M <= 4)

@pytest.fixture(scope="module")
def hg():
    handle = lcg.Handle(0)
    handle.set_option(lcg.OPT_PLAIN_KERNEL, 4)
    yield handle
    handle.close()


GEMV_SHAPES = [(1, 1, 1), (1, 7, 8), (2, 9, 24), (3, 1001, 1000), (4, 128, 4096), (1, 4096, 14336),
               (4, 14336, 4096), (2, 300, 4097), (1, 8, 3)]


@pytest.mark.parametrize("M,N,K", GEMV_SHAPES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemv_integer_bit_exact(hg, M, N, K, dtype):
    A, B = synthetic.operands(M, N, K, "int3", 84, dtype, "cuda")
    # rows padded to 16-byte starts (K need not be a multiple of 8)
    Ap, Bp = padded(M, K, dtype, A), padded(N, K, dtype, B)
    assert_bit_exact(_run(hg, Ap, Bp), oracle_c64(A, B, dtype), dtype)


@pytest.mark.parametrize("M,N,K", [(1, 14336, 4096), (4, 4096, 14336)])
def test_gemv_normal(hg, M, N, K):
    A = synthetic.matrix(M, K, "normal", 1004, "bf16", "cuda")
    B = synthetic.matrix(N, K, "normal", 2004, "bf16", "cuda", scale=0.02)
    assert_close(_run(hg, A, B), oracle_c64(A, B, "bf16"), "bf16", "plain")


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "gelu_tanh"])
def test_gemv_epilogue(hg, act):
    M, N, K = 3, 1000, 2048
    A, B = synthetic.operands(M, N, K, "int3", 85, "bf16", "cuda")
    A = (A.float() / 8).to(A.dtype)
    B = (B.float() / 8).to(B.dtype)
    b = (synthetic.matrix(1, N, "int3", 86, "bf16", "cuda")[0].float() / 8).to(torch.bfloat16)
    R = padded(M, N, "bf16", (synthetic.matrix(M, N, "int3", 87, "bf16", "cuda").float() / 8).to(torch.bfloat16))
    C = _run(hg, A, B, bias=b, residual=R, act=act)
    D64, pre = oracle_epilogue(A, B, "bf16", b, R, act)
    if act in ("none", "relu"):
        assert_bit_exact(C, D64, "bf16")
    else:
        assert_epilogue_close(C, D64, pre, "bf16", act)


def test_gemv_strided(hg):
    M, N, K = 4, 640, 1000
    Abig = synthetic.matrix(M, K + 24, "int3", 88, "bf16", "cuda")
    Bbig = synthetic.matrix(N, K + 40, "int3", 89, "bf16", "cuda")
    A, B = Abig[:, :K], Bbig[:, :K]
    assert_bit_exact(_run(hg, A, B), oracle_c64(A.contiguous(), B.contiguous(), "bf16"), "bf16")
