"""Parity of the fused epilogue C = act(A.B + bias) + residual against the CPU oracle
(GPU, through lcgemm_run_epilogue), for every algorithm and kernel variant."""
import ctypes

import numpy as np
import pytest
import torch

import complexity_matmul_gb300 as lcg
import oracle
import synthetic
from helpers import (MAXERR_SIGMA, assert_bit_exact, assert_epilogue_close, oracle_c64, oracle_epilogue,
                     padded)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[1, 2, 3, 4, 5], ids=["single_cta", "cta_pair", "skinny", "gemv", "cta_pair_512"])
def h(request):
    """Plain tests run on each plain kernel (3: the skinny kernel where M <= 256, 4: the GEMV where
    M <= 4), Strassen tests on both fused one-level kernels."""
    handle = lcg.Handle(0)
    handle.set_option(lcg.OPT_PLAIN_KERNEL, request.param)
    handle.set_option(lcg.OPT_LCMA_KERNEL, min(request.param, 2))
    yield handle
    handle.close()


def _vec(N, dist, seed, dtype, div=1):
    v = synthetic.matrix(1, N, dist, seed, dtype, "cuda")[0]
    return v if div == 1 else (v.float() / div).to(v.dtype)


def _mat(M, N, dist, seed, dtype, div=1):
    m = synthetic.matrix(M, N, dist, seed, dtype, "cuda")
    return padded(M, N, dtype, m if div == 1 else (m.float() / div).to(m.dtype))


def _int_operands(M, N, K, dtype, seed, div=1):
    """int3 operands, optionally divided by a power of two (exact): FP32 accumulation stays exact."""
    A, B = synthetic.operands(M, N, K, "int3", seed, dtype, "cuda")
    if div != 1:
        A = (A.float() / div).to(A.dtype)
        B = (B.float() / div).to(B.dtype)
    return A, B


def _run(h, A, B, algo="plain", **ep):
    C = h.run(A, B, algo=algo, **ep)
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert h.last_algo() == lcg.ALGOS[algo]
    return C


def _exact(h, M, N, K, dtype, act, algo="plain", bias=True, residual=True, seed=31, rows=None):
    A, B = _int_operands(M, N, K, dtype, seed)
    b = _vec(N, "int3", seed + 1, dtype) if bias else None
    R = _mat(M, N, "int3", seed + 2, dtype) if residual else None
    C = _run(h, A, B, algo, bias=b, residual=R, act=act)
    D64, _ = oracle_epilogue(A, B, dtype, b, R, act, rows=rows)
    assert_bit_exact(C, D64, dtype, rows=rows)


# ---------------------------------------------------------------- plain GEMM, bit-exact on integer inputs

SHAPES = [(256, 256, 256), (7, 9, 24), (129, 257, 72), (300, 130, 1000), (513, 384, 520), (1000, 24, 8),
          (64, 1024, 16)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", ["none", "relu"])
def test_plain_integer_bit_exact(h, M, N, K, dtype, act):
    # integer A, B, bias and residual: every FP32 step is exact, so D has one rounding on both sides
    _exact(h, M, N, K, dtype, act)


@pytest.mark.parametrize("bias,residual,act", [(True, False, "none"), (False, True, "none"),
                                               (False, False, "relu"), (True, False, "relu")])
def test_plain_each_part_alone(h, bias, residual, act):
    _exact(h, 300, 264, 136, "bf16", act, bias=bias, residual=residual)


# ---------------------------------------------------------------- GELU, exact product

@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (129, 257, 512), (7, 40, 256)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", ["gelu", "gelu_tanh"])
def test_plain_gelu_exact_product(h, M, N, K, dtype, act):
    """int3/8 operands: the product is exact in FP32 (multiples of 1/64) with sigma ~ sqrt(K)/16, so
    the pre-activation values fill GELU's curved region; only the activation and the cast differ."""
    A, B = _int_operands(M, N, K, dtype, 41, div=8)
    b = _vec(N, "int3", 42, dtype, div=8)
    R = _mat(M, N, "int3", 43, dtype, div=8)
    C = _run(h, A, B, bias=b, residual=R, act=act)
    D64, pre = oracle_epilogue(A, B, dtype, b, R, act)
    assert (np.abs(pre) < 2).mean() > 0.4
    assert_epilogue_close(C, D64, pre, dtype, act)
    if act == "gelu":
        # relative error ~1e-6 where |x| < 3: nearly every element is the correctly rounded value itself
        dt = 0 if dtype == "f16" else 1
        ref = oracle.decode(oracle.reference_output(D64, dt), dt)
        assert (C.cpu().double().numpy() == ref).mean() > 0.95


# ---------------------------------------------------------------- N(0,1) workload, scaled product

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", ["relu", "gelu", "gelu_tanh"])
def test_plain_normal_inputs(h, dtype, act):
    M, N, K = 1024, 1024, 1024
    A, B = synthetic.operands(M, N, K, "normal", 44, dtype, "cuda", scale_a=K ** -0.5)
    b = _vec(N, "normal", 45, dtype)
    R = _mat(M, N, "normal", 46, dtype)
    C = _run(h, A, B, bias=b, residual=R, act=act)
    D64, pre, C64 = oracle_epilogue(A, B, dtype, b, R, act, with_product=True)
    sigma = np.sqrt(np.mean(C64 ** 2))
    assert_epilogue_close(C, D64, pre, dtype, act, gemm_err=MAXERR_SIGMA * sigma)


def test_plain_full_size_sampled_rows(h):
    """The 8192^3 BF16 workload with bias + tanh GELU + residual, 64 sampled rows against the oracle."""
    M = N = K = 8192
    A, B = synthetic.operands(M, N, K, "normal", 47, "bf16", "cuda", scale_a=K ** -0.5)
    b = _vec(N, "normal", 48, "bf16")
    R = _mat(M, N, "normal", 49, "bf16")
    C = _run(h, A, B, bias=b, residual=R, act="gelu_tanh")
    rows = synthetic.row_sample(M, 64)
    D64, pre, C64 = oracle_epilogue(A, B, "bf16", b, R, "gelu_tanh", rows=rows, with_product=True)
    sigma = np.sqrt(np.mean(C64 ** 2))
    assert_epilogue_close(C, D64, pre, "bf16", "gelu_tanh", gemm_err=MAXERR_SIGMA * sigma, rows=rows)


# ---------------------------------------------------------------- split paths apply it once, after the sum

# single-CTA chunks: 4, 4, 8 (separate sum), 2 and 3 (last arriver), 4 with N < 64
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 4096), (128, 512, 8192), (16, 14336, 3072),
                                   (40, 300, 3072), (50, 40, 4160)])
def test_split_k_skinny(h, M, N, K):
    _exact(h, M, N, K, "bf16", "relu")


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 8192), (4352, 2560, 8200)])
def test_tail_split(h, M, N, K):
    _exact(h, M, N, K, "bf16", "relu", rows=synthetic.row_sample(M, 256))


# ---------------------------------------------------------------- Strassen paths

@pytest.mark.parametrize("algo", ["strassen1", "strassen1_unfused", "strassen2"])
@pytest.mark.parametrize("M,N,K", [(512, 768, 1024), (260, 392, 96), (2048, 2048, 1024)])
@pytest.mark.parametrize("act", ["none", "relu"])
def test_strassen_integer_bit_exact(h, algo, M, N, K, act):
    if algo == "strassen2" and (M % 4 or N % 4 or K % 32):
        pytest.skip("two levels need M, N multiples of 4 and K of 32")
    _exact(h, M, N, K, "bf16", act, algo=algo)


@pytest.mark.parametrize("algo", ["strassen1", "strassen1_unfused", "strassen2"])
@pytest.mark.parametrize("act", ["gelu", "gelu_tanh"])
def test_strassen_gelu_exact_product(h, algo, act):
    M, N, K = 1024, 512, 256
    A, B = _int_operands(M, N, K, "f16", 51, div=8)
    b = _vec(N, "int3", 52, "f16", div=8)
    R = _mat(M, N, "int3", 53, "f16", div=8)
    C = _run(h, A, B, algo, bias=b, residual=R, act=act)
    D64, pre = oracle_epilogue(A, B, "f16", b, R, act)
    assert_epilogue_close(C, D64, pre, "f16", act)


def test_strassen_split_tail_groups():
    """CTA-pair fused kernel with split tail Groups: the epilogue runs on whichever half finishes the value."""
    hp = lcg.Handle(0)
    hp.set_option(lcg.OPT_LCMA_KERNEL, 2)
    try:
        for split in (1, 0):
            hp.set_option(lcg.OPT_SPLIT, split)
            _exact(hp, 1536, 2560, 512, "bf16", "relu", algo="strassen1")
    finally:
        hp.close()


# ---------------------------------------------------------------- edge cases

def test_in_place_residual(h):
    M, N, K = 300, 264, 136
    A, B = _int_operands(M, N, K, "bf16", 61)
    b = _vec(N, "int3", 62, "bf16")
    R = _mat(M, N, "int3", 63, "bf16")
    D64, _ = oracle_epilogue(A, B, "bf16", b, R, "relu")
    C = R.clone() if R.is_contiguous() else padded(M, N, "bf16", R)
    out = _run(h, A, B, C=C, bias=b, residual=C, act="relu")
    assert out.data_ptr() == C.data_ptr()
    assert_bit_exact(C, D64, "bf16")


@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_empty_product(h, act):
    """K = 0: C = act(bias) + residual."""
    M, N = 37, 50
    A = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, 0), dtype=torch.bfloat16, device="cuda")
    b = _vec(N, "int3", 64, "bf16", div=4)
    R = _mat(M, N, "int3", 65, "bf16", div=4)
    C = _run(h, A, B, bias=b, residual=R, act=act)
    D64 = oracle.epilogue.apply(np.zeros((M, N)), oracle.decode(synthetic.bits(b), 1),
                                oracle.decode(synthetic.bits(R), 1), act)
    if act == "gelu":
        assert_epilogue_close(C, D64, np.zeros((M, N)) + oracle.decode(synthetic.bits(b), 1), "bf16", act)
    else:
        assert_bit_exact(C, D64, "bf16")


def test_empty_epilogue_equals_plain_run(h):
    A, B = synthetic.operands(513, 384, 520, "normal", 66, "bf16", "cuda")
    C0 = _run(h, A, B)
    C1 = torch.empty_like(C0)
    rc = h.run_epilogue_raw(513, 384, 520, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C1.data_ptr(),
                            C1.stride(0), lcg.BF16, lcg.PLAIN)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(C0, C1)


def test_argument_errors(h):
    M, N, K = 64, 64, 64
    A, B = synthetic.operands(M, N, K, "int3", 67, "bf16", "cuda")
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(N + 8, dtype=torch.bfloat16, device="cuda")
    R = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    args = (M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), N, lcg.BF16, lcg.PLAIN)
    run = h.run_epilogue_raw
    assert run(*args, act=4) == lcg.ERR_ARG
    assert run(*args, act=-1) == lcg.ERR_ARG
    assert run(*args, bias=bias.data_ptr() + 2) == lcg.ERR_ALIGN
    assert run(*args, residual=R.data_ptr(), ldr=N - 8) == lcg.ERR_ARG
    assert run(*args, residual=R.data_ptr(), ldr=N + 4) == lcg.ERR_ALIGN
    assert run(*args, residual=R.data_ptr() + 2, ldr=N) == lcg.ERR_ALIGN
    assert run(*args, bias=C.data_ptr() + 16 * N) == lcg.ERR_ALIAS                 # bias inside C
    assert run(*args, residual=C.data_ptr() + 16, ldr=N) == lcg.ERR_ALIAS          # shifted by 8 columns
    assert run(*args, residual=C.data_ptr(), ldr=N + 8) == lcg.ERR_ALIAS           # same start, other stride
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert not C.any(), "rejected calls launch nothing"
    # a null epilogue pointer through the raw ABI is a plain run
    L = lcg.lib()
    rc = L.lcgemm_run_epilogue(h.ptr, *args, None, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "gelu_tanh"])
def test_special_values_propagate_like_the_oracle(h, act):
    """Bias entries of +inf, -inf and NaN: every output column takes the oracle's value class (NaN,
    +inf, -inf or the finite value), e.g. ReLU(NaN) = +0 (x > 0 ? x : 0), GELU(-inf) = NaN."""
    M, N, K = 64, 256, 64
    A, B = _int_operands(M, N, K, "bf16", 71)
    b = _vec(N, "int3", 72, "bf16")
    b[0], b[1], b[2] = float("inf"), float("-inf"), float("nan")
    C = _run(h, A, B, bias=b, act=act)
    D64, pre = oracle_epilogue(A, B, "bf16", b, None, act)
    got = C.cpu().double().numpy()
    assert (np.isnan(got) == np.isnan(D64)).all()
    fin = np.isfinite(D64)
    assert (np.isinf(got) == np.isinf(D64)).all() and (np.sign(got[~fin & ~np.isnan(D64)]) ==
                                                       np.sign(D64[~fin & ~np.isnan(D64)])).all()
    assert_epilogue_close(C[:, 3:], D64[:, 3:], pre[:, 3:], "bf16", act)
