"""Parity of the Strassen (LCMA) paths against the CPU oracle (GPU, through the C ABI)."""
import numpy as np
import pytest
import torch

import complexity_matmul_gb300 as lcg
import oracle
import synthetic
from helpers import assert_bit_exact, assert_close, errors, oracle_c64, oracle_epilogue, padded

pytestmark = pytest.mark.gpu

STRASSEN = ["strassen1", "strassen1_unfused", "strassen2"]


@pytest.fixture(scope="module", params=[1, 2], ids=["single_cta", "cta_pair"])
def h(request):
    """Every Strassen test runs with both fused one-level kernels (single-CTA and CTA-pair Groups)."""
    handle = lcg.Handle(0)
    handle.set_option(lcg.OPT_LCMA_KERNEL, request.param)
    yield handle
    handle.close()


def _run(h, A, B, algo):
    C = h.run(A, B, algo=algo)
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert h.last_algo() == lcg.ALGOS[algo]
    return C


# ---------------------------------------------------------------- 256^3 FP16 (small square workload)

@pytest.mark.parametrize("algo", STRASSEN)
@pytest.mark.parametrize("dist", ["int3", "binary"])
def test_small_square_integer_bit_exact(h, algo, dist):
    # {-3..3}, K = 256: operand sums <= 12 in magnitude, C-block sums < 2^24 -> exact everywhere
    A, B = synthetic.operands(256, 256, 256, dist, 1, "f16", "cuda")
    assert_bit_exact(_run(h, A, B, algo), oracle_c64(A, B, "f16"), "f16")


@pytest.mark.parametrize("algo", STRASSEN)
def test_small_square_uniform(h, algo):
    A, B = synthetic.operands(256, 256, 256, "uniform", 1, "f16", "cuda")
    assert_close(_run(h, A, B, algo), oracle_c64(A, B, "f16"), "f16", algo)


@pytest.mark.parametrize("algo", STRASSEN)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_bit_exact_k1024(h, algo, dtype):
    A, B = synthetic.operands(512, 768, 1024, "int3", 3, dtype, "cuda")
    assert_bit_exact(_run(h, A, B, algo), oracle_c64(A, B, dtype), dtype)


# ---------------------------------------------------------------- ragged block sizes

RAGGED = [(260, 388, 160), (4, 4, 32), (132, 68, 64), (300, 516, 96), (1000, 24, 544), (68, 1028, 32)]
RAGGED_S1 = [(258, 390, 160), (2, 6, 16), (130, 66, 48)]   # even, but not multiples of 4


@pytest.mark.parametrize("M,N,K", RAGGED_S1)
@pytest.mark.parametrize("algo", ["strassen1", "strassen1_unfused"])
def test_ragged_one_level_only(h, M, N, K, algo):
    A, B = synthetic.operands(M, N, K, "int3", 4, "f16", "cuda")
    assert_bit_exact(_run(h, A, B, algo), oracle_c64(A, B, "f16"), "f16")


@pytest.mark.parametrize("M,N,K", RAGGED)
@pytest.mark.parametrize("algo", STRASSEN)
def test_ragged_integer_bit_exact(h, M, N, K, algo):
    A, B = synthetic.operands(M, N, K, "int3", 4, "bf16", "cuda")
    assert_bit_exact(_run(h, A, B, algo), oracle_c64(A, B, "bf16"), "bf16")


def test_strided_operands(h):
    M, N, K = 256, 192, 320
    Abig = synthetic.matrix(M, 400, "int3", 5, "bf16", "cuda")
    Bbig = synthetic.matrix(N, 336, "int3", 6, "bf16", "cuda")
    Cbig = torch.full((M, 264), 7.0, dtype=torch.bfloat16, device="cuda")
    A, B, C = Abig[:, 16:16 + K], Bbig[:, :K], Cbig[:, 8:8 + N]
    for algo in STRASSEN:
        h.run(A, B, C, algo=algo)
        torch.cuda.synchronize()
        assert_bit_exact(C, oracle_c64(A.contiguous(), B.contiguous(), "bf16"), "bf16")
        assert (Cbig[:, :8] == 7).all() and (Cbig[:, 8 + N:] == 7).all()


# ---------------------------------------------------------------- square sweep and large rectangles (BF16 N(0,1))

@pytest.mark.parametrize("algo", STRASSEN)
def test_square_2048_full(h, algo):
    A, B = synthetic.operands(2048, 2048, 2048, "normal", 2, "bf16", "cuda")
    assert_close(_run(h, A, B, algo), oracle_c64(A, B, "bf16"), "bf16", algo)


@pytest.mark.parametrize("n", [4096, 8192, 16384])
@pytest.mark.parametrize("algo", ["strassen1", "strassen2"])
def test_square_sampled_rows(h, n, algo):
    A, B = synthetic.operands(n, n, n, "normal", 2, "bf16", "cuda")
    C = _run(h, A, B, algo)
    rows = synthetic.row_sample(n, 64)
    assert_close(C, oracle_c64(A, B, "bf16", rows=rows), "bf16", algo, rows=rows)


@pytest.mark.parametrize("M,N,K", [(16384, 16384, 8192), (8192, 28672, 8192), (32768, 8192, 4096)])
def test_large_rectangular_error_growth(h, M, N, K):
    """Error against FP64 on a seeded 256-row sample grows with the Strassen level but stays in tolerance."""
    A, B = synthetic.operands(M, N, K, "normal", 5, "bf16", "cuda")
    rows = synthetic.row_sample(M, 256, seed=5)
    ref = oracle_c64(A, B, "bf16", rows=rows)
    err = {}
    for algo in ["plain", "strassen1", "strassen2"]:
        C = _run(h, A, B, algo)
        err[algo] = assert_close(C, ref, "bf16", algo, rows=rows)[0]
        del C
    assert err["plain"] <= err["strassen1"] * 1.05 + 1e-4
    print("normwise error per level:", {k: f"{v:.3e}" for k, v in err.items()})


# ---------------------------------------------------------------- against the dtype-emulating Strassen oracle

@pytest.mark.parametrize("levels,algo", [(1, "strassen1"), (2, "strassen2"), (1, "strassen1_unfused")])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_matches_emulating_oracle(h, levels, algo, dtype):
    """The GPU forms the summed operands exactly like the oracle's emulating Strassen
    (FP32 sums in ascending block order, one rounding to the input type); after the one
    final rounding the two agree element-wise except for rare one-ulp flips caused by
    FP32 (GPU) versus FP64 (oracle) accumulation of the products."""
    dt = oracle.F16 if dtype == "f16" else oracle.BF16
    M, N, K = 512, 512, 1024
    A, B = synthetic.operands(M, N, K, "normal", 6, dtype, "cuda")
    Ab, Bb = synthetic.bits(A), synthetic.bits(B)
    C64 = oracle.gemm(Ab, Bb, dt)
    emu = oracle.strassen.strassen(oracle.decode(Ab, dt), oracle.decode(Bb, dt).T, levels, "emulate", dt)
    emu_r = oracle.rounding.rne_values(emu, dt)
    got = _run(h, A, B, algo).cpu().double().numpy()
    to_exact = np.linalg.norm(got - C64) / np.linalg.norm(C64)
    to_emul = np.linalg.norm(got - emu_r) / np.linalg.norm(C64)
    assert (got == emu_r).mean() > 0.95
    assert to_emul < 0.25 * to_exact


# ---------------------------------------------------------------- identities, fusion and edge cases

@pytest.mark.parametrize("algo", STRASSEN)
def test_identity_on_integer_inputs(h, algo):
    n = 256
    A = synthetic.matrix(n, n, "int3", 7, "bf16", "cuda")
    eye = torch.eye(n, dtype=torch.bfloat16, device="cuda")
    assert torch.equal(_run(h, A, eye, algo), A)


def test_fused_at_least_as_accurate_as_unfused(h):
    A, B = synthetic.operands(1024, 1024, 2048, "normal", 8, "bf16", "cuda")
    C64 = oracle_c64(A, B, "bf16")
    e_f = errors(_run(h, A, B, "strassen1"), C64)[0]
    e_u = errors(_run(h, A, B, "strassen1_unfused"), C64)[0]
    assert e_f <= e_u * 1.02


# ---------------------------------------------------------------- non-divisible shapes (zero-padded operands)

PADDED = [(130, 66, 72), (131, 67, 40), (1, 1, 1), (257, 129, 1000), (7, 300, 33), (513, 390, 520),
          (1001, 24, 17), (300, 1001, 4097)]


@pytest.mark.parametrize("M,N,K", PADDED)
@pytest.mark.parametrize("algo", STRASSEN)
def test_padded_integer_bit_exact(h, M, N, K, algo):
    """Dimensions the block split cannot divide run on zero-padded copies of A and B: on integer inputs
    every FP32 step stays exact and C (only its M x N elements) matches the oracle bit for bit."""
    A, B = synthetic.operands(M, N, K, "int3", 9, "bf16", "cuda")
    Ap, Bp = padded(M, K, "bf16", A), padded(N, K, "bf16", B)   # 16-byte row starts for any K
    C = _run(h, Ap, Bp, algo)
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")


@pytest.mark.parametrize("algo", ["strassen1", "strassen2"])
def test_padded_float_and_untouched_padding(h, algo):
    """N(0,1) inputs on an odd shape stay within the Strassen tolerances, and no element of C's row
    padding (columns N .. ldc) is written."""
    M, N, K = 1023, 777, 1001
    A, B = synthetic.operands(M, N, K, "normal", 10, "bf16", "cuda")
    Ap, Bp = padded(M, K, "bf16", A), padded(N, K, "bf16", B)
    Cfull = torch.full((M, 784), 7.0, dtype=torch.bfloat16, device="cuda")
    C = h.run(Ap, Bp, Cfull[:, :N], algo=algo)
    torch.cuda.synchronize()
    assert h.sync_status() == 0 and h.last_algo() == lcg.ALGOS[algo]
    assert_close(C, oracle_c64(A, B, "bf16"), "bf16", algo)
    assert bool((Cfull[:, N:] == 7.0).all())


def test_padded_epilogue(h):
    M, N, K = 131, 67, 200
    A, B = synthetic.operands(M, N, K, "int3", 11, "bf16", "cuda")
    Ap, Bp = padded(M, K, "bf16", A), padded(N, K, "bf16", B)
    b = synthetic.matrix(1, N, "int3", 12, "bf16", "cuda")[0]
    R = padded(M, N, "bf16", synthetic.matrix(M, N, "int3", 13, "bf16", "cuda"))
    D64, _ = oracle_epilogue(A, B, "bf16", b, R, "relu")
    for algo in STRASSEN:
        C = h.run(Ap, Bp, algo=algo, bias=b, residual=R, act="relu")
        torch.cuda.synchronize()
        assert h.sync_status() == 0 and h.last_algo() == lcg.ALGOS[algo]
        assert_bit_exact(C, D64, "bf16")


def test_auto_on_non_divisible_shape(h):
    A = synthetic.matrix(130, 72, "int3", 9, "bf16", "cuda")
    B = synthetic.matrix(66, 72, "int3", 10, "bf16", "cuda")
    C = torch.empty((130, 72), dtype=torch.bfloat16, device="cuda")[:, :66]
    h.run(A, B, C, algo="auto")
    torch.cuda.synchronize()
    assert h.last_algo() == lcg.PLAIN            # small shape: the cost model keeps plain
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")


def test_repeated_and_interleaved_launches(h):
    """Workspace reuse and growth across shapes and algorithms, many launches in a row."""
    shapes = [(512, 512, 512), (1024, 768, 256), (256, 256, 2048)]
    data = [synthetic.operands(M, N, K, "int3", 11 + i, "f16", "cuda") for i, (M, N, K) in enumerate(shapes)]
    refs = [oracle_c64(A, B, "f16") for A, B in data]
    outs = []
    for _ in range(4):
        for i, (A, B) in enumerate(data):
            for algo in STRASSEN:
                outs.append((i, h.run(A, B, algo=algo)))
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    for i, C in outs[-len(shapes) * len(STRASSEN):]:
        assert_bit_exact(C, refs[i], "f16")


# ---------------------------------------------------------------- Stream-K split of tail Groups (CTA-pair kernel)

@pytest.fixture(scope="module")
def hp():
    handle = lcg.Handle(0)
    handle.set_option(lcg.OPT_LCMA_KERNEL, 2)
    yield handle
    handle.close()


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 1024), (1536, 2560, 512), (8704, 8704, 256), (512, 768, 1024)])
def test_split_on_off_integer_bit_exact(hp, M, N, K):
    """Split tail Groups (two halves on two CTA pairs, fixed up through L2) give the exact result."""
    A, B = synthetic.operands(M, N, K, "int3", 12, "bf16", "cuda")
    rows = None if M * N <= 4096 * 4096 else synthetic.row_sample(M, 128)
    ref = oracle_c64(A, B, "bf16", rows=rows)
    for split in (1, 0):
        hp.set_option(lcg.OPT_SPLIT, split)
        C = _run(hp, A, B, "strassen1")
        assert_bit_exact(C, ref, "bf16", rows=rows)
    hp.set_option(lcg.OPT_SPLIT, 1)


def test_split_float_tolerance(hp):
    A, B = synthetic.operands(2048, 2048, 2048, "normal", 13, "bf16", "cuda")
    ref = oracle_c64(A, B, "bf16")
    hp.set_option(lcg.OPT_SPLIT, 1)
    assert_close(_run(hp, A, B, "strassen1"), ref, "bf16", "strassen1")


def test_partner_signal_timeout_is_reported_and_recovered():
    """Failure detection without a GPU fault: the second halves of split Groups never publish,
    so the first halves' bounded waits run out; the kernel ends, the next status call reports
    LCGEMM_ERR_TIMEOUT, and the handle keeps working."""
    h2 = lcg.Handle(0)
    h2.set_option(lcg.OPT_LCMA_KERNEL, 2)
    h2.set_option(lcg.OPT_WAIT_TIMEOUT_US, 50000)
    A, B = synthetic.operands(2048, 2048, 1024, "int3", 14, "bf16", "cuda")
    h2.set_option(lcg.OPT_DEBUG_DROP_SIGNAL, 1)
    h2.run(A, B, algo="strassen1")
    torch.cuda.synchronize()
    assert h2.sync_status() == lcg.ERR_TIMEOUT
    assert h2.sync_status() == lcg.OK          # reported once, then cleared
    h2.set_option(lcg.OPT_DEBUG_DROP_SIGNAL, 0)
    C = h2.run(A, B, algo="strassen1")
    torch.cuda.synchronize()
    assert h2.sync_status() == lcg.OK
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")
    h2.close()


@pytest.mark.parametrize("algo", ["strassen1", "strassen1_unfused", "strassen2"])
def test_programmatic_dependent_launch_on_off(h, algo):
    """The product kernel launched as a programmatic dependent of the pre-pass (default) reads the
    pre-pass's sums only after the pre-pass completes: same bits as plain stream order."""
    A, B = synthetic.operands(1024, 768, 512, "normal", 14, "bf16", "cuda")
    out = {}
    for pdl in (1, 0):
        h.set_option(lcg.OPT_PDL, pdl)
        out[pdl] = _run(h, A, B, algo).cpu()
    h.set_option(lcg.OPT_PDL, 1)
    assert torch.equal(out[0], out[1])
    assert_close(out[1].cuda(), oracle_c64(A, B, "bf16"), "bf16", algo)


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 1024), (4096, 4096, 512), (8704, 8704, 256)])
def test_group_order_on_off(hp, M, N, K):
    """Group ordering off puts the odd CTA pairs on another product order (every wave then mixes two
    product types): the integer result is still exact, and N(0,1) results are the same bits as with
    ordering on (both orders form every quadrant sum in the same FP32 order)."""
    A, B = synthetic.operands(M, N, K, "int3", 15, "bf16", "cuda")
    rows = None if M * N <= 4096 * 4096 else synthetic.row_sample(M, 128)
    ref = oracle_c64(A, B, "bf16", rows=rows)
    An, Bn = synthetic.operands(M, N, K, "normal", 16, "bf16", "cuda")
    out = {}
    for order in (0, 1):
        hp.set_option(lcg.OPT_GROUP_ORDER, order)
        assert_bit_exact(_run(hp, A, B, "strassen1"), ref, "bf16", rows=rows)
        out[order] = _run(hp, An, Bn, "strassen1").cpu()
    hp.set_option(lcg.OPT_GROUP_ORDER, 1)
    assert torch.equal(out[0], out[1])


@pytest.mark.parametrize("split", [1, 0])
@pytest.mark.parametrize("order", [1, 0])
def test_two_level_hierarchical_options(hp, split, order):
    """Two levels on the CTA-pair kernel run as seven launches (one per outer product) whose inner
    quadrants go to FP32 outer slots: exact on integer inputs with the tail split and the Group
    ordering on or off (each launch's 4 Groups form a tail that is split), and for a ragged shape
    whose inner blocks are not multiples of the 256 x 256 Group tile."""
    hp.set_option(lcg.OPT_SPLIT, split)
    hp.set_option(lcg.OPT_GROUP_ORDER, order)
    for (M, N, K) in ((2048, 2048, 1024), (1160, 1096, 544)):
        A, B = synthetic.operands(M, N, K, "int3", 17, "bf16", "cuda")
        assert_bit_exact(_run(hp, A, B, "strassen2"), oracle_c64(A, B, "bf16"), "bf16")
    hp.set_option(lcg.OPT_SPLIT, 1)
    hp.set_option(lcg.OPT_GROUP_ORDER, 1)


def test_two_level_partner_timeout_is_reported_and_recovered():
    """The split-Group fix-up inside the seven two-level launches: second halves that never publish
    make the first halves' bounded waits run out; the status reports LCGEMM_ERR_TIMEOUT once and the
    next run is exact."""
    h2 = lcg.Handle(0)
    h2.set_option(lcg.OPT_LCMA_KERNEL, 2)
    h2.set_option(lcg.OPT_WAIT_TIMEOUT_US, 50000)
    A, B = synthetic.operands(2048, 2048, 1024, "int3", 18, "bf16", "cuda")
    h2.set_option(lcg.OPT_DEBUG_DROP_SIGNAL, 1)
    h2.run(A, B, algo="strassen2")
    torch.cuda.synchronize()
    assert h2.sync_status() == lcg.ERR_TIMEOUT
    assert h2.sync_status() == lcg.OK
    h2.set_option(lcg.OPT_DEBUG_DROP_SIGNAL, 0)
    C = h2.run(A, B, algo="strassen2")
    torch.cuda.synchronize()
    assert h2.sync_status() == lcg.OK
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")
    h2.close()
