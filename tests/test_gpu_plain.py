"""Parity of the plain persistent GEMM against the CPU oracle (GPU, through the C ABI)."""
import ctypes

import numpy as np
import pytest
import torch

import complexity_matmul_gb300 as lcg
import synthetic
from helpers import assert_bit_exact, assert_close, assert_epilogue_close, oracle_c64, oracle_epilogue, padded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[1, 2, 3, 4, 5], ids=["single_cta", "cta_pair", "skinny", "gemv", "cta_pair_512"])
def h(request):
    """Every plain test runs on each kernel: single-CTA 128x256 tiles, CTA-pair 256x256 tiles, the
    stream-K skinny kernel (M <= 256), the CUDA-core GEMV (M <= 4; other M choose) and CTA-pair
    256x512 tiles."""
    handle = lcg.Handle(0)
    handle.set_option(lcg.OPT_PLAIN_KERNEL, request.param)
    yield handle
    handle.close()


def _run(h, A, B, algo="plain"):
    C = h.run(A, B, algo=algo)
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    return C


# ---------------------------------------------------------------- 256^3 FP16 (small square workload)

@pytest.mark.parametrize("dist", ["int3", "binary"])
def test_small_square_integer_bit_exact(h, dist):
    A, B = synthetic.operands(256, 256, 256, dist, 1, "f16", "cuda")
    assert_bit_exact(_run(h, A, B), oracle_c64(A, B, "f16"), "f16")


def test_small_square_uniform(h):
    A, B = synthetic.operands(256, 256, 256, "uniform", 1, "f16", "cuda")
    C = _run(h, A, B)
    C64 = oracle_c64(A, B, "f16")
    assert_close(C, C64, "f16", "plain")
    # FP32 accumulation sits far below one FP16 ulp: nearly every element is the correctly rounded value
    ref = torch.from_numpy(C64).to(torch.float16)
    assert (C.cpu() == ref).float().mean().item() > 0.98


# ---------------------------------------------------------------- ragged shapes (tiles, tails, K tails)

RAGGED = [(1, 128, 4096), (1, 8, 8), (7, 9, 24), (129, 257, 72), (200, 300, 136), (128, 256, 64),
          (300, 130, 1000), (513, 384, 520), (64, 1024, 16), (1000, 24, 8)]


@pytest.mark.parametrize("M,N,K", RAGGED)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_ragged_integer_bit_exact(h, M, N, K, dtype):
    # integer inputs, K <= 4096: |C| <= 9K < 2^24 so FP32 accumulation is exact; one rounding either side
    A, B = synthetic.operands(M, N, K, "int3", 7, dtype, "cuda")
    assert_bit_exact(_run(h, A, B), oracle_c64(A, B, dtype), dtype)


def _padded(rows, cols, dist, seed, dtype):
    """rows x cols view of a buffer whose rows are padded to a multiple of 8 elements."""
    buf = synthetic.matrix(rows, (cols + 7) // 8 * 8, dist, seed, dtype, "cuda")
    return buf[:, :cols]


@pytest.mark.parametrize("M,N,K", [(33, 40, 100), (5, 3, 1), (130, 70, 7), (257, 129, 65)])
def test_k_not_multiple_of_8(h, M, N, K):
    """K that is not a multiple of 8 (rows padded in storage): exercises the K-tail zero fill."""
    A = _padded(M, K, "int3", 17, "bf16")
    B = _padded(N, K, "int3", 18, "bf16")
    assert_bit_exact(_run(h, A, B), oracle_c64(A.contiguous(), B.contiguous(), "bf16"), "bf16")


@pytest.mark.parametrize("M,N,K", [(129, 257, 72), (513, 384, 520), (300, 130, 1000)])
def test_ragged_normal(h, M, N, K):
    A, B = synthetic.operands(M, N, K, "normal", 8, "bf16", "cuda")
    assert_close(_run(h, A, B), oracle_c64(A, B, "bf16"), "bf16", "plain")


def test_strided_operands(h):
    """Leading dimensions larger than the row length (sub-matrix views)."""
    M, N, K = 192, 320, 200
    Abig = synthetic.matrix(M, 264, "int3", 9, "bf16", "cuda")
    Bbig = synthetic.matrix(N, 216, "int3", 10, "bf16", "cuda")
    Cbig = torch.full((M, 400), 7.0, dtype=torch.bfloat16, device="cuda")
    A, B, C = Abig[:, :K], Bbig[:, :K], Cbig[:, 16:16 + N]
    h.run(A, B, C)
    torch.cuda.synchronize()
    assert_bit_exact(C, oracle_c64(A.contiguous(), B.contiguous(), "bf16"), "bf16")
    # nothing outside the C view was written
    assert (Cbig[:, :16] == 7).all() and (Cbig[:, 16 + N:] == 7).all()


@pytest.mark.parametrize("M,N,K", [(300, 777, 200), (520, 1001, 136), (64, 5, 72)])
def test_ragged_n_leaves_neighbours_untouched(h, M, N, K):
    """C as a column view of a wider matrix, N not a multiple of 8: C matches the oracle bit for bit,
    with and without a fused epilogue, and no element outside the view is written (a tensor store
    writes whole 16-byte units of a row, so a row's last partial unit must not go through one)."""
    A, B = synthetic.operands(M, N, K, "int3", 21, "bf16", "cuda")
    ldc = (N + 7) // 8 * 8 + 16
    b = synthetic.matrix(1, N, "int3", 22, "bf16", "cuda")[0]
    R = padded(M, N, "bf16", synthetic.matrix(M, N, "int3", 23, "bf16", "cuda"))   # 16-byte row starts
    D64, _ = oracle_epilogue(A, B, "bf16", b, R, "relu")
    for kw, want in (({}, oracle_c64(A, B, "bf16")), ({"bias": b, "residual": R, "act": "relu"}, D64)):
        Cbig = torch.full((M, ldc), 7.0, dtype=torch.bfloat16, device="cuda")
        C = Cbig[:, 8:8 + N]
        h.run(A, B, C, **kw)
        torch.cuda.synchronize()
        assert h.sync_status() == 0
        assert_bit_exact(C, want, "bf16")
        assert bool((Cbig[:, :8] == 7).all()) and bool((Cbig[:, 8 + N:] == 7).all())


# Weight-streaming shapes whose K chunks the single-CTA kernel sums inside clusters of four
# (M <= 32, N about 4096, deep K), ragged M, N and K included; with the grid capped below the
# 128 CTAs the same shapes take the split-K path with a separate reduction, and at M = 77 the
# deep split-K runs regardless.
CLUSTER_SHAPES = [(16, 4096, 14336, "bf16"), (32, 4096, 14336, "bf16"), (5, 4096, 4096, "f16"),
                  (23, 4000, 8200, "bf16"), (9, 4001, 4104, "bf16"), (77, 4000, 8200, "bf16")]


@pytest.mark.parametrize("M,N,K,dtype", CLUSTER_SHAPES)
@pytest.mark.parametrize("max_ctas", [0, 64], ids=["cluster_sum", "capped_grid"])
def test_k_chunks_summed_in_cluster(M, N, K, dtype, max_ctas):
    hc = lcg.Handle(0)
    try:
        hc.set_option(lcg.OPT_MAX_CTAS, max_ctas)
        A, B = synthetic.operands(M, N, K, "int3", 31, dtype, "cuda")
        C = hc.run(A, B, algo="plain")
        torch.cuda.synchronize()
        assert hc.sync_status() == 0
        assert_bit_exact(C, oracle_c64(A, B, dtype), dtype)
        if M == 16:
            b = synthetic.matrix(1, N, "int3", 32, dtype, "cuda")[0]
            R = synthetic.matrix(M, N, "int3", 33, dtype, "cuda")
            D64, _ = oracle_epilogue(A, B, dtype, b, R, "relu")
            D = hc.run(A, B, algo="plain", bias=b, residual=R, act="relu")
            torch.cuda.synchronize()
            assert hc.sync_status() == 0
            assert_bit_exact(D, D64, dtype)
    finally:
        hc.close()


@pytest.mark.parametrize("M,dtype", [(1, "bf16"), (2, "f16")])
def test_k_chunks_summed_in_cluster_one_or_two_rows(M, dtype):
    """The single-CTA kernel forced for one or two rows (the default takes the GEMV there): an A box
    of 8 rows, K chunks summed in clusters of four, with and without a fused epilogue."""
    hc = lcg.Handle(0)
    try:
        hc.set_option(lcg.OPT_PLAIN_KERNEL, 1)
        N, K = 4096, 4096
        A, B = synthetic.operands(M, N, K, "int3", 35, dtype, "cuda")
        C = hc.run(A, B, algo="plain")
        torch.cuda.synchronize()
        assert hc.sync_status() == 0
        assert_bit_exact(C, oracle_c64(A, B, dtype), dtype)
        b = synthetic.matrix(1, N, "int3", 36, dtype, "cuda")[0]
        R = synthetic.matrix(M, N, "int3", 37, dtype, "cuda")
        act = "gelu_tanh" if dtype == "f16" else "relu"
        D64, pre64 = oracle_epilogue(A, B, dtype, b, R, act)
        D = hc.run(A, B, algo="plain", bias=b, residual=R, act=act)
        torch.cuda.synchronize()
        assert hc.sync_status() == 0
        if act == "relu":
            assert_bit_exact(D, D64, dtype)
        else:
            assert_epilogue_close(D, D64, pre64, dtype, act)
    finally:
        hc.close()


def test_k_chunks_summed_in_cluster_normal():
    """N(0,1) at the weight-streaming shape: the chunk sums in FP32 stay within the plain tolerance."""
    hc = lcg.Handle(0)
    try:
        A, B = synthetic.operands(16, 4096, 14336, "normal", 34, "bf16", "cuda")
        C = hc.run(A, B, algo="plain")
        torch.cuda.synchronize()
        assert hc.sync_status() == 0
        assert_close(C, oracle_c64(A, B, "bf16"), "bf16", "plain")
    finally:
        hc.close()


# ---------------------------------------------------------------- square sweep (BF16 N(0,1))

def test_square_2048_full(h):
    A, B = synthetic.operands(2048, 2048, 2048, "normal", 2, "bf16", "cuda")
    assert_close(_run(h, A, B), oracle_c64(A, B, "bf16"), "bf16", "plain")


@pytest.mark.parametrize("n", [4096, 8192, 16384])
def test_square_sampled_rows(h, n):
    A, B = synthetic.operands(n, n, n, "normal", 2, "bf16", "cuda")
    C = _run(h, A, B)
    rows = synthetic.row_sample(n, 64 if n == 16384 else 128)
    assert_close(C, oracle_c64(A, B, "bf16", rows=rows), "bf16", "plain", rows=rows)


@pytest.mark.parametrize("M,N,K", [(1, 14336, 4096), (16, 4096, 14336), (128, 14336, 4096), (1024, 4096, 14336)])
def test_llm_skinny(h, M, N, K):
    A = synthetic.matrix(M, K, "normal", 1004, "bf16", "cuda")
    B = synthetic.matrix(N, K, "normal", 2004, "bf16", "cuda", scale=0.02)
    C = _run(h, A, B)
    rows = synthetic.row_sample(M, 32)
    assert_close(C, oracle_c64(A, B, "bf16", rows=rows), "bf16", "plain", rows=rows)


# ---------------------------------------------------------------- split-K (few tiles, long K)

# chunks on the single-CTA kernel: 9 (separate sum), none (32 slabs), 4, 4, 8 (separate), none,
# 3 with a ragged last column chunk (last arriver), 3 on 128-wide tiles with partial row quarters,
# 4 with N < 64, 2 (56 tiles: last arriver)
SPLITK = [(1, 4096, 14336), (16, 1000, 2048), (100, 128, 4096), (1, 128, 4096), (128, 256, 8192), (3, 24, 1024),
          (40, 300, 3072), (200, 64, 3200), (50, 40, 4160), (16, 14336, 3072)]


@pytest.mark.parametrize("M,N,K", SPLITK)
def test_split_k_integer_bit_exact(h, M, N, K):
    """Shapes with fewer tiles than SMs cut K into chunks; partial sums meet in FP32 (exact here)."""
    A, B = synthetic.operands(M, N, K, "int3", 19, "bf16", "cuda")
    ref = oracle_c64(A, B, "bf16")
    for _ in range(3):                      # counters must be back at zero for every launch
        assert_bit_exact(_run(h, A, B), ref, "bf16")


def test_split_k_float(h):
    A = synthetic.matrix(16, 14336, "normal", 1004, "bf16", "cuda")
    B = synthetic.matrix(4096, 14336, "normal", 2004, "bf16", "cuda", scale=0.02)
    assert_close(_run(h, A, B), oracle_c64(A, B, "bf16"), "bf16", "plain")


# ---------------------------------------------------------------- tail split of the CTA-pair kernel

@pytest.mark.parametrize("M,N,K", [(4096, 4096, 8192), (4352, 2560, 8200), (2560, 4352, 9000), (4352, 2560, 6200)])
def test_tail_split_integer_bit_exact(h, M, N, K):
    """Tiles of a partial last wave run as two K halves on two pairs (summed by the later one)."""
    A, B = synthetic.operands(M, N, K, "int3", 21, "bf16", "cuda")
    rows = synthetic.row_sample(M, 256)
    ref = oracle_c64(A, B, "bf16", rows=rows)
    for split in (1, 0, 1):
        h.set_option(lcg.OPT_SPLIT, split)
        assert_bit_exact(_run(h, A, B), ref, "bf16", rows=rows)
    h.set_option(lcg.OPT_SPLIT, 1)


@pytest.mark.parametrize("kernel", [2, 5], ids=["tiles256", "tiles512"])
def test_tail_split_fp16(kernel):
    """FP16 through the exchanging tail halves (4352 x 2560 x 6200: 170 tiles of 256 x 256 = 2 waves
    + 18 split; on 256 x 512 tiles 85 = 1 wave + 9 split), split on and off, bit-exact on integers."""
    hs = lcg.Handle(0)
    try:
        hs.set_option(lcg.OPT_PLAIN_KERNEL, kernel)
        M, N, K = 4352, 2560, 6200
        A, B = synthetic.operands(M, N, K, "int3", 27, "f16", "cuda")
        rows = synthetic.row_sample(M, 256)
        ref = oracle_c64(A, B, "f16", rows=rows)
        for split in (1, 0):
            hs.set_option(lcg.OPT_SPLIT, split)
            C = hs.run(A, B, algo="plain")
            torch.cuda.synchronize()
            assert hs.sync_status() == 0
            assert_bit_exact(C, ref, "f16", rows=rows)
    finally:
        hs.close()


# ---------------------------------------------------------------- identities and edge cases

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_bit_exact(h, dtype):
    n = 384
    A = synthetic.matrix(n, n, "normal", 12, dtype, "cuda")
    eye = torch.eye(n, dtype=A.dtype, device="cuda")
    assert torch.equal(_run(h, A, eye), A)


def test_linearity(h):
    """(A1 + A2).B = A1.B + A2.B exactly: FP16 integers with |C| <= 6*3*64 < 2048 are all representable."""
    M, N, K = 256, 512, 64
    A1 = synthetic.matrix(M, K, "int3", 13, "f16", "cuda")
    A2 = synthetic.matrix(M, K, "int3", 14, "f16", "cuda")
    B = synthetic.matrix(N, K, "int3", 15, "f16", "cuda")
    lhs = _run(h, (A1.float() + A2.float()).to(torch.float16), B).float()
    rhs = _run(h, A1, B).float() + _run(h, A2, B).float()
    assert torch.equal(lhs, rhs)


def test_k_zero_writes_zeros_and_empty_is_noop(h):
    A = torch.empty((64, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((32, 0), dtype=torch.bfloat16, device="cuda")
    C = torch.full((64, 32), 3.0, dtype=torch.bfloat16, device="cuda")
    rc = h.run_raw(64, 32, 0, A.data_ptr(), 8, B.data_ptr(), 8, C.data_ptr(), 32, lcg.BF16, lcg.PLAIN,
                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and (C == 0).all()
    C.fill_(5.0)
    assert h.run_raw(0, 32, 16, None, 16, None, 16, C.data_ptr(), 32, lcg.BF16, lcg.PLAIN, None) == 0
    assert h.run_raw(64, 0, 16, None, 16, None, 16, C.data_ptr(), 32, lcg.BF16, lcg.PLAIN, None) == 0
    torch.cuda.synchronize()
    assert (C == 5).all()


def test_repeated_launches_stable(h):
    """Many back-to-back launches (mbarrier phase logic across CTAs' tile loops) stay exact."""
    A, B = synthetic.operands(1024, 1536, 704, "int3", 16, "f16", "cuda")
    ref = oracle_c64(A, B, "f16")
    Cs = [h.run(A, B) for _ in range(20)]
    torch.cuda.synchronize()
    for C in Cs[::5]:
        assert_bit_exact(C, ref, "f16")
    assert all(torch.equal(Cs[0], C) for C in Cs)


# ---------------------------------------------------------------- argument errors (host-side only)

def test_argument_errors(h):
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    a, b, c = A.data_ptr(), B.data_ptr(), C.data_ptr()
    run = h.run_raw
    assert run(-1, 64, 64, a, 64, b, 64, c, 64, 1, 0) == lcg.ERR_ARG
    assert run(64, 64, 64, a, 63, b, 64, c, 64, 1, 0) == lcg.ERR_ARG          # lda < K
    assert run(64, 64, 64, a, 64, b, 64, c, 60, 1, 0) == lcg.ERR_ARG          # ldc < N
    assert run(64, 64, 64, None, 64, b, 64, c, 64, 1, 0) == lcg.ERR_ARG
    assert run(64, 64, 64, a, 64, b, 64, c, 64, 2, 0) == lcg.ERR_ARG          # dtype
    assert run(64, 64, 64, a, 64, b, 64, c, 64, 1, 9) == lcg.ERR_ARG          # algo
    assert run(64, 64, 64, a + 2, 64, b, 64, c, 64, 1, 0) == lcg.ERR_ALIGN    # 2-byte offset
    assert run(60, 60, 60, a, 68, b, 64, c, 64, 1, 0) == lcg.ERR_ALIGN        # ld not multiple of 8
    assert run(64, 64, 64, a, 64, b, 64, a, 64, 1, 0) == lcg.ERR_ALIAS        # C == A
    assert run(32, 64, 64, a, 64, b, 64, a + 32 * 64 * 2 - 16, 64, 1, 0) == lcg.ERR_ALIAS
    torch.cuda.synchronize()
    assert h.sync_status() == 0


# ---------------------------------------------------------------- extreme aspect ratios

@pytest.mark.parametrize("M,N,K", [(131072, 64, 64), (64, 131072, 64), (64, 64, 1 << 20), (3, 5, 1 << 18)])
def test_extreme_aspect_ratios_bit_exact(h, M, N, K):
    """Very tall, very wide and very deep products: thousands of tiles along one dimension, or one
    tile with a million-deep K (split into the maximum number of chunks)."""
    A, B = synthetic.operands(M, N, K, "int3", 23, "bf16", "cuda")
    if K > 1 << 16:
        A = (A.float() / 8).to(A.dtype)           # |C| <= 9K/8 < 2^24 * 2^-3: exact in FP32
    assert_bit_exact(_run(h, A, B), oracle_c64(A, B, "bf16"), "bf16")


# ---------------------------------------------------------------- FP16 shape grid (A ~ N(0,1)/sqrt(K), B ~ N(0,1))

@pytest.mark.parametrize("M,N,K", [(16384, 16384, 16384), (12288, 16384, 64), (64, 12288, 16384),
                                   (16384, 64, 12288), (8192, 12288, 4096)])
def test_fp16_grid_shapes_sampled_rows(h, M, N, K):
    """FP16 grid workload at its largest extents, in the launch configuration the grid times
    (algo auto), against the oracle on 64 sampled rows."""
    A = synthetic.matrix(M, K, "normal", 1003, "f16", "cuda", scale=1.0 / K ** 0.5)
    B = synthetic.matrix(N, K, "normal", 2003, "f16", "cuda")
    C = h.run(A, B, algo="auto")
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    rows = synthetic.row_sample(M, 64)
    assert_close(C, oracle_c64(A, B, "f16", rows=rows), "f16", "plain", rows=rows)


# ---------------------------------------------------------------- one tile row on 96-column tiles

@pytest.mark.parametrize("M,N,K", [(16, 14336, 4096), (128, 14336, 4096), (3, 14300, 4104), (100, 13000, 520)])
def test_one_row_96_column_tiles(M, N, K):
    """C with one 128-row tile row whose 96-column tiles about fill the SMs (150 tiles for N = 14336)
    runs on the single-CTA kernel with BN = 96 and no split-K: integer inputs bit-exact, ragged N and
    K included; and the fused epilogue on the same tiles."""
    h = lcg.Handle(0)
    A, B = synthetic.operands(M, N, K, "int3", 71, "bf16", "cuda")
    Ap, Bp = padded(M, K, "bf16", A), padded(N, K, "bf16", B)
    C = h.run(Ap, Bp, algo="plain")
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert_bit_exact(C, oracle_c64(A, B, "bf16"), "bf16")
    if M == 100:
        b = synthetic.matrix(1, N, "int3", 72, "bf16", "cuda")[0]
        R = padded(M, N, "bf16", synthetic.matrix(M, N, "int3", 73, "bf16", "cuda"))
        D64, _ = oracle_epilogue(A, B, "bf16", b, R, "relu")
        C = h.run(Ap, Bp, algo="plain", bias=b, residual=R, act="relu")
        torch.cuda.synchronize()
        assert h.sync_status() == 0
        assert_bit_exact(C, D64, "bf16")
    h.close()


# ---------------------------------------------------------------- claimed items (CTA-pair kernel, many waves)

@pytest.mark.parametrize("kernel", [2, 5], ids=["tiles256", "tiles512"])
@pytest.mark.parametrize("ctas,M,N,K,dtype", [(8, 2048, 2048, 512, "bf16"), (8, 1900, 2100, 700, "f16"),
                                              (16, 2560, 3328, 6144, "bf16")])
def test_claimed_items_bit_exact(kernel, ctas, M, N, K, dtype):
    """With at least 16 waves of items the CTA-pair kernel claims every pair's later items from a
    counter.  A cap of 8 or 16 CTAs (4 or 8 pairs) puts small shapes there: exactly 16 waves, a
    ragged edge, and 130 tiles with the tail split (16 full waves + 2 tiles as K halves).  Integer
    inputs bit-exact against the oracle, the same bits as the static order on the full machine, and
    stable over back-to-back launches (the counter starts from zero each time).  On both tile widths;
    the 256 x 512 tiles run on half the CTAs (2 or 4 pairs), so that the same shapes have 16 waves."""
    A, B = synthetic.operands(M, N, K, "int3", 81, dtype, "cuda")
    rows = None if M * N * K <= 4e9 else synthetic.row_sample(M, 256)
    ref = oracle_c64(A, B, dtype, rows=rows)
    A, B = padded(M, K, dtype, A), padded(N, K, dtype, B)   # 16-byte row starts for any K
    h = lcg.Handle(0)
    h.set_option(lcg.OPT_PLAIN_KERNEL, kernel)
    h.set_option(lcg.OPT_MAX_CTAS, ctas if kernel == 2 else ctas // 2)
    Cs = [h.run(A, B, algo="plain") for _ in range(4)]
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert_bit_exact(Cs[0], ref, dtype, rows=rows)
    assert all(torch.equal(Cs[0], C) for C in Cs[1:])
    full = lcg.Handle(0)
    full.set_option(lcg.OPT_PLAIN_KERNEL, kernel)
    assert torch.equal(_run(full, A, B), Cs[0])
    full.close()
    h.close()


@pytest.mark.parametrize("kernel,ctas", [(2, 8), (5, 4)], ids=["tiles256", "tiles512"])
def test_claimed_items_with_epilogue(kernel, ctas):
    """The fused epilogue on claimed items (bias, residual, GELU; exact integer product) against the
    oracle's FP64 D, and the same bits as the static order (1792 x 2560: 70 narrow tiles on 4 pairs,
    35 wide ones on 2: at least 16 waves either way)."""
    M, N, K = 1792, 2560, 640
    A, B = synthetic.operands(M, N, K, "int3", 82, "bf16", "cuda")
    b = synthetic.matrix(1, N, "int3", 83, "bf16", "cuda")[0]
    R = synthetic.matrix(M, N, "int3", 84, "bf16", "cuda")
    D64, pre = oracle_epilogue(A, B, "bf16", b, R, "gelu")
    h = lcg.Handle(0)
    h.set_option(lcg.OPT_PLAIN_KERNEL, kernel)
    h.set_option(lcg.OPT_MAX_CTAS, ctas)
    C = h.run(A, B, algo="plain", bias=b, residual=R, act="gelu")
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert_epilogue_close(C, D64, pre, "bf16", "gelu")
    h.set_option(lcg.OPT_MAX_CTAS, 0)
    C2 = h.run(A, B, algo="plain", bias=b, residual=R, act="gelu")
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert torch.equal(C, C2)
    h.close()


@pytest.mark.parametrize("kernel", [2, 5], ids=["tiles256", "tiles512"])
def test_tail_split_partner_timeout_is_reported_and_recovered(kernel):
    """Failure detection without a GPU fault: the second K halves of the split tail tiles never
    raise their flags, so the first halves' bounded waits run out; the kernel ends, the next status
    call reports LCGEMM_ERR_TIMEOUT once, and the handle keeps working (same shape, exact again)."""
    h = lcg.Handle(0)
    h.set_option(lcg.OPT_PLAIN_KERNEL, kernel)
    h.set_option(lcg.OPT_WAIT_TIMEOUT_US, 50000)
    # 256 x 256 tiles: 256 = 3 waves of 76 pairs + 28 split; 256 x 512 tiles: 128 = 1 wave of 76 + 52,
    # which do not fit twice over, so 24 pairs (48 CTAs) run them: 5 waves + 8 split
    M, N, K = 4096, 4096, 8192
    if kernel == 5:
        h.set_option(lcg.OPT_MAX_CTAS, 48)
    A, B = synthetic.operands(M, N, K, "int3", 23, "bf16", "cuda")
    h.set_option(lcg.OPT_DEBUG_DROP_SIGNAL, 1)
    h.run(A, B, algo="plain")
    torch.cuda.synchronize()
    assert h.sync_status() == lcg.ERR_TIMEOUT
    assert h.sync_status() == lcg.OK
    h.set_option(lcg.OPT_DEBUG_DROP_SIGNAL, 0)
    C = h.run(A, B, algo="plain")
    torch.cuda.synchronize()
    assert h.sync_status() == lcg.OK
    rows = synthetic.row_sample(M, 256)
    assert_bit_exact(C, oracle_c64(A, B, "bf16", rows=rows), "bf16", rows=rows)
    h.close()
