"""Pins for O1, the plain-definition oracle (CPU only)."""
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_cases(path):
    cases, cur, lines = {}, None, [l.split("#")[0].strip() for l in open(path)]
    lines = [l for l in lines if l]
    i = 0
    while i < len(lines):
        tok = lines[i].split()
        if tok[0] == "case":
            cur = cases.setdefault(tok[1], {})
            i += 1
            continue
        name, r, c = tok[0], int(tok[1]), int(tok[2])
        cur[name] = np.array([[float(v) for v in lines[i + 1 + k].split()] for k in range(r)])
        assert cur[name].shape == (r, c)
        i += 1 + r
    return cases


def _enc(x, dtype):
    return oracle.rounding.rne_bits(np.asarray(x, np.float64), dtype)


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_golden_hand_computed(dtype):
    for name, cs in _parse_cases(os.path.join(GOLDEN, "gemm_small.txt")).items():
        A = _enc(cs["A"], dtype)
        Bnk = _enc(cs["B"].T.copy(), dtype)            # B stored N x K
        C = oracle.gemm(A, Bnk, dtype)
        np.testing.assert_array_equal(C, cs["C"], err_msg=name)


def test_decoders_exhaustive():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dtype in (oracle.F16, oracle.BF16):
        ref = oracle.decode(allbits, dtype)
        got = np.array([oracle.decode_c(int(b), dtype) for b in allbits])
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), (dtype, np.nonzero(~same)[0][:5])
        sign_ok = np.signbit(got[~np.isnan(got)]) == np.signbit(ref[~np.isnan(ref)])
        assert sign_ok.all()


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_identity(dtype):
    M, K = 37, 53
    A = synthetic.bits(synthetic.matrix(M, K, "uniform", 11, "f16" if dtype == 0 else "bf16"))
    eye = _enc(np.eye(K), dtype)                       # I is symmetric: stored N x K = I
    C = oracle.gemm(A, eye, dtype)
    np.testing.assert_array_equal(C, oracle.decode(A, dtype))


def test_linearity_exact_on_integers():
    M, N, K = 19, 23, 64
    dt = oracle.BF16
    A1 = synthetic.matrix(M, K, "int3", 1, "bf16")
    A2 = synthetic.matrix(M, K, "int3", 2, "bf16")
    B = synthetic.bits(synthetic.matrix(N, K, "int3", 3, "bf16"))
    S = synthetic.bits((A1.float() + A2.float()).to(torch.bfloat16))   # entries in {-6..6}: exact
    lhs = oracle.gemm(S, B, dt)
    rhs = oracle.gemm(synthetic.bits(A1), B, dt) + oracle.gemm(synthetic.bits(A2), B, dt)
    np.testing.assert_array_equal(lhs, rhs)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_against_numpy_matmul(dtype):
    dt = oracle.F16 if dtype == "f16" else oracle.BF16
    M, N, K = 45, 70, 129
    A = synthetic.bits(synthetic.matrix(M, K, "normal", 4, dtype))
    B = synthetic.bits(synthetic.matrix(N, K, "normal", 5, dtype))
    C = oracle.gemm(A, B, dt)
    ref = oracle.decode(A, dt) @ oracle.decode(B, dt).T
    np.testing.assert_allclose(C, ref, rtol=1e-12, atol=1e-12)


def test_transposed_operand_detected():
    """B must be read as stored N x K: reading it as K x N gives another product."""
    cs = _parse_cases(os.path.join(GOLDEN, "gemm_small.txt"))["fractional_2x2x2"]
    dt = oracle.BF16
    A = _enc(cs["A"], dt)
    wrong = oracle.gemm(A, _enc(cs["B"], dt), dt)      # B passed without the N x K transpose
    assert not np.array_equal(wrong, cs["C"])


def test_row_sample_matches_full():
    M, N, K = 64, 48, 80
    A = synthetic.bits(synthetic.matrix(M, K, "normal", 6, "bf16"))
    B = synthetic.bits(synthetic.matrix(N, K, "normal", 7, "bf16"))
    full = oracle.gemm(A, B, oracle.BF16)
    rows = np.array([63, 0, 17, 17, 40])
    np.testing.assert_array_equal(oracle.gemm(A, B, oracle.BF16, rows=rows), full[rows])


def test_degenerate_sizes():
    A = np.zeros((3, 0), np.uint16)
    B = np.zeros((4, 0), np.uint16)
    np.testing.assert_array_equal(oracle.gemm(A, B, oracle.F16), np.zeros((3, 4)))
    assert oracle.gemm(np.zeros((0, 5), np.uint16), np.zeros((2, 5), np.uint16), oracle.F16).shape == (0, 2)
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((3, 5), np.uint16), np.zeros((2, 4), np.uint16), oracle.F16)
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((3, 5), np.uint16), np.zeros((2, 5), np.uint16), oracle.F16, rows=[3])


def test_binary_inputs_exact():
    """Binary {0,1} inputs: every C entry is an integer count (exact match criterion)."""
    M, N, K = 16, 16, 256
    A = synthetic.matrix(M, K, "binary", 8, "f16")
    B = synthetic.matrix(N, K, "binary", 9, "f16")
    C = oracle.gemm(synthetic.bits(A), synthetic.bits(B), oracle.F16)
    ref = A.numpy().astype(np.int64) @ B.numpy().astype(np.int64).T
    np.testing.assert_array_equal(C, ref)
