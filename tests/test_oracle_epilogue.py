"""Pins for O3, the FP64 epilogue oracle D = act(A.B + bias) + R (CPU only)."""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import epilogue as ep

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse(path):
    cases, cur = {}, None
    lines = [l.split("#")[0].strip() for l in open(path)]
    lines = [l for l in lines if l]
    i = 0
    while i < len(lines):
        tok = lines[i].split()
        if tok[0] == "case":
            cur = cases.setdefault(tok[1], {})
            i += 1
        elif tok[0] == "act":
            cur["act"] = tok[1]
            i += 1
        else:
            name, r, c = tok[0], int(tok[1]), int(tok[2])
            cur[name] = np.array([[float(v) for v in lines[i + 1 + k].split()] for k in range(r)])
            assert cur[name].shape == (r, c)
            i += 1 + r
    return cases


CASES = _parse(os.path.join(GOLDEN, "epilogue_small.txt"))


def _run_case(cs, dtype):
    A = oracle.rounding.rne_bits(cs["A"], dtype)
    Bnk = oracle.rounding.rne_bits(cs["B"].T.copy(), dtype)
    C64 = oracle.gemm(A, Bnk, dtype)
    bias = cs["bias"][0] if "bias" in cs else None
    return ep.apply(C64, bias=bias, residual=cs.get("R"), act=cs["act"])


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_golden_hand_computed(name, dtype):
    cs = CASES[name]
    np.testing.assert_allclose(_run_case(cs, dtype), cs["D"], rtol=1e-12, atol=0)


def test_bias_is_per_column_and_residual_after_activation():
    cs = CASES["relu_2x3x2"]
    A = oracle.rounding.rne_bits(cs["A"], oracle.BF16)
    Bnk = oracle.rounding.rne_bits(cs["B"].T.copy(), oracle.BF16)
    C64 = oracle.gemm(A, Bnk, oracle.BF16)
    bias, R = cs["bias"][0], cs["R"]
    by_row = ep.relu(C64 + bias[:, None]) + R               # bias indexed by row
    res_inside = ep.relu(C64 + bias[None, :] + R)           # residual before the activation
    for wrong in (by_row, res_inside):
        assert not np.array_equal(wrong, cs["D"])
    np.testing.assert_array_equal(ep.apply(C64, bias, R, "relu"), cs["D"])


def test_no_epilogue_is_identity():
    C = np.random.default_rng(0).standard_normal((5, 7))
    np.testing.assert_array_equal(ep.apply(C), C)
    np.testing.assert_array_equal(ep.apply(C, act="none"), C)


def test_relu_invariants():
    x = np.array([-3.5, -0.0, 0.0, 1e-300, 2.0, -1e300])
    r = ep.relu(x)
    np.testing.assert_array_equal(r, (x + np.abs(x)) / 2)
    assert not np.signbit(r).any(), "ReLU of a non-positive value is +0"


@pytest.mark.parametrize("fn", [ep.gelu, ep.gelu_tanh])
def test_gelu_symmetry_and_limits(fn):
    # x Phi(x) - (-x) Phi(-x) = x (Phi(x) + Phi(-x)) = x, and the tanh form keeps it (tanh is odd)
    x = np.linspace(-7, 7, 1401)
    np.testing.assert_allclose(fn(x) - fn(-x), x, rtol=0, atol=1e-12)
    assert fn(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(fn(np.array([12.0])), [12.0], rtol=1e-15)
    assert abs(fn(np.array([-12.0]))[0]) < 1e-20
    # monotone for x >= 0 and bounded below by its minimum near x = -0.75 (about -0.17)
    assert np.all(np.diff(fn(np.linspace(0, 7, 701))) > 0)
    assert -0.18 < fn(x).min() < -0.16


def test_gelu_table_values():
    # standard normal table: Phi(0.5) = 0.691462461274013, Phi(1.5) = 0.933192798731142
    np.testing.assert_allclose(ep.gelu(np.array([0.5, 1.5, -1.5])),
                               [0.5 * 0.691462461274013, 1.5 * 0.933192798731142,
                                -1.5 * (1 - 0.933192798731142)], rtol=1e-12)


def test_gelu_tanh_close_to_gelu():
    """The tanh form approximates x Phi(x) to within 5e-4 everywhere (largest gap near |x| = 2.7);
    a wrong constant (0.05 for 0.044715: 3e-3) or a dropped cubic term (3e-2) breaks this."""
    x = np.linspace(-10, 10, 200001)
    gap = np.abs(ep.gelu_tanh(x) - ep.gelu(x))
    assert 1e-4 < gap.max() < 5e-4
    assert abs(abs(x[np.argmax(gap)]) - 2.7) < 0.1


def test_shape_checks():
    C = np.zeros((2, 3))
    with pytest.raises(ValueError):
        ep.apply(C, bias=np.zeros(2))
    with pytest.raises(ValueError):
        ep.apply(C, residual=np.zeros((3, 2)))
    with pytest.raises(ValueError):
        ep.activation(C, 7)
    assert math.isclose(ep.apply(np.array([[1.0]]), act="gelu")[0, 0], 0.841344746068543, rel_tol=1e-12)
