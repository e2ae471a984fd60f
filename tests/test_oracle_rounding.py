"""Pins for the oracle's round-to-nearest-even (CPU only)."""
import numpy as np
import torch

import oracle
from oracle.rounding import rne_bits, rne_values


def _edge_values_f16():
    v = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e6, -1e6,
         2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25,
         np.inf, -np.inf]
    # exact ties and near-ties between neighbouring FP16 values in several binades
    for e in (-20, -14, -3, 0, 4, 15):
        ulp = 2.0 ** (max(e, -14) - 10)
        base = 2.0 ** e
        for k in (0, 1, 2, 3, 1023):
            x = base + k * ulp
            v += [x + ulp / 2, x + ulp / 2 * (1 - 2 ** -30), x + ulp / 2 * (1 + 2 ** -30)]
    return np.array(v + [-x for x in v])


def test_f16_matches_numpy():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, 200000),
                        _edge_values_f16()])
    got = rne_bits(x, oracle.F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref), x[got != ref][:5]


def _edge_values_bf16():
    v = [0.0, 1.0, 3.3895314e38, 3.3961775e38, 3.4e38, 1e-40, 9.18355e-41, 1e-45,
         2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -126]
    for e in (-130, -126, -1, 0, 7, 127):
        ulp = 2.0 ** (max(e, -126) - 7)
        base = 2.0 ** e
        for k in (0, 1, 2, 127):
            x = base + k * ulp
            v += [x + ulp / 2, x + ulp / 2 - ulp * 2 ** -16, x + ulp / 2 + ulp * 2 ** -16]
    v = np.array(v, np.float64)
    v = v[np.isfinite(v.astype(np.float32))]
    return np.concatenate([v, -v]).astype(np.float32)


def test_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    x = np.concatenate([(rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32),
                        rng.integers(0, 2 ** 32 - 1, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32),
                        _edge_values_bf16()])
    x = x[np.isfinite(x)]
    got = rne_bits(x.astype(np.float64), oracle.BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref), x[got != ref][:5]


def test_special_values():
    for dt in (oracle.F16, oracle.BF16):
        r = rne_values(np.array([np.nan, np.inf, -np.inf, -0.0]), dt)
        assert np.isnan(r[0]) and r[1] == np.inf and r[2] == -np.inf and np.signbit(r[3])
    assert rne_bits(np.array([2.0 ** 128]), oracle.BF16)[0] == 0x7F80
    assert rne_bits(np.array([np.nan]), oracle.BF16)[0] & 0x7FC0 == 0x7FC0


def test_ties_go_to_even():
    # 1 + 2^-11 lies halfway between 1 and 1 + 2^-10 (FP16): even neighbour is 1
    assert rne_values(np.array([1 + 2.0 ** -11]), oracle.F16)[0] == 1.0
    # 1 + 3*2^-11 lies halfway between 1+2^-10 (odd) and 1+2^-9 (even)
    assert rne_values(np.array([1 + 3 * 2.0 ** -11]), oracle.F16)[0] == 1 + 2.0 ** -9
    # BF16 keeps 8 significant bits: 1 + 2^-8 is a tie that goes to 1
    assert rne_values(np.array([1 + 2.0 ** -8]), oracle.BF16)[0] == 1.0
    assert rne_values(np.array([1 + 3 * 2.0 ** -8]), oracle.BF16)[0] == 1 + 2.0 ** -6
