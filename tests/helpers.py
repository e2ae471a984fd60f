"""Shared helpers for the parity tests: run the library, run the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synthetic

# Floating-point tolerances on N(0,1)-type inputs, normwise relative Frobenius
# error against the unrounded FP64 product, per algorithm family and dtype.
NORMWISE_TOL = {
    ("plain", "f16"): 2e-3,
    ("plain", "bf16"): 8e-3,
    ("strassen", "f16"): 4e-3,
    ("strassen", "bf16"): 1.6e-2,
}
# max_ij |C_gpu - C64| <= MAXERR_SIGMA * sigma_C, sigma_C = RMS(C64).  0.05 everywhere except
# two-level Strassen in BF16: rounding the 4-term operand sums to BF16 alone (the oracle's
# emulating Strassen, exact products) already reaches max/sigma_C = 0.071 on 1024^3 and
# 2048^3 N(0,1) inputs, so that algorithm/dtype pair is held to 0.10.
MAXERR_SIGMA = 0.05
MAXERR_SIGMA_OVERRIDE = {("strassen2", "bf16"): 0.10}


def family(algo: str) -> str:
    return "plain" if algo == "plain" else "strassen"


def dt_code(dtype: str) -> int:
    return oracle.F16 if dtype == "f16" else oracle.BF16


def oracle_c64(A: torch.Tensor, B: torch.Tensor, dtype: str, rows=None) -> np.ndarray:
    return oracle.gemm(synthetic.bits(A), synthetic.bits(B), dt_code(dtype), rows=rows)


def gpu_values(C: torch.Tensor, rows=None) -> np.ndarray:
    Ch = C.detach().cpu()
    if rows is not None:
        Ch = Ch[torch.as_tensor(rows)]
    return Ch.to(torch.float64).numpy()


def assert_bit_exact(C: torch.Tensor, C64: np.ndarray, dtype: str, rows=None):
    ref = oracle.reference_output(C64, dt_code(dtype))
    got = synthetic.bits(C if rows is None else C.detach().cpu()[torch.as_tensor(rows)])
    bad = np.nonzero(got != ref)
    assert bad[0].size == 0, f"{bad[0].size} mismatches, first at {bad[0][0]},{bad[1][0]}: " \
                             f"got {got[bad][0]:#06x} want {ref[bad][0]:#06x}"


def errors(C: torch.Tensor, C64: np.ndarray, rows=None):
    got = gpu_values(C, rows)
    diff = got - C64
    nrm = np.linalg.norm(C64)
    normwise = np.linalg.norm(diff) / nrm if nrm > 0 else np.linalg.norm(diff)
    sigma = np.sqrt(np.mean(C64 ** 2))
    return normwise, float(np.max(np.abs(diff))) if diff.size else 0.0, sigma


def assert_close(C: torch.Tensor, C64: np.ndarray, dtype: str, algo: str, rows=None):
    assert np.isfinite(gpu_values(C, rows)).all(), "non-finite output"
    normwise, maxerr, sigma = errors(C, C64, rows)
    tol = NORMWISE_TOL[(family(algo), dtype)]
    assert normwise <= tol, f"normwise error {normwise:.3e} > {tol:.1e} ({algo}, {dtype})"
    bound = MAXERR_SIGMA_OVERRIDE.get((algo, dtype), MAXERR_SIGMA)
    assert maxerr <= bound * sigma, f"max error {maxerr:.3e} > {bound} * sigma_C ({sigma:.3e})"
    return normwise, maxerr, sigma


# ---------------------------------------------------------------- fused epilogue

# GELU's derivative x phi(x) + Phi(x) peaks at 1.129 (x = sqrt 2): an error e in the
# pre-activation value moves GELU by at most 1.13 e; ReLU and the identity by at most e.
ACT_LIPSCHITZ = 1.13
# Absolute error of the hardware tanh approximation used by GELU_TANH: below 2^-10 over the
# whole range (the library header's stated bound); it moves x/2 (1 + tanh) by |x| 2^-11.
TANH_HW_ABS = 2.0 ** -10
# GELU's erfc (Abramowitz-Stegun 7.1.26, absolute error <= 1.5e-7, times a fast exponential):
# it moves x Phi(x) by at most |x| 2^-22 (the usual FP32 erf evaluation has the same order).
GELU_ERFC_ABS = 2.0 ** -22


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` values at |x| (FP16: 11-bit significand, BF16: 8; subnormals included)."""
    p, emin = (11, -14) if dtype == "f16" else (8, -126)
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return 2.0 ** (np.maximum(e, emin) - (p - 1))


def padded(M: int, N: int, dtype: str, fill=None, device="cuda") -> torch.Tensor:
    """An M x N view with rows padded to a multiple of 8 elements (16-byte row starts)."""
    t = torch.zeros((M, (N + 7) // 8 * 8), dtype=synthetic.DTYPES[dtype], device=device)[:, :N]
    if fill is not None:
        t.copy_(fill)
    return t


def oracle_epilogue(A, B, dtype: str, bias=None, residual=None, act="none", rows=None, with_product=False):
    """(D64, pre64[, C64]): the oracle's FP64 D = act(A.B + bias) + residual, its pre-activation
    A.B + bias and (with_product) the product A.B itself."""
    dt = dt_code(dtype)
    C64 = oracle_c64(A, B, dtype, rows=rows)
    b = None if bias is None else oracle.decode(synthetic.bits(bias), dt)
    R = None
    if residual is not None:
        Rh = residual.detach().cpu()
        if rows is not None:
            Rh = Rh[torch.as_tensor(rows)]
        R = oracle.decode(synthetic.bits(Rh), dt)
    pre = C64 if b is None else C64 + b[None, :]
    D64 = oracle.epilogue.apply(C64, b, R, act)
    return (D64, pre, C64) if with_product else (D64, pre)


def assert_epilogue_close(C, D64, pre64, dtype: str, act: str, gemm_err: float = 0.0, rows=None):
    """Elementwise |C - D64| <= ACT_LIPSCHITZ * gemm_err + ulp(D) (+ the hardware tanh term).

    ``gemm_err`` bounds the error of the FP32 product itself (0 where it is exact)."""
    got = gpu_values(C, rows)
    assert np.isfinite(got).all(), "non-finite output"
    tol = ACT_LIPSCHITZ * gemm_err + ulp(np.maximum(np.abs(got), np.abs(D64)), dtype)
    if act == "gelu_tanh":
        tol = tol + 0.5 * np.abs(pre64) * TANH_HW_ABS
    elif act == "gelu":
        tol = tol + np.abs(pre64) * GELU_ERFC_ABS
    bad = np.abs(got - D64) > tol
    assert not bad.any(), (f"{bad.sum()} elements off, worst at {np.unravel_index(np.argmax(np.abs(got - D64) - tol), got.shape)}: "
                           f"got {got[bad][0]} want {D64[bad][0]} (tol {tol[bad][0]:.3e})")
