"""O3: the element-wise GEMM epilogue in FP64 -- oracle, test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
use this module; the product library shares no code with it.

What it computes (one output element at a time, C64 the exact product A.B):

    D[m, n] = act(C64[m, n] + bias[n]) + residual[m, n]

Sources:
* DeepGEMM tuning blog (kwkr.cn news 553926), section 3.3 (算子融合): a GEMM
  is usually followed by a bias add and a GeLU (Transformer) or a ReLU (CNN);
  the fused kernel adds the bias, broadcast, to the finished C tile while it
  is still on chip, applies a tanh-approximated GeLU, and only then stores.
* "Kernel 与性能" (wineandchord.com kernels-performance), section "Fusion":
  bias + activation, and residual add, as element-wise work folded into the
  producing kernel.

Readings (the pages give no formulas for these steps):
* ``bias`` is one value per output column (length N), added to every row.
* The order is bias, then activation, then the residual.
* ReLU(x) = x if x > 0 else +0.
* GELU is x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)) (Hendrycks and Gimpel,
  "Gaussian Error Linear Units", 2016); GELU_TANH is that paper's tanh
  approximation x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))), the form
  section 3.3 of the DeepGEMM page evaluates with a fast hardware tanh.
* The result is rounded once to the output type (``oracle.reference_output``).
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

ACT_NONE, ACT_RELU, ACT_GELU, ACT_GELU_TANH = 0, 1, 2, 3
ACTS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU, "gelu_tanh": ACT_GELU_TANH}


def relu(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    return np.where(x > 0, x, 0.0)


def gelu(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


_ACT_FN = {ACT_NONE: lambda x: np.asarray(x, np.float64), ACT_RELU: relu, ACT_GELU: gelu,
           ACT_GELU_TANH: gelu_tanh}


def activation(x: np.ndarray, act) -> np.ndarray:
    act = ACTS[act] if isinstance(act, str) else int(act)
    if act not in _ACT_FN:
        raise ValueError(f"unknown activation {act}")
    with np.errstate(invalid="ignore", over="ignore"):   # IEEE results for inf and NaN inputs, silently
        return _ACT_FN[act](x)


def apply(C64: np.ndarray, bias=None, residual=None, act=ACT_NONE) -> np.ndarray:
    """D = act(C64 + bias[None, :]) + residual, all in FP64.

    ``C64``: M x N (or a sample of rows of it); ``bias``: N values or None;
    ``residual``: an array of C64's shape or None.  Inputs are values (decode
    16-bit operands with ``oracle.decode`` first).
    """
    D = np.array(C64, np.float64, copy=True)
    if bias is not None:
        bias = np.asarray(bias, np.float64)
        if bias.shape != (D.shape[1],):
            raise ValueError(f"bias must have {D.shape[1]} values, got shape {bias.shape}")
        D = D + bias[None, :]
    D = activation(D, act)
    if residual is not None:
        residual = np.asarray(residual, np.float64)
        if residual.shape != D.shape:
            raise ValueError(f"residual must be {D.shape}, got {residual.shape}")
        D = D + residual
    return D
