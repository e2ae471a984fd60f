"""O2: one- and two-level Strassen -- oracle, test infrastructure only.

Source: FalconGEMM write-up (hyper.ai news 54396), section "从 Strassen 出发":
a 2x2 block product needs 8 block multiplications; Strassen (1969) recombines
the inputs so that 7 suffice, then recovers C with extra additions; applied
recursively, a 4x4 block product needs 49 instead of 64 multiplications.  The
LCMA description of such an algorithm states which input sub-blocks are
combined, how many products run and how the products recombine into C.  The
write-up prints no formulas, so this module uses the textbook 1969 scheme:

    M1 = (A11 + A22)(B11 + B22)    C11 = M1 + M4 - M5 + M7
    M2 = (A21 + A22) B11           C12 = M3 + M5
    M3 = A11 (B12 - B22)           C21 = M2 + M4
    M4 = A22 (B21 - B11)           C22 = M1 - M2 + M3 + M6
    M5 = (A11 + A12) B22
    M6 = (A21 - A11)(B11 + B12)
    M7 = (A12 - A22)(B21 + B22)

written as coefficient tables U (7 x 4, A blocks), V (7 x 4, B blocks) and
W (4 x 7, C blocks), block index ``2*row + col``.  Two levels apply the scheme
inside every product, which is the Kronecker product of the tables (49
products over a 4x4 block grid; block row ``2*r_outer + r_inner``).

The algorithm runs in the three steps the write-up gives for the basic GPU
pipeline (section "从 LCMA 到 FalconGEMM"): combine the A and B sub-blocks into
the product operands, run the products, combine the products into C.

Modes
-----
``"f64"``     every step in FP64 -- equal to the plain product up to FP64
              rounding (the algebra check).
``"emulate"`` the operand sums of step 1 are formed in FP32 in ascending block
              order and rounded once to the input type (round to nearest
              even); products and the combination are FP64 with one final
              rounding by the caller.  This models the error the low-precision
              operand sums add (numerics paragraph of the write-up).
"""
from __future__ import annotations

import numpy as np

from .rounding import rne_values

# Block index q = 2*r + c:  0 -> X11, 1 -> X12, 2 -> X21, 3 -> X22.
U1 = np.array([
    [1, 0, 0, 1],    # M1: A11 + A22
    [0, 0, 1, 1],    # M2: A21 + A22
    [1, 0, 0, 0],    # M3: A11
    [0, 0, 0, 1],    # M4: A22
    [1, 1, 0, 0],    # M5: A11 + A12
    [-1, 0, 1, 0],   # M6: A21 - A11
    [0, 1, 0, -1],   # M7: A12 - A22
], dtype=np.int64)

V1 = np.array([
    [1, 0, 0, 1],    # M1: B11 + B22
    [1, 0, 0, 0],    # M2: B11
    [0, 1, 0, -1],   # M3: B12 - B22
    [-1, 0, 1, 0],   # M4: B21 - B11
    [0, 0, 0, 1],    # M5: B22
    [1, 1, 0, 0],    # M6: B11 + B12
    [0, 0, 1, 1],    # M7: B21 + B22
], dtype=np.int64)

W1 = np.array([
    [1, 0, 0, 1, -1, 0, 1],   # C11 = M1 + M4 - M5 + M7
    [0, 0, 1, 0, 1, 0, 0],    # C12 = M3 + M5
    [0, 1, 0, 1, 0, 0, 0],    # C21 = M2 + M4
    [1, -1, 1, 0, 0, 1, 0],   # C22 = M1 - M2 + M3 + M6
], dtype=np.int64)


def tables(levels: int):
    """(U, V, W) for ``levels`` nested Strassen levels over a 2^L x 2^L block grid.

    Returns integer arrays ``U[p, R, C]``, ``V[p, R, C]`` (product p, block row R,
    block column C of A resp. B) and ``W[R, C, p]`` (block of C).  For L = 0 the
    single "product" is the whole matrix.
    """
    g = 1
    U = np.ones((1, 1, 1), np.int64)
    V = np.ones((1, 1, 1), np.int64)
    W = np.ones((1, 1, 1), np.int64)
    for _ in range(levels):
        U = _kron_level(U, U1.reshape(7, 2, 2), g)
        V = _kron_level(V, V1.reshape(7, 2, 2), g)
        Wt = _kron_level(np.transpose(W, (2, 0, 1)), np.transpose(W1.reshape(2, 2, 7), (2, 0, 1)), g)
        W = np.transpose(Wt, (1, 2, 0))
        g *= 2
    return U, V, W


def _kron_level(outer, inner, g):
    """Compose an outer table (P x g x g) with a one-level table (R x 2 x 2).

    New product index ``p_outer * R + p_inner``; new block row
    ``2 * r_outer + r_inner`` and column ``2 * c_outer + c_inner``.
    """
    P = outer.shape[0]
    R = inner.shape[0]
    out = np.zeros((P * R, 2 * g, 2 * g), np.int64)
    for po in range(P):
        for pi in range(R):
            for ro in range(g):
                for co in range(g):
                    for ri in range(2):
                        for ci in range(2):
                            out[po * R + pi, 2 * ro + ri, 2 * co + ci] = outer[po, ro, co] * inner[pi, ri, ci]
    return out


def _blocks(X, g):
    r, c = X.shape
    return [[X[i * (r // g):(i + 1) * (r // g), j * (c // g):(j + 1) * (c // g)] for j in range(g)]
            for i in range(g)]


def _combine(coef, blocks, mode, dtype):
    """Step 1 for one product: sum_q coef[q] * block_q."""
    g = coef.shape[0]
    if mode == "f64":
        s = None
        for R in range(g):
            for C in range(g):
                if coef[R, C]:
                    t = coef[R, C] * blocks[R][C]
                    s = t if s is None else s + t
        return s
    # "emulate": FP32 sum in ascending block order, then one rounding to the input type
    s = None
    for R in range(g):
        for C in range(g):
            if coef[R, C]:
                t = np.float32(coef[R, C]) * blocks[R][C].astype(np.float32)
                s = t if s is None else (s + t).astype(np.float32)
    return rne_values(s.astype(np.float64), dtype)


def strassen(A: np.ndarray, B: np.ndarray, levels: int, mode: str = "f64", dtype=None, rows=None):
    """C = A @ B by ``levels``-level Strassen (float64 result).

    ``A``: M x K float64 values; ``B``: K x N float64 values (mathematical
    layout).  M, N, K must be divisible by 2^levels.  ``rows``: optional output
    row indices; only the product rows they need are formed.  ``dtype``
    (oracle.F16 / oracle.BF16) is required for mode "emulate".
    """
    if mode not in ("f64", "emulate"):
        raise ValueError(mode)
    if mode == "emulate" and dtype is None:
        raise ValueError("mode 'emulate' needs the input dtype")
    M, K = A.shape
    K2, N = B.shape
    g = 2 ** levels
    if K2 != K or M % g or N % g or K % g:
        raise ValueError("dimensions must be divisible by 2^levels")
    Mb, Nb = M // g, N // g
    U, V, W = tables(levels)
    if rows is None:
        rows = np.arange(M)
    rows = np.asarray(rows, dtype=np.int64)
    local = np.unique(rows % Mb)          # product rows the sample needs
    A_loc = A.reshape(g, Mb, K)[:, local, :].reshape(g * local.size, K)
    Ab = _blocks(A_loc, g)
    Bb = _blocks(B, g)
    P = U.shape[0]
    prods = []
    for p in range(P):                    # step 1 (combine A/B) and step 2 (products)
        At = _combine(U[p], Ab, mode, dtype)
        Bt = _combine(V[p], Bb, mode, dtype)
        prods.append(At @ Bt)
    out = np.zeros((rows.size, N), np.float64)
    pos = {int(l): i for i, l in enumerate(local)}
    for R in range(g):                    # step 3 (combine the products into C)
        for C in range(g):
            acc = np.zeros((local.size, Nb), np.float64)
            for p in range(P):
                if W[R, C, p]:
                    acc = acc + W[R, C, p] * prods[p]
            sel = np.nonzero(rows // Mb == R)[0]
            if sel.size:
                idx = [pos[int(r % Mb)] for r in rows[sel]]
                out[sel, C * Nb:(C + 1) * Nb] = acc[idx]
    return out
