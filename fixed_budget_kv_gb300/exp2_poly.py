"""Coefficients of the polynomial 2^x that the CUDA kernels evaluate on the FMA pipe.

The kernels take part of their exponentials off the special-function unit
(MUFU, 32 results per clock per SM) and compute them with fused multiply-adds
instead, so that both pipes work at once.  The method is the textbook one:

    x = j + f,  j = round(x) (an integer),  f in [-1/2, 1/2]
    2^x = 2^j * 2^f,  2^f ~ p(f) = c0 + c1 f + c2 f^2 + c3 f^3

where 2^j is applied by adding j to the binary exponent of p(f), and the
coefficients of p minimise the largest relative error |p(f) / 2^f - 1| over
[-1/2, 1/2] (the Remez exchange algorithm for a weighted minimax fit).  This
module derives them; `python -m fixed_budget_kv_gb300.exp2_poly` prints the
fp32 values written into csrc/common.cuh, and the CPU tests check the two
agree and that the error stays below the stated bound.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def _rel_err(c, x):
    return np.polyval(c[::-1], x) / np.exp2(x) - 1.0


def remez(degree: int = DEGREE, iters: int = 30) -> tuple[np.ndarray, float]:
    """Minimax coefficients (c0 .. c_degree) of 2^f on [LO, HI] for relative error,
    and the size of the equioscillating error."""
    n = degree + 2
    # Chebyshev extrema as the first reference
    k = np.arange(n)
    ref = (LO + HI) / 2 + (HI - LO) / 2 * -np.cos(np.pi * k / (n - 1))
    grid = np.linspace(LO, HI, 20001)
    E = 0.0
    c = np.zeros(degree + 1)
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i E 2^x_i  ->  unknowns c_0..c_d, E
        A = np.zeros((n, n))
        for i, xi in enumerate(ref):
            A[i, :degree + 1] = xi ** np.arange(degree + 1)
            A[i, degree + 1] = -((-1) ** i) * np.exp2(xi)
        sol = np.linalg.solve(A, np.exp2(ref))
        c, E = sol[:degree + 1], sol[degree + 1]
        err = _rel_err(c, grid)
        # new reference: the extremum of each sign run of the error
        sgn = np.sign(err)
        runs = np.split(np.arange(grid.size), np.nonzero(np.diff(sgn))[0] + 1)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        if len(ext) < n:
            break
        # keep n consecutive extrema containing the largest one
        ext = np.array(ext)
        best = int(np.argmax(np.abs(err[ext])))
        start = min(max(0, best - n // 2), len(ext) - n)
        ref = grid[ext[start:start + n]]
    return c, float(abs(E))


def fp32_coefficients() -> list[float]:
    c, _ = remez()
    return [float(np.float32(v)) for v in c]


def max_rel_error_fp32(coef=None, samples: int = 200001) -> float:
    """Largest relative error of p(f) with fp32 coefficients (evaluated in fp64)."""
    c = np.array(fp32_coefficients() if coef is None else coef, dtype=np.float64)
    x = np.linspace(LO, HI, samples)
    return float(np.abs(_rel_err(c, x)).max())


if __name__ == "__main__":
    c, e = remez()
    print("minimax relative error", e)
    for i, v in enumerate(fp32_coefficients()):
        print(f"c{i} = {v!r}  ({np.float32(v).view(np.uint32):#010x})")
    print("with fp32 coefficients", max_rel_error_fp32())
