"""Fit the polynomial used by the FMA-pipe 2^x (exp2_fma in sv_device.cuh).

Method: 2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]
(Cody and Waite's argument reduction), and 2^f approximated by a degree-5
polynomial whose maximum RELATIVE error on [-1/2, 1/2] is minimised with the
Remez exchange algorithm (equioscillation on 7 reference points; all six
coefficients free).

Run: python fit_exp2_poly.py  -> prints the coefficients (float32) and the
relative error of the float32-rounded polynomial evaluated in float64.
"""
import numpy as np

DEG = 5
LO, HI = -0.5, 0.5


def remez_relative(deg=DEG, iters=30):
    f = np.exp2
    n = deg + 2  # reference points: deg+1 coefficients and the levelled error
    ref = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(LO, HI, 200001)
    c = None
    for _ in range(iters):
        A = np.zeros((n, deg + 2))
        for i, x in enumerate(ref):
            # (sum_j c_j x^j - 2^x) / 2^x = (-1)^i E
            for j in range(deg + 1):
                A[i, j] = x ** j / f(x)
            A[i, deg + 1] = -((-1) ** i)
        sol = np.linalg.solve(A, np.ones(n))
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - f(grid)) / f(grid)
        # new reference: the largest |error| between consecutive sign changes
        idx, best, sign = [], 0, np.sign(err[0])
        for k in range(1, grid.size):
            s = np.sign(err[k])
            if s == sign or s == 0:
                if abs(err[k]) > abs(err[best]):
                    best = k
            else:
                idx.append(best)
                best, sign = k, s
        idx.append(best)
        while len(idx) > n:
            idx.pop(0 if abs(err[idx[0]]) < abs(err[idx[-1]]) else -1)
        if len(idx) == n:
            ref = grid[idx]
    return c, np.abs(err).max()


def main():
    c, e = remez_relative()
    c32 = c.astype(np.float32)
    grid = np.linspace(LO, HI, 400001)
    rel = np.abs(np.polyval(c32.astype(np.float64)[::-1], grid) / np.exp2(grid) - 1).max()
    print("coefficients c0..c5 (float32):")
    for i, v in enumerate(c32):
        print(f"  c{i} = {float(v)!r}")
    print(f"max relative error: exact coefficients {e:.3e}, float32 coefficients {rel:.3e}")


if __name__ == "__main__":
    main()
