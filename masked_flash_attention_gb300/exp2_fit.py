"""Coefficients of the cubic that the prefill kernel uses for part of its
base-2 exponentials.

The kernel splits v = n + f with n = floor(v) and f in [0, 1), evaluates
2^f ~ 1 + f (c1 + f (c2 + f c3)) with fused multiply-adds in fp32 and adds n
to the exponent field of the result.  p(0) = 1 is fixed, so that exact powers
of two come out exact.  c1..c3 minimise the largest relative error
max |p(f) / 2^f - 1| over [0, 1]: a discrete Chebyshev (minimax) fit, solved
as a linear program over a dense grid of f.

Running this file prints the coefficients and the bound; the test suite
re-runs the fit and checks that the constants in the kernel source match it.
"""
import numpy as np


def fit(degree: int = 3, n_grid: int = 4097):
    """Return (coefficients c1..c_degree, max relative error on the grid)."""
    from scipy.optimize import linprog

    f = np.linspace(0.0, 1.0, n_grid)
    w = np.exp2(-f)  # relative error = (p(f) - 2^f) / 2^f
    # variables: c1..c_deg, t ; minimise t
    A = np.stack([f ** k * w for k in range(1, degree + 1)], axis=1)
    r = 1.0 - (1.0 * w)  # p(f)/2^f - 1 = A c + w - 1
    ones = np.ones((n_grid, 1))
    # A c + (w - 1) <= t   and   -(A c + (w - 1)) <= t
    A_ub = np.vstack([np.hstack([A, -ones]), np.hstack([-A, -ones])])
    b_ub = np.concatenate([r, -r])
    c = np.zeros(degree + 1)
    c[-1] = 1.0
    res = linprog(c, A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * (degree + 1), method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return res.x[:degree], float(res.x[degree])


def exp2_fp32(v: np.ndarray, coeffs) -> np.ndarray:
    """The kernel's steps in fp32 (clamp, floor, fraction, Horner, exponent add)."""
    v = np.maximum(np.asarray(v, dtype=np.float32), np.float32(-127.0))
    n = np.floor(v).astype(np.float32)
    f = (v - n).astype(np.float32)
    q = np.float32(coeffs[-1])
    for ck in reversed(list(coeffs[:-1])):
        q = (q * f + np.float32(ck)).astype(np.float32)
    q = (q * f + np.float32(1.0)).astype(np.float32)
    bits = q.view(np.int32) + (n.astype(np.int32) << 23)
    return bits.view(np.float32)


if __name__ == "__main__":
    cs, err = fit()
    for k, ck in enumerate(cs, 1):
        print("c%d = %.9e  (fp32 %r)" % (k, ck, np.float32(ck)))
    print("max relative error on the grid: %.3e" % err)
