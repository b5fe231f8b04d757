"""Coefficients of the FMA-pipe exp2 used by the block-wise kernels' exp split
(blockwise_common.cuh, ex2_fma).

2^x is computed as 2^n * p(f) with n = rint(x), f = x - n in [-1/2, 1/2] and
p(f) = 1 + f*(c1 + f*(c2 + f*(c3 + f*c4))): a polynomial with p(0) = 1
exactly whose maximum relative error |p(f) - 2^f| / 2^f on [-1/2, 1/2] is as
small as possible.  The coefficients come from the Remez exchange algorithm
(E. Remez, 1934) applied to q(f) = (2^f - 1) / f with weight |f| / 2^f, so
that the weighted error of q is the relative error of p: solve for q and the
levelled error E on a reference set of deg + 1 points, move the reference to
the extrema of the new error curve, repeat.  The result is rounded to fp32.

Run as a script to print the coefficients as C++ hex-float literals and the
maximum relative error of the fp32 polynomial; tests re-derive them and
compare with the constants in the header.  Needs mpmath.
"""
import numpy as np

DEGREE = 4


def remez_exp2(degree=DEGREE, iterations=30, grid=8000):
    """fp32 coefficients [1, c1, ..., c_degree] of p and the Remez levelled error."""
    import mpmath as mp
    mp.mp.dps = 40
    nq = degree              # q has degree - 1 + 1 = degree coefficients
    n_ref = nq + 1

    def target(f):           # q's target (2^f - 1) / f, ln 2 at f = 0
        return (mp.power(2, f) - 1) / f if f != 0 else mp.log(2)

    def weight(f):
        return abs(f) / mp.power(2, f)

    # initial reference: Chebyshev points of [-1/2, 1/2], moved off 0 (where the weight vanishes)
    ref = [mp.mpf("0.5") * mp.cos(mp.pi * (i + mp.mpf("0.5")) / n_ref) for i in range(n_ref)][::-1]
    ref = [x if abs(x) > mp.mpf("1e-3") else mp.mpf("1e-3") for x in ref]
    xs = [mp.mpf(-0.5) + mp.mpf(k) / grid for k in range(grid + 1)]
    coef, level = None, None
    for _ in range(iterations):
        a = mp.matrix(n_ref, n_ref)
        b = mp.matrix(n_ref, 1)
        for i, x in enumerate(ref):
            for j in range(nq):
                a[i, j] = x ** j
            a[i, nq] = (-1) ** i / weight(x)
            b[i] = target(x)
        sol = mp.lu_solve(a, b)
        coef = [sol[j] for j in range(nq)]
        level = abs(sol[nq])

        def weighted_err(x):  # weight * (q - target): |it| is p's relative error, its sign that of q's error
            if x == 0:
                return mp.mpf(0)
            return weight(x) * (sum(c * x ** j for j, c in enumerate(coef)) - target(x))

        # new reference: the largest |error| of each run of one sign
        runs = []
        for x in xs:
            e = weighted_err(x)
            if e == 0:
                continue
            sign = 1 if e > 0 else -1
            if runs and runs[-1][0] == sign:
                if abs(e) > runs[-1][2]:
                    runs[-1][1], runs[-1][2] = x, abs(e)
            else:
                runs.append([sign, x, abs(e)])
        if len(runs) < n_ref:
            break
        best = max(range(len(runs) - n_ref + 1), key=lambda k: min(r[2] for r in runs[k:k + n_ref]))
        new_ref = [r[1] for r in runs[best:best + n_ref]]
        if all(abs(u - v) < mp.mpf(1) / grid for u, v in zip(new_ref, ref)):
            break
        ref = new_ref
    coeffs = [1.0] + [float(np.float32(float(c))) for c in coef]
    return coeffs, float(level)


def fp32_relative_error(coeffs, n=400001):
    """Max relative error of the fp32-coefficient polynomial on [-1/2, 1/2] (fp64 evaluation)."""
    f = np.linspace(-0.5, 0.5, n)
    p = np.zeros_like(f)
    for c in reversed(coeffs):
        p = p * f + c
    return float(np.max(np.abs(p - np.exp2(f)) / np.exp2(f)))


if __name__ == "__main__":
    c, level = remez_exp2()
    for i, v in enumerate(c):
        print(f"c{i} = {float(np.float32(v)).hex()}f  ({v!r})")
    print(f"levelled relative error {level:.4e}; fp32 coefficients {fp32_relative_error(c):.4e}")
