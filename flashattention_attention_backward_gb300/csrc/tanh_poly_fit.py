"""Fits the polynomial of csrc/softcap_math.cuh: tanh(u) = u + u^3 Q(u^2) on
|u| <= 1, Q of degree 5, minimising the largest absolute error of tanh.

Method: Lawson's algorithm (iteratively reweighted least squares converging
to the minimax fit) on a dense grid, in float64. The coefficients are then
rounded to float32 and the fp32 evaluation the kernels perform (Horner with
fused multiply-adds, then t = (u x) q + u) is checked against float64 tanh.

Run: python csrc/tanh_poly_fit.py   (prints the coefficients and the error)
"""
import numpy as np

U0 = 1.0
DEG = 5


def fit(u0=U0, deg=DEG, iters=60):
    u = np.linspace(1e-4, u0, 40001)
    x = u * u
    target = (np.tanh(u) - u) / u ** 3
    w = u ** 3  # the absolute error of tanh is u^3 times that of Q
    V = np.vander(x, deg + 1, increasing=True)
    wt = np.ones_like(u)
    for _ in range(iters):
        A = V * (w * wt)[:, None]
        c, *_ = np.linalg.lstsq(A, target * w * wt, rcond=None)
        err = np.abs((V @ c - target) * w)
        wt = wt * err / err.mean() + 1e-3  # Lawson's update: weight by the error
        wt /= wt.mean()
    return c


def eval_fp32(c32, u):
    """The kernels' evaluation in float32 (fma rounding emulated in float64,
    which is exact for one product plus one addend of float32 values)."""
    u = np.asarray(u, dtype=np.float32)
    x = (u.astype(np.float64) * u).astype(np.float32)
    q = np.full_like(u, c32[-1])
    for ck in c32[-2::-1]:
        q = (q.astype(np.float64) * x + np.float64(ck)).astype(np.float32)
    ux = (u.astype(np.float64) * x).astype(np.float32)
    return (ux.astype(np.float64) * q + u).astype(np.float32)


def max_abs_error(c32, u0=U0):
    u = np.linspace(-u0, u0, 800001).astype(np.float32)
    return float(np.abs(eval_fp32(c32, u).astype(np.float64) - np.tanh(u.astype(np.float64))).max())


if __name__ == "__main__":
    c32 = fit().astype(np.float32)
    for i, ck in enumerate(c32):
        print("  C%d = %.9ef" % (i, ck))
    print("max |error| of the fp32 evaluation on |u| <= %g: %.3e" % (U0, max_abs_error(c32)))
