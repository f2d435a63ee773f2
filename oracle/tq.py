"""TurboQuant Q_mse codebook for the TQ4 cache variant (test infrastructure).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU legs may import
this module; the product library computes its own codebook and shares nothing
with this file.

Source: "TurboQuant 완전 정리" (juhoplayground.github.io), sections "랜덤 회전과
Beta 분포" and "Lloyd-Max 스칼라 양자화 (Q_mse)".  After a random rotation, one
coordinate X of a unit vector in R^d has the density

    f(x) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) * (1 - x^2)^((d-3)/2),  |x| <= 1

(X^2 ~ Beta(1/2, (d-1)/2)), and the Q_mse codebook is the Lloyd-Max quantiser
(continuous k-means) of that density with 2^b levels, computed once from the
pdf, without data.

Readings of this library (listed in the design doc):
  T1  the Lloyd-Max fixed point is found in fp64 by alternating the two
      optimality conditions (boundaries at centroid midpoints, centroids at
      cell conditional means) on the half-line [0, 1] and mirroring, so the
      codebook is exactly symmetric; cell masses use the regularised
      incomplete beta function, first moments their closed form
      int x (1-x^2)^k dx = -(1-x^2)^(k+1) / (2(k+1)).
  T2  the oracle quantises to, and reconstructs with, the fp64 centroids;
      `codebook` also gives their f16 roundings and the fp32 roundings of the
      midpoints, the form in which the library stores its table (checked
      against it exactly).
"""
import math

import numpy as np
from scipy import special


def pdf_const(d: int) -> float:
    """Normalising constant Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2))."""
    return math.exp(math.lgamma(d / 2.0) - math.lgamma((d - 1) / 2.0)) / math.sqrt(math.pi)


def pdf(x, d: int):
    x = np.asarray(x, np.float64)
    return pdf_const(d) * np.power(np.clip(1.0 - x * x, 0.0, None), (d - 3) / 2.0)


def mass(a: float, b: float, d: int) -> float:
    """P(a <= X <= b) for 0 <= a <= b <= 1: half the difference of
    I_{x^2}(1/2, (d-1)/2), since P(|X| <= x) = I_{x^2}(1/2, (d-1)/2)."""
    return 0.5 * (special.betainc(0.5, (d - 1) / 2.0, b * b) - special.betainc(0.5, (d - 1) / 2.0, a * a))


def first_moment(a: float, b: float, d: int) -> float:
    """int_a^b x f(x) dx (closed form)."""
    k1 = (d - 1) / 2.0  # k + 1 with k = (d - 3) / 2
    return pdf_const(d) * ((1.0 - a * a) ** k1 - (1.0 - b * b) ** k1) / (2.0 * k1)


def lloyd_max(d: int, bits: int, max_iter: int = 200000) -> np.ndarray:
    """Ascending fp64 centroids c_0 < ... < c_{2^bits - 1} of the Lloyd-Max
    quantiser of f (T1).  Symmetric: c_{L-1-i} = -c_i.  Iterates until no
    centroid moves by more than 1e-14 standard deviations (1/sqrt(d))."""
    L = 1 << bits
    h = L // 2
    sigma = 1.0 / math.sqrt(d)
    k1 = (d - 1) / 2.0
    C = pdf_const(d)
    # positive half: start on a uniform grid over [0, 3 sigma]
    c = np.array([(i + 0.5) * 3.0 * sigma / h for i in range(h)], np.float64)
    for _ in range(max_iter):
        edges = np.concatenate(([0.0], 0.5 * (c[:-1] + c[1:]), [1.0]))
        cdf = special.betainc(0.5, k1, edges * edges)        # P(|X| <= edge)
        m = 0.5 * (cdf[1:] - cdf[:-1])                        # cell masses on [0, 1]
        fm = C * ((1.0 - edges[:-1] ** 2) ** k1 - (1.0 - edges[1:] ** 2) ** k1) / (2.0 * k1)
        new = fm / m                                          # conditional means
        moved = np.max(np.abs(new - c))
        c = new
        if moved <= 1e-14 * sigma:
            break
    return np.concatenate((-c[::-1], c))


def distortion(c: np.ndarray, d: int) -> float:
    """E||x - x_hat||^2 of a unit vector quantised coordinate-wise with the
    centroids c: d times the per-coordinate MSE int (x - c(x))^2 f(x) dx."""
    L = len(c)
    edges = np.concatenate(([-1.0], 0.5 * (c[:-1] + c[1:]), [1.0]))
    mse = 0.0
    k1 = (d - 1) / 2.0
    C = pdf_const(d)
    for i in range(L):
        a, b = edges[i], edges[i + 1]
        # int (x - c)^2 f = int x^2 f - 2 c int x f + c^2 int f; int x^2 f by quadrature
        xs, ws = np.polynomial.legendre.leggauss(200)
        x = 0.5 * (b - a) * xs + 0.5 * (b + a)
        m2 = 0.5 * (b - a) * np.sum(ws * x * x * pdf(x, d))
        m1 = first_moment(a, b, d) if a >= 0 else -first_moment(-b, -a, d) if b <= 0 else \
            first_moment(0.0, b, d) - first_moment(0.0, -a, d)
        m0 = (mass(a, b, d) if a >= 0 else mass(-b, -a, d) if b <= 0 else mass(0.0, b, d) + mass(0.0, -a, d))
        mse += m2 - 2.0 * c[i] * m1 + c[i] * c[i] * m0
    return d * mse


def codebook(d: int, bits: int = 4):
    """(f16 roundings of the non-negative centroids, ascending, as float64;
    fp32 roundings of the midpoints tau_0 < ... < tau_{L-2}) per T2."""
    c = lloyd_max(d, bits)
    L = len(c)
    mags = np.array([float(np.float16(v)) for v in c[L // 2:]], np.float64)
    tau = np.array([np.float32(0.5 * (c[j] + c[j + 1])) for j in range(L - 1)], np.float32)
    return mags, tau
