"""Derivation of the PolarQuant angle tables in ``pq_codebook.inc``.

PolarQuant (Han et al., "PolarQuant: Quantizing KV Caches with Polar
Transformation", 2025) turns a rotated block into a tree of (radius, angle)
pairs and quantizes every angle with its level's codebook.  After the random
rotation the level-1 angles are uniform on the circle; a level-l angle (l >= 2)
is the angle between two independent k-dimensional Gaussian halves, k =
2^(l-1), with density proportional to sin(2 psi)^(k-1) on [0, pi/2]
(equivalently sin^2(psi) ~ Beta(k/2, k/2)).

Per width b (2..6) and level l (1..10, blocks up to 1024):

* level 1: 2^b uniform cells of the circle, reconstructed at their centres;
  the encoder decides within a quadrant against the 2^(b-2) - 1 boundaries
  j pi / 2^(b-1);
* level l >= 2: the minimum-MSE (Lloyd-Max) quantizer of the density, found
  here by solving the two optimality conditions directly
      level q = E[psi | t_(q-1) < psi < t_q],   t_q = (level q + level q+1) / 2
  with scipy's root finder and the analytic (tridiagonal) Jacobian, from the
  levels at the quantiles of f^(1/3) (the high-resolution optimum; f^(1/3) is
  the same family with k' = (k + 2) / 3, so the quantiles come from the
  inverse regularized incomplete beta function).  Cell integrals by adaptive
  quadrature.

The kernels hold cos and sin of every centroid and threshold, each rounded
once from float64 to float32.

Run:  python gen_pq_codebook.py > pq_codebook.inc
"""
import math
import sys

import numpy as np
from scipy import integrate, optimize, special

MAX_LEVEL = 10
BITS = range(2, 7)


def density(k):
    return lambda t: math.sin(2.0 * t) ** (k - 1)


def cell(k, a, b):
    f = density(k)
    pts = [math.pi / 4] if a < math.pi / 4 < b else None
    F = integrate.quad(f, a, b, epsabs=0, epsrel=2e-14, limit=400, points=pts)[0]
    M = integrate.quad(lambda t: t * f(t), a, b, epsabs=0, epsrel=2e-14, limit=400, points=pts)[0]
    return F, M


def start(k, L):
    kp = (k + 2) / 3.0
    u = special.betaincinv(kp / 2, kp / 2, (np.arange(L) + 0.5) / L)
    return np.arcsin(np.sqrt(u))


def lloyd_max(k, L):
    f = density(k)

    def conditions(c):
        th = 0.5 * (c[1:] + c[:-1])
        edges = np.concatenate([[0.0], th, [math.pi / 2]])
        g = np.empty(L)
        J = np.zeros((L, L))
        for q in range(L):
            F, M = cell(k, edges[q], edges[q + 1])
            mu = M / F
            g[q] = mu - c[q]
            da = f(edges[q]) * (mu - edges[q]) / F if q > 0 else 0.0
            db = f(edges[q + 1]) * (edges[q + 1] - mu) / F if q + 1 < L else 0.0
            if q > 0:
                J[q, q - 1] = 0.5 * da
            if q + 1 < L:
                J[q, q + 1] = 0.5 * db
            J[q, q] = 0.5 * (da + db) - 1.0
        return g, J

    sol = optimize.root(conditions, start(k, L), jac=True, method="hybr", options={"xtol": 1e-15})
    c = sol.x
    resid = np.max(np.abs(conditions(c)[0]))
    if resid > 1e-13:
        raise RuntimeError(f"k={k} L={L}: residual {resid}")
    return c, 0.5 * (c[1:] + c[:-1])


def f32_bits(v):
    return int(np.float32(v).view(np.uint32))


def tables():
    cent, thr, quad_th = {}, {}, {}
    for b in BITS:
        L = 1 << b
        step = 2 * math.pi / L
        cent[b] = {1: (np.arange(L) + 0.5) * step}
        thr[b] = {}
        for level in range(2, MAX_LEVEL + 1):
            c, t = lloyd_max(1 << (level - 1), L)
            cent[b][level] = c
            thr[b][level] = t
        quad_th[b] = np.arange(1, L // 4) * math.pi / (1 << (b - 1))
    return cent, thr, quad_th


def emit(out=sys.stdout):
    cent, thr, quad_th = tables()
    w = out.write
    w("// PolarQuant angle tables: cos and sin of every centroid and decision threshold,\n")
    w("// f32 bit patterns, written by gen_pq_codebook.py (see its docstring for the\n")
    w("// derivation).  Per width b = 2..6:\n")
    w("//   kPqCent:   levels 1..10, 2^b centroids each, (cos, sin) pairs\n")
    w("//   kPqThresh: levels 2..10, 2^b - 1 thresholds each, then the level-1\n")
    w("//              in-quadrant thresholds j pi / 2^(b-1), j = 1 .. 2^(b-2) - 1\n")
    w("// kPqCentOff[b] / kPqThreshOff[b] give the first pair of width b.\n")
    cent_words, th_words, coff, toff = [], [], [], []
    for b in BITS:
        coff.append(len(cent_words) // 2)
        toff.append(len(th_words) // 2)
        for level in range(1, MAX_LEVEL + 1):
            for v in cent[b][level]:
                cent_words += [f32_bits(math.cos(v)), f32_bits(math.sin(v))]
        for level in range(2, MAX_LEVEL + 1):
            for v in thr[b][level]:
                th_words += [f32_bits(math.cos(v)), f32_bits(math.sin(v))]
        for v in quad_th[b]:
            th_words += [f32_bits(math.cos(v)), f32_bits(math.sin(v))]
    w(f"constexpr int kPqCentOff[7] = {{0, 0, {', '.join(map(str, coff))}}};\n")
    w(f"constexpr int kPqThreshOff[7] = {{0, 0, {', '.join(map(str, toff))}}};\n")
    w(f"constexpr int kPqCentWords = {len(cent_words)};\n")
    w(f"constexpr int kPqThreshWords = {len(th_words)};\n")
    w("// The word lists, as macros: one list initializes both the device tables and\n")
    w("// the host copies.\n")
    for name, words in (("KVQ_PQ_CENT_WORDS", cent_words), ("KVQ_PQ_THRESH_WORDS", th_words)):
        w(f"#define {name} \\\n")
        lines = [", ".join(f"0x{x:08x}u" for x in words[i:i + 8]) for i in range(0, len(words), 8)]
        w(", \\\n".join("    " + ln for ln in lines) + "\n")

if __name__ == "__main__":
    emit()
