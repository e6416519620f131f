"""Derivation of the codebook constants hard-coded in ``kvq_codebooks.cuh``.

The TQ4 codec uses the 16-level, and the K2 codec the 4-level, minimum-MSE
(Lloyd-Max) quantizer of N(0,1).  The library stores them as f32 bit patterns;
this script is how those patterns were obtained.  It solves the two optimality
conditions directly with a root finder on the positive half-line (the optimum
is odd-symmetric, so for an even level count the middle threshold is 0):

    level k  = E[X | t_k < X < t_(k+1)]         (centroid condition)
    t_k      = (level_(k-1) + level_k) / 2       (nearest-neighbour condition)

Levels and thresholds are rounded once from float64 to float32.

Run:  python gen_codebook.py   (prints the C initialisers)
"""
import numpy as np
from scipy import optimize, stats


def solve(levels: int) -> np.ndarray:
    half = levels // 2

    def residual(pos):
        c = np.concatenate([-pos[::-1], pos])
        t = np.concatenate([[-np.inf], (c[1:] + c[:-1]) / 2, [np.inf]])
        a, b = t[half:-1], t[half + 1:]
        mass = stats.norm.cdf(b) - stats.norm.cdf(a)
        centroid = (stats.norm.pdf(a) - stats.norm.pdf(b)) / mass
        return centroid - pos

    start = np.linspace(0.5, 2.0, half) * (2.7 if levels > 4 else 1.0)
    pos = optimize.fsolve(residual, start, xtol=1e-15)
    pos = optimize.fsolve(residual, pos, xtol=1e-15)
    return np.concatenate([-pos[::-1], pos])


def emit(name: str, c: np.ndarray) -> None:
    lv = c.astype(np.float32)
    th = ((c[1:] + c[:-1]) / 2).astype(np.float32)
    hx = lambda a: ", ".join(f"0x{int(v):08x}u" for v in a.view(np.uint32))
    print(f"// {name}: levels {np.array2string(lv, precision=6)}")
    print(f"{name}_LEVELS_BITS = {{ {hx(lv)} }};")
    print(f"{name}_THRESH_BITS = {{ {hx(th)} }};")


if __name__ == "__main__":
    emit("TQ4", solve(16))
    emit("K2", solve(4))
