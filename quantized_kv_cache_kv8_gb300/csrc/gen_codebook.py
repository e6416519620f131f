"""Derivation of the codebook constants hard-coded in ``kvq_internal.cuh`` (kTq4LevelBits, kTq4ThreshBits, kK2LevelBits, kK2ThreshBits).

The TQ4 codec uses the 16-level, and the K2 codec the 4-level, minimum-MSE
(Lloyd-Max) quantizer of N(0,1).  The library stores them as f32 bit patterns;
this script is how those patterns were obtained.  It solves the two optimality
conditions directly with a root finder on the positive half-line (the optimum
is odd-symmetric, so for an even level count the middle threshold is 0):

    level k  = E[X | t_k < X < t_(k+1)]         (centroid condition)
    t_k      = (level_(k-1) + level_k) / 2       (nearest-neighbour condition)

Levels and thresholds are rounded once from float64 to float32.

The tensor-core TQ4 kernel multiplies the 16 levels by one scale before
rounding them to f16 (the MMA operand type), chosen so that all of them land
close to f16 values; --level-scale repeats that search: random scales in
[1, 2), then a fine grid around the best, minimising the largest relative
rounding error over the levels.

The tensor-core K2/V4 kernel does the same for the 4 K levels (searched over
the 1024 f16 values in [1, 2), so that the scale itself is exact in f16):
--k2-level-scale.

Run:  python gen_codebook.py   (prints the C initialisers)
      python gen_codebook.py --level-scale
      python gen_codebook.py --k2-level-scale
"""
import sys

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


def level_scale_error(g: np.ndarray, levels_f32: np.ndarray) -> np.ndarray:
    x = g[:, None] * np.abs(levels_f32.astype(np.float64))[None, :]
    return np.max(np.abs(x.astype(np.float16).astype(np.float64) - x) / x, axis=1)


def level_scale(levels: np.ndarray, seed: int = 1) -> tuple[float, float]:
    lv = levels.astype(np.float32)
    rng = np.random.default_rng(seed)
    cand = []
    for _ in range(20):
        g = 1.0 + rng.random(2_000_000)
        e = level_scale_error(g, lv)
        i = np.argsort(e)[:20]
        cand += list(zip(e[i], g[i]))
    cand.sort()
    best = cand[0]
    for _, g0 in cand[:50]:
        g = g0 + np.linspace(-2e-5, 2e-5, 400001)
        e = level_scale_error(g, lv)
        i = int(np.argmin(e))
        if e[i] < best[0]:
            best = (e[i], g[i])
    return float(np.float32(best[1])), float(best[0])


if __name__ == "__main__":
    if "--k2-level-scale" in sys.argv:
        lv = solve(4).astype(np.float32)
        cand = np.array([1.0 + k / 1024 for k in range(1024)], np.float64)
        best = None
        for g in cand:
            x = np.abs(lv[2:]).astype(np.float64) * g
            h = (np.abs(lv[2:]) * np.float32(g)).astype(np.float32).astype(np.float16).astype(np.float64)
            e = float(np.max(np.abs(h - x) / x))
            if best is None or e < best[0]:
                best = (e, g)
        print(f"K2 level scale {float(best[1])!r} (exact in f16), largest relative f16 rounding error {best[0]:.3e}")
    elif "--level-scale" in sys.argv:
        g, err = level_scale(solve(16))
        print(f"TQ4 level scale {g!r} (f32), largest relative f16 rounding error {err:.3e}")
    else:
        emit("TQ4", solve(16))
        emit("K2", solve(4))
