"""Pins of the oracle's scalar and row codecs against sources other than itself.

Each test names what it pins to: a published table or specification (golden
fixtures), a library routine (numpy casts, an explicit Hadamard matrix), a
brute-force search, or a number the pages print.
"""
import math

import numpy as np
import pytest

from conftest import golden_lines
from quantized_kv_cache_kv8_gb300 import synth


# -- fp8 e4m3 -----------------------------------------------------------------

def _grid_pos():
    """Positive e4m3 magnitudes for codes 0x00..0x7E built by enumerating the
    format's fields the way the OCP specification describes them (independent
    of the oracle's decoder)."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def _brute_e4m3(u):
    """Nearest grid value by exhaustive search; ties to the even code; >=448 saturates."""
    grid = _grid_pos()
    a = abs(float(u))
    sign = 0x80 if math.copysign(1.0, float(u)) < 0 else 0
    if a >= 448.0:
        return sign | 0x7E
    d = np.abs(grid - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return sign | code


def test_e4m3_spec_values(oracle):
    for line in golden_lines("e4m3_values.txt"):
        code, val = line.split()
        v = oracle.e4m3_value(int(code, 16))
        assert v == float(val), (code, v, val)
        assert math.copysign(1.0, v) == math.copysign(1.0, float(val))


def test_e4m3_grid_monotone_and_complete(oracle):
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert vals[-1] == 448.0
    np.testing.assert_array_equal(np.array(vals), _grid_pos())


def test_e4m3_roundtrip_all_codes(oracle):
    for code in range(256):
        if code & 0x7F == 0x7F:
            continue                      # the NaN pattern is never produced
        v = oracle.e4m3_value(code)
        assert oracle.e4m3_encode(np.float32(v)) == code, hex(code)


def test_e4m3_midpoints_round_to_even(oracle):
    grid = _grid_pos()
    for c in range(0x7E):
        mid = np.float32((grid[c] + grid[c + 1]) / 2)
        assert float(mid) == (grid[c] + grid[c + 1]) / 2           # midpoints are exact in f32
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even
        assert oracle.e4m3_encode(-mid) == 0x80 | even


def test_e4m3_saturation(oracle):
    for u in [448.0, 448.5, 463.9, 464.0, 480.0, 1e6, 3.4e38, float("inf")]:
        assert oracle.e4m3_encode(np.float32(u)) == 0x7E
        assert oracle.e4m3_encode(np.float32(-u)) == 0xFE


def test_e4m3_brute_force_random(oracle):
    rng = np.random.default_rng(7)
    exps = rng.uniform(-14, 10, 4000)
    u = (rng.choice([-1, 1], 4000) * 2.0 ** exps).astype(np.float32)
    got = oracle.e4m3_encode_array(u)
    for x, g in zip(u, got):
        assert g == _brute_e4m3(x), (x, hex(g))


# -- IEEE binary16 ------------------------------------------------------------

def test_f16_matches_numpy_cast(oracle):
    rng = np.random.default_rng(3)
    x = np.concatenate([(rng.standard_normal(3000) * 2.0 ** rng.uniform(-26, 17, 3000)),
                        [0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e6, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]]
                       ).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_encode(v) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
    for h in list(range(0, 65536, 97)) + [0x7BFF, 0x0001, 0x8001, 0x3C00]:
        if (h & 0x7C00) == 0x7C00 and (h & 0x3FF):
            continue
        assert oracle.f16_value(h) == float(np.array([h], np.uint16).view(np.float16)[0])


# -- splitmix64 ---------------------------------------------------------------

def test_splitmix64_published_outputs(oracle):
    for line in golden_lines("splitmix64.txt"):
        seed, outs = line.split(":")
        want = [int(w, 0) for w in outs.split()]
        assert oracle.splitmix64(int(seed), len(want)) == want


def test_tq4_signs_follow_words(oracle):
    """Sign i of the 512 block is bit i%64 of splitmix64 word i//64; the 64 block uses word 8."""
    words = [int(w) for w in oracle.splitmix64(0, 9)]
    sig = oracle.tq4_signs(0, (512, 64))
    for i in range(576):
        w = words[i // 64] if i < 512 else words[8]
        j = i % 64
        assert sig[i] == (-1 if (w >> j) & 1 else 1)


# -- Lloyd-Max ----------------------------------------------------------------

def test_lloyd_max_matches_max_1960(oracle):
    from scipy import integrate, stats
    for line in golden_lines("lloyd_max_max1960.txt"):
        parts = line.split()
        n, mse_tab, levels = int(parts[0]), float(parts[1]), [float(v) for v in parts[2:]]
        c, mse, _ = oracle.lloyd_max(n)
        np.testing.assert_allclose(c[n // 2:], levels, atol=6e-4)
        np.testing.assert_allclose(c, -c[::-1], atol=0)                   # odd symmetry
        # the 1960 figures carry about three and a half significant digits
        assert abs(mse - mse_tab) / mse_tab < 1e-3
        # the levels are centroids of their cells (checked by quadrature, not by the solver)
        t = np.concatenate([[-np.inf], (c[1:] + c[:-1]) / 2, [np.inf]])
        for k in range(n):
            m1 = integrate.quad(lambda x: x * stats.norm.pdf(x), t[k], t[k + 1], epsabs=1e-13)[0]
            m0 = stats.norm.cdf(t[k + 1]) - stats.norm.cdf(t[k])
            assert abs(m1 / m0 - c[k]) < 1e-9
        # the MSE agrees with direct quadrature of (x - Q(x))^2
        q_mse = sum(integrate.quad(lambda x, ck=c[k]: (x - ck) ** 2 * stats.norm.pdf(x), t[k], t[k + 1],
                                   epsabs=1e-13)[0] for k in range(n))
        assert abs(q_mse - mse) < 1e-9


def test_codebook_f32_rounding(oracle):
    c, _, _ = oracle.lloyd_max(16)
    lv, th = oracle.tq4_codebook()
    np.testing.assert_array_equal(lv, c.astype(np.float32))
    np.testing.assert_array_equal(th, ((c[1:] + c[:-1]) / 2).astype(np.float32))
    assert th[7] == 0.0


# -- FWHT and the rotation ----------------------------------------------------

def _sylvester(n):
    H = np.array([[1.0]])
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


@pytest.mark.parametrize("n", [2, 4, 8, 64, 512])
def test_fwht_equals_hadamard_matrix(oracle, n):
    rng = np.random.default_rng(n)
    v = rng.standard_normal((3, n))
    np.testing.assert_allclose(oracle.fwht(v), v @ _sylvester(n).T, rtol=0, atol=1e-11 * n)
    e0 = np.zeros(n, np.float32)
    e0[0] = 1
    np.testing.assert_array_equal(oracle.fwht(e0), np.ones(n, np.float32))
    ints = rng.integers(-50, 50, n).astype(np.float32)
    np.testing.assert_array_equal(oracle.fwht(oracle.fwht(ints)), ints * n)     # H H = n I, exact


def test_rotation_is_orthogonal(oracle):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((20, 576))
    y = oracle.tq4_rotate(x, seed=5)
    np.testing.assert_allclose(np.linalg.norm(y[:, :512], axis=1), np.linalg.norm(x[:, :512], axis=1), rtol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(y[:, 512:], axis=1), np.linalg.norm(x[:, 512:], axis=1), rtol=1e-12)
    np.testing.assert_allclose(oracle.tq4_rotate(y, seed=5, inverse=True), x, atol=1e-12)
    # rotate(e_0) = sigma_0 * (1/sqrt n) * ones over the first block
    e = np.zeros((1, 576))
    e[0, 0] = 1
    r = oracle.tq4_rotate(e, seed=5)
    s0 = oracle.tq4_signs(5, (512, 64))[0]
    np.testing.assert_allclose(r[0, :512], s0 / math.sqrt(512), rtol=1e-15)
    np.testing.assert_array_equal(r[0, 512:], 0)


# -- KV8 row codec ------------------------------------------------------------

def test_kv8_scale_and_codes_by_definition(oracle):
    x = synth.mla_rows(11, 40)
    codes, scales = oracle.kv8_encode(x)
    assert codes.shape == (40, 576) and scales.shape == (40, 2)
    for t in range(40):
        for b, (lo, hi) in enumerate([(0, 512), (512, 576)]):
            amax = np.max(np.abs(x[t, lo:hi]))
            s = np.float32(amax) / np.float32(448.0)                 # numpy IEEE f32 division
            assert scales[t, b] == s
            u = (x[t, lo:hi] / s).astype(np.float32)
            for i in range(0, hi - lo, 7):
                assert codes[t, lo + i] == _brute_e4m3(u[i])
            vals = np.array([oracle.e4m3_value(c) for c in codes[t, lo:hi]])
            assert np.max(np.abs(vals)) == 448.0


def test_kv8_inert_and_tiny_blocks(oracle):
    x = np.zeros((3, 576), np.float32)
    x[1, 600 - 576 + 512] = 3.0                                 # only the rope block is live
    x[2, 5] = 1e-44                                              # amax/448 underflows to 0
    codes, scales = oracle.kv8_encode(x)
    assert np.all(codes[0] == 0) and np.all(scales[0] == 0)
    assert scales[1, 0] == 0 and np.all(codes[1, :512] == 0) and scales[1, 1] == np.float32(3.0) / np.float32(448)
    assert scales[2, 0] == 0 and np.all(codes[2] == 0)
    xh = oracle.kv8_decode(codes, scales)
    assert np.all(xh[0] == 0) and xh[1, 536] == pytest.approx(3.0, rel=1e-6)


def test_kv8_single_scale_layout(oracle):
    x = synth.mla_rows(2, 5)
    codes, scales = oracle.kv8_encode(x, bdims=(576,))
    assert scales.shape == (5, 1)
    np.testing.assert_array_equal(scales[:, 0], np.max(np.abs(x), axis=1) / np.float32(448))


def test_kv8_reconstruction_error_bound(oracle):
    x = synth.mla_rows(12, 64)
    codes, scales = oracle.kv8_encode(x)
    xh = oracle.kv8_decode(codes, scales)
    for b, (lo, hi) in enumerate([(0, 512), (512, 576)]):
        s = scales[:, b:b + 1].astype(np.float64)
        u = np.abs(x[:, lo:hi]) / s
        # half a grid step: 2^-4 relative in the normal range, 2^-10 absolute (in units of s) below it
        bound = np.maximum(u * 2.0 ** -4, 2.0 ** -10) * s * (1 + 1e-6)
        assert np.all(np.abs(xh[:, lo:hi] - x[:, lo:hi]) <= bound)


def test_byte_counts_from_the_pages():
    counts = {l.split()[0]: float(l.split()[1]) for l in golden_lines("page_byte_counts.txt")}
    kv8_row = 576 + 2 * 4
    tq4_row = 576 // 2 + 2 * 4
    assert (kv8_row, tq4_row) == (584, 296)
    assert round(2304 / kv8_row, 1) == counts["kv8_ratio_vs_f32"]
    assert round(2304 / tq4_row, 1) == counts["tq4_ratio_vs_f32"]


# -- TQ4 row codec ------------------------------------------------------------

def test_tq4_distortion_near_page_value(oracle):
    """The KV cache quantization page (Why rotated-int4) and its CPU split both
    quote ~0.096 rel-L2 for rotated-int4 at 4 bits on Gaussian rows."""
    z = synth.normal(21, 9, 4000 * 512).reshape(4000, 512).astype(np.float32)
    packed, scales = oracle.tq4_encode(z, bdims=(512,), seed=3)
    xh = oracle.tq4_decode(packed, scales, bdims=(512,), seed=3)
    rel = np.linalg.norm(xh - z, axis=1) / np.linalg.norm(z, axis=1)
    assert 0.090 <= rel.mean() <= 0.100, rel.mean()


def test_tq4_codes_are_nearest_levels(oracle):
    x = synth.mla_rows(13, 16)
    packed, scales = oracle.tq4_encode(x, seed=7)
    c, _, _ = oracle.lloyd_max(16)
    y = oracle.tq4_rotate(x.astype(np.float64), seed=7)
    for t in range(16):
        for b, (lo, hi) in enumerate([(0, 512), (512, 576)]):
            s = float(scales[t, b])
            n = hi - lo
            assert s == pytest.approx(np.linalg.norm(x[t, lo:hi].astype(np.float64)) / math.sqrt(n), rel=2e-7)
            for i in range(lo, hi, 5):
                code = (packed[t, i // 2] >> 4) if i % 2 else (packed[t, i // 2] & 15)
                u = y[t, i] / s
                d = np.abs(c - u)
                assert d[code] <= d.min() + 1e-5, (t, i)


def test_tq4_inert_rows(oracle):
    x = np.zeros((2, 576), np.float32)
    x[1, :512] = 1.0
    packed, scales = oracle.tq4_encode(x)
    assert np.all(scales[0] == 0) and np.all(packed[0] == 0)
    assert scales[1, 1] == 0 and np.all(packed[1, 256:] == 0)
    xh = oracle.tq4_decode(packed, scales)
    assert np.all(xh[0] == 0) and np.all(xh[1, 512:] == 0)


def test_tq4_refuses_non_power_of_two(oracle):
    """Both pages: a width that is not a power of two would make every row inert;
    the codec refuses instead, at every entry point."""
    for bd in [(576,), (500, 76), (512, 60), (1,)]:
        x = np.ones((2, sum(bd)), np.float32)
        assert oracle.tq4_encode_status(x, bd) == 2
        with pytest.raises(ValueError):
            oracle.tq4_decode(np.zeros((1, sum(bd) // 2), np.uint8), np.zeros((1, len(bd)), np.float32), bd)
        with pytest.raises(ValueError):
            oracle.tq4_rotate(np.zeros((1, sum(bd))), bd)
        with pytest.raises(ValueError):
            oracle.attn_method(2, np.zeros((1, sum(bd) // 2), np.uint8), np.zeros((1, len(bd)), np.float32),
                               np.zeros((1, sum(bd)), np.float32), 1.0, v_dim=min(bd), bdims=bd)


def test_tq4_scale_and_sign_invariance(oracle):
    """Scaling a row by a power of two scales only the stored scale (every f32
    step of the encoder is exact under such scaling); negating it mirrors every
    code k -> 15-k (the codebook and its thresholds are odd-symmetric)."""
    x = synth.mla_rows(14, 12)
    p0, s0 = oracle.tq4_encode(x, seed=4)
    for a in (0.25, 8.0, 2.0 ** 20):
        p1, s1 = oracle.tq4_encode((x * np.float32(a)).astype(np.float32), seed=4)
        np.testing.assert_array_equal(p1, p0)
        np.testing.assert_array_equal(s1, s0 * np.float32(a))
    pn, sn = oracle.tq4_encode(-x, seed=4)
    np.testing.assert_array_equal(sn, s0)
    lo, hi = p0 & 15, p0 >> 4
    np.testing.assert_array_equal(pn & 15, 15 - lo)
    np.testing.assert_array_equal(pn >> 4, 15 - hi)
