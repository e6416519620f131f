"""Pins of the oracle's K2/V4 GQA codec and FP16 overlay (Strata pull request
"KV cache: FP16 sliding window + attention sinks, and an optional 2-bit K /
4-bit V cache scheme (--kv q2k)")."""
import math

import numpy as np
import pytest

from conftest import golden_lines
from quantized_kv_cache_kv8_gb300 import synth


def _counts():
    return {l.split()[0]: float(l.split()[1]) for l in golden_lines("page_byte_counts.txt")}


def test_byte_counts_and_footprints_match_page():
    c = _counts()
    D, H = 256, 2
    per_head = D // 4 + (D * 2) // 32 + (D // 32) * 18            # K codes + K scales per cell + V blocks
    assert per_head == c["q2k_bytes_per_cell_head"]
    assert H * per_head == c["q2k_bytes_per_cell_2heads"]
    assert H * (D // 32) * 18 * 2 == c["q4_0_bytes_per_cell_2heads"]
    assert H * D * 2 * 2 == c["fp16_bytes_per_cell_2heads"]
    fp16_cell = H * D * 2 * 2
    slots128 = 8 + 128 + 16
    assert slots128 * fp16_cell / 1024 == c["overlay_kib_per_layer_w128_s8"]
    assert round(12 * slots128 * fp16_cell / 2 ** 20, 2) == c["overlay_mib_12_layers_w128_s8"]
    assert round(12 * (8 + 256 + 16) * fp16_cell / 2 ** 20, 2) == c["overlay_mib_12_layers_w256_s8"]
    ctx = 262144
    assert round(ctx * 448 * 12 / 2 ** 30, 2) == c["q2k_gib_262144_12_layers"]
    assert round(ctx * 576 * 12 / 2 ** 30, 2) == c["q4_0_gib_262144_12_layers"]
    assert round(ctx * 2048 * 12 / 2 ** 30, 2) == c["fp16_gib_262144_12_layers"]


def test_q4_0_nibble_order_fixture(oracle):
    lines = {l.split()[0]: l.split()[1:] for l in golden_lines("q4_0_block.txt")}
    d_bits = int(lines["d"][0], 16)
    body = [int(b, 16) for b in lines["bytes"]]
    want = [float(v) for v in lines["values"]]
    L = oracle.k2v4_layout(n_kv_heads=1, head_dim=32, n_sink=0, n_window=0, n_slack=0)
    kc = np.zeros((1, 32, 8), np.uint8)
    ks = np.zeros((1, 1, 32), np.uint16)
    vb = np.zeros((1, 32, 1, 18), np.uint8)
    vb[0, 0, 0, 0] = d_bits & 255
    vb[0, 0, 0, 1] = d_bits >> 8
    vb[0, 0, 0, 2:] = body
    kw = np.zeros((1, 1, 32), np.uint16)
    _, V = oracle.k2v4_reconstruct(kc, ks, vb, kw, kw, 32, L, use_overlay=False)
    np.testing.assert_array_equal(V[0, 0], want)


def test_k2_codebook_is_four_level_max(oracle):
    lv, th = oracle.k2_codebook()
    np.testing.assert_allclose(lv, [-1.510, -0.4528, 0.4528, 1.510], atol=6e-4)
    assert th[1] == 0.0 and th[0] == -th[2]


def _small_case(oracle, T=96, D=64, H=2, gain=1.10, sink=4, window=16, slack=16, seed=31):
    k, v = synth.gqa_kv(seed, 1, H, T, D)
    L = oracle.k2v4_layout(n_kv_heads=H, head_dim=D, k_gain=gain, n_sink=sink, n_window=window, n_slack=slack)
    enc = oracle.k2v4_encode(k[0], v[0], L)
    return k[0], v[0], L, enc


def test_k2_scale_rule_and_gain(oracle):
    """Stored scale = fp16(gain * rms over the 32 cells of a channel); the codes
    are chosen against the un-gained scale, so they do not depend on the gain."""
    k, v, L1, enc1 = _small_case(oracle, gain=1.0)
    _, _, L2, enc2 = _small_case(oracle, gain=1.10)
    np.testing.assert_array_equal(enc1[0], enc2[0])                       # K codes identical
    s1 = np.vectorize(oracle.f16_value)(enc1[1])
    s2 = np.vectorize(oracle.f16_value)(enc2[1])
    rms = np.sqrt((k.astype(np.float64).reshape(2, 3, 32, 64) ** 2).mean(axis=2))
    np.testing.assert_allclose(s1, rms, rtol=2 ** -10)
    np.testing.assert_allclose(s2, 1.10 * rms, rtol=2 ** -10 + 1e-6)


def test_k2_codes_are_nearest_levels(oracle):
    k, v, L, (kc, ks, vb, kw, vw) = _small_case(oracle, gain=1.0)
    lv, _ = oracle.k2_codebook()
    rms = np.sqrt((k.astype(np.float64).reshape(2, 3, 32, 64) ** 2).mean(axis=2))
    for h in range(2):
        for t in range(0, 96, 5):
            for d in range(0, 64, 3):
                code = (kc[h, t, d // 4] >> (2 * (d % 4))) & 3
                u = k[h, t, d] / rms[h, t // 32, d]
                dist = np.abs(lv - u)
                assert dist[code] <= dist.min() + 1e-6


def test_v_q4_0_error_bound(oracle):
    k, v, L, enc = _small_case(oracle)
    K, V = oracle.k2v4_reconstruct(*enc, 96, L, use_overlay=False)
    blocks = v.astype(np.float64).reshape(2, 96, 2, 32)
    dmag = np.abs(blocks).max(axis=3, keepdims=True) / 8
    err = np.abs(V.reshape(2, 96, 2, 32) - blocks)
    assert np.all(err <= dmag * (1.0 + 2 ** -9) + 1e-12)      # one grid step at most (the clamped top)
    assert np.mean(err <= dmag / 2 * (1 + 2 ** -9) + 1e-12) > 0.95


def test_overlay_slots_and_exact_cells(oracle):
    T = 96
    k, v, L, enc = _small_case(oracle, T=T)
    slots = [oracle.k2v4_slot(c, T, L) for c in range(T)]
    live = [s for s in slots if s >= 0]
    assert len(live) == len(set(live)) == L.n_sink + L.n_window
    assert all(0 <= s < L.n_sink + L.n_window + L.n_slack for s in live)
    for c in range(T):
        assert (slots[c] >= 0) == (c < L.n_sink or c >= T - L.n_window)
    K1, V1 = oracle.k2v4_reconstruct(*enc, T, L, use_overlay=True)
    K0, V0 = oracle.k2v4_reconstruct(*enc, T, L, use_overlay=False)
    for c in range(T):
        if slots[c] >= 0:                              # overlay cells read exact fp16
            np.testing.assert_array_equal(K1[:, c], k[:, c].astype(np.float16).astype(np.float64))
            np.testing.assert_array_equal(V1[:, c], v[:, c].astype(np.float16).astype(np.float64))
        else:                                          # the bulk is untouched
            np.testing.assert_array_equal(K1[:, c], K0[:, c])
            np.testing.assert_array_equal(V1[:, c], V0[:, c])


def test_overlay_cells_match_fp16_attention(oracle):
    """With every cell inside the overlay, attention equals attention over an all-fp16 cache."""
    T = 64
    k, v = synth.gqa_kv(41, 1, 2, T, 64)
    L = oracle.k2v4_layout(n_kv_heads=2, head_dim=64, n_sink=8, n_window=T, n_slack=16)
    enc = oracle.k2v4_encode(k[0], v[0], L)
    K, V = oracle.k2v4_reconstruct(*enc, T, L)
    q = synth.queries(42, (16, 64))
    got = oracle.k2v4_attn(K, V, q, 1 / 8)
    Kf = k[0].astype(np.float16).astype(np.float64)
    Vf = v[0].astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, oracle.k2v4_attn(Kf, Vf, q, 1 / 8))
