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


# --- appends and the partial-group scale rule ([P3] "Review fixes", item
# "Fresh partial-group scale"; "Attention error under the engine's append
# patterns") ---------------------------------------------------------------

def _empty_pools(H, cap, D, slots):
    return (np.zeros((H, cap, D // 4), np.uint8), np.zeros((H, cap // 32, D), np.uint16),
            np.zeros((H, cap, D // 32, 18), np.uint8), np.zeros((H, slots, D), np.uint16),
            np.zeros((H, slots, D), np.uint16))


def _append_all(oracle, L, k, v, cuts, cap):
    """Append k[:, a:b], v[:, a:b] for consecutive cut points, from an empty pool."""
    H, _, D = k.shape
    pools = _empty_pools(H, cap, D, L.n_sink + L.n_window + L.n_slack)
    for a, b in zip(cuts[:-1], cuts[1:]):
        pools = oracle.k2v4_append(*pools, k[:, a:b], v[:, a:b], a, L)
    return pools


def _f16(x):
    return int(np.float16(x).view(np.uint16))


def test_append_of_whole_groups_equals_encoder(oracle):
    """Appends of whole 32-cell groups never run the partial rule: the pools
    equal the encoder's (bulk bit for bit, the reader's view through the
    overlay identical)."""
    H, T, D, cap = 2, 96, 64, 128
    k, v = synth.gqa_kv(41, 1, H, T, D)
    L = oracle.k2v4_layout(H, D, 1.10, 4, 16, 16)
    enc = oracle.k2v4_encode(k[0], v[0], L, cap)
    for cuts in ([0, 96], [0, 32, 96], [0, 32, 64, 96]):
        app = _append_all(oracle, L, k[0], v[0], cuts, cap)
        for a, b in zip(enc[:3], app[:3]):
            np.testing.assert_array_equal(a, b)
        ke, ve = oracle.k2v4_reconstruct(*enc, T, L)
        ka, va = oracle.k2v4_reconstruct(*app, T, L)
        np.testing.assert_array_equal(ke, ka)
        np.testing.assert_array_equal(ve, va)


def test_partial_group_closed_forms_at_constant_magnitude(oracle):
    """Every cell of magnitude c: the previous group's mean square equals the
    present cells', so the shrink rule returns c for any n, and the /n rule of
    a partial first group returns c too; a later append into a started group
    keeps its scale."""
    H, D, cap, c = 1, 32, 160, 0.75
    rng = np.random.default_rng(3)
    k = (c * rng.choice([-1.0, 1.0], size=(H, 150, D))).astype(np.float32)
    v = rng.standard_normal((H, 150, D)).astype(np.float32)
    L = oracle.k2v4_layout(H, D, 1.0, 0, 0, 0)
    for cuts in ([0, 5], [0, 40], [0, 40, 43, 93], [0, 1, 2, 3, 35, 150]):
        kc, ks, vb, kw, vw = _append_all(oracle, L, k, v, cuts, cap)
        n_groups = (cuts[-1] + 31) // 32
        assert np.all(ks[0, :n_groups] == _f16(c)), cuts
        # codes: x / s = +-1 is nearest the outer levels +-1.510 (|1 - 1.510| <
        # |1 - 0.4528|), read back as +-1.510 c
        K, _ = oracle.k2v4_reconstruct(kc, ks, vb, kw, vw, cuts[-1], L, use_overlay=False)
        lv, _ = oracle.k2_codebook()
        want = np.where(k[0, :cuts[-1]] > 0, lv[3], lv[0]) * c
        np.testing.assert_allclose(K[0], want, rtol=1e-6)


def test_partial_group_shrinks_toward_previous_scale(oracle):
    """A fresh group of n zero cells after a group of magnitude c: s =
    c * sqrt((32 - n) / 32) (no present energy, the previous mean square
    fills the 32 - n missing cells), to one fp16 step after the f32 steps."""
    H, D, cap, c = 1, 32, 64, 0.75
    for gain in (1.0, 1.10):
        L = oracle.k2v4_layout(H, D, gain, 0, 0, 0)
        for n in (1, 3, 17, 31):
            k = np.zeros((H, 32 + n, D), np.float32)
            k[:, :32] = c
            v = np.zeros_like(k)
            _, ks, _, _, _ = _append_all(oracle, L, k, v, [0, 32 + n], cap)
            prev = float(np.float16(gain * c)) / gain
            want = gain * prev * math.sqrt((32 - n) / 32)
            got = float(ks[0, 1, 0].view(np.float16))
            assert abs(got - want) <= 2 ** -10 * want + 1e-12, (gain, n, got, want)
            assert ks[0, 0, 0] == _f16(gain * c)


def test_partial_first_group_is_rms_of_present_cells(oracle):
    """Group 0 written by a partial batch has no previous group: its scale is
    the RMS of the n cells present (3, 4, 0, 0 -> sqrt(25 / 4) = 2.5)."""
    H, D, cap = 1, 32, 64
    L = oracle.k2v4_layout(H, D, 1.0, 0, 0, 0)
    k = np.zeros((H, 4, D), np.float32)
    k[0, 0], k[0, 1] = 3.0, 4.0
    _, ks, _, _, _ = _append_all(oracle, L, k, np.zeros_like(k), [0, 4], cap)
    assert np.all(ks[0, 0] == _f16(2.5))


def test_one_call_equals_two_calls_split_at_a_group_boundary(oracle):
    """The previous group's scale enters the partial rule identically whether
    it was stored by an earlier call or in the same call ([P3]: two-call and
    one-call appends store the same scale)."""
    H, D, cap = 2, 64, 192
    k, v = synth.gqa_kv(43, 1, H, 180, D)
    L = oracle.k2v4_layout(H, D, 1.10, 4, 16, 16)
    for total, split in ((70, 64), (101, 96), (180, 128), (40, 32)):
        one = _append_all(oracle, L, k[0, :, :total], v[0, :, :total], [0, total], cap)
        two = _append_all(oracle, L, k[0, :, :total], v[0, :, :total], [0, split, total], cap)
        for a, b in zip(one[:3], two[:3]):
            np.testing.assert_array_equal(a, b)


def test_append_into_started_group_keeps_its_scale(oracle):
    """Cells appended into a group that already holds cells are coded against
    the stored scale, which stays as it was."""
    H, D, cap = 2, 64, 128
    k, v = synth.gqa_kv(47, 1, H, 100, D)
    L = oracle.k2v4_layout(H, D, 1.10, 4, 16, 16)
    first = _append_all(oracle, L, k[0, :, :45], v[0, :, :45], [0, 45], cap)
    after = oracle.k2v4_append(*first, k[0, :, 45:50], v[0, :, 45:50], 45, L)
    np.testing.assert_array_equal(first[1][:, :2], after[1][:, :2])
    np.testing.assert_array_equal(first[0][:, :45], after[0][:, :45])
