"""Pins of the oracle's attention: closed forms, a library softmax, and the
orthogonality identities the KV cache quantization pages state for the
consumers (q.x_hat == rotate(q).c and sum w x_hat == unrotate(sum w c))."""
import math

import numpy as np
import pytest
from scipy.special import softmax

from quantized_kv_cache_kv8_gb300 import synth

SM = 1.0 / math.sqrt(192.0)


def test_single_row_returns_that_row(oracle):
    K = synth.mla_rows(1, 1).astype(np.float64)
    q = synth.queries(2, (3, 576))
    out = oracle.attn_dense(K, q, SM, 512)
    for j in range(3):
        np.testing.assert_array_equal(out[j], K[0, :512])


def test_zero_query_averages_rows(oracle):
    K = synth.mla_rows(3, 37).astype(np.float64)
    out = oracle.attn_dense(K, np.zeros((1, 576), np.float32), SM, 512)
    np.testing.assert_allclose(out[0], K[:, :512].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_identical_rows(oracle):
    row = synth.mla_rows(4, 1).astype(np.float64)
    K = np.repeat(row, 9, axis=0)
    out = oracle.attn_dense(K, synth.queries(5, (2, 576)), SM, 512)
    np.testing.assert_allclose(out, np.repeat(row[:, :512], 2, axis=0), rtol=1e-14)


def test_two_rows_weights_three_to_one(oracle):
    """Scores differing by ln 3 give weights 3/4 and 1/4."""
    K = np.zeros((2, 576))
    K[0, 0] = 2.0
    K[0, 10] = 5.0
    K[1, 10] = -7.0
    q = np.zeros((1, 576), np.float32)
    q[0, 0] = np.float32(math.log(3.0) / (SM * 2.0))
    out = oracle.attn_dense(K, q, SM, 512)
    z0 = SM * float(q[0, 0]) * 2.0
    w0 = math.exp(z0) / (math.exp(z0) + 1.0)
    assert w0 == pytest.approx(0.75, abs=1e-7)
    np.testing.assert_allclose(out[0, [0, 10]], [w0 * 2.0, w0 * 5.0 + (1 - w0) * -7.0], rtol=1e-14)


def test_matches_library_softmax(oracle):
    K = synth.mla_rows(6, 300).astype(np.float64)
    q = synth.queries(7, (4, 576))
    out = oracle.attn_dense(K, q, SM, 512)
    ref = softmax(SM * (q.astype(np.float64) @ K.T), axis=1) @ K[:, :512]
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_empty_range_gives_zeros(oracle):
    out = oracle.attn_dense(np.zeros((0, 576)), synth.queries(8, (2, 576)), SM, 512)
    assert np.all(out == 0)


@pytest.mark.parametrize("fmt", [1, 2])
def test_method_path_identities(oracle, fmt):
    """The consumers' own arithmetic (KV8: row scale factored out of both sums;
    TQ4: rotated query, codebook dots, one unrotation of the context) equals
    attention over the reconstructed cache."""
    x = synth.mla_rows(9, 200)
    q = synth.queries(10, (5, 576))
    if fmt == 1:
        codes, scales = oracle.kv8_encode(x)
        xh = oracle.kv8_decode(codes, scales)
    else:
        codes, scales = oracle.tq4_encode(x, seed=17)
        xh = oracle.tq4_decode(codes, scales, seed=17)
    plain = oracle.attn_dense(xh, q, SM, 512)
    method = oracle.attn_method(fmt, codes, scales, q, SM, seed=17)
    np.testing.assert_allclose(method, plain, rtol=1e-10, atol=1e-12 * np.abs(plain).max())
    # and the score identity itself, row by row
    if fmt == 2:
        lv, _ = oracle.tq4_codebook()
        qr = oracle.tq4_rotate(q.astype(np.float64), seed=17)
        idx = np.zeros((200, 576), np.int64)
        idx[:, 0::2] = codes & 15
        idx[:, 1::2] = codes >> 4
        chat = lv[idx].astype(np.float64)
        chat[:, :512] *= scales[:, :1]
        chat[:, 512:] *= scales[:, 1:]
        np.testing.assert_allclose(qr @ chat.T, q.astype(np.float64) @ xh.T, rtol=1e-9, atol=1e-9)


def test_ragged_decode_groups_by_sequence(oracle):
    lens = [3, 0, 17, 1]
    cu = synth.cu_seqlens(lens)
    x = synth.mla_rows(12, int(cu[-1]))
    codes, scales = oracle.kv8_encode(x)
    q = synth.queries(13, (4, 2, 576))
    out = oracle.attn_decode(1, codes, scales, q, cu, SM)
    xh = oracle.kv8_decode(codes, scales)
    for b in range(4):
        for h in range(2):
            lo, hi = cu[b], cu[b + 1]
            if hi == lo:
                assert np.all(out[(b, h)] == 0)
            else:
                ref = softmax(SM * (xh[lo:hi] @ q[b, h].astype(np.float64))) @ xh[lo:hi, :512]
                np.testing.assert_allclose(out[(b, h)], ref, rtol=1e-11, atol=1e-13)
