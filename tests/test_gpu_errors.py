"""The device-side error contract on the GPU, through the C ABI.

* Non-finite inputs: the pages define no code for a NaN or an infinity, so an
  encoder that meets one sets KVQ_ERR_NONFINITE in the error word it is given
  (the attention calls give theirs: the workspace's first 4 bytes); the other
  rows are encoded exactly as the oracle encodes them.
* A bounded wait that runs out: the testing hook makes every tensor-core
  attention launch first wait on a barrier that nothing arrives on, with a
  short poll limit.  The wait runs out, the kernel leaves its tiles, drains the
  tensor-core work it issued, frees its tensor memory and sets KVQ_ERR_TIMEOUT;
  the next call without the hook runs normally and matches the oracle.
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import TENSOR_TOL, gpu_encode, kvq_module, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)
NONFINITE, TIMEOUT = 9, 10


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def bad_rows(seed, n=64):
    x = synth.mla_rows(seed, n)
    x[3, 17] = np.nan
    x[7, 300] = np.inf
    x[11, 530] = -np.inf
    return x, {3, 7, 11}


@pytest.mark.parametrize("fmt", [1, 2], ids=["kv8", "tq4"])
def test_encoder_flags_non_finite_rows(kvq, oracle, fmt):
    x, bad = bad_rows(51)
    layout = kvq.mla_layout(seed=3)
    n = x.shape[0]
    row = 576 if fmt == 1 else 288
    codes = torch.empty((n, row), dtype=torch.uint8, device="cuda")
    scales = torch.empty((n, 2), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    enc = kvq.kv8_encode if fmt == 1 else kvq.tq4_encode
    enc(to_dev(x), codes, scales, layout, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == NONFINITE
    good = np.array([i for i in range(n) if i not in bad])
    xg = np.ascontiguousarray(x[good])
    oc, os_ = oracle.kv8_encode(xg) if fmt == 1 else oracle.tq4_encode(xg, seed=3)
    np.testing.assert_array_equal(codes.cpu().numpy()[good], oc)
    np.testing.assert_array_equal(scales.cpu().numpy()[good].view(np.uint32), os_.view(np.uint32))
    # finite rows leave the word as it was; without a word nothing is reported
    err.zero_()
    enc(to_dev(xg), codes[:len(good)], scales[:len(good)], layout, err_word=err)
    enc(to_dev(x), codes, scales, layout)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_tq4_radius_past_f32_range_is_flagged(kvq):
    x = synth.mla_rows(52, 8)
    x[2, :512] = np.float32(3e19)   # the sum of squares overflows f32
    codes = torch.empty((8, 288), dtype=torch.uint8, device="cuda")
    scales = torch.empty((8, 2), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.tq4_encode(to_dev(x), codes, scales, kvq.mla_layout(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == NONFINITE


@pytest.mark.parametrize("fmt", [1, 2], ids=["kv8-fused", "tq4"])
def test_decode_append_reports_a_non_finite_new_row(kvq, fmt):
    B, T, H = 4, 512, 128
    layout = kvq.mla_layout()
    x = synth.mla_rows(53, B * T)
    codes, scales = gpu_encode(kvq, fmt, x, layout)
    x_new = synth.mla_rows(54, B)
    x_new[2, 5] = np.nan
    cu = synth.cu_seqlens([T] * B)
    bits = synth.bf16_bits(synth.queries(55, (B, H, 576)))
    q = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty((B, H, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, B, H, B * T, layout), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_decode_append(fmt, to_dev(x_new), to_dev(cu[1:] - 1), q, codes, scales, to_dev(cu), out, ws, B * T,
                              SM, layout)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == NONFINITE


def test_prefill_reports_a_non_finite_new_row(kvq):
    P, N, H = 256, 16, 64
    layout = kvq.mla_layout()
    x = synth.mla_rows(56, P + N)
    x[P + 4, 100] = np.inf
    codes = torch.zeros((P + N, 576), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((P + N, 2), dtype=torch.float32, device="cuda")
    pc, ps = gpu_encode(kvq, 1, x[:P], layout)
    codes[:P], scales[:P] = pc, ps
    bits = synth.bf16_bits(synth.queries(57, (N, H, 576)))
    q = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty((N, H, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_prefill_workspace_size(1, H, P, N, layout), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_prefill(1, to_dev(x[P:]), q, codes, scales, P, out, ws, SM, layout)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == NONFINITE


@pytest.mark.parametrize("fmt,q_bf16", [(1, True), (1, False), (2, True)], ids=["kv8-bf16", "kv8-f32", "tq4"])
def test_a_wait_that_runs_out_reports_timeout_and_the_next_call_runs(kvq, oracle, fmt, q_bf16):
    B, T, H = 2, 1000, 128
    layout = kvq.mla_layout(seed=7)
    x = synth.mla_rows(58, B * T)
    codes, scales = gpu_encode(kvq, fmt, x, layout)
    q32 = synth.queries(59, (B, H, 576))
    if q_bf16:
        bits = synth.bf16_bits(q32)
        q = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        qo = synth.bf16_to_f32(bits)
    else:
        q, qo = to_dev(q32), q32
    cu = synth.cu_seqlens([T] * B)
    out = torch.empty((B, H, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, B, H, B * T, layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    try:
        kvq.test_stall_waits(2000)
        kvq.kv_attn_decode(fmt, q, codes, scales, to_dev(cu), out, ws, B * T, SM, layout, kvq.PATH_TENSOR)
        torch.cuda.synchronize()
    finally:
        kvq.test_stall_waits(0)
    assert kvq.read_device_error(ws, clear=True) == TIMEOUT
    out.fill_(float("nan"))
    kvq.kv_attn_decode(fmt, q, codes, scales, to_dev(cu), out, ws, B * T, SM, layout, kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    oc, os_ = oracle.kv8_encode(x) if fmt == 1 else oracle.tq4_encode(x, seed=7)
    xh = oracle.reconstruct(fmt, oc, os_, seed=7)
    got = out.cpu().numpy()
    for b in range(B):
        heads = [0, 63, 64, 127]
        ref = oracle.attn_dense(xh[cu[b]:cu[b + 1]], np.ascontiguousarray(qo[b, heads]), SM, 512)
        for i, h in enumerate(heads):
            assert rel_err(got[b, h], ref[i]) <= TENSOR_TOL, (b, h)



def test_k2v4_producers_flag_non_finite_values(kvq, oracle):
    """The K2/V4 encoder and append report a NaN in K or an infinity in V through
    the error word; a sequence without one is encoded exactly as the oracle
    encodes it; clean calls leave the word at 0."""
    B, H, T, D = 2, 2, 64, 128
    layout = kvq.k2v4_layout(H, D, 1.10, 4, 16, 16)
    OL = oracle.k2v4_layout(H, D, 1.10, 4, 16, 16)
    k, v = synth.gqa_kv(71, B, H, T, D)
    slots = 4 + 16 + 16

    def pools():
        return (torch.zeros((B, H, T, D // 4), dtype=torch.uint8, device="cuda"),
                torch.zeros((B, H, T // 32, D), dtype=torch.int16, device="cuda"),
                torch.zeros((B, H, T, D // 32, 18), dtype=torch.uint8, device="cuda"),
                torch.zeros((B, H, slots, D), dtype=torch.int16, device="cuda"),
                torch.zeros((B, H, slots, D), dtype=torch.int16, device="cuda"))
    for case in ("k_nan", "v_inf", "v_nan"):
        kb, vb = k.copy(), v.copy()
        if case == "k_nan":
            kb[1, 0, 40, 7] = np.nan
        elif case == "v_inf":
            vb[1, 1, 50, 3] = np.inf
        else:
            vb[1, 0, 20, 100] = np.nan
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        enc = pools()
        kvq.k2v4_encode(layout, to_dev(kb), to_dev(vb), *enc, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == NONFINITE
        oenc = oracle.k2v4_encode(k[0], v[0], OL)
        for g, o in zip(enc, oenc):
            np.testing.assert_array_equal(g[0].cpu().numpy().view(o.dtype), o)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    enc = pools()
    kvq.k2v4_encode(layout, to_dev(k), to_dev(v), *enc, err_word=err)
    k_new, v_new = synth.gqa_kv(72, B, H, 8, D)
    kvq.k2v4_append(layout, to_dev(k_new), to_dev(v_new), 32, *enc, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k_new[0, 1, 3, 9] = np.inf
    kvq.k2v4_append(layout, to_dev(k_new), to_dev(v_new), 40, *enc, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == NONFINITE
