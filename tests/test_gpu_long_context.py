"""Long-context workloads at full size, on the GPU against the oracle.

Ragged decode: 32 sequences with lengths drawn uniformly from [1024, 131072]
(seed 4, about 2.26 M rows in total), 128 heads, bf16 query, KV8 and TQ4.
Drawing 2.26 M fresh latent rows on the host would take minutes, so the pool is
built from one master block of 131072 seeded rows: sequence b holds master rows
(o_b + t) mod 131072 for t < T_b, with a different start o_b per sequence, so
no two sequences hold the same row at the same position.  Encoding is per row,
so gathering encoded master rows is the same as encoding the gathered rows.

Chunked causal prefill: 2048 new rows appended to a cache of 124 x 1024 =
126,976 rows, 128 heads, bf16 query; token j attends rows [0, P + j].

Outputs are checked on sampled (sequence or token, head) pairs, which the
oracle computes one by one in float64 over its own encoding of the same rows.
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, TENSOR_TOL, gpu_encode, kvq_module, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)
H = 128
MASTER = 131072
B = 32


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


@pytest.fixture(scope="module")
def ragged_inputs():
    lens = synth.ragged_lengths(4, B, 1024, 131072)
    cu = synth.cu_seqlens(lens)
    offs = (np.arange(B, dtype=np.int64) * 40961) % MASTER
    x = synth.mla_rows(4, MASTER)
    bits = synth.bf16_bits(synth.queries(5, (B, H, 576)))
    return dict(lens=lens, cu=cu, offs=offs, x=x, q_bits=bits, q=synth.bf16_to_f32(bits))


def _bf16_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("path", ["simt", "tensor"])
@pytest.mark.parametrize("fmt", [1, 2])
def test_config4_ragged_decode(kvq, oracle, ragged_inputs, fmt, path):
    d = ragged_inputs
    lens, cu, offs, x = d["lens"], d["cu"], d["offs"], d["x"]
    seed = 4
    layout = kvq.mla_layout(seed=seed)
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    tol = SIMT_TOL if path == "simt" else TENSOR_TOL
    mc, ms = gpu_encode(kvq, fmt, x, layout)
    idx = np.concatenate([(o + np.arange(T, dtype=np.int64)) % MASTER for o, T in zip(offs, lens)])
    idx_t = torch.from_numpy(idx).cuda()
    codes = mc[idx_t].contiguous()
    scales = ms[idx_t].contiguous()
    del idx_t
    total = int(cu[-1])
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, B, H, total, layout, pth), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_decode(fmt, _bf16_dev(d["q_bits"]), codes, scales, to_dev(cu), out, ws, total, SM, layout, pth)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    if fmt == 1:
        oc, os_ = oracle.kv8_encode(x)
    else:
        oc, os_ = oracle.tq4_encode(x, seed=seed)
    np.testing.assert_array_equal(mc.cpu().numpy(), oc)
    np.testing.assert_array_equal(ms.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, 13})
    for b in seqs:
        rows = (offs[b] + np.arange(lens[b], dtype=np.int64)) % MASTER
        xh = oracle.reconstruct(fmt, oc[rows], os_[rows], seed=seed)
        heads = [0, 63, 64, 127]
        ref = oracle.attn_dense(xh, d["q"][b, heads], SM, 512)
        for i, h in enumerate(heads):
            e = rel_err(got[b, h], ref[i])
            assert e <= tol, (b, h, int(lens[b]), e)


@pytest.mark.parametrize("fmt", [1, 2])
def test_config4_ragged_decode_append(kvq, oracle, ragged_inputs, fmt):
    """The step the benchmark times: kv_attn_decode_append on the tensor path
    over the ragged batch, each sequence's new row written at its last
    position (KV8: encoded inside the decode launch).  The appended rows are
    bit-exact against the oracle's encoding; sampled outputs are checked
    against the oracle over the master rows plus the new row."""
    d = ragged_inputs
    lens, cu, offs, x = d["lens"], d["cu"], d["offs"], d["x"]
    seed = 4
    layout = kvq.mla_layout(seed=seed)
    mc, ms = gpu_encode(kvq, fmt, x, layout)
    idx = np.concatenate([(o + np.arange(T, dtype=np.int64)) % MASTER for o, T in zip(offs, lens)])
    idx_t = torch.from_numpy(idx).cuda()
    codes = mc[idx_t].contiguous()
    scales = ms[idx_t].contiguous()
    del idx_t, mc, ms
    total = int(cu[-1])
    x_new = synth.mla_rows(7, B)
    dst = (cu[1:] - 1).astype(np.int64)
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, B, H, total, layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_decode_append(fmt, to_dev(x_new), to_dev(dst), _bf16_dev(d["q_bits"]), codes, scales, to_dev(cu),
                              out, ws, total, SM, layout, kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    if fmt == 1:
        oc, os_ = oracle.kv8_encode(x)
        nc, ns = oracle.kv8_encode(x_new)
    else:
        oc, os_ = oracle.tq4_encode(x, seed=seed)
        nc, ns = oracle.tq4_encode(x_new, seed=seed)
    np.testing.assert_array_equal(codes[torch.from_numpy(dst).cuda()].cpu().numpy(), nc)
    np.testing.assert_array_equal(scales[torch.from_numpy(dst).cuda()].cpu().numpy().view(np.uint32),
                                  ns.view(np.uint32))
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, 21})
    for b in seqs:
        rows = (offs[b] + np.arange(lens[b] - 1, dtype=np.int64)) % MASTER
        xh = np.concatenate([oracle.reconstruct(fmt, oc[rows], os_[rows], seed=seed),
                             oracle.reconstruct(fmt, nc[b:b + 1], ns[b:b + 1], seed=seed)])
        heads = [0, 63, 64, 127]
        ref = oracle.attn_dense(xh, d["q"][b, heads], SM, 512)
        for i, h in enumerate(heads):
            e = rel_err(got[b, h], ref[i])
            assert e <= TENSOR_TOL, (b, h, int(lens[b]), e)


@pytest.fixture(scope="module")
def prefill_inputs():
    n_past, n_new = 124 * 1024, 2048
    x = synth.mla_rows(41, n_past + n_new)
    bits = synth.bf16_bits(synth.queries(42, (n_new, H, 576)))
    return dict(n_past=n_past, n_new=n_new, x=x, q_bits=bits)


@pytest.mark.parametrize("fmt,path", [(1, "tensor"), (2, "tensor"), (1, "simt")])
def test_config4_prefill(kvq, oracle, prefill_inputs, fmt, path):
    d = prefill_inputs
    n_past, n_new, x = d["n_past"], d["n_new"], d["x"]
    seed = 4
    layout = kvq.mla_layout(seed=seed)
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    tol = SIMT_TOL if path == "simt" else TENSOR_TOL
    row = 576 if fmt == 1 else 288
    codes = torch.zeros((n_past + n_new, row), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((n_past + n_new, 2), dtype=torch.float32, device="cuda")
    pc, ps = gpu_encode(kvq, fmt, x[:n_past], layout)
    codes[:n_past] = pc
    scales[:n_past] = ps
    del pc, ps
    out = torch.full((n_new, H, 512), float("nan"), device="cuda")
    ws = torch.zeros(kvq.kv_attn_prefill_workspace_size(fmt, H, n_past, n_new, layout, pth), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_prefill(fmt, to_dev(x[n_past:]), _bf16_dev(d["q_bits"]), codes, scales, n_past, out, ws, SM,
                        layout, pth)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    if fmt == 1:
        oc, os_ = oracle.kv8_encode(x)
    else:
        oc, os_ = oracle.tq4_encode(x, seed=seed)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    toks = [0, 1, 1023, 2047]
    heads = [0, 77, 127]
    got = out[toks].cpu().numpy()
    assert np.all(np.isfinite(got))
    xh = oracle.reconstruct(fmt, oc, os_, seed=seed)
    qv = synth.bf16_to_f32(d["q_bits"][toks][:, heads])
    for i, j in enumerate(toks):
        ref = oracle.attn_dense(xh[:n_past + j + 1], qv[i], SM, 512)
        for k, h in enumerate(heads):
            e = rel_err(got[i, h], ref[k])
            assert e <= tol, (j, h, e)
