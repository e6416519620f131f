"""Decode and prefill attention on the GPU against the oracle (plain f64
softmax attention over the oracle's own reconstruction of the oracle's own
encoding of the same seeded rows)."""
import math

import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, TENSOR_TOL, gpu_encode, kvq_module, queries, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def run_decode(kvq, fmt, lens, H, bf16, seed, path, layout=None, max_rows=None):
    layout = layout or kvq.mla_layout(seed=seed)
    cu = synth.cu_seqlens(lens)
    x = synth.mla_rows(seed, int(cu[-1]))
    codes, scales = gpu_encode(kvq, fmt, x, layout)
    qd, qv = queries(seed + 1, (len(lens), H, 576), bf16)
    out = torch.full((len(lens), H, 512), float("nan"), device="cuda")
    max_rows = int(cu[-1]) if max_rows is None else max_rows
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, len(lens), H, max_rows, layout, path), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_decode(fmt, qd, codes, scales, to_dev(cu), out, ws, max_rows, SM, layout, path)
    torch.cuda.synchronize()
    return x, cu, qv, out.cpu().numpy(), ws


def check_decode(oracle, fmt, x, cu, qv, got, pairs=None, seed=0, tol=SIMT_TOL):
    if fmt == 1:
        codes, scales = oracle.kv8_encode(x)
    else:
        codes, scales = oracle.tq4_encode(x, seed=seed)
    ref = oracle.attn_decode(fmt, codes, scales, qv, cu, SM, pairs=pairs, seed=seed)
    worst = 0.0
    for (b, h), r in ref.items():
        e = rel_err(got[b, h], r)
        worst = max(worst, e)
        assert e <= tol, (b, h, e)
    return worst


@pytest.mark.parametrize("fmt", [1, 2])
def test_config1_tiny(kvq, oracle, fmt):
    """1 sequence x 256 rows, 16 heads, f32 query; TQ4 with sign seed 0."""
    x, cu, qv, got, _ = run_decode(kvq, fmt, [256], 16, False, 0, kvq.PATH_SIMT)
    check_decode(oracle, fmt, x, cu, qv, got, seed=0)


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("bf16", [False, True])
def test_ragged_small_with_edges(kvq, oracle, fmt, bf16):
    lens = [1, 0, 17, 300, 64, 33]
    x, cu, qv, got, ws = run_decode(kvq, fmt, lens, 20, bf16, 11, kvq.PATH_SIMT)
    check_decode(oracle, fmt, x, cu, qv, got, seed=11)
    assert np.all(got[1] == 0.0)                      # the empty sequence
    assert kvq.read_device_error(ws) == 0


def test_single_scale_kv8_layout(kvq, oracle):
    layout = kvq.mla_layout((576,))
    lens = [40, 129]
    x, cu, qv, got, _ = run_decode(kvq, 1, lens, 16, True, 21, kvq.PATH_SIMT, layout=layout)
    codes, scales = oracle.kv8_encode(x, (576,))
    ref = oracle.attn_decode(1, codes, scales, qv, cu, SM, bdims=(576,))
    for (b, h), r in ref.items():
        assert rel_err(got[b, h], r) <= SIMT_TOL


@pytest.mark.parametrize("path", ["simt", "tensor"])
@pytest.mark.parametrize("fmt", [1, 2])
def test_config2_3_full_size_sampled(kvq, oracle, fmt, path):
    """8 sequences x 4096 rows, 128 heads, bf16 query (KV8 = config 2, TQ4 = config 3)."""
    lens = [4096] * 8
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    x, cu, qv, got, _ = run_decode(kvq, fmt, lens, 128, True, 2 if fmt == 1 else 3, pth)
    pairs = [(b, h) for b in range(8) for h in (0, 37, 64, 127)]
    check_decode(oracle, fmt, x, cu, qv, got, pairs=pairs, seed=2 if fmt == 1 else 3,
                 tol=SIMT_TOL if path == "simt" else TENSOR_TOL)
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("bf16", [False, True])
def test_tensor_ragged_with_edges(kvq, oracle, fmt, bf16):
    """Tensor-core path: ragged lengths with an empty, a one-row and tail-tile sequences, 128 heads."""
    lens = [1, 0, 127, 129, 700, 256, 3000]
    x, cu, qv, got, ws = run_decode(kvq, fmt, lens, 128, bf16, 13, kvq.PATH_TENSOR)
    pairs = [(b, h) for b in range(len(lens)) for h in (0, 31, 32, 63, 64, 100, 127)]
    check_decode(oracle, fmt, x, cu, qv, got, pairs=pairs, seed=13, tol=TENSOR_TOL)
    assert np.all(got[1] == 0.0)
    assert np.all(np.isfinite(got))
    assert kvq.read_device_error(ws) == 0


@pytest.mark.parametrize("fmt", [1, 2])
def test_tensor_many_sequences(kvq, oracle, fmt):
    """More sequences than the device-side chunk balancing handles (1024): the
    tensor path falls back to the host's chunk; lengths 0..300."""
    rng = np.random.default_rng(23)
    lens = [int(v) for v in rng.integers(0, 301, size=1100)]
    x, cu, qv, got, ws = run_decode(kvq, fmt, lens, 64, True, 23, kvq.PATH_TENSOR)
    pairs = [(b, h) for b in (0, 1, 517, 1023, 1024, 1099) for h in (0, 31, 32, 63)]
    pairs += [(b, 5) for b in range(0, 1100, 97)]
    check_decode(oracle, fmt, x, cu, qv, got, pairs=pairs, seed=23, tol=TENSOR_TOL)
    for b, T in enumerate(lens):
        if T == 0:
            assert np.all(got[b] == 0.0)
    assert kvq.read_device_error(ws) == 0


@pytest.mark.parametrize("fmt", [1, 2])
def test_tensor_balanced_chunks_skewed(kvq, oracle, fmt):
    """One long sequence among short ones: the device-chosen chunk splits the
    long one across many CTAs (several items per sequence, one wave)."""
    lens = [20000, 5, 300, 0, 129, 1]
    x, cu, qv, got, ws = run_decode(kvq, fmt, lens, 128, True, 29, kvq.PATH_TENSOR)
    pairs = [(b, h) for b in range(len(lens)) for h in (0, 33, 64, 127)]
    check_decode(oracle, fmt, x, cu, qv, got, pairs=pairs, seed=29, tol=TENSOR_TOL)
    assert np.all(got[3] == 0.0)
    assert kvq.read_device_error(ws) == 0


def test_tensor_matches_simt_closely(kvq):
    """The two kernel families on the same inputs agree to the tensor path's tolerance."""
    lens = [777, 2048, 5]
    outs = []
    for pth in (kvq.PATH_SIMT, kvq.PATH_TENSOR):
        _, _, _, got, _ = run_decode(kvq, 1, lens, 64, True, 17, pth)
        outs.append(got)
    for b in range(3):
        for h in range(64):
            assert rel_err(outs[1][b, h], outs[0][b, h]) <= TENSOR_TOL


@pytest.mark.parametrize("H,path", [(16, "simt"), (64, "tensor")])
def test_device_error_when_rows_exceed_bound(kvq, H, path):
    """A ragged batch larger than the bound the call was sized for sets the
    device error word instead of reading or writing out of bounds."""
    lens = [600, 600]
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    x, cu, qv, got, ws = run_decode(kvq, 1, lens, H, False, 5, pth, max_rows=100)
    assert kvq.read_device_error(ws) == 6
    assert kvq.read_device_error(ws) == 0             # cleared by the first read


@pytest.mark.parametrize("fmt,H,path", [(1, 16, "simt"), (2, 16, "simt"), (1, 64, "tensor"), (2, 64, "tensor")])
def test_prefill_small(kvq, oracle, fmt, H, path):
    n_past, n_new = 200, 37
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    tol = SIMT_TOL if path == "simt" else TENSOR_TOL
    layout = kvq.mla_layout(seed=4)
    x_all = synth.mla_rows(31, n_past + n_new)
    row = 576 if fmt == 1 else 288
    codes = torch.zeros((n_past + n_new, row), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((n_past + n_new, 2), dtype=torch.float32, device="cuda")
    pc, ps = gpu_encode(kvq, fmt, x_all[:n_past], layout)
    codes[:n_past] = pc
    scales[:n_past] = ps
    qd, qv = queries(32, (n_new, H, 576), False)
    out = torch.empty((n_new, H, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_prefill_workspace_size(fmt, H, n_past, n_new, layout, pth), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_prefill(fmt, to_dev(x_all[n_past:]), qd, codes, scales, n_past, out, ws, SM, layout, pth)
    torch.cuda.synchronize()
    if fmt == 1:
        oc, os_ = oracle.kv8_encode(x_all)
    else:
        oc, os_ = oracle.tq4_encode(x_all, seed=4)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)          # the new rows were encoded bit-exactly
    xh = oracle.reconstruct(fmt, oc, os_, seed=4)
    got = out.cpu().numpy()
    for j in range(n_new):
        ref = oracle.attn_dense(xh[:n_past + j + 1], qv[j], SM, 512)
        for h in range(H):
            assert rel_err(got[j, h], ref[h]) <= tol, (j, h)
