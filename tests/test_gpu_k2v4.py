"""K2/V4 GQA cache on the GPU against the oracle: encode bit for bit, decode
within 1e-5 on the fp32 path and 2e-3 on the tensor-core path (f16 operands),
overlay cells exact."""
import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, TENSOR_TOL, kvq_module, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def gpu_k2v4(kvq, k, v, layout, cap=None):
    B, H, T, D = k.shape
    cap = T if cap is None else cap
    slots = layout.n_sink + layout.n_window + layout.n_slack
    kc = torch.zeros((B, H, cap, D // 4), dtype=torch.uint8, device="cuda")
    ks = torch.zeros((B, H, cap // 32, D), dtype=torch.int16, device="cuda")
    vb = torch.zeros((B, H, cap, D // 32, 18), dtype=torch.uint8, device="cuda")
    kw = torch.zeros((B, H, slots, D), dtype=torch.int16, device="cuda")
    vw = torch.zeros((B, H, slots, D), dtype=torch.int16, device="cuda")
    kvq.k2v4_encode(layout, to_dev(k), to_dev(v), kc, ks, vb, kw, vw, capacity=cap)
    return kc, ks, vb, kw, vw


def oracle_layout(oracle, layout):
    return oracle.k2v4_layout(layout.n_kv_heads, layout.head_dim, layout.k_gain, layout.n_sink, layout.n_window,
                              layout.n_slack)


def run_case(kvq, oracle, B, H, T, D, Hq, sink, window, seed, path, full_check=True, pairs=None):
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    tol = SIMT_TOL if path == "simt" else TENSOR_TOL
    layout = kvq.k2v4_layout(H, D, 1.10, sink, window, 16)
    OL = oracle_layout(oracle, layout)
    k, v = synth.gqa_kv(seed, B, H, T, D)
    enc = gpu_k2v4(kvq, k, v, layout)
    for b in range(B):
        oenc = oracle.k2v4_encode(k[b], v[b], OL)
        for name, g, o in zip(("k_codes", "k_scales", "v_blocks", "k_win", "v_win"), enc, oenc):
            np.testing.assert_array_equal(g[b].cpu().numpy().view(o.dtype), o, err_msg=f"{name} seq {b}")
    q = synth.queries(seed + 1, (B, Hq, D))
    out = torch.empty((B, Hq, D), device="cuda")
    ws = torch.zeros(kvq.kv_attn_decode_k2v4_workspace_size(layout, B, Hq, T, pth), dtype=torch.uint8, device="cuda")
    sm = 1.0 / np.sqrt(D)
    kvq.kv_attn_decode_k2v4(layout, to_dev(q), T, *enc, out, ws, sm, path=pth)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    got = out.cpu().numpy()
    grp = Hq // H
    for b in range(B):
        oenc = oracle.k2v4_encode(k[b], v[b], OL)
        K, V = oracle.k2v4_reconstruct(*oenc, T, OL)
        ref = oracle.k2v4_attn(K, V, q[b], sm)
        for h in range(Hq):
            if pairs is not None and (b, h) not in pairs:
                continue
            assert rel_err(got[b, h], ref[h]) <= tol, (b, h, path)
    return got


@pytest.mark.parametrize("path", ["simt", "tensor"])
def test_k2v4_small(kvq, oracle, path):
    run_case(kvq, oracle, B=2, H=2, T=96, D=128, Hq=16, sink=4, window=16, seed=51, path=path)


@pytest.mark.parametrize("path", ["simt", "tensor"])
def test_k2v4_half_group_and_tail_tile(kvq, oracle, path):
    """4 query heads per kv head (half of a group), 416 cells: three full
    128-cell tensor tiles and a 32-cell tail."""
    run_case(kvq, oracle, B=1, H=2, T=416, D=256, Hq=8, sink=8, window=64, seed=53, path=path)


def test_k2v4_tensor_odd_chunk_counts(kvq, oracle):
    """The tensor kernel runs two chunks per CTA.  320 cells of one kv head
    make 3 chunks of one tile (the second CTA's second pipeline has no chunk;
    the last tile holds 64 cells); 40000 cells at head_dim 128 make 157 chunks
    of two tiles each (every pipeline refills its raw K and V buffers)."""
    run_case(kvq, oracle, B=1, H=1, T=320, D=256, Hq=8, sink=8, window=32, seed=57, path="tensor")
    run_case(kvq, oracle, B=1, H=1, T=40000, D=128, Hq=8, sink=8, window=256, seed=58, path="tensor")


@pytest.mark.parametrize("path", ["simt", "tensor"])
def test_k2v4_window_covers_all(kvq, oracle, path):
    """Every cell inside the overlay: output equals attention over fp16 K/V."""
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    tol = SIMT_TOL if path == "simt" else TENSOR_TOL
    B, H, T, D, Hq = 1, 2, 64, 128, 8
    layout = kvq.k2v4_layout(H, D, 1.10, 8, T, 16)
    k, v = synth.gqa_kv(61, B, H, T, D)
    enc = gpu_k2v4(kvq, k, v, layout)
    q = synth.queries(62, (B, Hq, D))
    out = torch.empty((B, Hq, D), device="cuda")
    ws = torch.zeros(kvq.kv_attn_decode_k2v4_workspace_size(layout, B, Hq, T, pth), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_decode_k2v4(layout, to_dev(q), T, *enc, out, ws, 1 / np.sqrt(D), path=pth)
    Kf = k[0].astype(np.float16).astype(np.float64)
    Vf = v[0].astype(np.float16).astype(np.float64)
    ref = oracle.k2v4_attn(Kf, Vf, q[0], 1 / np.sqrt(D))
    got = out.cpu().numpy()[0]
    for h in range(Hq):
        assert rel_err(got[h], ref[h]) <= tol


@pytest.mark.parametrize("path", ["simt", "tensor"])
def test_config5_full_size(kvq, oracle, path):
    """4 sequences x 32768 cells, 2 kv heads x 256, 16 query heads, sinks 8, window 256, gain 1.10."""
    run_case(kvq, oracle, B=4, H=2, T=32768, D=256, Hq=16, sink=8, window=256, seed=5, path=path)
