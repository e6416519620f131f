"""K2/V4 appends on the GPU against the oracle (the Strata page's append
patterns and its "Fresh partial-group scale" rule): pools bit for bit after
every call, then the decode over a length that ends inside a 32-cell group
within 1e-5 (fp32 path) and 2e-3 (tensor-core path)."""
import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, TENSOR_TOL, kvq_module, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu

CAP = 512


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def _pools_gpu(B, H, D, slots):
    return (torch.zeros((B, H, CAP, D // 4), dtype=torch.uint8, device="cuda"),
            torch.zeros((B, H, CAP // 32, D), dtype=torch.int16, device="cuda"),
            torch.zeros((B, H, CAP, D // 32, 18), dtype=torch.uint8, device="cuda"),
            torch.zeros((B, H, slots, D), dtype=torch.int16, device="cuda"),
            torch.zeros((B, H, slots, D), dtype=torch.int16, device="cuda"))


def _pools_oracle(H, D, slots):
    return (np.zeros((H, CAP, D // 4), np.uint8), np.zeros((H, CAP // 32, D), np.uint16),
            np.zeros((H, CAP, D // 32, 18), np.uint8), np.zeros((H, slots, D), np.uint16),
            np.zeros((H, slots, D), np.uint16))


def _replay(kvq, oracle, cuts, D=256, H=2, B=2, gain=1.10, sink=8, window=64, seed=71):
    """Append the cells between consecutive cut points on both sides; compare
    every pool after every call; return the GPU pools, the oracle pools, the
    layouts and the K/V the cells came from."""
    layout = kvq.k2v4_layout(H, D, gain, sink, window, 16)
    OL = oracle.k2v4_layout(H, D, gain, sink, window, 16)
    slots = sink + window + 16
    k, v = synth.gqa_kv(seed, B, H, cuts[-1], D)
    gp = _pools_gpu(B, H, D, slots)
    op = [_pools_oracle(H, D, slots) for _ in range(B)]
    for a, b in zip(cuts[:-1], cuts[1:]):
        kvq.k2v4_append(layout, to_dev(k[:, :, a:b]), to_dev(v[:, :, a:b]), a, *gp)
        torch.cuda.synchronize()
        for s in range(B):
            op[s] = oracle.k2v4_append(*op[s], k[s, :, a:b], v[s, :, a:b], a, OL)
            for name, g, o in zip(("k_codes", "k_scales", "v_blocks", "k_win", "v_win"), gp, op[s]):
                np.testing.assert_array_equal(g[s].cpu().numpy().view(o.dtype), o,
                                              err_msg=f"{name} seq {s} after cells {a}..{b}")
    return gp, op, layout, OL, k, v


@pytest.mark.parametrize("name,cuts", [
    ("whole groups", [0, 32, 96]),
    ("partial group in one call", [0, 40]),
    ("first group partial", [0, 5, 6, 9, 32]),
    ("decode and verify windows", [0, 37, 38, 39, 42, 45, 64, 65, 68, 100, 101, 131]),
    ("prefill chunks mid-group", [0, 100, 200, 300, 400]),
    ("boundary split", [0, 64, 70]),
])
def test_append_patterns_bit_exact(kvq, oracle, name, cuts):
    _replay(kvq, oracle, cuts)


def test_append_head_dim_128(kvq, oracle):
    _replay(kvq, oracle, [0, 3, 35, 70, 133], D=128, H=2, B=3, seed=73)


@pytest.mark.parametrize("path", ["simt", "tensor"])
def test_decode_after_appends_ends_inside_a_group(kvq, oracle, path):
    """227 cells (7 groups and 3 cells of an eighth) written by appends, then
    decoded: the cells past the end of the last group are masked."""
    cuts = [0, 100, 131, 133, 200, 227]
    gp, op, layout, OL, k, v = _replay(kvq, oracle, cuts, seed=79)
    B, H, T, D = k.shape
    Hq = 16
    pth = kvq.PATH_SIMT if path == "simt" else kvq.PATH_TENSOR
    tol = SIMT_TOL if path == "simt" else TENSOR_TOL
    q = synth.queries(80, (B, Hq, D))
    out = torch.empty((B, Hq, D), device="cuda")
    ws = torch.zeros(kvq.kv_attn_decode_k2v4_workspace_size(layout, B, Hq, T, pth), dtype=torch.uint8, device="cuda")
    sm = 1.0 / np.sqrt(D)
    kvq.kv_attn_decode_k2v4(layout, to_dev(q), T, *gp, out, ws, sm, capacity=CAP, path=pth)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    got = out.cpu().numpy()
    for s in range(B):
        K, V = oracle.k2v4_reconstruct(*op[s], T, OL)
        ref = oracle.k2v4_attn(K, V, q[s], sm)
        for h in range(Hq):
            assert rel_err(got[s, h], ref[h]) <= tol, (s, h, path)
