"""kv_attn_decode_gather: decode over selected rows (absolute pool indices),
against the oracle over the same rows, against kv_attn_decode when the
selection is each sequence's own range (bit for bit), and its error word for
an index outside the pool."""
import math

import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, TENSOR_TOL, gpu_encode, kvq_module, queries, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)
POOL = 20000


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def selections(seed, ks):
    """Per sequence: k pool rows, unsorted, with a few repeats where k > 8."""
    rng = np.random.default_rng(seed)
    out = []
    for k in ks:
        s = rng.integers(0, POOL, size=k).astype(np.int64)
        if k > 8:
            s[-3:] = s[:3]
        out.append(s)
    return out


@pytest.mark.parametrize("fmt,path,bf16,H", [(1, "tensor", True, 128), (1, "simt", True, 16), (2, "auto", True, 128),
                                             (1, "auto", False, 64)])
def test_gather_matches_oracle(kvq, oracle, fmt, path, bf16, H):
    seed = 91
    layout = kvq.mla_layout(seed=seed)
    x = synth.mla_rows(seed, POOL)
    codes, scales = gpu_encode(kvq, fmt, x, layout)
    ks = [0, 1, 2048, 300, 129, 4096]
    sels = selections(seed, ks)
    cu_sel = synth.cu_seqlens(ks)
    sel = np.concatenate(sels)
    qd, qv = queries(seed + 1, (len(ks), H, 576), bf16)
    pth = {"tensor": kvq.PATH_TENSOR, "simt": kvq.PATH_SIMT, "auto": kvq.PATH_AUTO}[path]
    n = int(cu_sel[-1])
    ws = torch.zeros(kvq.kv_attn_gather_workspace_size(fmt, len(ks), H, n, bf16, layout, pth), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((len(ks), H, 512), float("nan"), device="cuda")
    kvq.kv_attn_decode_gather(fmt, qd, codes, scales, to_dev(sel), to_dev(cu_sel), out, ws, n, SM, layout, pth)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    got = out.cpu().numpy()
    assert np.all(got[0] == 0.0)                       # nothing selected
    if fmt == 1:
        oc, os_ = oracle.kv8_encode(x)
    else:
        oc, os_ = oracle.tq4_encode(x, seed=seed)
    tol = SIMT_TOL if (path == "simt" or not bf16 or fmt == 2) else TENSOR_TOL
    for b, s in enumerate(sels):
        if len(s) == 0:
            continue
        xh = oracle.reconstruct(fmt, oc[s], os_[s], seed=seed)
        heads = [0, H // 2, H - 1]
        ref = oracle.attn_dense(xh, qv[b, heads], SM, 512)
        for i, h in enumerate(heads):
            assert rel_err(got[b, h], ref[i]) <= tol, (b, h)


@pytest.mark.parametrize("path", ["tensor", "simt"])
def test_gather_of_own_ranges_equals_decode(kvq, path):
    lens = [700, 1, 4096, 129]
    cu = synth.cu_seqlens(lens)
    layout = kvq.mla_layout()
    x = synth.mla_rows(93, int(cu[-1]))
    codes, scales = gpu_encode(kvq, 1, x, layout)
    H = 128
    qd, _ = queries(94, (len(lens), H, 576), True)
    pth = kvq.PATH_TENSOR if path == "tensor" else kvq.PATH_SIMT
    n = int(cu[-1])
    outs = []
    for gather in (True, False):
        out = torch.empty((len(lens), H, 512), device="cuda")
        if gather:
            ws = torch.zeros(kvq.kv_attn_gather_workspace_size(1, len(lens), H, n, True, layout, pth),
                             dtype=torch.uint8, device="cuda")
            kvq.kv_attn_decode_gather(1, qd, codes, scales, to_dev(np.arange(n, dtype=np.int64)), to_dev(cu), out,
                                      ws, n, SM, layout, pth)
        else:
            ws = torch.zeros(kvq.kv_attn_workspace_size(1, len(lens), H, n, layout, pth), dtype=torch.uint8,
                             device="cuda")
            kvq.kv_attn_decode(1, qd, codes, scales, to_dev(cu), out, ws, n, SM, layout, pth)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])


def test_gather_index_outside_pool_sets_error(kvq):
    layout = kvq.mla_layout()
    x = synth.mla_rows(95, 1000)
    codes, scales = gpu_encode(kvq, 1, x, layout)
    sel = np.array([5, 999, 1000, 7, -3], np.int64)
    cu_sel = np.array([0, 2, 5], np.int64)
    qd, _ = queries(96, (2, 64, 576), True)
    ws = torch.zeros(kvq.kv_attn_gather_workspace_size(1, 2, 64, 5, True, layout), dtype=torch.uint8, device="cuda")
    out = torch.empty((2, 64, 512), device="cuda")
    kvq.kv_attn_decode_gather(1, qd, codes, scales, to_dev(sel), to_dev(cu_sel), out, ws, 5, SM, layout)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 1
    assert np.all(np.isfinite(out.cpu().numpy()))


def test_gather_tensor_path_limits(kvq):
    layout = kvq.mla_layout()
    assert kvq.kv_attn_gather_workspace_size(2, 2, 128, 100, True, layout, kvq.PATH_TENSOR) == 0
    assert kvq.kv_attn_gather_workspace_size(1, 2, 128, 100, False, layout, kvq.PATH_TENSOR) == 0
    assert kvq.kv_attn_gather_workspace_size(1, 2, 128, 100, True, layout, kvq.PATH_TENSOR) > 0
