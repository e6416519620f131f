"""kv_attn_decode_append: one decode step with its new rows, against the
encoder launch followed by kv_attn_decode (bit for bit: same codes, same
scales, same outputs) and against the oracle."""
import math

import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, TENSOR_TOL, kvq_module, queries, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def make_case(kvq, fmt, lens, dst, seed, layout):
    """Pool holding every row of old content (dst rows included), plus the
    new rows to append at dst."""
    cu = synth.cu_seqlens(lens)
    n = int(cu[-1])
    x_old = synth.mla_rows(seed, n)
    x_new = synth.mla_rows(seed + 50, len(lens))
    row = 576 if fmt == 1 else 288
    codes = torch.empty((n, row), dtype=torch.uint8, device="cuda")
    scales = torch.empty((n, 2), dtype=torch.float32, device="cuda")
    (kvq.kv8_encode if fmt == 1 else kvq.tq4_encode)(to_dev(x_old), codes, scales, layout)
    return cu, x_old, x_new, codes, scales, to_dev(np.asarray(dst, np.int64))


def run_both(kvq, fmt, lens, dst, seed, H, path, bf16=True):
    layout = kvq.mla_layout(seed=seed)
    cu, x_old, x_new, codes, scales, dst_t = make_case(kvq, fmt, lens, dst, seed, layout)
    n = int(cu[-1])
    qd, qv = queries(seed + 1, (len(lens), H, 576), bf16)
    cut, xn = to_dev(cu), to_dev(x_new)
    outs, pools = [], []
    for fused in (True, False):
        c, s = codes.clone(), scales.clone()
        out = torch.full((len(lens), H, 512), float("nan"), device="cuda")
        ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, len(lens), H, n, layout, path), dtype=torch.uint8,
                         device="cuda")
        if fused:
            kvq.kv_attn_decode_append(fmt, xn, dst_t, qd, c, s, cut, out, ws, n, SM, layout, path)
        else:
            (kvq.kv8_encode if fmt == 1 else kvq.tq4_encode)(xn, c, s, layout, dst_rows=dst_t)
            kvq.kv_attn_decode(fmt, qd, c, s, cut, out, ws, n, SM, layout, path)
        torch.cuda.synchronize()
        assert kvq.read_device_error(ws) == 0
        outs.append(out.cpu().numpy())
        pools.append((c.cpu().numpy(), s.cpu().numpy()))
    x_all = x_old.copy()
    x_all[np.asarray(dst)] = x_new
    return cu, x_all, qv, outs, pools


def check_oracle(oracle, fmt, x_all, cu, qv, got, seed, tol, pairs):
    if fmt == 1:
        oc, os_ = oracle.kv8_encode(x_all)
    else:
        oc, os_ = oracle.tq4_encode(x_all, seed=seed)
    ref = oracle.attn_decode(fmt, oc, os_, qv, cu, SM, pairs=pairs, seed=seed)
    for (b, h), r in ref.items():
        assert rel_err(got[b, h], r) <= tol, (b, h)
    return oc, os_


def test_fused_kv8_equals_encode_then_decode(kvq, oracle):
    """Tensor path, KV8, bf16 query (the one-launch kernel): new rows at the end,
    the start and the middle of sequences, a one-row sequence, 128 heads."""
    lens = [1, 129, 700, 4096, 2, 3000, 128]
    cu = synth.cu_seqlens(lens)
    dst = [int(cu[0]), int(cu[1]), int(cu[2]) + 350, int(cu[4]) - 1, int(cu[4]) + 1, int(cu[5]) + 2047,
           int(cu[7]) - 1]
    cu, x_all, qv, outs, pools = run_both(kvq, 1, lens, dst, 71, 128, kvq.PATH_TENSOR)
    np.testing.assert_array_equal(pools[0][0], pools[1][0])
    np.testing.assert_array_equal(pools[0][1].view(np.uint32), pools[1][1].view(np.uint32))
    np.testing.assert_array_equal(outs[0], outs[1])
    pairs = [(b, h) for b in range(len(lens)) for h in (0, 63, 64, 127)]
    oc, os_ = check_oracle(oracle, 1, x_all, cu, qv, outs[0], 71, TENSOR_TOL, pairs)
    np.testing.assert_array_equal(pools[0][0], oc)          # the appended rows, bit-exact


def test_fused_config2_step(kvq, oracle):
    """The decode step of the benchmark: 8 x 4096 rows, the new row last; the
    one-launch kernel against the two-call path (bit for bit) and, on sampled
    (sequence, head) pairs, against the oracle; the appended rows bit-exact."""
    lens = [4096] * 8
    cu = synth.cu_seqlens(lens)
    cu, x_all, qv, outs, pools = run_both(kvq, 1, lens, list(cu[1:] - 1), 2, 128, kvq.PATH_TENSOR)
    np.testing.assert_array_equal(pools[0][0], pools[1][0])
    np.testing.assert_array_equal(outs[0], outs[1])
    assert np.all(np.isfinite(outs[0]))
    pairs = [(b, h) for b in (0, 3, 7) for h in (0, 64, 127)]
    oc, os_ = check_oracle(oracle, 1, x_all, cu, qv, outs[0], 2, TENSOR_TOL, pairs)
    np.testing.assert_array_equal(pools[0][0], oc)


@pytest.mark.parametrize("fmt,path,bf16", [(2, "tensor", True), (1, "simt", True), (1, "tensor", False)])
def test_other_paths_encode_then_decode(kvq, oracle, fmt, path, bf16):
    """Formats and paths without a one-launch kernel give the same results as the two calls."""
    lens = [300, 1, 513]
    cu = synth.cu_seqlens(lens)
    dst = [int(cu[1]) - 1, int(cu[1]), int(cu[2]) + 7]
    H = 128 if path == "tensor" else 16
    pth = kvq.PATH_TENSOR if path == "tensor" else kvq.PATH_SIMT
    cu, x_all, qv, outs, pools = run_both(kvq, fmt, lens, dst, 73, H, pth, bf16)
    np.testing.assert_array_equal(pools[0][0], pools[1][0])
    np.testing.assert_array_equal(outs[0], outs[1])
    tol = TENSOR_TOL if path == "tensor" else SIMT_TOL
    check_oracle(oracle, fmt, x_all, cu, qv, outs[0], 73, tol, [(b, h) for b in range(3) for h in (0, H - 1)])


def test_fused_refuses_row_outside_its_sequence(kvq):
    layout = kvq.mla_layout()
    lens = [200, 300]
    cu, _, x_new, codes, scales, _ = make_case(kvq, 1, lens, [0, 0], 81, layout)
    before = codes.clone()
    dst = to_dev(np.array([250, 499], np.int64))            # row 250 belongs to sequence 1
    qd, _ = queries(82, (2, 64, 576), True)
    out = torch.empty((2, 64, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(1, 2, 64, 500, layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_decode_append(1, to_dev(x_new), dst, qd, codes, scales, to_dev(cu), out, ws, 500, SM, layout,
                              kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 1
    np.testing.assert_array_equal(codes[:300].cpu().numpy(), before[:300].cpu().numpy())   # row 250 untouched
    assert not np.array_equal(codes[499].cpu().numpy(), before[499].cpu().numpy())         # row 499 appended
