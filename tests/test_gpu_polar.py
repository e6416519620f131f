"""PolarQuant (codec 0 of the TQ tier) on the GPU against the oracle.

* encoder: codes and radii bit for bit at every width (2..6 bits), on the
  workload's rows, ragged row counts, edge rows and other block widths, with a
  scattered destination; a non-finite radius sets KVQ_ERR_NONFINITE;
* dequantizer: rows within 2e-6 of the oracle's float64 reconstruction
  (rotated and unrotated; f32 products down a tree of at most 9 levels);
* the fp32 attention consumer (trees rebuilt per tile in the rotated domain,
  the context unrotated once) within the fp32 bound 1e-5 of exact attention
  over the oracle's reconstruction: ragged decode with empty and one-row
  sequences, bf16 and f32 queries, the append step, the gather decode and a
  small chunked prefill;
* the tensor-core consumer of 4-bit rows (the TQ4 kernel with the trees
  rebuilt into f16 operands; KVQ_PATH_TENSOR only) within 4e-3: each leaf is
  an f32 product rounded once to f16 (up to 2^-11 relative, about five times
  the 9.3e-5 of TQ4's scaled levels), so the bound is twice the 2e-3 of the
  KV8/TQ4 tensor path (worst measured 2.7e-3, on 300- and 900-row sequences):
  the same ragged decode, the append step at the benchmark's size, a prefill.
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, TENSOR_TOL, gpu_encode, kvq_module, queries, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)
PQ_TENSOR_TOL = 2 * TENSOR_TOL
NONFINITE = 9


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def edge_rows(D=576):
    rows = [np.zeros(D), np.full(D, 3.0), np.full(D, -1e-3)]
    one = np.zeros(D)
    one[5] = -7.25
    rows.append(one)
    rows.append(np.full(D, 1e-39))                       # subnormal inputs
    big = synth.mla_rows(77, 1, D)[0] * 1e15             # large, squares still finite
    rows.append(big)
    mixed = synth.mla_rows(78, 1, D)[0]
    mixed[512:] = 0                                      # inert rope block
    rows.append(mixed)
    pairs = synth.mla_rows(79, 1, D)[0]
    pairs[0:64:2] = 0                                    # zero and axis-aligned pairs
    pairs[1:64:4] = -0.0
    rows.append(pairs)
    return np.array(rows, np.float32)


def cases():
    yield "rows", synth.mla_rows(1, 512)
    yield "prefill_rows", synth.mla_rows(4, 1024, row_offset=126976)
    yield "edge", edge_rows()
    for n in (1, 7, 33):
        yield f"n{n}", synth.mla_rows(100 + n, n)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
def test_encode_bit_exact(kvq, oracle, bits):
    fmt = kvq.pq_format(bits)
    layout = kvq.mla_layout(seed=3)
    for name, x in cases():
        codes, radii = gpu_encode(kvq, fmt, x, layout)
        oc, orr = oracle.pq_encode(x, bits, seed=3)
        np.testing.assert_array_equal(codes.cpu().numpy(), oc, err_msg=name)
        np.testing.assert_array_equal(radii.cpu().numpy().view(np.uint32), orr.view(np.uint32), err_msg=name)


@pytest.mark.parametrize("bd,seed,bits", [((64,), 3, 3), ((1024,), 5, 4), ((2,), 1, 5), ((16, 32), 9, 6),
                                          ((256, 256), 12345, 2), ((8, 512), 7, 4)])
def test_other_widths(kvq, oracle, bd, seed, bits):
    layout = kvq.mla_layout(bd, v_dim=bd[0], seed=seed)
    x = synth.mla_rows(seed, 50, sum(bd))
    codes, radii = gpu_encode(kvq, kvq.pq_format(bits), x, layout)
    oc, orr = oracle.pq_encode(x, bits, bd, seed=seed)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(radii.cpu().numpy().view(np.uint32), orr.view(np.uint32))


def test_scattered_destination_rows(kvq, oracle):
    layout = kvq.mla_layout(seed=2)
    x = synth.mla_rows(11, 40)
    dst = np.random.default_rng(0).permutation(64)[:40].astype(np.int64)
    codes = torch.zeros((64, kvq.row_bytes(14)), dtype=torch.uint8, device="cuda")
    radii = torch.zeros((64, 2), dtype=torch.float32, device="cuda")
    kvq.pq_encode(14, to_dev(x), codes, radii, layout, dst_rows=to_dev(dst))
    oc, orr = oracle.pq_encode(x, 4, seed=2)
    np.testing.assert_array_equal(codes.cpu().numpy()[dst], oc)
    np.testing.assert_array_equal(radii.cpu().numpy()[dst].view(np.uint32), orr.view(np.uint32))


def test_non_finite_radius_is_flagged(kvq, oracle):
    x = synth.mla_rows(12, 16)
    x[3, 7] = np.nan
    x[9, :64] = np.float32(1e30)          # squares past the f32 range
    layout = kvq.mla_layout()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes = torch.empty((16, kvq.row_bytes(13)), dtype=torch.uint8, device="cuda")
    radii = torch.empty((16, 2), dtype=torch.float32, device="cuda")
    kvq.pq_encode(13, to_dev(x), codes, radii, layout, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == NONFINITE
    good = [i for i in range(16) if i not in (3, 9)]
    oc, orr = oracle.pq_encode(x[good], 3)
    np.testing.assert_array_equal(codes.cpu().numpy()[good], oc)
    np.testing.assert_array_equal(radii.cpu().numpy()[good].view(np.uint32), orr.view(np.uint32))


@pytest.mark.parametrize("bits", [2, 3, 4, 6])
@pytest.mark.parametrize("rotated", [False, True])
def test_decode_matches_oracle(kvq, oracle, bits, rotated):
    layout = kvq.mla_layout(seed=5)
    # the subnormal row is left out: its f32 products keep fewer significant bits
    x = np.concatenate([synth.mla_rows(13, 300), np.delete(edge_rows(), 4, axis=0)])
    fmt = kvq.pq_format(bits)
    codes, radii = gpu_encode(kvq, fmt, x, layout)
    out = torch.full((x.shape[0], 576), float("nan"), device="cuda")
    kvq.pq_decode(fmt, codes, radii, out, layout, rotated=rotated)
    oc, orr = oracle.pq_encode(x, bits, seed=5)
    ref = oracle.pq_decode(oc, orr, bits, seed=5, rotated=rotated)
    got = out.cpu().numpy()
    for t in range(x.shape[0]):
        assert rel_err(got[t], ref[t]) <= 2e-6, t


def ragged_case(seed, lengths):
    cu = synth.cu_seqlens(lengths)
    x = synth.mla_rows(seed, int(cu[-1]))
    return x, cu


@pytest.mark.parametrize("bits,bf16", [(4, True), (4, False), (2, True), (6, False), (3, True), (5, False)])
def test_ragged_decode_against_oracle(kvq, oracle, bits, bf16):
    lengths = [0, 1, 17, 300, 1000, 129]
    x, cu = ragged_case(20 + bits, lengths)
    B, H = len(lengths), 128
    fmt = kvq.pq_format(bits)
    layout = kvq.mla_layout(seed=6)
    codes, radii = gpu_encode(kvq, fmt, x, layout)
    q_dev, q = queries(21 + bits, (B, H, 576), bf16)
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    S = kvq.PATH_SIMT
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, B, H, int(cu[-1]), layout, S), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_decode(fmt, q_dev, codes, radii, to_dev(cu), out, ws, int(cu[-1]), SM, layout, S)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    oc, orr = oracle.pq_encode(x, bits, seed=6)
    xh = oracle.pq_decode(oc, orr, bits, seed=6)
    got = out.cpu().numpy()
    for b in range(B):
        ref = oracle.attn_dense(xh[cu[b]:cu[b + 1]], np.ascontiguousarray(q[b]), SM, 512)
        for h in range(H):
            assert rel_err(got[b, h], ref[h]) <= SIMT_TOL, (b, h)


def test_tensor_path_serves_four_bits_only(kvq):
    layout = kvq.mla_layout()
    for bits in (2, 3, 5, 6):
        assert kvq.kv_attn_workspace_size(kvq.pq_format(bits), 2, 128, 100, layout, path=kvq.PATH_TENSOR) == 0
    assert kvq.kv_attn_workspace_size(14, 2, 128, 100, layout, path=kvq.PATH_TENSOR) > 0
    # AUTO keeps PolarQuant on the fp32 consumer
    assert kvq.kv_attn_workspace_size(14, 2, 128, 100, layout) == \
        kvq.kv_attn_workspace_size(14, 2, 128, 100, layout, path=kvq.PATH_SIMT)


def test_append_step_and_gather(kvq, oracle):
    lengths = [5, 260, 800]
    x, cu = ragged_case(30, lengths)
    B, H = 3, 64
    layout = kvq.mla_layout(seed=8)
    codes, radii = gpu_encode(kvq, 14, x, layout)
    x_new = synth.mla_rows(31, B)
    dst = (cu[1:] - 1).astype(np.int64)
    q_dev, q = queries(32, (B, H, 576), True)
    out = torch.empty((B, H, 512), device="cuda")
    S = kvq.PATH_SIMT
    ws = torch.zeros(kvq.kv_attn_workspace_size(14, B, H, int(cu[-1]), layout, S), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_decode_append(14, to_dev(x_new), to_dev(dst), q_dev, codes, radii, to_dev(cu), out, ws, int(cu[-1]),
                              SM, layout, S)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    xa = x.copy()
    xa[dst] = x_new
    oc, orr = oracle.pq_encode(xa, 4, seed=8)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    xh = oracle.pq_decode(oc, orr, 4, seed=8)
    got = out.cpu().numpy()
    for b in range(B):
        ref = oracle.attn_dense(xh[cu[b]:cu[b + 1]], np.ascontiguousarray(q[b]), SM, 512)
        for h in range(H):
            assert rel_err(got[b, h], ref[h]) <= SIMT_TOL, (b, h)
    # gather: unsorted rows with a repeat, across sequences
    sel = np.array([1000, 3, 3, 517, 64, 900, 2, 265], np.int64)
    cu_sel = synth.cu_seqlens([3, 0, 5])
    ws2 = torch.zeros(kvq.kv_attn_gather_workspace_size(14, B, H, 8, True, layout), dtype=torch.uint8,
                      device="cuda")
    kvq.kv_attn_decode_gather(14, q_dev, codes, radii, to_dev(sel), to_dev(cu_sel), out, ws2, 8, SM, layout)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws2) == 0
    got = out.cpu().numpy()
    for b in range(B):
        rows = sel[cu_sel[b]:cu_sel[b + 1]]
        ref = oracle.attn_dense(np.ascontiguousarray(xh[rows]), np.ascontiguousarray(q[b]), SM, 512)
        for h in range(H):
            assert rel_err(got[b, h], ref[h]) <= SIMT_TOL, (b, h)


def test_small_prefill(kvq, oracle):
    P, N, H = 700, 24, 32
    layout = kvq.mla_layout(seed=9)
    x = synth.mla_rows(40, P + N)
    rb = kvq.row_bytes(15)
    codes = torch.zeros((P + N, rb), dtype=torch.uint8, device="cuda")
    radii = torch.zeros((P + N, 2), dtype=torch.float32, device="cuda")
    pc, pr = gpu_encode(kvq, 15, x[:P], layout)
    codes[:P], radii[:P] = pc, pr
    q_dev, q = queries(41, (N, H, 576), False)
    out = torch.empty((N, H, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_prefill_workspace_size(15, H, P, N, layout), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_prefill(15, to_dev(x[P:]), q_dev, codes, radii, P, out, ws, SM, layout)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    oc, orr = oracle.pq_encode(x, 5, seed=9)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    xh = oracle.pq_decode(oc, orr, 5, seed=9)
    got = out.cpu().numpy()
    for j in range(N):
        ref = oracle.attn_dense(np.ascontiguousarray(xh[:P + j + 1]), np.ascontiguousarray(q[j]), SM, 512)
        for h in range(H):
            assert rel_err(got[j, h], ref[h]) <= SIMT_TOL, (j, h)


def test_bench_step_at_full_size(kvq, oracle):
    """The PolarQuant-4 step the benchmark times (8 x 4096 rows, 128 heads,
    bf16 queries, the step's 8 rows appended; fp32 consumer), every
    (sequence, head) against the oracle."""
    B, T, H = 8, 4096, 128
    layout = kvq.mla_layout(seed=4)
    x = synth.mla_rows(2, B * T)
    codes, radii = gpu_encode(kvq, 14, x, layout)
    cu = synth.cu_seqlens([T] * B)
    dst = (cu[1:] - 1).astype(np.int64)
    x_new = synth.mla_rows(102, B)
    q_dev, q = queries(3, (B, H, 576), True)
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    S = kvq.PATH_SIMT
    ws = torch.zeros(kvq.kv_attn_workspace_size(14, B, H, B * T, layout, S), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_decode_append(14, to_dev(x_new), to_dev(dst), q_dev, codes, radii, to_dev(cu), out, ws, B * T, SM,
                              layout, S)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    xa = x.copy()
    xa[dst] = x_new
    oc, orr = oracle.pq_encode(xa, 4, seed=4)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(radii.cpu().numpy().view(np.uint32), orr.view(np.uint32))
    xh = oracle.pq_decode(oc, orr, 4, seed=4)
    got = out.cpu().numpy()
    for b in range(B):
        ref = oracle.attn_dense(np.ascontiguousarray(xh[cu[b]:cu[b + 1]]), np.ascontiguousarray(q[b]), SM, 512)
        for h in range(H):
            assert rel_err(got[b, h], ref[h]) <= SIMT_TOL, (b, h)


@pytest.mark.parametrize("bits", [2, 6])
def test_encode_at_ragged_pool_scale(kvq, oracle, bits):
    """An encode of the ragged workload's 131072-row master block; 3000
    sampled rows bit for bit against the oracle."""
    layout = kvq.mla_layout(seed=4)
    x = synth.mla_rows(4, 131072)
    codes, radii = gpu_encode(kvq, kvq.pq_format(bits), x, layout)
    rows = np.sort(np.random.default_rng(bits).choice(131072, 3000, replace=False))
    oc, orr = oracle.pq_encode(np.ascontiguousarray(x[rows]), bits, seed=4)
    np.testing.assert_array_equal(codes.cpu().numpy()[rows], oc)
    np.testing.assert_array_equal(radii.cpu().numpy()[rows].view(np.uint32), orr.view(np.uint32))


@pytest.mark.parametrize("bf16", [True, False], ids=["bf16", "f32"])
def test_tensor_ragged_decode_against_oracle(kvq, oracle, bf16):
    lengths = [0, 1, 17, 300, 1000, 129, 2048]
    x, cu = ragged_case(60, lengths)
    B, H = len(lengths), 128
    layout = kvq.mla_layout(seed=6)
    codes, radii = gpu_encode(kvq, 14, x, layout)
    q_dev, q = queries(61, (B, H, 576), bf16)
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(14, B, H, int(cu[-1]), layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_decode(14, q_dev, codes, radii, to_dev(cu), out, ws, int(cu[-1]), SM, layout, kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    oc, orr = oracle.pq_encode(x, 4, seed=6)
    xh = oracle.pq_decode(oc, orr, 4, seed=6)
    got = out.cpu().numpy()
    for b in range(B):
        ref = oracle.attn_dense(np.ascontiguousarray(xh[cu[b]:cu[b + 1]]), np.ascontiguousarray(q[b]), SM, 512)
        for h in range(H):
            assert rel_err(got[b, h], ref[h]) <= PQ_TENSOR_TOL, (b, h)


def test_tensor_bench_step_at_full_size(kvq, oracle):
    """The benchmark's PolarQuant-4 step (8 x 4096 rows, 128 heads, bf16, the
    step's rows appended) on the tensor-core path, every (sequence, head)."""
    B, T, H = 8, 4096, 128
    layout = kvq.mla_layout(seed=4)
    x = synth.mla_rows(2, B * T)
    codes, radii = gpu_encode(kvq, 14, x, layout)
    cu = synth.cu_seqlens([T] * B)
    dst = (cu[1:] - 1).astype(np.int64)
    x_new = synth.mla_rows(102, B)
    q_dev, q = queries(3, (B, H, 576), True)
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(14, B, H, B * T, layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_decode_append(14, to_dev(x_new), to_dev(dst), q_dev, codes, radii, to_dev(cu), out, ws, B * T, SM,
                              layout, kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    xa = x.copy()
    xa[dst] = x_new
    oc, orr = oracle.pq_encode(xa, 4, seed=4)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    xh = oracle.pq_decode(oc, orr, 4, seed=4)
    got = out.cpu().numpy()
    for b in range(B):
        ref = oracle.attn_dense(np.ascontiguousarray(xh[cu[b]:cu[b + 1]]), np.ascontiguousarray(q[b]), SM, 512)
        for h in range(H):
            assert rel_err(got[b, h], ref[h]) <= PQ_TENSOR_TOL, (b, h)


def test_tensor_prefill(kvq, oracle):
    P, N, H = 900, 20, 64
    layout = kvq.mla_layout(seed=9)
    x = synth.mla_rows(62, P + N)
    rb = kvq.row_bytes(14)
    codes = torch.zeros((P + N, rb), dtype=torch.uint8, device="cuda")
    radii = torch.zeros((P + N, 2), dtype=torch.float32, device="cuda")
    pc, pr = gpu_encode(kvq, 14, x[:P], layout)
    codes[:P], radii[:P] = pc, pr
    q_dev, q = queries(63, (N, H, 576), True)
    out = torch.empty((N, H, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_prefill_workspace_size(14, H, P, N, layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_prefill(14, to_dev(x[P:]), q_dev, codes, radii, P, out, ws, SM, layout, kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    oc, orr = oracle.pq_encode(x, 4, seed=9)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    xh = oracle.pq_decode(oc, orr, 4, seed=9)
    got = out.cpu().numpy()
    for j in range(N):
        ref = oracle.attn_dense(np.ascontiguousarray(xh[:P + j + 1]), np.ascontiguousarray(q[j]), SM, 512)
        for h in range(H):
            assert rel_err(got[j, h], ref[h]) <= PQ_TENSOR_TOL, (j, h)
