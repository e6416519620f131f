"""Producers on the GPU against the oracle: codes and scales bit for bit."""
import numpy as np
import pytest
import torch

from gpu_common import gpu_encode, kvq_module, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def edge_rows(D=576):
    rows = [np.zeros(D), np.full(D, 3.0), np.full(D, -1e-3)]
    one = np.zeros(D)
    one[5] = -7.25
    rows.append(one)
    tiny = np.zeros(D)
    tiny[0] = 1e-44                      # scale underflows to zero
    rows.append(tiny)
    den = np.full(D, 1e-39)              # subnormal inputs
    rows.append(den)
    big = synth.mla_rows(77, 1, D)[0] * 1e30
    rows.append(big)
    mixed = synth.mla_rows(78, 1, D)[0]
    mixed[512:] = 0
    rows.append(mixed)
    return np.array(rows, np.float32)


def cases():
    yield "config1", synth.mla_rows(1, 256)
    yield "prefill_rows", synth.mla_rows(4, 2048, row_offset=126976)
    yield "edge", edge_rows()
    for n in (1, 7, 33):
        yield f"n{n}", synth.mla_rows(100 + n, n)


@pytest.mark.parametrize("fmt", ["kv8", "tq4"])
@pytest.mark.parametrize("bd", [(512, 64), (576,)])
def test_encode_bit_exact(kvq, oracle, fmt, bd):
    if fmt == "tq4" and bd == (576,):
        pytest.skip("576 is not a power of two (covered by the refusal tests)")
    layout = kvq.mla_layout(bd, seed=0)
    f = kvq.KVQ_KV8 if fmt == "kv8" else kvq.KVQ_TQ4
    for name, x in cases():
        codes, scales = gpu_encode(kvq, f, x, layout)
        if fmt == "kv8":
            oc, os_ = oracle.kv8_encode(x, bd)
        else:
            oc, os_ = oracle.tq4_encode(x, bd, seed=0)
        np.testing.assert_array_equal(codes.cpu().numpy(), oc, err_msg=name)
        np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32), err_msg=name)


@pytest.mark.parametrize("bd,seed", [((128,), 3), ((1024,), 5), ((2,), 1), ((16, 32), 9), ((256, 256), 12345)])
def test_tq4_other_widths(kvq, oracle, bd, seed):
    layout = kvq.mla_layout(bd, v_dim=bd[0], seed=seed)
    x = synth.mla_rows(seed, 50, sum(bd))
    codes, scales = gpu_encode(kvq, kvq.KVQ_TQ4, x, layout)
    oc, os_ = oracle.tq4_encode(x, bd, seed=seed)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_tq4_refuses_non_power_of_two(kvq):
    for bd in [(576,), (500, 76)]:
        layout = kvq.mla_layout(bd, v_dim=min(bd[0], 512))
        x = torch.ones((2, sum(bd)), device="cuda")
        assert kvq.tq4_encode_status(x, torch.empty(2, sum(bd) // 2, dtype=torch.uint8, device="cuda"),
                                     torch.empty(2, len(bd), device="cuda"), layout) == 2


def test_e4m3_conversion_matches_oracle_densely(kvq, oracle):
    """The oracle's e4m3 rounding against CUDA's own conversion instruction:
    rows whose amax is 448 get scale 1 exactly, so every other element is
    converted as it is.  Covers a dense stride of all f32 in [0, 448] plus
    every midpoint of the grid and its 8 neighbours on each side, both signs."""
    top = np.array([448.0], np.float32).view(np.uint32)[0]
    bits = np.arange(0, int(top), 29, dtype=np.uint32)
    grid = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32).view(np.uint32)
    near = (mids[:, None].astype(np.int64) + np.arange(-8, 9)[None, :]).ravel()
    near = near[(near >= 0) & (near <= int(top))].astype(np.uint32)
    vals = np.concatenate([bits, near]).view(np.float32)
    vals = np.concatenate([vals, -vals])
    per = 575
    n_rows = (len(vals) + per - 1) // per
    pad = np.zeros(n_rows * per, np.float32)
    pad[:len(vals)] = vals
    x = np.empty((n_rows, 576), np.float32)
    x[:, 0] = 448.0
    x[:, 1:] = pad.reshape(n_rows, per)
    layout = kvq.mla_layout((576,))
    codes, scales = gpu_encode(kvq, kvq.KVQ_KV8, x, layout)
    assert torch.all(scales == 1.0)
    got = codes.cpu().numpy()[:, 1:].ravel()[:len(vals)]
    want = oracle.e4m3_encode_array(vals)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(want[i])) for i in bad[:10]]


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("inverse", [False, True])
def test_tq4_rotate_matches_oracle(kvq, oracle, bf16, inverse):
    from gpu_common import queries
    layout = kvq.mla_layout(seed=7)
    qd, qv = queries(5, (40, 576), bf16)
    out = torch.empty((40, 576), dtype=torch.float32, device="cuda")
    kvq.tq4_rotate(qd, out, layout, inverse=inverse)
    ref = oracle.tq4_rotate(qv.astype(np.float64), seed=7, inverse=inverse)
    got = out.cpu().numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=2e-6 * np.abs(ref).max())
