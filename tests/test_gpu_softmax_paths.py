"""The tensor-core kernels' softmax paths, on inputs built to reach them, against
the oracle on every (sequence, head).

The kernels weight each tile against lagged running maxima: m over the scores
(row sums) and R over the scores plus log2 of the row's latent scale (the f16
context weights).  A tile whose values pass a reference by more than the lag
takes the exact path: column maxima over the tile, then the context
accumulator rescaled in tensor memory.  On the first tile of a work item that
path is always taken and rescales nothing; these tests make later tiles take
it, and read the kernels' counter of such tiles to show that they did.

* ``rescale``: sequences whose rows are scaled tile by tile -- alternating
  0.05 and 1.5 (even sequences) or growing 0.05 x 4^(k mod 4) (odd ones) -- so
  that a later tile's scores pass the running maximum by far more than 2^14.
* ``spread``: latent scales spanning 10^6 within every tile, with the scores
  carried by the rope block: rows with a 10^-3 latent block and a normal rope
  block (which hold the attention), rows with a 10^3 latent block and no rope
  (whose latent products rival them), and rows whose latent block is all zero
  (an inert block, latent scale 0).  The f16 context weights must stay exact to
  f16 precision relative to the largest weight.  For KV8 the query's rope part
  is scaled by 4, so that the attention-holding rows' weights sit near 10^-9
  of the largest-scale rows' (a chunk-wide weight reference fails there: its
  f16 weights underflow).  For TQ4 it stays at 1: the TQ4 levels enter the
  tensor cores as f16 (within 9.3e-5 of the codebook), and that rounding
  grows with the magnitude of the scores, which a rope part scaled by 4 pushes
  to 50 nats and past the 2e-3 bound (float64 emulation of the kernel's
  operands: 2.3e-3 at 4, 5.6e-4 at 1).

Shapes: 8 sequences x 4096 rows, 128 heads (work items of several 128-row
tiles).  Tolerance: the tensor-core bound, 2e-3 of each output vector's
largest magnitude.
"""
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from gpu_common import TENSOR_TOL, gpu_encode, kvq_module, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)
B, T, H = 8, 4096, 128


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


def rescale_rows(seed):
    x = synth.mla_rows(seed, B * T).reshape(B, T, 576)
    tile = np.arange(T) // 128
    for b in range(B):
        if b % 2 == 0:
            a = np.where(tile % 2 == 0, 0.05, 1.5)
        else:
            a = 0.05 * 4.0 ** (tile % 4)
        x[b] *= a.astype(np.float32)[:, None]
    return x.reshape(B * T, 576)


def spread_rows(seed):
    x = synth.mla_rows(seed, B * T)
    r = np.arange(B * T)
    big = r % 2 == 1
    inert = r % 7 == 3
    x[~big, :512] *= np.float32(1e-3)
    x[big, :512] *= np.float32(1e3)
    x[big, 512:] = 0.0
    x[inert, :512] = 0.0
    return x


def spread_queries(seed, rope_gain):
    q = synth.queries(seed, (B, H, 576))
    q[..., :512] *= np.float32(1e-4)
    q[..., 512:] *= np.float32(rope_gain)
    return q


def oracle_outputs(oracle, fmt, x, q, seed):
    """Every (sequence, head) output of the oracle over its own encoding of x."""
    oc, os_ = oracle.kv8_encode(x) if fmt == 1 else oracle.tq4_encode(x, seed=seed)
    xh = oracle.reconstruct(fmt, oc, os_, seed=seed)

    def one(b):
        return oracle.attn_dense(np.ascontiguousarray(xh[b * T:(b + 1) * T]), np.ascontiguousarray(q[b]), SM, 512)
    with ThreadPoolExecutor(max_workers=8) as ex:
        ref = list(ex.map(one, range(B)))
    return oc, os_, np.stack(ref)


def run_case(kvq, oracle, fmt, q_bf16, x, q32, seed):
    layout = kvq.mla_layout(seed=seed)
    codes, scales = gpu_encode(kvq, fmt, x, layout)
    if q_bf16:
        bits = synth.bf16_bits(q32)
        q_dev = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        q_or = synth.bf16_to_f32(bits)
    else:
        q_dev, q_or = to_dev(q32), q32
    cu = synth.cu_seqlens([T] * B)
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, B, H, B * T, layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_decode(fmt, q_dev, codes, scales, to_dev(cu), out, ws, B * T, SM, layout, kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    exact = kvq.read_exact_rescales(ws)
    oc, os_, ref = oracle_outputs(oracle, fmt, x, q_or, seed)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    worst = max(rel_err(got[b, h], ref[b, h]) for b in range(B) for h in range(H))
    return worst, exact


CASES = [(1, True), (1, False), (2, True), (2, False)]
IDS = ["kv8-bf16", "kv8-f32", "tq4-bf16", "tq4-f32"]


@pytest.mark.parametrize("fmt,q_bf16", CASES, ids=IDS)
def test_exact_rescale_path_on_later_tiles(kvq, oracle, fmt, q_bf16):
    x = rescale_rows(31)
    q = synth.queries(32, (B, H, 576))
    worst, exact = run_case(kvq, oracle, fmt, q_bf16, x, q, seed=5)
    assert exact > 0, "no tile after a work item's first took the exact path"
    assert worst <= TENSOR_TOL, worst


@pytest.mark.parametrize("fmt,q_bf16", CASES, ids=IDS)
def test_latent_scales_spanning_six_decades(kvq, oracle, fmt, q_bf16):
    x = spread_rows(33)
    q = spread_queries(34, 4.0 if fmt == 1 else 1.0)
    worst, _ = run_case(kvq, oracle, fmt, q_bf16, x, q, seed=6)
    assert worst <= TENSOR_TOL, worst


def test_plain_inputs_keep_the_lagged_path(kvq, oracle):
    """On the workloads' own value distribution later tiles rarely pass the lag:
    the counter stays well below the number of tiles."""
    x = synth.mla_rows(35, B * T)
    q = synth.queries(36, (B, H, 576))
    worst, exact = run_case(kvq, oracle, 1, True, x, q, seed=5)
    assert worst <= TENSOR_TOL, worst
    assert exact < B * T // 128, exact


def test_fused_append_step_against_the_oracle(kvq, oracle):
    """The one-launch decode step (new rows encoded inside the tensor-core
    decode) at 8 x 4096 rows, 128 heads, bf16 queries, checked directly against
    the oracle on every (sequence, head)."""
    layout = kvq.mla_layout()
    x = synth.mla_rows(37, B * T)
    x_new = synth.mla_rows(38, B)
    codes, scales = gpu_encode(kvq, 1, x, layout)
    cu = synth.cu_seqlens([T] * B)
    dst = cu[1:] - 1
    bits = synth.bf16_bits(synth.queries(39, (B, H, 576)))
    q_dev = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full((B, H, 512), float("nan"), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(1, B, H, B * T, layout, kvq.PATH_TENSOR), dtype=torch.uint8,
                     device="cuda")
    kvq.kv_attn_decode_append(1, to_dev(x_new), to_dev(dst), q_dev, codes, scales, to_dev(cu), out, ws, B * T, SM,
                              layout, kvq.PATH_TENSOR)
    torch.cuda.synchronize()
    assert kvq.read_device_error(ws) == 0
    xa = x.copy()
    xa[dst] = x_new
    oc, os_, ref = oracle_outputs(oracle, 1, xa, synth.bf16_to_f32(bits), 0)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    got = out.cpu().numpy()
    worst = max(rel_err(got[b, h], ref[b, h]) for b in range(B) for h in range(H))
    assert worst <= TENSOR_TOL, worst
