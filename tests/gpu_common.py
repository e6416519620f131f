"""Helpers shared by the GPU parity tests (the tests themselves carry the gpu mark).

Parity metric for attention outputs: for every output vector (one per
sequence-or-token and head), max_d |gpu - oracle| / max_d |oracle|.  The
bounds are 1e-5 for the fp32 SIMT path and 2e-3 for the tensor-core path.
"""
import numpy as np
import pytest
import torch

from quantized_kv_cache_kv8_gb300 import synth

SIMT_TOL = 1e-5
TENSOR_TOL = 2e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def kvq_module():
    need_gpu()
    from quantized_kv_cache_kv8_gb300 import kvq
    kvq.lib()
    return kvq


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.max(np.abs(ref))
    if scale == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / scale)


def queries(seed, shape, bf16: bool):
    """(device tensor, f32 numpy values the oracle sees)."""
    q = synth.queries(seed, shape)
    if not bf16:
        return to_dev(q), q
    bits = synth.bf16_bits(q)
    t = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    return t, synth.bf16_to_f32(bits)


def gpu_encode(kvq, fmt, x: np.ndarray, layout):
    D = x.shape[1]
    n = x.shape[0]
    nb = layout.n_blocks
    row = kvq.row_bytes(fmt, layout)
    codes = torch.empty((n, row), dtype=torch.uint8, device="cuda")
    scales = torch.empty((n, nb), dtype=torch.float32, device="cuda")
    xt = to_dev(x)
    if fmt == kvq.KVQ_KV8:
        kvq.kv8_encode(xt, codes, scales, layout)
    elif fmt == kvq.KVQ_TQ4:
        kvq.tq4_encode(xt, codes, scales, layout)
    else:
        kvq.pq_encode(fmt, xt, codes, scales, layout)
    return codes, scales
