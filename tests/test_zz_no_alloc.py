"""The allocation-free decode entry point against the regular one.

kv_attn_decode_noalloc serves callers that cannot allocate device memory (for
instance code running under CUDA graph capture, or a plugin whose host owns
all allocations): it keeps its scratch in the library's own fixed device
array instead of a caller workspace.  Two calls in a row, with different
shapes and formats, must give the regular entry point's outputs, and an
oversized request must be refused before any launch.  This file is collected
last so that a failure here comes after every other test has run.
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import SIMT_TOL, gpu_encode, kvq_module, queries, rel_err, to_dev
from quantized_kv_cache_kv8_gb300 import synth

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(192.0)


def _case(kvq, fmt, lens, H, bf16, seed):
    layout = kvq.mla_layout(seed=seed)
    cu = synth.cu_seqlens(lens)
    total = int(cu[-1])
    codes, scales = gpu_encode(kvq, fmt, synth.mla_rows(seed, total), layout)
    qd, _ = queries(seed + 1, (len(lens), H, 576), bf16)
    cu_d = to_dev(cu)
    ref = torch.empty((len(lens), H, 512), device="cuda")
    ws = torch.zeros(kvq.kv_attn_workspace_size(fmt, len(lens), H, total, layout), dtype=torch.uint8, device="cuda")
    kvq.kv_attn_decode(fmt, qd, codes, scales, cu_d, ref, ws, total, SM, layout)
    got = torch.full((len(lens), H, 512), float("nan"), device="cuda")
    kvq.kv_attn_decode_noalloc(fmt, qd, codes, scales, cu_d, got, total, SM, layout)
    torch.cuda.synchronize()
    return got.cpu().numpy(), ref.cpu().numpy()


def test_noalloc_matches_regular_entry_on_two_calls():
    kvq = kvq_module()
    for fmt, lens, H, bf16, seed in ((kvq.KVQ_KV8, [300, 0, 17, 1000], 32, True, 71),
                                     (kvq.KVQ_TQ4, [4096, 1, 2048], 128, False, 72)):
        got, ref = _case(kvq, fmt, lens, H, bf16, seed)
        assert np.all(np.isfinite(got))
        for b in range(len(lens)):
            for h in range(H):
                assert rel_err(got[b, h], ref[b, h]) <= SIMT_TOL, (fmt, b, h)


def test_noalloc_refuses_requests_beyond_its_scratch():
    kvq = kvq_module()
    # 100 sequences take two waves of 76 work items: 152 x 128 x 514 floats > 32 MiB
    q = torch.zeros((100, 128, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((100, 128, 512), device="cuda")
    cu = torch.zeros(101, dtype=torch.int64, device="cuda")
    codes = torch.zeros((16, 576), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((16, 2), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_attn_decode_noalloc(kvq.KVQ_KV8, q, codes, scales, cu, out, 50_000_000)
    assert e.value.status == 3
    assert torch.all(out == 0)
