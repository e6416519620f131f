"""The opt-in launch timing hook: each timed decode call yields one record
with a positive partial-kernel time and a positive merge time, results are the
same as untimed, and nothing is recorded once it is turned off."""
import numpy as np
import pytest
import torch

from gpu_common import kvq_module
from test_gpu_attention import run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    return kvq_module()


@pytest.mark.parametrize("path_name", ["simt", "tensor"])
def test_timing_records_each_call(kvq, path_name):
    path = {"simt": kvq.PATH_SIMT, "tensor": kvq.PATH_TENSOR}[path_name]
    _, _, _, untimed, _ = run_decode(kvq, 1, [300, 1000, 129], 64, True, 71, path)
    kvq.timing_enable(8)
    try:
        for _ in range(3):
            _, _, _, timed, _ = run_decode(kvq, 1, [300, 1000, 129], 64, True, 71, path)
        part, merge, n = kvq.timing_read()
    finally:
        kvq.timing_enable(0)
    assert n == 3
    assert part > 0.0 and merge > 0.0
    np.testing.assert_array_equal(timed, untimed)
    # ring emptied by the read, and nothing recorded while off
    run_decode(kvq, 1, [300], 64, True, 71, path)
    assert kvq.timing_read() == (0.0, 0.0, 0)


def test_timing_ring_keeps_the_last_calls(kvq):
    kvq.timing_enable(2)
    try:
        for _ in range(5):
            run_decode(kvq, 1, [256], 64, True, 72, kvq.PATH_TENSOR)
        torch.cuda.synchronize()
        _, _, n = kvq.timing_read()
    finally:
        kvq.timing_enable(0)
    assert n == 2
