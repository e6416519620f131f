"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and its host-side logic (validation, workspace sizing, the
codebook constants) behaves.  No call here launches a kernel."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def kvq():
    from quantized_kv_cache_kv8_gb300 import kvq as K
    K.lib()
    return K


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(kvq):
    names = declared_functions()
    assert len(names) >= 14, names
    for n in names:
        assert hasattr(kvq.lib(), n), n


def test_status_strings_and_version(kvq):
    assert kvq.version() == "0.1.0"
    for s in range(11):
        assert kvq.status_string(s)


def test_codebook_constants_equal_the_oracle(kvq, oracle):
    lv, th = kvq.codebook(16)
    olv, oth = oracle.tq4_codebook()
    np.testing.assert_array_equal(np.array(lv, np.float32).view(np.uint32), olv.view(np.uint32))
    np.testing.assert_array_equal(np.array(th, np.float32).view(np.uint32), oth.view(np.uint32))
    lv, th = kvq.codebook(4)
    olv, oth = oracle.k2_codebook()
    np.testing.assert_array_equal(np.array(lv, np.float32).view(np.uint32), olv.view(np.uint32))
    np.testing.assert_array_equal(np.array(th, np.float32).view(np.uint32), oth.view(np.uint32))


def test_tq4_refuses_non_power_of_two_before_launch(kvq):
    L = kvq.lib()
    for bd in [(576,), (500, 76), (512, 60)]:
        lay = kvq.mla_layout(bd, v_dim=min(bd[0], 512))
        assert L.tq4_encode(None, 4, C.byref(lay), None, None, None, None, None) == 2
        assert L.tq4_rotate(None, 0, 4, C.byref(lay), 0, None, None) == 2
        assert L.kv_attn_workspace_size(2, C.byref(lay), 1, 16, 100, 0) == 0
        assert L.kv_attn_decode(2, C.byref(lay), None, 0, 1, 16, None, None, None, 100, 0.1, None, None, 0, 0,
                                None) == 2


def test_argument_validation(kvq):
    L = kvq.lib()
    lay = kvq.mla_layout()
    assert L.kv8_encode(None, -1, C.byref(lay), None, None, None, None, None) == 1
    assert L.kv8_encode(None, 0, C.byref(lay), None, None, None, None, None) == 0    # empty is a no-op
    assert L.kv8_encode(None, 3, C.byref(lay), None, None, None, None, None) == 1    # null pointers
    assert L.kv8_encode(None, 3, None, None, None, None, None, None) == 1
    # workspace too small is reported before any launch
    need = kvq.kv_attn_workspace_size(1, 8, 128, 32768)
    assert need > 0
    d = C.c_void_p(256)     # a dummy device address, aligned for every operand (never dereferenced)
    assert L.kv_attn_decode(1, C.byref(lay), d, 1, 8, 128, d, d, d, 32768, 0.07, d, d, need - 1, 0, None) == 3
    # unsupported attention layouts
    odd = kvq.mla_layout((256, 64), v_dim=256)
    assert kvq.kv_attn_workspace_size(1, 1, 16, 100, layout=odd) == 0
    k2 = kvq.k2v4_layout()
    k2.group = 16
    assert L.k2v4_encode(C.byref(k2), None, None, 1, 64, 64, None, None, None, None, None, None, None) == 5


def test_workspace_sizes_grow_with_work(kvq):
    item = 128 * 514 * 4                      # one work item's partial state, 128 heads
    a = kvq.kv_attn_workspace_size(1, 8, 128, 32768)
    b = kvq.kv_attn_workspace_size(1, 32, 128, 2_100_000)
    assert 0 < a
    # tensor-core split: a host chunk when it guarantees one wave (76 items of
    # 64 heads per wave for KV8) near the ideal size: 8 x 4096 rows -> 512-row
    # chunks, 64 + 8 items; otherwise the device balances items over at most
    # 4 waves for KV8 and 6 for TQ4 (76 items of 64 heads, 38 items of 32
    # heads per wave; whole waves per 76 / 38 sequences), never more than one
    # per 128-row tile plus one per sequence
    assert a == 256 + (64 + 8) * item
    assert b == 256 + 4 * 76 * item
    assert kvq.kv_attn_workspace_size(2, 8, 128, 32768) == 256 + 6 * 38 * item
    # the PolarQuant-4 tensor consumer runs the TQ4 kernel's 32-head CTAs
    assert kvq.kv_attn_workspace_size(kvq.KVQ_PQ4, 8, 128, 32768, path=kvq.PATH_TENSOR) == 256 + 6 * 38 * item
    # a ragged batch of 32 sequences: one wave holds 38 of them, so 6 waves of 38
    assert kvq.kv_attn_workspace_size(2, 32, 128, 2_100_000) == 256 + 6 * 38 * item
    assert kvq.kv_attn_workspace_size(1, 8, 128, 1000) == 256 + (8 + 8) * item
    assert kvq.kv_attn_workspace_size(1, 100, 128, 10**6) == 256 + 4 * 152 * item
    # the SIMT split grows with the rows
    s1 = kvq.kv_attn_workspace_size(1, 8, 128, 32768, path=kvq.PATH_SIMT)
    s2 = kvq.kv_attn_workspace_size(1, 32, 128, 2_100_000, path=kvq.PATH_SIMT)
    assert 0 < s1 < s2
    p = kvq.kv_attn_prefill_workspace_size(2, 128, 126976, 2048)
    assert p >= 2048 * 128 * 514 * 4
    k = kvq.kv_attn_decode_k2v4_workspace_size(kvq.k2v4_layout(), 4, 16, 32768)
    assert k > 0


def test_decode_append_validates_before_launch(kvq):
    L = kvq.lib()
    lay = kvq.mla_layout()
    # null x_new / dst_rows, fewer rows than sequences, no workspace: refused on the host
    assert L.kv_attn_decode_append(1, C.byref(lay), None, None, None, 1, 2, 64, None, None, None, 10, 0.1, None,
                                   None, 0, 0, None) == 1
    dummy = C.c_void_p(256)
    assert L.kv_attn_decode_append(1, C.byref(lay), dummy, dummy, dummy, 1, 4, 64, dummy, dummy, dummy, 3, 0.1,
                                   dummy, dummy, 1 << 30, 0, None) == 1
    assert L.kv_attn_decode_append(1, C.byref(lay), dummy, dummy, dummy, 1, 2, 64, dummy, dummy, dummy, 10, 0.1,
                                   dummy, None, 0, 0, None) == 3
    bad = kvq.mla_layout((500, 76))
    assert L.kv_attn_decode_append(2, C.byref(bad), dummy, dummy, dummy, 1, 2, 64, dummy, dummy, dummy, 10, 0.1,
                                   dummy, dummy, 1 << 30, 0, None) == 2
    # empty batch: nothing to do
    assert L.kv_attn_decode_append(1, C.byref(lay), None, None, None, 1, 0, 64, None, None, None, 0, 0.1, None,
                                   None, 0, 0, None) == 0


def test_attention_refuses_misaligned_pointers(kvq):
    """Checked on the host before any launch (no GPU needed)."""
    L = kvq.lib()
    lay = kvq.mla_layout()
    ok, odd = C.c_void_p(1 << 20), C.c_void_p((1 << 20) + 16)     # 16-byte but not 32-byte aligned
    ws = C.c_void_p(1 << 21)
    # codes pointer off a 32-byte boundary
    assert L.kv_attn_decode(1, C.byref(lay), ok, 1, 2, 64, odd, ok, ok, 10, 0.1, ok, ws, 1 << 30, 0, None) == 1
    # query off a 16-byte boundary
    assert L.kv_attn_decode(1, C.byref(lay), C.c_void_p((1 << 20) + 8), 1, 2, 64, ok, ok, ok, 10, 0.1, ok, ws,
                            1 << 30, 0, None) == 1
    assert L.kv_attn_decode_append(1, C.byref(lay), C.c_void_p((1 << 20) + 4), ok, ok, 1, 2, 64, ok, ok, ok, 10,
                                   0.1, ok, ws, 1 << 30, 0, None) == 1


def test_tq4_tensor_level_scale_keeps_levels_near_f16(oracle):
    """The tensor-core TQ4 kernel feeds f16(f32(level * scale)) to the MMA; the
    scale in its source keeps every level within 1e-4 relative of its f16 copy
    (unscaled levels are off by up to 3.2e-4)."""
    src = open(os.path.join(ROOT, "quantized_kv_cache_kv8_gb300", "csrc", "attn_tc_tq4.cu")).read()
    g = np.float32(float(re.search(r"constexpr float kTq4Gamma = ([0-9.]+)f;", src).group(1)))
    lv, _ = oracle.tq4_codebook()
    scaled = (lv.astype(np.float32) * g).astype(np.float32)
    rel = np.abs(scaled.astype(np.float16).astype(np.float64) - lv.astype(np.float64) * float(g)) / \
        np.abs(lv.astype(np.float64) * float(g))
    assert rel.max() <= 1e-4, rel.max()
    plain = np.abs(lv.astype(np.float16).astype(np.float64) - lv) / np.abs(lv)
    assert plain.max() > 3e-4


def test_k2_tensor_level_scale_is_f16_exact_and_tight(oracle):
    """The tensor-core K2/V4 kernel scales bulk K levels by a constant (an f16
    value) that keeps both level magnitudes within 2e-5 of their f16 copies."""
    src = open(os.path.join(ROOT, "quantized_kv_cache_kv8_gb300", "csrc", "k2v4.cu")).read()
    g = float(re.search(r"constexpr float kK2Gamma = ([0-9.]+)f;", src).group(1))
    assert float(np.float16(g)) == g
    lv, _ = oracle.k2_codebook()
    prod = (np.abs(lv).astype(np.float32) * np.float32(g)).astype(np.float32)
    rel = np.abs(prod.astype(np.float16).astype(np.float64) - np.abs(lv) * g) / (np.abs(lv) * g)
    assert rel.max() <= 2e-5, rel.max()


def test_k2v4_append_validates_before_launch(kvq):
    """Refused on the host, nothing launched: a range past the capacity, a
    negative position, a capacity that is not whole groups, missing pools."""
    L = kvq.lib()
    lay = kvq.k2v4_layout()
    d = C.c_void_p(256)
    assert L.k2v4_append(C.byref(lay), d, d, 1, 60, 10, 64, d, d, d, d, d, None, None) == 1      # 70 > 64 cells
    assert L.k2v4_append(C.byref(lay), d, d, 1, -1, 10, 64, d, d, d, d, d, None, None) == 1
    assert L.k2v4_append(C.byref(lay), d, d, 1, 0, 10, 40, d, d, d, d, d, None, None) == 5       # capacity 40
    assert L.k2v4_append(C.byref(lay), None, d, 1, 0, 10, 64, d, d, d, d, d, None, None) == 1
    assert L.k2v4_append(C.byref(lay), d, d, 1, 0, 10, 64, d, d, d, None, d, None, None) == 1  # overlay pools
    assert L.k2v4_append(C.byref(lay), None, None, 1, 5, 0, 64, None, None, None, None, None, None, None) == 0


def test_k2v4_decode_refuses_unaligned_pools(kvq):
    """Refused on the host before any launch: a K2/V4 pool that is not 16-byte
    aligned (the decode stages whole cell groups by 16-byte bulk copies)."""
    L = kvq.lib()
    lay = kvq.k2v4_layout()
    d = C.c_void_p(256)     # dummy device addresses, never dereferenced
    odd = C.c_void_p(264)
    ws = C.c_void_p(4096)
    for kc, ks, vb in ((odd, d, d), (d, odd, d), (d, d, odd)):
        assert L.kv_attn_decode_k2v4(C.byref(lay), d, 1, 16, 64, 64, kc, ks, vb, d, d, 0.1, d, ws, 1 << 30,
                                     kvq.PATH_TENSOR, None) == 1


def test_timing_hook_host_side(kvq):
    """The launch timing hook: off by default (an empty read), a negative
    capacity and null outputs refused, capacity 0 always accepted."""
    L = kvq.lib()
    a, b, n = C.c_double(1.0), C.c_double(1.0), C.c_int32(7)
    assert L.kvq_timing_read(C.byref(a), C.byref(b), C.byref(n)) == 0
    assert (a.value, b.value, n.value) == (0.0, 0.0, 0)
    assert L.kvq_timing_enable(-1) == 1
    assert L.kvq_timing_read(None, C.byref(b), C.byref(n)) == 1
    assert L.kvq_timing_enable(0) == 0


def test_stall_hook_rejects_a_negative_count(kvq):
    L = kvq.lib()
    assert L.kvq_test_stall_waits(-1) == 1
    assert L.kvq_test_stall_waits(0) == 0


def test_new_status_strings(kvq):
    assert "NaN" in kvq.status_string(9)
    assert "wait" in kvq.status_string(10)


def test_polar_tables_equal_the_oracle(kvq, oracle):
    """The f32 cos/sin tables compiled into the library (derived by
    csrc/gen_pq_codebook.py) against the oracle's own codebooks, bit for bit:
    centroids as f32(cos), f32(sin) of the oracle's f64 centroids, thresholds
    as the oracle's f32 decision tables."""
    for bits in range(2, 7):
        for level in range(1, 11):
            c, t = kvq.pq_codebook(bits, level)
            lv, _, _ = oracle.pq_codebook(level, bits)
            want = np.stack([np.cos(lv), np.sin(lv)], 1).astype(np.float32)
            np.testing.assert_array_equal(c.view(np.uint32), want.view(np.uint32))
            ct, st = oracle.pq_decision_table(level, bits)
            np.testing.assert_array_equal(t[:, 0].view(np.uint32), ct.view(np.uint32))
            np.testing.assert_array_equal(t[:, 1].view(np.uint32), st.view(np.uint32))


def test_polar_row_bytes_and_validation(kvq, oracle):
    L = kvq.lib()
    lay = kvq.mla_layout()
    for bits in range(2, 7):
        fmt = kvq.pq_format(bits)
        assert kvq.row_bytes(fmt) == 72 * bits == oracle.pq_row_bytes(bits)
        for bd in [(64,), (2,), (1024,), (16, 32)]:
            lo = kvq.mla_layout(bd, v_dim=bd[0])
            assert kvq.row_bytes(fmt, lo) == oracle.pq_row_bytes(bits, bd)
    assert kvq.row_bytes(kvq.KVQ_KV8) == 576 and kvq.row_bytes(kvq.KVQ_TQ4) == 288
    assert L.kvq_row_bytes(11, C.byref(lay)) == 0 and L.kvq_row_bytes(17, C.byref(lay)) == 0
    d = C.c_void_p(256)
    assert L.pq_encode(kvq.KVQ_TQ4, d, 4, C.byref(lay), None, d, d, None, None) == 1     # not a PolarQuant format
    assert L.pq_encode(14, None, 0, C.byref(lay), None, None, None, None, None) == 0       # empty
    assert L.pq_encode(14, None, 4, C.byref(lay), None, d, d, None, None) == 1             # null x
    odd = kvq.mla_layout((500, 76), v_dim=500)
    assert L.pq_encode(14, d, 4, C.byref(odd), None, d, d, None, None) == 2
    assert L.pq_decode(14, d, d, 4, C.byref(odd), 0, d, None) == 2
    assert L.pq_decode(2, d, d, 4, C.byref(lay), 0, d, None) == 1
    # attention: the fp32 path serves every PolarQuant width, the tensor path 4 bits only
    assert kvq.kv_attn_workspace_size(13, 8, 128, 32768) == kvq.kv_attn_workspace_size(13, 8, 128, 32768,
                                                                                        path=kvq.PATH_SIMT) > 0
    assert kvq.kv_attn_workspace_size(13, 8, 128, 32768, path=kvq.PATH_TENSOR) == 0
    assert kvq.kv_attn_workspace_size(14, 8, 128, 32768, path=kvq.PATH_TENSOR) == \
        kvq.kv_attn_workspace_size(2, 8, 128, 32768, path=kvq.PATH_TENSOR) > 0
    assert kvq.kv_attn_workspace_size(14, 8, 128, 32768) == kvq.kv_attn_workspace_size(14, 8, 128, 32768,
                                                                                        path=kvq.PATH_SIMT)
    ws = C.c_void_p(1 << 21)
    assert L.kv_attn_decode(12, C.byref(lay), d, 1, 2, 128, d, d, d, 10, 0.1, d, ws, 1 << 30, kvq.PATH_TENSOR,
                            None) == 5
