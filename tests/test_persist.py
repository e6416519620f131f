"""Persistence of quantized pools (host code, no GPU): the versioned file the
KV cache quantization pages describe -- tier in the magic, TQ codec and bits in
header word 7, refusal of any mismatch, quantize-on-load of f32 files,
in-place appends that heal a torn tail."""
import os

import numpy as np
import pytest

from quantized_kv_cache_kv8_gb300 import synth

KV8, TQ4 = 1, 2
MISMATCH, IO, WORKSPACE = 7, 8, 3


@pytest.fixture(scope="module")
def kvq():
    from quantized_kv_cache_kv8_gb300 import kvq as K
    K.lib()
    return K


def pool(oracle, fmt, n, seed=3):
    x = synth.mla_rows(seed, n)
    return oracle.kv8_encode(x) if fmt == KV8 else oracle.tq4_encode(x, seed=seed)


@pytest.mark.parametrize("fmt,rec", [(KV8, 584), (TQ4, 296)])
def test_round_trip_and_byte_layout(kvq, oracle, tmp_path, fmt, rec):
    codes, scales = pool(oracle, fmt, 37)
    path = str(tmp_path / "kv.bin")
    lay = kvq.mla_layout(seed=3)
    kvq.cache_save(path, fmt, codes, scales, lay)
    assert os.path.getsize(path) == 8 + 64 + 37 * rec          # magic, 8 header words, one record per row
    raw = open(path, "rb").read()
    assert raw[:8] == (b"COLIKV2\0" if fmt == KV8 else b"COLIKV3\0")
    h = np.frombuffer(raw[8:72], np.int64)
    assert list(h[:6]) == [37, 576, 2, 512, 64, 512]
    assert h[7] == (0 if fmt == KV8 else (1 << 8 | 4))          # codec << 8 | bits
    assert h[6] == (0 if fmt == KV8 else 3)                      # the TQ sign seed
    first = np.frombuffer(raw[72:72 + rec], np.uint8)
    np.testing.assert_array_equal(first[:rec - 8], codes[0])
    np.testing.assert_array_equal(first[rec - 8:].view(np.float32), scales[0])
    c2, s2 = kvq.cache_load(path, fmt, 64, lay)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2.view(np.uint32), scales.view(np.uint32))
    assert kvq.cache_info(path)[:2] == (2 if fmt == KV8 else 3, 37)


def test_other_tier_is_refused_both_ways(kvq, oracle, tmp_path):
    lay = kvq.mla_layout(seed=3)
    p8, p4 = str(tmp_path / "a"), str(tmp_path / "b")
    kvq.cache_save(p8, KV8, *pool(oracle, KV8, 5), lay)
    kvq.cache_save(p4, TQ4, *pool(oracle, TQ4, 5), lay)
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(p8, TQ4, 10, lay)
    assert e.value.status == MISMATCH and "fp8 (KV8)" in e.value.msg
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(p4, KV8, 10, lay)
    assert e.value.status == MISMATCH and "KV_TQ" in e.value.msg
    with pytest.raises(kvq.CacheFileError) as e:               # a quantized file under the f32 tier
        kvq.cache_load_f32(p8, 10, lay)
    assert e.value.status == MISMATCH


def test_tq_codec_bits_seed_and_layout_mismatch_refused(kvq, oracle, tmp_path):
    lay = kvq.mla_layout(seed=3)
    path = str(tmp_path / "t")
    kvq.cache_save(path, TQ4, *pool(oracle, TQ4, 4), lay)
    raw = bytearray(open(path, "rb").read())
    bad = bytearray(raw)
    bad[8 + 7 * 8:8 + 8 * 8] = np.array([1 << 8 | 3], np.int64).tobytes()     # same codec, 3 bits
    open(path, "wb").write(bad)
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(path, TQ4, 10, lay)
    assert e.value.status == MISMATCH and "codec 1, 3-bit" in e.value.msg and "codec 1, 4-bit" in e.value.msg
    open(path, "wb").write(raw)
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(path, TQ4, 10, kvq.mla_layout(seed=4))              # another rotation
    assert e.value.status == MISMATCH
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(path, TQ4, 10, kvq.mla_layout(seed=3, v_dim=256))   # another layout
    assert e.value.status == MISMATCH
    kvq.cache_load(path, TQ4, 10, lay)                                     # the original still loads


def test_size_and_magic_checks(kvq, oracle, tmp_path):
    lay = kvq.mla_layout()
    path = str(tmp_path / "k")
    kvq.cache_save(path, KV8, *pool(oracle, KV8, 6), lay)
    raw = open(path, "rb").read()
    open(path, "wb").write(raw[:-1])                                       # truncated
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(path, KV8, 10, lay)
    assert e.value.status == IO
    open(path, "wb").write(raw + b"\0" * 584)                              # a row the header does not count
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(path, KV8, 10, lay)
    assert e.value.status == IO
    open(path, "wb").write(b"NOTAKVCF" + raw[8:])
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(path, KV8, 10, lay)
    assert e.value.status == IO and "magic" in e.value.msg
    open(path, "wb").write(raw)
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(path, KV8, 5, lay)                                  # 6 rows, room for 5
    assert e.value.status == WORKSPACE


def test_f32_file_upgrades_on_load(kvq, oracle, tmp_path):
    """A v1 (f32) file is read under KV8 by encoding its rows; it is not
    touched until the first save rewrites it as v2."""
    lay = kvq.mla_layout()
    x = synth.mla_rows(7, 9)
    path = str(tmp_path / "v1")
    kvq.cache_save_f32(path, x, lay)
    before = open(path, "rb").read()
    assert before[:8] == b"COLIKV\0\0"
    rows = kvq.cache_load_f32(path, 16, lay)
    np.testing.assert_array_equal(rows, x)
    with pytest.raises(kvq.CacheFileError):
        kvq.cache_load(path, KV8, 16, lay)                                 # not misread as KV8
    codes, scales = oracle.kv8_encode(rows)                                # quantize on load
    assert open(path, "rb").read() == before                               # untouched so far
    kvq.cache_save(path, KV8, codes, scales, lay)
    assert kvq.cache_info(path)[0] == 2
    c2, _ = kvq.cache_load(path, KV8, 16, lay)
    np.testing.assert_array_equal(c2, codes)


def test_append_in_place_and_self_heal(kvq, oracle, tmp_path):
    lay = kvq.mla_layout()
    codes, scales = pool(oracle, KV8, 12)
    path = str(tmp_path / "ap")
    kvq.cache_save(path, KV8, codes[:5], scales[:5], lay)
    n, msg = kvq.cache_append(path, KV8, codes[5:8], scales[5:8], lay)
    assert n == 8 and msg == ""
    # an append interrupted after writing one and a half records, before its header update
    with open(path, "ab") as f:
        f.write(bytes(584 + 300))
    n, msg = kvq.cache_append(path, KV8, codes[8:12], scales[8:12], lay)
    assert n == 12 and "interrupted" in msg
    c2, s2 = kvq.cache_load(path, KV8, 20, lay)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2.view(np.uint32), scales.view(np.uint32))
    with pytest.raises(kvq.CacheFileError) as e:                          # appends check the mode too
        kvq.cache_append(path, TQ4, codes[:1, :288], scales[:1], lay)
    assert e.value.status == MISMATCH


@pytest.mark.parametrize("rows", [-5, 2 ** 62, 2 ** 63 - 1])
def test_header_row_count_out_of_range_is_refused(kvq, oracle, tmp_path, rows):
    """A header whose row count is negative, or so large that the file size it
    implies overflows, is refused as corrupt by every reader, never misread."""
    codes, scales = pool(oracle, KV8, 4)
    path = str(tmp_path / "kv.bin")
    lay = kvq.mla_layout(seed=3)
    kvq.cache_save(path, KV8, codes, scales, lay)
    raw = bytearray(open(path, "rb").read())
    raw[8:16] = np.array([rows], np.int64).tobytes()
    open(path, "wb").write(bytes(raw))
    for call in (lambda: kvq.cache_info(path), lambda: kvq.cache_load(path, KV8, 8, lay),
                 lambda: kvq.cache_append(path, KV8, codes, scales, lay)):
        with pytest.raises(kvq.CacheFileError) as e:
            call()
        assert e.value.status == IO


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6])
def test_polar_pools_round_trip_under_codec_0(kvq, oracle, tmp_path, bits):
    """PolarQuant pools persist in the TQ tier (COLIKV3) with h[7] = 0 << 8 | b
    and records of 72 b code bytes + 8 radius bytes."""
    x = synth.mla_rows(9, 23)
    codes, radii = oracle.pq_encode(x, bits, seed=4)
    fmt = 10 + bits
    lay = kvq.mla_layout(seed=4)
    path = str(tmp_path / f"pq{bits}")
    kvq.cache_save(path, fmt, codes, radii, lay)
    raw = open(path, "rb").read()
    assert raw[:8] == b"COLIKV3\0" and len(raw) == 72 + 23 * (72 * bits + 8)
    h = np.frombuffer(raw[8:72], np.int64)
    assert h[7] == bits and h[6] == 4
    c2, r2 = kvq.cache_load(path, fmt, 30, lay)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(r2.view(np.uint32), radii.view(np.uint32))
    kvq.cache_append(path, fmt, codes[:3], radii[:3], lay)
    c3, _ = kvq.cache_load(path, fmt, 30, lay)
    np.testing.assert_array_equal(c3[23:], codes[:3])


def test_polar_and_rotated_int4_refuse_each_other(kvq, oracle, tmp_path):
    lay = kvq.mla_layout(seed=4)
    x = synth.mla_rows(10, 5)
    pq, pr = oracle.pq_encode(x, 4, seed=4)
    tq, ts = oracle.tq4_encode(x, seed=4)
    p_pq, p_tq = str(tmp_path / "pq"), str(tmp_path / "tq")
    kvq.cache_save(p_pq, 14, pq, pr, lay)
    kvq.cache_save(p_tq, TQ4, tq, ts, lay)
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(p_pq, TQ4, 10, lay)
    assert e.value.status == MISMATCH and "codec 0, 4-bit" in e.value.msg and "codec 1, 4-bit" in e.value.msg
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(p_tq, 14, 10, lay)
    assert e.value.status == MISMATCH
    with pytest.raises(kvq.CacheFileError) as e:
        kvq.cache_load(p_pq, 13, 10, lay)
    assert e.value.status == MISMATCH and "codec 0, 3-bit" in e.value.msg
