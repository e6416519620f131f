"""ctypes front end of the CPU oracle (``kvq_oracle.c``) -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path never does.

The C file is compiled on first use with gcc into ``oracle/_build/``.  The
flags keep IEEE semantics: no fast-math and no contraction of a multiply and an
add into one fused operation (gcc contracts by default on AArch64 in GNU mode).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvq_oracle.so")
CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

KV8, TQ4 = 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


class K2V4Layout(C.Structure):
    _fields_ = [("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("group", C.c_int32),
                ("k_gain", C.c_float), ("n_sink", C.c_int32), ("n_window", C.c_int32),
                ("n_slack", C.c_int32)]


def _declare(L):
    P = C.c_void_p
    L.kvqo_e4m3_value.restype = C.c_double
    L.kvqo_e4m3_value.argtypes = [C.c_uint]
    L.kvqo_e4m3_encode.restype = C.c_uint
    L.kvqo_e4m3_encode.argtypes = [C.c_float]
    L.kvqo_e4m3_encode_array.restype = None
    L.kvqo_e4m3_encode_array.argtypes = [P, C.c_int64, P]
    L.kvqo_f16_value.restype = C.c_double
    L.kvqo_f16_value.argtypes = [C.c_uint]
    L.kvqo_f16_encode.restype = C.c_uint
    L.kvqo_f16_encode.argtypes = [C.c_float]
    L.kvqo_splitmix64_next.restype = C.c_uint64
    L.kvqo_splitmix64_next.argtypes = [C.POINTER(C.c_uint64)]
    L.kvqo_tq4_signs.restype = None
    L.kvqo_tq4_signs.argtypes = [C.c_uint64, C.c_int, P, P]
    L.kvqo_lloyd_max_gaussian.restype = C.c_int
    L.kvqo_lloyd_max_gaussian.argtypes = [C.c_int, P, P]
    L.kvqo_tq4_codebook.restype = None
    L.kvqo_tq4_codebook.argtypes = [P, P]
    L.kvqo_k2_codebook.restype = None
    L.kvqo_k2_codebook.argtypes = [P, P]
    L.kvqo_fwht_f32.restype = None
    L.kvqo_fwht_f32.argtypes = [P, C.c_int]
    L.kvqo_fwht_f64.restype = None
    L.kvqo_fwht_f64.argtypes = [P, C.c_int]
    L.kvqo_kv8_encode.restype = C.c_int
    L.kvqo_kv8_encode.argtypes = [P, C.c_int64, C.c_int, P, P, P]
    L.kvqo_kv8_decode.restype = None
    L.kvqo_kv8_decode.argtypes = [P, P, C.c_int64, C.c_int, P, P]
    L.kvqo_tq4_encode.restype = C.c_int
    L.kvqo_tq4_encode.argtypes = [P, C.c_int64, C.c_int, P, C.c_uint64, P, P]
    L.kvqo_tq4_decode.restype = C.c_int
    L.kvqo_tq4_decode.argtypes = [P, P, C.c_int64, C.c_int, P, C.c_uint64, P]
    L.kvqo_tq4_rotate.restype = C.c_int
    L.kvqo_tq4_rotate.argtypes = [P, P, C.c_int64, C.c_int, P, C.c_uint64, C.c_int]
    L.kvqo_attn_dense.restype = C.c_int
    L.kvqo_attn_dense.argtypes = [P, C.c_int64, C.c_int, P, C.c_int64, C.c_int, C.c_int64,
                                  P, C.c_int, C.c_double, P]
    L.kvqo_attn_method.restype = C.c_int
    L.kvqo_attn_method.argtypes = [C.c_int, C.c_int, P, C.c_uint64, C.c_int, P, P, C.c_int64,
                                   P, C.c_int, C.c_double, P]
    L.kvqo_k2v4_slot.restype = C.c_int64
    L.kvqo_k2v4_slot.argtypes = [C.c_int64, C.c_int64, C.POINTER(K2V4Layout)]
    L.kvqo_k2v4_encode.restype = C.c_int
    L.kvqo_k2v4_encode.argtypes = [P, P, C.c_int64, C.c_int64, C.POINTER(K2V4Layout), P, P, P, P, P]
    L.kvqo_k2v4_append.restype = C.c_int
    L.kvqo_k2v4_append.argtypes = [P, P, C.c_int64, C.c_int64, C.c_int64, C.POINTER(K2V4Layout), P, P, P, P, P]
    L.kvqo_pq_codebook.restype = C.c_int
    L.kvqo_pq_codebook.argtypes = [C.c_int, C.c_int, P, P, P]
    L.kvqo_pq_decision_table.restype = C.c_int
    L.kvqo_pq_decision_table.argtypes = [C.c_int, C.c_int, P, P]
    L.kvqo_pq_row_bytes.restype = C.c_int64
    L.kvqo_pq_row_bytes.argtypes = [C.c_int, P, C.c_int]
    L.kvqo_pq_encode.restype = C.c_int
    L.kvqo_pq_encode.argtypes = [P, C.c_int64, C.c_int, P, C.c_uint64, C.c_int, P, P]
    L.kvqo_pq_decode.restype = C.c_int
    L.kvqo_pq_decode.argtypes = [P, P, C.c_int64, C.c_int, P, C.c_uint64, C.c_int, C.c_int, P]
    L.kvqo_polar_forward.restype = C.c_int
    L.kvqo_polar_forward.argtypes = [P, C.c_int, P, P]
    L.kvqo_polar_inverse.restype = C.c_int
    L.kvqo_polar_inverse.argtypes = [P, C.c_double, C.c_int, P]
    L.kvqo_k2v4_reconstruct.restype = C.c_int
    L.kvqo_k2v4_reconstruct.argtypes = [P, P, P, P, P, C.c_int64, C.c_int64, C.POINTER(K2V4Layout),
                                        C.c_int, P, P]


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _dims(bdims):
    return np.ascontiguousarray(np.asarray(bdims, dtype=np.int32))


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} returned status {rc}")


# -- scalar codecs -----------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().kvqo_e4m3_value(int(code))


def e4m3_encode(u: float) -> int:
    return lib().kvqo_e4m3_encode(float(u))


def e4m3_encode_array(u: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(u, dtype=np.float32)
    out = np.empty(u.shape, dtype=np.uint8)
    lib().kvqo_e4m3_encode_array(_p(u), u.size, _p(out))
    return out


def f16_value(h: int) -> float:
    return lib().kvqo_f16_value(int(h))


def f16_encode(x: float) -> int:
    return lib().kvqo_f16_encode(float(x))


def splitmix64(seed: int, n: int) -> list[int]:
    st = C.c_uint64(seed)
    return [lib().kvqo_splitmix64_next(C.byref(st)) for _ in range(n)]


def tq4_signs(seed: int, bdims) -> np.ndarray:
    d = _dims(bdims)
    out = np.empty(int(d.sum()), dtype=np.int8)
    lib().kvqo_tq4_signs(seed, d.size, _p(d), _p(out))
    return out


def lloyd_max(levels: int):
    c = np.empty(levels, dtype=np.float64)
    mse = np.empty(1, dtype=np.float64)
    it = lib().kvqo_lloyd_max_gaussian(levels, _p(c), _p(mse))
    return c, float(mse[0]), it


def tq4_codebook():
    lv = np.empty(16, np.float32)
    th = np.empty(15, np.float32)
    lib().kvqo_tq4_codebook(_p(lv), _p(th))
    return lv, th


def k2_codebook():
    lv = np.empty(4, np.float32)
    th = np.empty(3, np.float32)
    lib().kvqo_k2_codebook(_p(lv), _p(th))
    return lv, th


def fwht(v: np.ndarray) -> np.ndarray:
    """Unnormalized FWHT along the last axis, in the array's precision (f32 or f64)."""
    dt = np.float32 if v.dtype == np.float32 else np.float64
    out = np.array(v, dtype=dt, copy=True, order="C")
    n = out.shape[-1]
    rows = out.reshape(-1, n)
    fn = lib().kvqo_fwht_f32 if dt == np.float32 else lib().kvqo_fwht_f64
    for r in range(rows.shape[0]):
        fn(rows[r].ctypes.data_as(C.c_void_p), n)
    return out


# -- row codecs --------------------------------------------------------------

def kv8_encode(x: np.ndarray, bdims=(512, 64)):
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = _dims(bdims)
    n = x.shape[0]
    codes = np.empty((n, int(d.sum())), np.uint8)
    scales = np.empty((n, d.size), np.float32)
    _check(lib().kvqo_kv8_encode(_p(x), n, d.size, _p(d), _p(codes), _p(scales)), "kv8_encode")
    return codes, scales


def kv8_decode(codes, scales, bdims=(512, 64)) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    d = _dims(bdims)
    out = np.empty((codes.shape[0], int(d.sum())), np.float64)
    lib().kvqo_kv8_decode(_p(codes), _p(scales), codes.shape[0], d.size, _p(d), _p(out))
    return out


def tq4_encode(x: np.ndarray, bdims=(512, 64), seed: int = 0):
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = _dims(bdims)
    n = x.shape[0]
    packed = np.empty((n, int(d.sum()) // 2), np.uint8)
    scales = np.empty((n, d.size), np.float32)
    _check(lib().kvqo_tq4_encode(_p(x), n, d.size, _p(d), seed, _p(packed), _p(scales)), "tq4_encode")
    return packed, scales


def tq4_encode_status(x: np.ndarray, bdims, seed: int = 0) -> int:
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = _dims(bdims)
    n = x.shape[0]
    packed = np.zeros((max(n, 1), max(int(d.sum()) // 2, 1)), np.uint8)
    scales = np.zeros((max(n, 1), d.size), np.float32)
    return lib().kvqo_tq4_encode(_p(x), n, d.size, _p(d), seed, _p(packed), _p(scales))


def tq4_decode(packed, scales, bdims=(512, 64), seed: int = 0) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    d = _dims(bdims)
    out = np.empty((packed.shape[0], int(d.sum())), np.float64)
    _check(lib().kvqo_tq4_decode(_p(packed), _p(scales), packed.shape[0], d.size, _p(d), seed, _p(out)),
           "tq4_decode")
    return out


def tq4_rotate(v: np.ndarray, bdims=(512, 64), seed: int = 0, inverse: bool = False) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float64)
    d = _dims(bdims)
    out = np.empty_like(v)
    n = v.size // int(d.sum())
    _check(lib().kvqo_tq4_rotate(_p(v), _p(out), n, d.size, _p(d), seed, int(inverse)), "tq4_rotate")
    return out


# -- PolarQuant (codec 0 of the TQ tier) ------------------------------------

NONFINITE = 3   # kvqo_pq_encode: some block's radius is not finite


def pq_format(bits: int) -> int:
    """Format number of the PolarQuant tier at ``bits`` bits per angle."""
    return 10 + bits


def pq_bits(fmt: int) -> int:
    return fmt - 10 if 12 <= fmt <= 16 else 0


def pq_codebook(level: int, bits: int):
    """Centroids (2^bits) and thresholds (2^bits - 1) of one level's angle
    quantizer in radians, and its mean squared error (rad^2)."""
    lv = np.empty(1 << bits, np.float64)
    th = np.empty((1 << bits) - 1, np.float64)
    mse = C.c_double()
    _check(lib().kvqo_pq_codebook(level, bits, _p(lv), _p(th), C.byref(mse)), "pq_codebook")
    return lv, th, mse.value


def pq_decision_table(level: int, bits: int):
    """f32 cosines and sines of the thresholds the encoder compares against
    (level 1: the in-quadrant thresholds)."""
    ct = np.zeros(64, np.float32)
    st = np.zeros(64, np.float32)
    n = lib().kvqo_pq_decision_table(level, bits, _p(ct), _p(st))
    if n < 0:
        raise ValueError("oracle pq_decision_table failed")
    return ct[:n].copy(), st[:n].copy()


def pq_row_bytes(bits: int, bdims=(512, 64)) -> int:
    d = _dims(bdims)
    return int(lib().kvqo_pq_row_bytes(d.size, _p(d), bits))


def pq_encode(x: np.ndarray, bits: int, bdims=(512, 64), seed: int = 0, allow_nonfinite: bool = False):
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = _dims(bdims)
    n = x.shape[0]
    codes = np.zeros((n, pq_row_bytes(bits, bdims)), np.uint8)
    radii = np.zeros((n, d.size), np.float32)
    rc = lib().kvqo_pq_encode(_p(x), n, d.size, _p(d), seed, bits, _p(codes), _p(radii))
    if not (rc == 0 or (allow_nonfinite and rc == NONFINITE)):
        _check(rc, "pq_encode")
    return codes, radii


def pq_decode(codes, radii, bits: int, bdims=(512, 64), seed: int = 0, rotated: bool = False) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    radii = np.ascontiguousarray(radii, np.float32)
    d = _dims(bdims)
    out = np.empty((codes.shape[0], int(d.sum())), np.float64)
    _check(lib().kvqo_pq_decode(_p(codes), _p(radii), codes.shape[0], d.size, _p(d), seed, bits, int(rotated),
                                _p(out)), "pq_decode")
    return out


def polar_forward(v: np.ndarray):
    """Angles (level 1 first) and radius of the exact polar transform of v."""
    v = np.ascontiguousarray(v, np.float64)
    ang = np.empty(v.size - 1, np.float64)
    r = C.c_double()
    _check(lib().kvqo_polar_forward(_p(v), v.size, _p(ang), C.byref(r)), "polar_forward")
    return ang, r.value


def polar_inverse(angles: np.ndarray, radius: float) -> np.ndarray:
    angles = np.ascontiguousarray(angles, np.float64)
    out = np.empty(angles.size + 1, np.float64)
    _check(lib().kvqo_polar_inverse(_p(angles), float(radius), out.size, _p(out)), "polar_inverse")
    return out


def reconstruct(fmt: int, codes, scales, bdims=(512, 64), seed: int = 0) -> np.ndarray:
    if fmt == KV8:
        return kv8_decode(codes, scales, bdims)
    if fmt == TQ4:
        return tq4_decode(codes, scales, bdims, seed)
    return pq_decode(codes, scales, pq_bits(fmt), bdims, seed)


# -- attention ---------------------------------------------------------------

def attn_dense(K: np.ndarray, q: np.ndarray, sm_scale: float, dv: int, V: np.ndarray | None = None) -> np.ndarray:
    """Plain softmax attention of each query row of ``q`` over all rows of ``K``.

    ``K`` is [T, dk] float64; ``V`` defaults to ``K`` (the MLA latent is both key
    and value) and its leading ``dv`` columns are the value.
    """
    K = np.ascontiguousarray(K, np.float64)
    V = K if V is None else np.ascontiguousarray(V, np.float64)
    q = np.ascontiguousarray(q, np.float32).reshape(-1, K.shape[1])
    out = np.empty((q.shape[0], dv), np.float64)
    _check(lib().kvqo_attn_dense(_p(K), K.shape[1], K.shape[1], _p(V), V.shape[1], dv, K.shape[0],
                                 _p(q), q.shape[0], float(sm_scale), _p(out)), "attn_dense")
    return out


def attn_method(fmt: int, codes, scales, q, sm_scale: float, v_dim: int = 512, bdims=(512, 64),
                seed: int = 0) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    d = _dims(bdims)
    q = np.ascontiguousarray(q, np.float32).reshape(-1, int(d.sum()))
    out = np.empty((q.shape[0], v_dim), np.float64)
    _check(lib().kvqo_attn_method(fmt, d.size, _p(d), seed, v_dim, _p(codes), _p(scales), codes.shape[0],
                                  _p(q), q.shape[0], float(sm_scale), _p(out)), "attn_method")
    return out


def attn_decode(fmt: int, codes, scales, q, cu_seqlens, sm_scale: float, pairs=None, v_dim: int = 512,
                bdims=(512, 64), seed: int = 0) -> dict:
    """Ragged decode: q is [B, H, D]; rows of sequence b are [cu[b], cu[b+1]).

    Returns {(b, h): out[v_dim]} for the requested (b, h) pairs (all if None).
    Each sequence's rows are reconstructed once.
    """
    q = np.asarray(q, np.float32)
    B, H, D = q.shape
    cu = np.asarray(cu_seqlens, np.int64)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    by_seq: dict[int, list[int]] = {}
    for b, h in pairs:
        by_seq.setdefault(int(b), []).append(int(h))
    out = {}
    for b, heads in by_seq.items():
        lo, hi = int(cu[b]), int(cu[b + 1])
        xhat = reconstruct(fmt, codes[lo:hi], scales[lo:hi], bdims, seed)
        res = attn_dense(xhat, q[b, heads], sm_scale, v_dim)
        for i, h in enumerate(heads):
            out[(b, h)] = res[i]
    return out


# -- K2/V4 -------------------------------------------------------------------

def k2v4_layout(n_kv_heads=2, head_dim=256, k_gain=1.10, n_sink=8, n_window=256, n_slack=16):
    return K2V4Layout(n_kv_heads, head_dim, 32, k_gain, n_sink, n_window, n_slack)


def k2v4_slot(cell: int, T: int, L: K2V4Layout) -> int:
    return lib().kvqo_k2v4_slot(cell, T, C.byref(L))


def k2v4_encode(k: np.ndarray, v: np.ndarray, L: K2V4Layout, cap: int | None = None):
    """Encode one sequence: k, v are [Hkv, T, D] float32."""
    k = np.ascontiguousarray(k, np.float32)
    v = np.ascontiguousarray(v, np.float32)
    H, T, D = k.shape
    cap = T if cap is None else cap
    slots = L.n_sink + L.n_window + L.n_slack
    kc = np.zeros((H, cap, D // 4), np.uint8)
    ks = np.zeros((H, cap // 32, D), np.uint16)
    vb = np.zeros((H, cap, D // 32, 18), np.uint8)
    kw = np.zeros((H, slots, D), np.uint16)
    vw = np.zeros((H, slots, D), np.uint16)
    _check(lib().kvqo_k2v4_encode(_p(k), _p(v), T, cap, C.byref(L), _p(kc), _p(ks), _p(vb), _p(kw), _p(vw)),
           "k2v4_encode")
    return kc, ks, vb, kw, vw


def k2v4_append(kc, ks, vb, kw, vw, k_new: np.ndarray, v_new: np.ndarray, T_old: int, L: K2V4Layout):
    """Append k_new, v_new ([Hkv, n, D] float32) at cells T_old .. T_old + n - 1 of
    one sequence's pools; returns updated copies (kc, ks, vb, kw, vw)."""
    kc, ks, vb, kw, vw = (np.array(a, copy=True) for a in (kc, ks, vb, kw, vw))
    k_new = np.ascontiguousarray(k_new, np.float32)
    v_new = np.ascontiguousarray(v_new, np.float32)
    cap = kc.shape[1]
    _check(lib().kvqo_k2v4_append(_p(k_new), _p(v_new), int(T_old), k_new.shape[1], cap, C.byref(L), _p(kc),
                                  _p(ks), _p(vb), _p(kw), _p(vw)), "k2v4_append")
    return kc, ks, vb, kw, vw


def k2v4_reconstruct(kc, ks, vb, kw, vw, T: int, L: K2V4Layout, use_overlay: bool = True):
    H = L.n_kv_heads
    D = L.head_dim
    cap = kc.shape[1]
    K = np.empty((H, T, D), np.float64)
    V = np.empty((H, T, D), np.float64)
    _check(lib().kvqo_k2v4_reconstruct(_p(np.ascontiguousarray(kc)), _p(np.ascontiguousarray(ks)),
                                       _p(np.ascontiguousarray(vb)), _p(np.ascontiguousarray(kw)),
                                       _p(np.ascontiguousarray(vw)), T, cap, C.byref(L), int(use_overlay),
                                       _p(K), _p(V)), "k2v4_reconstruct")
    return K, V


def k2v4_attn(K: np.ndarray, V: np.ndarray, q: np.ndarray, sm_scale: float) -> np.ndarray:
    """GQA attention of one sequence: K, V [Hkv, T, D]; q [Hq, D]; q head h reads kv head h // (Hq/Hkv)."""
    Hkv, T, D = K.shape
    Hq = q.shape[0]
    grp = Hq // Hkv
    out = np.empty((Hq, D), np.float64)
    for g in range(Hkv):
        out[g * grp:(g + 1) * grp] = attn_dense(K[g], q[g * grp:(g + 1) * grp], sm_scale, D, V=V[g])
    return out
