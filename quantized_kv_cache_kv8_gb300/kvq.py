"""Python binding of libkvq's C ABI (include/kvq.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Tensors must be contiguous CUDA tensors of the stated dtypes; the
calls are asynchronous on the current torch stream (or the one given).  There
is no CPU path: if the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import math
import threading

import torch

from . import build as _build

KVQ_KV8, KVQ_TQ4 = 1, 2
KVQ_PQ2, KVQ_PQ3, KVQ_PQ4, KVQ_PQ5, KVQ_PQ6 = 12, 13, 14, 15, 16   # PolarQuant, 10 + bits
KVQ_F32, KVQ_BF16 = 0, 1
PATH_AUTO, PATH_SIMT, PATH_TENSOR = 0, 1, 2
SM_SCALE_MLA = 1.0 / math.sqrt(192.0)


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: kvq status {status} ({status_string(status)})")
        self.status = status


class MLALayout(C.Structure):
    _fields_ = [("n_blocks", C.c_int32), ("block_dim", C.c_int32 * 2), ("v_dim", C.c_int32),
                ("seed", C.c_uint64)]


class K2V4Layout(C.Structure):
    _fields_ = [("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("group", C.c_int32),
                ("k_gain", C.c_float), ("n_sink", C.c_int32), ("n_window", C.c_int32), ("n_slack", C.c_int32)]


def mla_layout(block_dims=(512, 64), v_dim=512, seed=0) -> MLALayout:
    bd = (C.c_int32 * 2)(block_dims[0], block_dims[1] if len(block_dims) > 1 else 0)
    return MLALayout(len(block_dims), bd, v_dim, seed)


def k2v4_layout(n_kv_heads=2, head_dim=256, k_gain=1.10, n_sink=8, n_window=256, n_slack=16) -> K2V4Layout:
    return K2V4Layout(n_kv_heads, head_dim, 32, k_gain, n_sink, n_window, n_slack)


_lock = threading.Lock()
_lib = None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = C.CDLL(path)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    P, S, I32, I64 = C.c_void_p, C.c_size_t, C.c_int32, C.c_int64
    pl, pk = C.POINTER(MLALayout), C.POINTER(K2V4Layout)
    L.kvq_status_string.restype = C.c_char_p
    L.kvq_status_string.argtypes = [C.c_int]
    L.kvq_version.restype = C.c_char_p
    L.kvq_codebook.restype = C.c_int
    L.kvq_codebook.argtypes = [I32, P, P]
    L.kv8_encode.restype = C.c_int
    L.kv8_encode.argtypes = [P, I64, pl, P, P, P, P, P]
    L.tq4_encode.restype = C.c_int
    L.tq4_encode.argtypes = [P, I64, pl, P, P, P, P, P]
    L.kvq_test_stall_waits.restype = C.c_int
    L.kvq_test_stall_waits.argtypes = [I64]
    L.pq_encode.restype = C.c_int
    L.pq_encode.argtypes = [C.c_int, P, I64, pl, P, P, P, P, P]
    L.pq_decode.restype = C.c_int
    L.pq_decode.argtypes = [C.c_int, P, P, I64, pl, I32, P, P]
    L.kvq_row_bytes.restype = I64
    L.kvq_row_bytes.argtypes = [C.c_int, pl]
    L.kvq_pq_codebook.restype = C.c_int
    L.kvq_pq_codebook.argtypes = [I32, I32, P, P]
    L.tq4_rotate.restype = C.c_int
    L.tq4_rotate.argtypes = [P, C.c_int, I64, pl, I32, P, P]
    L.kv_attn_workspace_size.restype = S
    L.kv_attn_workspace_size.argtypes = [C.c_int, pl, I32, I32, I64, C.c_int]
    L.kv_attn_decode.restype = C.c_int
    L.kv_attn_decode.argtypes = [C.c_int, pl, P, C.c_int, I32, I32, P, P, P, I64, C.c_float, P, P, S, C.c_int, P]
    for name in ("kvq_cache_save", "kvq_cache_save_f32", "kvq_cache_info", "kvq_cache_load", "kvq_cache_load_f32",
                 "kvq_cache_append"):
        getattr(L, name).restype = C.c_int
    L.kvq_cache_save.argtypes = [C.c_char_p, C.c_int, pl, I64, P, P]
    L.kvq_cache_save_f32.argtypes = [C.c_char_p, pl, I64, P]
    L.kvq_cache_info.argtypes = [C.c_char_p, P, P, P, C.c_char_p, S]
    L.kvq_cache_load.argtypes = [C.c_char_p, C.c_int, pl, I64, P, P, P, C.c_char_p, S]
    L.kvq_cache_load_f32.argtypes = [C.c_char_p, pl, I64, P, P, C.c_char_p, S]
    L.kvq_cache_append.argtypes = [C.c_char_p, C.c_int, pl, I64, P, P, P, C.c_char_p, S]
    L.kv_attn_gather_workspace_size.restype = S
    L.kv_attn_gather_workspace_size.argtypes = [C.c_int, pl, C.c_int, I32, I32, I64, C.c_int]
    L.kv_attn_decode_gather.restype = C.c_int
    L.kv_attn_decode_gather.argtypes = [C.c_int, pl, P, C.c_int, I32, I32, P, P, I64, P, P, I64, C.c_float, P, P, S,
                                        C.c_int, P]
    L.kv_attn_decode_append.restype = C.c_int
    L.kv_attn_decode_append.argtypes = [C.c_int, pl, P, P, P, C.c_int, I32, I32, P, P, P, I64, C.c_float, P, P, S,
                                        C.c_int, P]
    L.kv_attn_decode_noalloc.restype = C.c_int
    L.kv_attn_decode_noalloc.argtypes = [C.c_int, pl, P, C.c_int, I32, I32, P, P, P, I64, C.c_float, P, C.c_int, P]
    L.kv_attn_prefill_workspace_size.restype = S
    L.kv_attn_prefill_workspace_size.argtypes = [C.c_int, pl, I32, I64, I64, C.c_int]
    L.kv_attn_prefill.restype = C.c_int
    L.kv_attn_prefill.argtypes = [C.c_int, pl, P, P, C.c_int, I64, I64, I32, P, P, C.c_float, P, P, S, C.c_int, P]
    L.kvq_read_device_error.restype = I32
    L.kvq_read_device_error.argtypes = [P, I32, P]
    L.kvq_read_exact_rescales.restype = I64
    L.kvq_read_exact_rescales.argtypes = [P, I32, P]
    L.kvq_timing_enable.restype = C.c_int
    L.kvq_timing_enable.argtypes = [I32]
    L.kvq_timing_read.restype = C.c_int
    L.kvq_timing_read.argtypes = [C.POINTER(C.c_double), C.POINTER(C.c_double), C.POINTER(I32)]
    L.k2v4_encode.restype = C.c_int
    L.k2v4_encode.argtypes = [pk, P, P, I32, I64, I64, P, P, P, P, P, P, P]
    L.k2v4_append.restype = C.c_int
    L.k2v4_append.argtypes = [pk, P, P, I32, I64, I64, I64, P, P, P, P, P, P, P]
    L.kv_attn_decode_k2v4_workspace_size.restype = S
    L.kv_attn_decode_k2v4_workspace_size.argtypes = [pk, I32, I32, I64, C.c_int]
    L.kv_attn_decode_k2v4.restype = C.c_int
    L.kv_attn_decode_k2v4.argtypes = [pk, P, I32, I32, I64, I64, P, P, P, P, P, C.c_float, P, P, S, C.c_int, P]


def status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


def version() -> str:
    return lib().kvq_version().decode()


def _ok(status: int, what: str):
    if status != 0:
        raise KvqError(status, what)


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _qdtype(q: torch.Tensor) -> int:
    if q.dtype == torch.float32:
        return KVQ_F32
    if q.dtype == torch.bfloat16:
        return KVQ_BF16
    raise ValueError("query must be float32 or bfloat16")


def codebook(which: int):
    n = 16 if which == 16 else 4
    lv = (C.c_float * n)()
    th = (C.c_float * (n - 1))()
    _ok(lib().kvq_codebook(which, lv, th), "kvq_codebook")
    return list(lv), list(th)


# -- producers ---------------------------------------------------------------

def _err_ptr(err_word):
    """A device int32 error word: an int32 tensor, or a uint8 workspace (its first 4 bytes)."""
    if err_word is None:
        return None
    if err_word.dtype not in (torch.int32, torch.uint8):
        raise ValueError("err_word must be an int32 tensor or a uint8 workspace")
    return _ptr(err_word, None, "err_word")


def kv8_encode(x, codes, scales, layout: MLALayout | None = None, dst_rows=None, stream=None, err_word=None):
    """Encode rows of x into the pool; row i goes to pool row dst_rows[i] (or i).
    A non-finite row sets err_word (if given) to KVQ_ERR_NONFINITE."""
    layout = layout or mla_layout()
    _ok(lib().kv8_encode(_ptr(x, torch.float32, "x"), x.shape[0], C.byref(layout),
                         _ptr(dst_rows, torch.int64, "dst_rows"), _ptr(codes, torch.uint8, "codes"),
                         _ptr(scales, torch.float32, "scales"), _err_ptr(err_word), _stream(stream)), "kv8_encode")


def tq4_encode(x, packed, scales, layout: MLALayout | None = None, dst_rows=None, stream=None, err_word=None):
    layout = layout or mla_layout()
    _ok(lib().tq4_encode(_ptr(x, torch.float32, "x"), x.shape[0], C.byref(layout),
                         _ptr(dst_rows, torch.int64, "dst_rows"), _ptr(packed, torch.uint8, "packed"),
                         _ptr(scales, torch.float32, "scales"), _err_ptr(err_word), _stream(stream)), "tq4_encode")


def tq4_encode_status(x, packed, scales, layout: MLALayout, stream=None) -> int:
    return lib().tq4_encode(_ptr(x, torch.float32, "x"), x.shape[0], C.byref(layout), None, _ptr(packed),
                            _ptr(scales), None, _stream(stream))


def pq_format(bits: int) -> int:
    """The PolarQuant format at `bits` (2..6) bits per angle."""
    if not 2 <= bits <= 6:
        raise ValueError("PolarQuant widths are 2..6 bits")
    return 10 + bits


def row_bytes(fmt: int, layout: MLALayout | None = None) -> int:
    """Code bytes of one row of `fmt` (scales excluded); raises for an invalid pair."""
    layout = layout or mla_layout()
    n = lib().kvq_row_bytes(fmt, C.byref(layout))
    if n <= 0:
        raise KvqError(1, "kvq_row_bytes")
    return n


def pq_codebook(bits: int, level: int):
    """The library's f32 PolarQuant tables of one width and level: centroids
    [2^bits][2] and thresholds [2^bits - 1][2] (cos, sin); level 1 gives its
    2^(bits-2) - 1 in-quadrant thresholds."""
    import numpy as np
    n = 1 << bits
    c = np.zeros((n, 2), np.float32)
    t = np.zeros((n - 1, 2), np.float32)
    _ok(lib().kvq_pq_codebook(bits, level, c.ctypes.data_as(C.c_void_p), t.ctypes.data_as(C.c_void_p)),
        "kvq_pq_codebook")
    return c, (t[: n // 4 - 1] if level == 1 else t)


def pq_encode(fmt: int, x, codes, radii, layout: MLALayout | None = None, dst_rows=None, stream=None,
              err_word=None):
    """PolarQuant-encode rows of x into the pool (codes [*][row_bytes], radii
    [*][n_blocks]); row i goes to pool row dst_rows[i] (or i)."""
    layout = layout or mla_layout()
    _ok(lib().pq_encode(fmt, _ptr(x, torch.float32, "x"), x.shape[0], C.byref(layout),
                        _ptr(dst_rows, torch.int64, "dst_rows"), _ptr(codes, torch.uint8, "codes"),
                        _ptr(radii, torch.float32, "radii"), _err_ptr(err_word), _stream(stream)), "pq_encode")


def pq_decode(fmt: int, codes, radii, out, layout: MLALayout | None = None, rotated: bool = False, stream=None):
    """Rebuild PolarQuant rows as f32 (unrotated, or in the rotated domain)."""
    layout = layout or mla_layout()
    _ok(lib().pq_decode(fmt, _ptr(codes, torch.uint8, "codes"), _ptr(radii, torch.float32, "radii"),
                        codes.shape[0], C.byref(layout), int(rotated), _ptr(out, torch.float32, "out"),
                        _stream(stream)), "pq_decode")


def test_stall_waits(polls: int) -> None:
    """Testing hook: later tensor-core attention launches stall on a barrier
    nothing arrives on for `polls` polls (then report KVQ_ERR_TIMEOUT); 0 = off."""
    _ok(lib().kvq_test_stall_waits(int(polls)), "kvq_test_stall_waits")


def tq4_rotate(inp, out, layout: MLALayout | None = None, inverse=False, stream=None):
    layout = layout or mla_layout()
    D = layout.block_dim[0] + (layout.block_dim[1] if layout.n_blocks > 1 else 0)
    n = inp.numel() // D
    _ok(lib().tq4_rotate(_ptr(inp, None, "in"), _qdtype(inp), n, C.byref(layout), int(inverse),
                         _ptr(out, torch.float32, "out"), _stream(stream)), "tq4_rotate")


# -- consumers ---------------------------------------------------------------

def kv_attn_workspace_size(fmt: int, batch: int, n_heads: int, max_total_rows: int,
                           layout: MLALayout | None = None, path: int = PATH_AUTO) -> int:
    layout = layout or mla_layout()
    return lib().kv_attn_workspace_size(fmt, C.byref(layout), batch, n_heads, max_total_rows, path)


def kv_attn_decode(fmt: int, q, codes, scales, cu_seqlens, out, workspace, max_total_rows: int,
                   sm_scale: float = SM_SCALE_MLA, layout: MLALayout | None = None, path: int = PATH_AUTO,
                   stream=None):
    layout = layout or mla_layout()
    B, H = q.shape[0], q.shape[1]
    _ok(lib().kv_attn_decode(fmt, C.byref(layout), _ptr(q, None, "q"), _qdtype(q), B, H,
                             _ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"),
                             _ptr(cu_seqlens, torch.int64, "cu_seqlens"), int(max_total_rows), float(sm_scale),
                             _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
                             workspace.numel(), path, _stream(stream)), "kv_attn_decode")


def kv_attn_decode_append(fmt: int, x_new, dst_rows, q, codes, scales, cu_seqlens, out, workspace,
                          max_total_rows: int, sm_scale: float = SM_SCALE_MLA, layout: MLALayout | None = None,
                          path: int = PATH_AUTO, stream=None):
    """One decode step with its new rows: x_new[b] is encoded into pool row
    dst_rows[b] (inside sequence b), then attention runs over the pool."""
    layout = layout or mla_layout()
    B, H = q.shape[0], q.shape[1]
    _ok(lib().kv_attn_decode_append(fmt, C.byref(layout), _ptr(x_new, torch.float32, "x_new"),
                                    _ptr(dst_rows, torch.int64, "dst_rows"), _ptr(q, None, "q"), _qdtype(q), B, H,
                                    _ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"),
                                    _ptr(cu_seqlens, torch.int64, "cu_seqlens"), int(max_total_rows),
                                    float(sm_scale), _ptr(out, torch.float32, "out"),
                                    _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), path,
                                    _stream(stream)), "kv_attn_decode_append")


def kv_attn_gather_workspace_size(fmt: int, batch: int, n_heads: int, max_total_selected: int, bf16: bool = True,
                                  layout: MLALayout | None = None, path: int = PATH_AUTO) -> int:
    layout = layout or mla_layout()
    return lib().kv_attn_gather_workspace_size(fmt, C.byref(layout), KVQ_BF16 if bf16 else KVQ_F32, batch, n_heads,
                                               max_total_selected, path)


def kv_attn_decode_gather(fmt: int, q, codes, scales, sel_rows, cu_sel, out, workspace, max_total_selected: int,
                          sm_scale: float = SM_SCALE_MLA, layout: MLALayout | None = None, path: int = PATH_AUTO,
                          stream=None):
    """Decode over selected rows: sequence b attends the pool rows
    sel_rows[cu_sel[b]:cu_sel[b+1]] (absolute indices)."""
    layout = layout or mla_layout()
    B, H = q.shape[0], q.shape[1]
    _ok(lib().kv_attn_decode_gather(fmt, C.byref(layout), _ptr(q, None, "q"), _qdtype(q), B, H,
                                    _ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"),
                                    int(codes.shape[0]), _ptr(sel_rows, torch.int64, "sel_rows"),
                                    _ptr(cu_sel, torch.int64, "cu_sel"), int(max_total_selected), float(sm_scale),
                                    _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
                                    workspace.numel(), path, _stream(stream)), "kv_attn_decode_gather")


def kv_attn_decode_noalloc(fmt: int, q, codes, scales, cu_seqlens, out, max_total_rows: int,
                           sm_scale: float = SM_SCALE_MLA, layout: MLALayout | None = None, path: int = PATH_AUTO,
                           stream=None):
    """kv_attn_decode without a caller-provided workspace (the library's fixed
    32 MiB device scratch is used; concurrent calls race)."""
    layout = layout or mla_layout()
    B, H = q.shape[0], q.shape[1]
    _ok(lib().kv_attn_decode_noalloc(fmt, C.byref(layout), _ptr(q, None, "q"), _qdtype(q), B, H,
                                     _ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"),
                                     _ptr(cu_seqlens, torch.int64, "cu_seqlens"), int(max_total_rows),
                                     float(sm_scale), _ptr(out, torch.float32, "out"), path, _stream(stream)),
        "kv_attn_decode_noalloc")


def kv_attn_prefill_workspace_size(fmt: int, n_heads: int, n_past: int, n_new: int,
                                   layout: MLALayout | None = None, path: int = PATH_AUTO) -> int:
    layout = layout or mla_layout()
    return lib().kv_attn_prefill_workspace_size(fmt, C.byref(layout), n_heads, n_past, n_new, path)


def kv_attn_prefill(fmt: int, x_new, q, codes, scales, n_past: int, out, workspace,
                    sm_scale: float = SM_SCALE_MLA, layout: MLALayout | None = None, path: int = PATH_AUTO,
                    stream=None):
    layout = layout or mla_layout()
    n_new, H = q.shape[0], q.shape[1]
    _ok(lib().kv_attn_prefill(fmt, C.byref(layout), _ptr(x_new, torch.float32, "x_new"), _ptr(q, None, "q"),
                              _qdtype(q), int(n_past), n_new, H, _ptr(codes, torch.uint8, "codes"),
                              _ptr(scales, torch.float32, "scales"), float(sm_scale), _ptr(out, torch.float32, "out"),
                              _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), path, _stream(stream)),
        "kv_attn_prefill")


def read_device_error(workspace, clear: bool = True, stream=None) -> int:
    return lib().kvq_read_device_error(_ptr(workspace, torch.uint8, "workspace"), int(clear), _stream(stream))


def read_exact_rescales(workspace, clear: bool = True, stream=None) -> int:
    """Tiles after a work item's first that took the tensor kernels' exact
    rescale path since the counter was last cleared."""
    v = lib().kvq_read_exact_rescales(_ptr(workspace, torch.uint8, "workspace"), int(clear), _stream(stream))
    if v < 0:
        raise KvqError(4, "kvq_read_exact_rescales")
    return v


def timing_enable(capacity: int) -> None:
    """Opt-in launch timing of the attention calls (events before the partial
    kernel, before and after the merge); 0 turns it off."""
    _ok(lib().kvq_timing_enable(int(capacity)), "kvq_timing_enable")


def timing_read() -> tuple[float, float, int]:
    """(partial kernel ms, merge ms, calls) summed over the recorded calls;
    waits for them and empties the record."""
    a, b, n = C.c_double(), C.c_double(), C.c_int32()
    _ok(lib().kvq_timing_read(C.byref(a), C.byref(b), C.byref(n)), "kvq_timing_read")
    return a.value, b.value, n.value


# -- K2/V4 -------------------------------------------------------------------

def k2v4_encode(layout: K2V4Layout, k, v, k_codes, k_scales, v_blocks, k_win, v_win, capacity: int | None = None,
                stream=None, err_word=None):
    B, H, T, D = k.shape
    cap = T if capacity is None else capacity
    _ok(lib().k2v4_encode(C.byref(layout), _ptr(k, torch.float32, "k"), _ptr(v, torch.float32, "v"), B, T, cap,
                          _ptr(k_codes, torch.uint8, "k_codes"), _ptr(k_scales, torch.int16, "k_scales"),
                          _ptr(v_blocks, torch.uint8, "v_blocks"), _ptr(k_win, torch.int16, "k_win"),
                          _ptr(v_win, torch.int16, "v_win"), _err_ptr(err_word), _stream(stream)), "k2v4_encode")


def k2v4_append(layout: K2V4Layout, k_new, v_new, n_past: int, k_codes, k_scales, v_blocks, k_win, v_win,
                stream=None, err_word=None):
    """Append k_new, v_new ([B, Hkv, n_new, D] f32) at cells n_past .. n_past + n_new - 1 of every
    sequence; the pools' capacity is their cell dimension."""
    B, H, n_new, D = k_new.shape
    cap = k_codes.shape[2]
    _ok(lib().k2v4_append(C.byref(layout), _ptr(k_new, torch.float32, "k_new"), _ptr(v_new, torch.float32, "v_new"),
                          B, n_past, n_new, cap, _ptr(k_codes, torch.uint8, "k_codes"),
                          _ptr(k_scales, torch.int16, "k_scales"), _ptr(v_blocks, torch.uint8, "v_blocks"),
                          _ptr(k_win, torch.int16, "k_win"), _ptr(v_win, torch.int16, "v_win"), _err_ptr(err_word),
                          _stream(stream)),
        "k2v4_append")


def kv_attn_decode_k2v4_workspace_size(layout: K2V4Layout, batch: int, n_q_heads: int, n_cells: int,
                                       path: int = PATH_AUTO) -> int:
    return lib().kv_attn_decode_k2v4_workspace_size(C.byref(layout), batch, n_q_heads, n_cells, path)


def kv_attn_decode_k2v4(layout: K2V4Layout, q, n_cells: int, k_codes, k_scales, v_blocks, k_win, v_win, out,
                        workspace, sm_scale: float, capacity: int | None = None, path: int = PATH_AUTO, stream=None):
    B, Hq, D = q.shape
    cap = n_cells if capacity is None else capacity
    _ok(lib().kv_attn_decode_k2v4(C.byref(layout), _ptr(q, torch.float32, "q"), B, Hq, n_cells, cap,
                                  _ptr(k_codes, torch.uint8, "k_codes"), _ptr(k_scales, torch.int16, "k_scales"),
                                  _ptr(v_blocks, torch.uint8, "v_blocks"), _ptr(k_win, torch.int16, "k_win"),
                                  _ptr(v_win, torch.int16, "v_win"), float(sm_scale), _ptr(out, torch.float32, "out"),
                                  _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), path,
                                  _stream(stream)), "kv_attn_decode_k2v4")


# -- persistence of quantized pools (host arrays) ------------------------------

class CacheFileError(KvqError):
    """A cache file was refused (another tier/codec/layout) or unreadable; .msg says why."""

    def __init__(self, status: int, what: str, msg: str):
        super().__init__(status, what)
        self.msg = msg

    def __str__(self):
        return f"{super().__str__()}: {self.msg}"


def _np_ptr(a):
    return None if a is None else C.c_void_p(a.ctypes.data)


def _row_bytes(fmt: int, layout: MLALayout) -> int:
    return row_bytes(fmt, layout)


def cache_save(path: str, fmt: int, codes, scales, layout: MLALayout | None = None):
    import numpy as np
    layout = layout or mla_layout()
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    _ok(lib().kvq_cache_save(path.encode(), fmt, C.byref(layout), codes.shape[0], _np_ptr(codes), _np_ptr(scales)),
        "kvq_cache_save")


def cache_save_f32(path: str, rows, layout: MLALayout | None = None):
    import numpy as np
    layout = layout or mla_layout()
    rows = np.ascontiguousarray(rows, np.float32)
    _ok(lib().kvq_cache_save_f32(path.encode(), C.byref(layout), rows.shape[0], _np_ptr(rows)), "kvq_cache_save_f32")


def cache_info(path: str):
    """(version, rows, header words)."""
    import numpy as np
    v, n, h = C.c_int32(), C.c_int64(), np.zeros(8, np.int64)
    msg = C.create_string_buffer(256)
    st = lib().kvq_cache_info(path.encode(), C.byref(v), C.byref(n), _np_ptr(h), msg, 256)
    if st != 0:
        raise CacheFileError(st, "kvq_cache_info", msg.value.decode())
    return v.value, n.value, h


def cache_load(path: str, fmt: int, capacity: int, layout: MLALayout | None = None):
    """(codes [n][row_bytes] u8, scales [n][n_blocks] f32); raises CacheFileError on refusal."""
    import numpy as np
    layout = layout or mla_layout()
    codes = np.zeros((capacity, _row_bytes(fmt, layout)), np.uint8)
    scales = np.zeros((capacity, layout.n_blocks), np.float32)
    n = C.c_int64()
    msg = C.create_string_buffer(256)
    st = lib().kvq_cache_load(path.encode(), fmt, C.byref(layout), capacity, _np_ptr(codes), _np_ptr(scales),
                              C.byref(n), msg, 256)
    if st != 0:
        raise CacheFileError(st, "kvq_cache_load", msg.value.decode())
    return codes[:n.value], scales[:n.value]


def cache_load_f32(path: str, capacity: int, layout: MLALayout | None = None):
    import numpy as np
    layout = layout or mla_layout()
    D = sum(layout.block_dim[b] for b in range(layout.n_blocks))
    rows = np.zeros((capacity, D), np.float32)
    n = C.c_int64()
    msg = C.create_string_buffer(256)
    st = lib().kvq_cache_load_f32(path.encode(), C.byref(layout), capacity, _np_ptr(rows), C.byref(n), msg, 256)
    if st != 0:
        raise CacheFileError(st, "kvq_cache_load_f32", msg.value.decode())
    return rows[:n.value]


def cache_append(path: str, fmt: int, codes, scales, layout: MLALayout | None = None):
    """Appends rows in place; returns (total rows, message)."""
    import numpy as np
    layout = layout or mla_layout()
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    n = C.c_int64()
    msg = C.create_string_buffer(256)
    st = lib().kvq_cache_append(path.encode(), fmt, C.byref(layout), codes.shape[0], _np_ptr(codes), _np_ptr(scales),
                                C.byref(n), msg, 256)
    if st != 0:
        raise CacheFileError(st, "kvq_cache_append", msg.value.decode())
    return n.value, msg.value.decode()

