"""Seeded synthetic inputs for the quantized-KV MLA workloads.

This module only draws numbers; it holds none of the codecs' or attention's
arithmetic.  Both the CUDA path and the CPU oracle are fed from it.

Generator: counter-based splitmix64 (Steele, Lea, Flood 2014).  Each named
stream gets its own key, output i of a stream is mix(key + (i+1) * golden).
Normals come from Box-Muller in float64 and are rounded once to float32.

Workload recipes (shapes from the benchmark configurations; value statistics
from the pages: latent rows are N(0,1) times a per-channel log-normal gain, the
channel-outlier structure that the Strata pull request measures as 5.8x-74.9x
max/median channel RMS on real K):

* ``mla_rows``   latent rows [n, 576]: x[t,i] = g_i * z[t,i], z ~ N(0,1),
                 g_i = exp(sigma * n_i), n_i ~ N(0,1), sigma = 1.
* ``queries``    [*, 576] N(0,1), optionally rounded to bfloat16 (RNE).
* ``ragged_lengths`` uniform integers in [lo, hi].
* ``gqa_kv``     K [B, Hkv, T, D] with per-(kv head, channel) log-normal gains,
                 V [B, Hkv, T, D] N(0,1).
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream identifiers
S_GAIN, S_ROWS, S_QUERY, S_LEN, S_KGAIN, S_K, S_V = range(1, 8)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed * 1000003 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(base + GOLDEN)[0]


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+n-1 of stream ``stream`` of seed ``seed``."""
    k = _key(seed, stream)
    with np.errstate(over="ignore"):
        idx = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix(k + idx * GOLDEN)


def uniform(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Doubles in [0, 1) with 53 random bits."""
    return (u64(seed, stream, n, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Float64 N(0,1) samples (one Box-Muller draw per pair of uniforms)."""
    u = uniform(seed, stream, 2 * n, 2 * offset)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)


def channel_gains(seed: int, dim: int, sigma: float = 1.0, stream: int = S_GAIN) -> np.ndarray:
    return np.exp(sigma * normal(seed, stream, dim))


def mla_rows(seed: int, n_rows: int, dim: int = 576, sigma: float = 1.0, row_offset: int = 0) -> np.ndarray:
    """Latent rows [n_rows, dim] float32; rows row_offset.. of the seed's row stream."""
    g = channel_gains(seed, dim, sigma)
    z = normal(seed, S_ROWS, n_rows * dim, row_offset * dim).reshape(n_rows, dim)
    return (z * g[None, :]).astype(np.float32)


def queries(seed: int, shape, stream: int = S_QUERY) -> np.ndarray:
    n = int(np.prod(shape))
    return normal(seed, stream, n).astype(np.float32).reshape(shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the 16-bit patterns."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """batch integers uniform in [lo, hi]."""
    span = np.uint64(hi - lo + 1)
    return (u64(seed, S_LEN, batch) % span).astype(np.int64) + lo


def cu_seqlens(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, np.int64))
    return cu


def gqa_kv(seed: int, batch: int, n_kv_heads: int, n_cells: int, head_dim: int, sigma: float = 1.0):
    """K [B, Hkv, T, D] with log-normal channel gains per kv head; V [B, Hkv, T, D] N(0,1)."""
    g = np.exp(sigma * normal(seed, S_KGAIN, n_kv_heads * head_dim)).reshape(1, n_kv_heads, 1, head_dim)
    n = batch * n_kv_heads * n_cells * head_dim
    k = (normal(seed, S_K, n).reshape(batch, n_kv_heads, n_cells, head_dim) * g).astype(np.float32)
    v = normal(seed, S_V, n).astype(np.float32).reshape(batch, n_kv_heads, n_cells, head_dim)
    return k, v


# ----------------------------------------------------------------------------
# The five workloads (one Python description each; sizes only).
# ----------------------------------------------------------------------------
CONFIGS = {
    1: dict(name="tiny: 1 seq x 256 rows, 16 heads, KV8 then TQ4 (sign seed 0)",
            batch=1, seqlen=256, heads=16, q_dtype="f32"),
    2: dict(name="KV8 decode: 8 seqs x 4096 rows, 128 heads, bf16 query",
            batch=8, seqlen=4096, heads=128, q_dtype="bf16", fmt="kv8"),
    3: dict(name="TQ4 decode: 8 seqs x 4096 rows, 128 heads, bf16 query",
            batch=8, seqlen=4096, heads=128, q_dtype="bf16", fmt="tq4"),
    4: dict(name="ragged decode: 32 seqs, lengths U[1024,131072] (seed 4), 128 heads; "
                 "prefill 2048 new tokens over 126976 past rows",
            batch=32, len_lo=1024, len_hi=131072, heads=128, q_dtype="bf16",
            prefill_past=126976, prefill_new=2048),
    5: dict(name="K2/V4 GQA: 4 seqs x 32768 cells, 2 kv heads x 256, 16 q heads, "
                 "sinks 8, window 256, K gain 1.10",
            batch=4, seqlen=32768, kv_heads=2, q_heads=16, head_dim=256, n_sink=8, n_window=256,
            k_gain=1.10),
}
