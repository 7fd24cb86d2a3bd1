"""Seeded, counter-based synthetic inputs for the CSA2 decode path.

This module is shared by the CPU oracle and the GPU path and holds none of the
method's arithmetic: it only draws numbers.  Every value is a pure function of
(seed, stream, sub-stream, counter), so any row of any tensor can be produced on
its own, in any order, on the host (this module) or on the device (the CUDA
twin in ``gen_cuda.cu``, which must give the same bits; a GPU test checks it).

Building blocks (all integer, so both sides agree bit for bit):

* ``mix64`` -- the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).  Counter i of
  a stream with key K gives ``mix64(K + (i + 1) * GOLDEN)``.
* Normal variates come from the top 20 bits of that word used as an index into
  a table of 2**20 standard-normal quantiles, ``Phi^-1((i + 0.5) / 2**20)``,
  each rounded to bfloat16.  The table is data: the device gets a copy of these
  exact bytes, so no transcendental function is evaluated twice.
* Zipf ranks use a seeded bijection of [0, 2**b) (a 4-round Feistel network
  whose round function is ``mix64``) with cycle walking down to [0, N).
* Scaled values (Zipf keys, indexer weights) are one IEEE fp32 multiply (and for
  Zipf one fp32 division) followed by round-to-nearest-even to bfloat16, all
  correctly rounded operations that every IEEE machine computes identically.

Workload recipes (which stream feeds which tensor, and the distributions) live
in ``gen/workloads.py``.
"""
from __future__ import annotations

import numpy as np

MASK64 = np.uint64(0xFFFFFFFFFFFFFFFF)
GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
TABLE_BITS = 20

# stream ids (one per independent random tensor kind)
S_LATENT = 1      # 512-wide k=v latents, bf16 N(0,1)
S_IDX_KEY = 2     # 128-wide indexer keys (direction part), bf16 N(0,1)
S_Q = 3           # attention queries [64 x 512], bf16 N(0,1)
S_QIDX = 4        # indexer queries [32 x 128], bf16 N(0,1) before FP4 packing
S_W = 5           # indexer per-head weights, N(0, 1/32)
S_SWA = 6         # sliding-window entries [512], bf16 N(0,1)
S_GATE = 7        # m=2 gate logits, N(0,1) (fp32 holding bf16 values)
S_ZIPF = 8        # Zipf rank permutation of cache positions
S_QIDX_RE = 9     # Reindex-layer indexer queries
S_W_RE = 10       # Reindex-layer indexer weights
S_SCORES = 11     # raw fp32 scores for top-k tests
S_MISC = 12       # anything else a test needs
S_LQ = 13         # attention queries of the decoder step's other layers (sub = layer * 65536 + query)
S_LSWA = 14       # sliding-window entries of those layers (sub = layer * 65536 + sequence)
LAYER_SUB = 65536  # sub-stream stride per layer (Reindex layer r: S_QIDX_RE / S_W_RE with sub r * 65536 + query)

W_STD_F32 = np.float32(1.0 / np.sqrt(32.0))   # weights ~ N(0, variance 1/32)


def mix64(z):
    """SplitMix64 output function on uint64 (array or scalar), wrapping."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, stream: int, sub: int = 0) -> int:
    """64-bit key of (seed, stream, sub-stream); returned as a Python int."""
    with np.errstate(over="ignore"):
        a = mix64(np.uint64(seed & 0xFFFFFFFF) ^ (np.uint64(stream & 0xFFFF) << np.uint64(32)))
        b = mix64(a + np.uint64(sub & 0xFFFFFFFFFFFF) * GOLDEN)
    return int(b)


def words(key: int, counters) -> np.ndarray:
    """Random uint64 word for each counter of the stream with this key."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + (c + np.uint64(1)) * GOLDEN)


_TABLE = None


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (nearest, ties to even); finite inputs only."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_table() -> np.ndarray:
    """2**20 standard-normal quantiles as bfloat16 bit patterns (uint16)."""
    global _TABLE
    if _TABLE is None:
        from scipy.special import ndtri
        p = (np.arange(1 << TABLE_BITS, dtype=np.float64) + 0.5) / float(1 << TABLE_BITS)
        _TABLE = _f32_to_bf16_bits(ndtri(p).astype(np.float32))
    return _TABLE


def normal_bf16(key: int, counters) -> np.ndarray:
    """bf16 bit patterns of N(0,1) variates for the given counters."""
    w = words(key, counters)
    return normal_table()[(w >> np.uint64(64 - TABLE_BITS)).astype(np.int64)]


def normal_rows_bf16(seed: int, stream: int, sub: int, rows, ncols: int) -> np.ndarray:
    """[len(rows), ncols] bf16 bits; element (r, c) uses counter r*ncols + c."""
    rows = np.asarray(rows, dtype=np.uint64).reshape(-1, 1)
    ctr = rows * np.uint64(ncols) + np.arange(ncols, dtype=np.uint64).reshape(1, -1)
    return normal_bf16(stream_key(seed, stream, sub), ctr)


def normal_block_bf16(seed: int, stream: int, sub: int, row0: int, nrows: int, ncols: int) -> np.ndarray:
    return normal_rows_bf16(seed, stream, sub, np.arange(row0, row0 + nrows, dtype=np.uint64), ncols)


# ---------------------------------------------------------------- Zipf ranks
def _bits_for(n: int) -> int:
    b = max(2, int(n - 1).bit_length())
    return b + (b & 1)          # even, so the Feistel halves are equal


def _feistel(x: np.ndarray, key: int, bits: int) -> np.ndarray:
    half = bits // 2
    mask = np.uint64((1 << half) - 1)
    L = (x >> np.uint64(half)) & mask
    R = x & mask
    k = np.uint64(key)
    for rnd in range(4):
        with np.errstate(over="ignore"):
            f = mix64(k ^ (np.uint64(rnd) << np.uint64(56)) ^ R) & mask
        L, R = R, L ^ f
    return (L << np.uint64(half)) | R


def zipf_rank(seed: int, sub: int, n: int, positions) -> np.ndarray:
    """rank in 1..n of each cache position (a seeded permutation of 1..n)."""
    bits = _bits_for(n)
    key = stream_key(seed, S_ZIPF, sub)
    x = np.asarray(positions, dtype=np.uint64).copy()
    x = _feistel(x, key, bits)
    todo = x >= np.uint64(n)
    while np.any(todo):                 # cycle walking back into [0, n)
        x[todo] = _feistel(x[todo], key, bits)
        todo = x >= np.uint64(n)
    return x.astype(np.int64) + 1


def zipf_keys_bf16(seed: int, sub: int, n: int, positions, ncols: int = 128) -> np.ndarray:
    """Indexer keys with Zipf norms: bf16(fp32(g) * fp32(1 / rank)), g ~ N(0,1)."""
    positions = np.asarray(positions, dtype=np.int64)
    g = bf16_bits_to_f32(normal_rows_bf16(seed, S_IDX_KEY, sub, positions, ncols))
    r = np.float32(1.0) / zipf_rank(seed, sub, n, positions).astype(np.float32)
    return _f32_to_bf16_bits(g * r.reshape(-1, 1))


def weights_f32(seed: int, stream: int, sub: int, rows, ncols: int = 32) -> np.ndarray:
    """Indexer per-head weights, fp32(g) * fp32(1/sqrt(32)), g ~ N(0,1)."""
    g = bf16_bits_to_f32(normal_rows_bf16(seed, stream, sub, rows, ncols))
    return (g * W_STD_F32).astype(np.float32)


def gate_logits_f32(seed: int, sub: int, rows, ncols: int = 512) -> np.ndarray:
    return bf16_bits_to_f32(normal_rows_bf16(seed, S_GATE, sub, rows, ncols))


def uniform_f32_scores(seed: int, sub: int, n: int, levels: int = 0) -> np.ndarray:
    """fp32 test scores in [-1, 1); with ``levels`` > 0 they are quantised to
    that many values so that exact ties are common."""
    w = words(stream_key(seed, S_SCORES, sub), np.arange(n, dtype=np.uint64))
    u = (w >> np.uint64(40)).astype(np.float64) / float(1 << 24)      # 24-bit uniform in [0,1)
    if levels:
        u = np.floor(u * levels) / levels
    return (2.0 * u - 1.0).astype(np.float32)
