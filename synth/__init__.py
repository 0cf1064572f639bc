"""Seeded synthetic inputs for the CSA2 decode path.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It holds none of the method's arithmetic: it only draws numbers
and lays them out.  Every value is a pure function of (seed, stream,
coordinates), so any subset of a large workload (one sequence of a 1M-token
cache, a sample of query rows) can be regenerated on its own.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a hash of a 64-bit counter.  Uniforms
take the top 53 bits.  Normals come from the Box-Muller transform in double
precision, one (cos, sin) pair per two adjacent channels, then are rounded
double -> float32 -> bfloat16 (round to nearest even at each step).

Workload shapes follow the five configurations of the DeepSeek-V4.1-Flash
CSA2 decode path (origotech.dev deep dive, section "Compressed Sparse
Attention 2"): MQA main KV of 128 channels with 1% outlier channels scaled by
8, an 8-head x 64 indexer, 16 (or 64) query heads of dim 128, N(0,1) bf16
activations and U(0,1) head weights.
"""
from __future__ import annotations

import enum
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# coordinate packing: counter = ((layer << 35 | row) << 7) | pair
ROW_BITS = 35
PAIR_BITS = 7
POS_BITS = 22          # row = b << POS_BITS | position  (positions < 4M)
MAX_POS = 1 << POS_BITS


class Stream(enum.IntEnum):
    KV = 1
    KV_OUTLIER = 2
    IK = 3
    SWA = 4
    SWA_OUTLIER = 5
    Q = 6
    QIDX = 7
    W = 8
    LEN = 9
    TOPK = 10


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int, sub: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([(seed * 0x100000001B3 + stream * 0x1F3 + sub) & 0xFFFFFFFFFFFFFFFF],
                     dtype=np.uint64)
        return _mix64(_mix64(k) + _GAMMA)[0]


def _bits(seed: int, stream: int, sub: int, counter: np.ndarray) -> np.ndarray:
    key = _key(seed, stream, sub)
    with np.errstate(over="ignore"):
        return _mix64(key + (counter.astype(np.uint64) + np.uint64(1)) * _GAMMA)


def uniform(seed: int, stream: int, counter: np.ndarray, sub: int = 0) -> np.ndarray:
    """Uniform doubles in (0, 1], one per counter value."""
    b = _bits(seed, stream, sub, np.asarray(counter, dtype=np.uint64))
    return ((b >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_POOL: ThreadPoolExecutor | None = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _normals_chunk(seed, stream, layer, rows, n_ch, out, lo, hi, outliers, outlier_scale):
    n_pair = n_ch // 2
    r = rows[lo:hi].astype(np.uint64)
    base = ((np.uint64(layer) << np.uint64(ROW_BITS)) | r) << np.uint64(PAIR_BITS)
    ctr = base[:, None] + np.arange(n_pair, dtype=np.uint64)[None, :]
    u1 = uniform(seed, stream, ctr, sub=0)
    u2 = uniform(seed, stream, ctr, sub=1)
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * math.pi * u2
    z = np.empty((hi - lo, n_ch), dtype=np.float64)
    z[:, 0::2] = rad * np.cos(ang)
    z[:, 1::2] = rad * np.sin(ang)
    for c in outliers:
        z[:, c] *= outlier_scale
    out[lo:hi] = f32_to_bf16_bits(z.astype(np.float32))


def normals_bf16(seed: int, stream: int, layer: int, rows: np.ndarray, n_ch: int,
                 outliers=(), outlier_scale: float = 8.0, chunk: int = 32768) -> np.ndarray:
    """N(0,1) bf16 bit patterns, shape [len(rows), n_ch].

    ``rows`` are row coordinates (see ``row_id``); ``outliers`` lists channel
    ids multiplied by ``outlier_scale`` before rounding to bf16.
    """
    assert n_ch % 2 == 0 and n_ch // 2 <= (1 << PAIR_BITS)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.shape[0], n_ch), dtype=np.uint16)
    n = rows.shape[0]
    if n == 0:
        return out
    spans = [(lo, min(n, lo + chunk)) for lo in range(0, n, chunk)]
    if len(spans) == 1:
        _normals_chunk(seed, stream, layer, rows, n_ch, out, 0, n, tuple(outliers), outlier_scale)
    else:
        futs = [_pool().submit(_normals_chunk, seed, stream, layer, rows, n_ch, out, lo, hi,
                               tuple(outliers), outlier_scale) for lo, hi in spans]
        for f in futs:
            f.result()
    return out


def row_id(b, pos) -> np.ndarray:
    """Row coordinate of (sequence b, position pos)."""
    return (np.asarray(b, dtype=np.int64) << POS_BITS) | np.asarray(pos, dtype=np.int64)


def outlier_channels(seed: int, stream: int, n_ch: int = 128, count: int = 2) -> tuple:
    """``count`` distinct channel ids drawn from the seed (1% of 128 channels, rounded up)."""
    chosen = []
    j = 0
    while len(chosen) < count:
        c = int(uniform(seed, stream, np.array([j]))[0] * n_ch)
        c = min(c, n_ch - 1)
        if c not in chosen:
            chosen.append(c)
        j += 1
    return tuple(sorted(chosen))


def head_weights(seed: int, layer: int, b: int, n_heads: int = 8) -> np.ndarray:
    """Indexer head weights w ~ U(0,1), float32 [n_heads]."""
    ctr = ((np.uint64(layer) << np.uint64(ROW_BITS)) | np.uint64(b)) << np.uint64(PAIR_BITS)
    return uniform(seed, Stream.W, ctr + np.arange(n_heads, dtype=np.uint64)).astype(np.float32)


def ragged_lengths(seed: int, batch: int, lo: int = 4096, hi: int = 1048576) -> np.ndarray:
    """Context lengths log-uniform on [lo, hi]: floor(exp(U(ln lo, ln hi)))."""
    u = uniform(seed, Stream.LEN, np.arange(batch, dtype=np.uint64))
    lens = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return np.clip(lens, lo, hi).astype(np.int64)


def causal_topk(seed: int, q_pos: np.ndarray, k: int = 512, draws: int | None = None) -> np.ndarray:
    """Per query row, ``min(k, p+1)`` distinct positions in [0, p], ascending, -1 padded.

    Stands in for an indexer's causal selection when only the attention step
    is exercised (the chunked-query workload).
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    T = q_pos.shape[0]
    out = np.full((T, k), -1, dtype=np.int32)
    draws = draws or (k + k // 4 + 64)
    for t in range(T):
        p = int(q_pos[t])
        if p + 1 <= k:
            out[t, :p + 1] = np.arange(p + 1, dtype=np.int32)
            continue
        sel: list = []
        seen = set()
        start = 0
        while len(sel) < k:
            ctr = (np.uint64(t) << np.uint64(20)) + np.arange(start, start + draws, dtype=np.uint64)
            cand = np.minimum((uniform(seed, Stream.TOPK, ctr) * (p + 1)).astype(np.int64), p)
            for c in cand.tolist():
                if c not in seen:
                    seen.add(c)
                    sel.append(c)
                    if len(sel) == k:
                        break
            start += draws
        out[t] = np.sort(np.array(sel, dtype=np.int32))
    return out


def rope_table(n_pos: int, rot_dims: int = 64, base: float = 10000.0):
    """Rotation operand of the append: cos/sin float32 [n_pos][rot_dims/2].

    Angle of pair i at position p is p * base**(-2i/rot_dims), evaluated in
    double precision and rounded to float32.  The append takes these tables
    as inputs, so trigonometry stays outside its bit-exact contract.
    """
    half = rot_dims // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / rot_dims)
    cos = np.empty((n_pos, half), dtype=np.float32)
    sin = np.empty((n_pos, half), dtype=np.float32)
    step = 1 << 16

    def work(lo):
        hi = min(n_pos, lo + step)
        ang = np.arange(lo, hi, dtype=np.float64)[:, None] * inv[None, :]
        cos[lo:hi] = np.cos(ang).astype(np.float32)
        sin[lo:hi] = np.sin(ang).astype(np.float32)

    futs = [_pool().submit(work, lo) for lo in range(0, n_pos, step)]
    for f in futs:
        f.result()
    return cos, sin
