"""Pure-Python loops for tiny inputs (oracle side).

Written independently of the numpy oracle so each pins the other: the score
is summed term by term, blocks and top-k come from Python's ``sorted`` with
the key (-score, id), and attention is an explicit softmax loop.  Only for
contexts of a few dozen positions.
"""
from __future__ import annotations

import math


def e4m3(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 0:
        return s * m / 512.0
    return s * (8 + m) / 8.0 * 2.0 ** (e - 7)


def score(q, w, key_codes, key_scale) -> float:
    """q: 8 lists of 64 floats; w: 8 floats; key_codes: 64 ints; key_scale: float."""
    total = 0.0
    for h in range(len(q)):
        d = 0.0
        for i in range(len(key_codes)):
            d += q[h][i] * e4m3(key_codes[i])
        total += w[h] * (d if d > 0.0 else 0.0)
    return key_scale * total


def select(q, w, codes, scales, block, n_keep, topk):
    """(pool ascending, top-k ascending) for one tiny sequence."""
    L = len(codes)
    sig = [score(q, w, codes[t], scales[t]) for t in range(L)]
    blocks = []
    for j in range((L + block - 1) // block):
        members = sig[j * block:min(L, j * block + block)]
        blocks.append((max(members), j))
    best_blocks = sorted(blocks, key=lambda x: (-x[0], x[1]))[:n_keep]
    best_pos = sorted([(sig[t], t) for t in range(L)], key=lambda x: (-x[0], x[1]))[:topk]
    return sorted(j for _, j in best_blocks), sorted(t for _, t in best_pos), sig


def reselect(q, w, codes, scales, pool, block, topk):
    """Top-k over the pool's positions only."""
    L = len(codes)
    cand = [t for j in pool if j >= 0 for t in range(j * block, min(L, j * block + block))]
    ranked = sorted([(score(q, w, codes[t], scales[t]), t) for t in cand], key=lambda x: (-x[0], x[1]))
    return sorted(t for _, t in ranked[:topk])


def attend(q, rows, tau):
    """q: H lists of D floats; rows: list of D-float lists -> (o, lse)."""
    out, lses = [], []
    for qh in q:
        z = [tau * sum(a * b for a, b in zip(qh, r)) for r in rows]
        if not z:
            out.append([0.0] * len(qh))
            lses.append(-math.inf)
            continue
        m = max(z)
        e = [math.exp(v - m) for v in z]
        l = sum(e)
        out.append([sum(e[j] * rows[j][d] for j in range(len(rows))) / l for d in range(len(qh))])
        lses.append(m + math.log(l))
    return out, lses


def e2m1(code: int) -> float:
    """Value of a 4-bit E2M1 code (sign bit 3, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6)."""
    mag = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)[code & 7]
    return -mag if code & 8 else mag


def fp4_row(codes, scales):
    """One packed FP4 cache row (64 bytes, 8 E4M3 group scales) back to 128 floats."""
    out = []
    for j, byte in enumerate(codes):
        s = e4m3(scales[(2 * j) // 16])
        out.append(e2m1(byte & 0xF) * s)
        out.append(e2m1(byte >> 4) * s)
    return out


def fp8_row(codes, scale):
    """One FP8 row (E4M3 codes and a per-row float scale) back to floats."""
    return [e4m3(c) * scale for c in codes]
