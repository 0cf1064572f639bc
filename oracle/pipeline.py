"""One decode step of the CSA2 decoder for selected sequences (oracle side).

Composes the oracle's steps in the order the pages give (origotech.dev deep
dive, subsection "Compressed Sparse Attention 2(CSA2)"): quantise-and-append
of the new token, the first Full layer's indexer over every position (pool +
top-k), Reindex layers over the pool, Reuse layers passing indices on, and
every layer's sparse attention over its indices plus its own SWA window.

With ``wl.drafts`` = D > 1 the step verifies D drafted positions per session
(origotech.dev deep dive, section "아키텍처는 어떻게 KV 캐시를 줄이나", the DSpark
item): positions L-D..L-1 are all in the cache, each has its own query row, the
Full layer's pool is scored with the last row's queries, and each row's top-k
of every indexer layer comes from that pool up to the row's own position.

Inputs are regenerated from ``synth`` for each sequence on its own, so any
subset of a large batch can be checked.  TEST INFRASTRUCTURE ONLY.
"""
from __future__ import annotations

import numpy as np

import synth
from synth.workloads import FULL, REINDEX, DecodeWorkload

from . import append as ap
from . import indexer as ix
from . import attention as at


def sequence_cache(wl: DecodeWorkload, b: int, rope=None, chunk: int = 1 << 18):
    """(kv_codes, kv_scales, ik_codes, ik_scale) of sequence b's positions 0..L-1."""
    L = int(wl.lengths[b])
    cos, sin = rope if rope is not None else synth.rope_table(L)
    oc = synth.outlier_channels(wl.seed, synth.Stream.KV_OUTLIER)
    parts = []
    for lo in range(0, L, chunk):
        hi = min(L, lo + chunk)
        rows = synth.row_id(b, np.arange(lo, hi))
        kv = synth.normals_bf16(wl.seed, synth.Stream.KV, 0, rows, 128, oc)
        ik = synth.normals_bf16(wl.seed, synth.Stream.IK, 0, rows, 64)
        parts.append(ap.append_rows(kv, ik, cos[lo:hi], sin[lo:hi]))
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(4))


def sequence_swa(wl: DecodeWorkload, b: int, layer: int, rope=None):
    """Ring arrays (codes [ring][128], scale [ring]) of one layer after the step's append: the
    positions in the window of any of the step's query rows."""
    L = int(wl.lengths[b])
    cos, sin = rope if rope is not None else synth.rope_table(L)
    oc = synth.outlier_channels(wl.seed, synth.Stream.SWA_OUTLIER)
    lo = max(0, L - wl.drafts - wl.window + 1)
    pos = np.arange(lo, L)
    sw = synth.normals_bf16(wl.seed, synth.Stream.SWA, layer, synth.row_id(b, pos), 128, oc)
    codes, scale = ap.swa_rows(sw, cos[lo:L], sin[lo:L])
    rc = np.zeros((wl.ring, 128), np.uint8)
    rs = np.zeros(wl.ring, np.float32)
    rc[pos % wl.ring] = codes
    rs[pos % wl.ring] = scale
    return rc, rs


def layer_inputs(wl: DecodeWorkload, b: int, layer: int, j: int | None = None):
    """(attention q bf16 [H][128], indexer q bf16 [8][64], head weights [8]) of one layer for
    query row j of sequence b (default: its last row, position L-1); the row's id is b*D + j."""
    r = b * wl.drafts + (wl.drafts - 1 if j is None else j)
    q = synth.normals_bf16(wl.seed, synth.Stream.Q, layer, synth.row_id(r, np.arange(wl.H)), 128)
    qi = synth.normals_bf16(wl.seed, synth.Stream.QIDX, layer, synth.row_id(r, np.arange(8)), 64)
    w = synth.head_weights(wl.seed, layer, r)
    return q, qi, w


def new_token_inputs(wl: DecodeWorkload, b: int, rope=None):
    """The step's own inputs to the append: bf16 main KV [D][128], indexer key [D][64] and SWA
    KV of every layer [layers][D][128] of the D = wl.drafts new tokens (positions L-D..L-1),
    with their rows of the rotation tables."""
    L = int(wl.lengths[b])
    cos, sin = rope if rope is not None else synth.rope_table(L)
    pos = np.arange(L - wl.drafts, L)
    rows = synth.row_id(b, pos)
    kv = synth.normals_bf16(wl.seed, synth.Stream.KV, 0, rows, 128,
                            synth.outlier_channels(wl.seed, synth.Stream.KV_OUTLIER))
    ik = synth.normals_bf16(wl.seed, synth.Stream.IK, 0, rows, 64)
    oc = synth.outlier_channels(wl.seed, synth.Stream.SWA_OUTLIER)
    sw = [synth.normals_bf16(wl.seed, synth.Stream.SWA, l, rows, 128, oc) for l in range(wl.n_layers)]
    return kv, ik, sw, cos[pos], sin[pos]


def append_token(new_inputs):
    """Quantise-and-append of the step's new tokens (origotech.dev deep dive, subsection "FP4와
    SWA Bounded Replay"): their cache rows (FP4 main KV, FP8 indexer key) and one FP8 window
    row per layer."""
    kv, ik, sw, cos, sin = new_inputs
    return ap.append_rows(kv, ik, cos, sin), [ap.swa_rows(x, cos, sin) for x in sw]


def prepare(wl: DecodeWorkload, b: int, layers=None):
    """Per-sequence state that exists before the step: cache rows 0..L-1, window rings, layer
    inputs, and the new tokens' append inputs ('new')."""
    L = int(wl.lengths[b])
    rope = synth.rope_table(L)
    layers = list(range(wl.n_layers)) if layers is None else list(layers)
    return {
        "cache": sequence_cache(wl, b, rope),
        "swa": {l: sequence_swa(wl, b, l, rope) for l in layers},
        "inputs": {l: layer_inputs(wl, b, l) for l in range(max(layers) + 1)},
        "rows": ({l: [layer_inputs(wl, b, l, j) for j in range(wl.drafts)] for l in range(max(layers) + 1)}
                 if wl.drafts > 1 else None),
        "layers": layers,
        "new": new_token_inputs(wl, b, rope),
    }


def step(wl: DecodeWorkload, b: int, st: dict, with_attention: bool = True):
    """Selection and attention of every layer up to the last requested one.

    Returns dict with 'pool', 'topk' {layer: idx}, 'sigma' {layer: scores},
    'out' {layer: [H][128]}, 'lse' {layer: [H]}.
    """
    if wl.drafts > 1:
        return verify_step(wl, b, st, with_attention)
    L = int(wl.lengths[b])
    kc, ks, ic, isc = st["cache"]
    res = {"cache": st["cache"], "topk": {}, "sigma": {}, "out": {}, "lse": {}}
    cur = None
    pool = None
    layers = st["layers"]
    for l in range(max(layers) + 1):
        mode = wl.schedule[l]
        q, qi, w = st["inputs"][l]
        if mode == FULL:
            pool, cur, sig = ix.full_select(qi, w, ic, isc, wl.block, wl.n_keep, wl.topk)
            res["pool"] = pool
            res["topk"][l] = cur
            res["sigma"][l] = sig
        elif mode == REINDEX:
            cur, sig, pos = ix.reindex_select(qi, w, ic, isc, pool, wl.block, wl.topk)
            res["topk"][l] = cur
            res["sigma"][l] = (sig, pos)
        else:
            cur = ix.reuse(cur)
        if with_attention and l in layers:
            rc, rs = st["swa"][l]
            o, lse = at.decode_row(q, kc, ks, 0, cur, rc, rs, L - 1, wl.window)
            res["out"][l] = o
            res["lse"][l] = lse
    return res


def verify_step(wl: DecodeWorkload, b: int, st: dict, with_attention: bool = True):
    """The step with D = wl.drafts query rows at positions L-D..L-1 of sequence b.

    Returns dict with 'pool', 'sigma' {Full layer: scores of the last row's queries},
    'topk' {layer: [D][topk]}, 'out' {layer: [D][H][128]}, 'lse' {layer: [D][H]}.
    """
    L, D = int(wl.lengths[b]), wl.drafts
    kc, ks, ic, isc = st["cache"]
    res = {"cache": st["cache"], "topk": {}, "sigma": {}, "out": {}, "lse": {}}
    pos = [L - D + j for j in range(D)]
    cur, pool = None, None
    layers = st["layers"]
    for l in range(max(layers) + 1):
        mode = wl.schedule[l]
        rows = st["rows"][l]
        if mode == FULL:
            _, qi, w = st["inputs"][l]                           # the last row's indexer queries
            pool, _, sig = ix.full_select(qi, w, ic, isc, wl.block, wl.n_keep, wl.topk)
            res["pool"] = pool
            res["sigma"][l] = sig
        if mode in (FULL, REINDEX):
            cur = np.stack([ix.verify_select(rows[j][1], rows[j][2], ic, isc, pool, pos[j], wl.block, wl.topk)[0]
                            for j in range(D)])
            res["topk"][l] = cur
        else:
            cur = ix.reuse(cur)
        if with_attention and l in layers:
            rc, rs = st["swa"][l]
            outs = [at.decode_row(rows[j][0], kc, ks, 0, cur[j], rc, rs, pos[j], wl.window) for j in range(D)]
            res["out"][l] = np.stack([o for o, _ in outs])
            res["lse"][l] = np.stack([x for _, x in outs])
    return res


def decode_step(wl: DecodeWorkload, b: int, layers=None, with_attention: bool = True):
    """prepare + step for one sequence."""
    return step(wl, b, prepare(wl, b, layers), with_attention)
