"""One decode step of the CSA2 decoder for selected sequences (oracle side).

Composes the oracle's steps in the order the pages give (origotech.dev deep
dive, subsection "Compressed Sparse Attention 2(CSA2)"): quantise-and-append
of the new token, the first Full layer's indexer over every position (pool +
top-k), Reindex layers over the pool, Reuse layers passing indices on, and
every layer's sparse attention over its indices plus its own SWA window.

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
    """Ring arrays (codes [ring][128], scale [ring]) of one layer after the step's append."""
    L = int(wl.lengths[b])
    cos, sin = rope if rope is not None else synth.rope_table(L)
    oc = synth.outlier_channels(wl.seed, synth.Stream.SWA_OUTLIER)
    lo = max(0, L - wl.window)
    pos = np.arange(lo, L)
    sw = synth.normals_bf16(wl.seed, synth.Stream.SWA, layer, synth.row_id(b, pos), 128, oc)
    codes, scale = ap.swa_rows(sw, cos[lo:L], sin[lo:L])
    rc = np.zeros((wl.ring, 128), np.uint8)
    rs = np.zeros(wl.ring, np.float32)
    rc[pos % wl.ring] = codes
    rs[pos % wl.ring] = scale
    return rc, rs


def layer_inputs(wl: DecodeWorkload, b: int, layer: int):
    """(attention q bf16 [H][128], indexer q bf16 [8][64], head weights [8]) of one layer."""
    q = synth.normals_bf16(wl.seed, synth.Stream.Q, layer, synth.row_id(b, np.arange(wl.H)), 128)
    qi = synth.normals_bf16(wl.seed, synth.Stream.QIDX, layer, synth.row_id(b, np.arange(8)), 64)
    w = synth.head_weights(wl.seed, layer, b)
    return q, qi, w


def prepare(wl: DecodeWorkload, b: int, layers=None):
    """Per-sequence state that exists before the step: cache rows 0..L-1, window rings, layer inputs."""
    L = int(wl.lengths[b])
    rope = synth.rope_table(L)
    layers = list(range(wl.n_layers)) if layers is None else list(layers)
    return {
        "cache": sequence_cache(wl, b, rope),
        "swa": {l: sequence_swa(wl, b, l, rope) for l in layers},
        "inputs": {l: layer_inputs(wl, b, l) for l in range(max(layers) + 1)},
        "layers": layers,
    }


def step(wl: DecodeWorkload, b: int, st: dict, with_attention: bool = True):
    """Selection and attention of every layer up to the last requested one.

    Returns dict with 'pool', 'topk' {layer: idx}, 'sigma' {layer: scores},
    'out' {layer: [H][128]}, 'lse' {layer: [H]}.
    """
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


def decode_step(wl: DecodeWorkload, b: int, layers=None, with_attention: bool = True):
    """prepare + step for one sequence."""
    return step(wl, b, prepare(wl, b, layers), with_attention)
