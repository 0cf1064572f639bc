"""Pin for the oracle's decode-step composition (CPU only).

``oracle.pipeline.step`` wires the layers of the decoder together: the Full
layer's pool and top-k, each Reindex layer's own indexer queries over that
pool, Reuse layers passing the previous list on, and every layer's attention
over its own list plus its own SWA window (origotech.dev deep dive,
subsection "Compressed Sparse Attention 2(CSA2)"; ttj.kr, section "CSA2와
어텐션 재설계").  Here the same step is rebuilt for tiny contexts from the
pure-Python brute-force routines only, with every input regenerated straight
from the seeded generator, and compared element by element.  Three planted
mistakes in the composition (a Reindex layer ranking with the Full layer's
queries, an attention call fed the previous indexer layer's list, the SWA
ring filled one slot off) must each make the comparison fail.
"""
import math

import numpy as np
import pytest

import synth
from oracle import append as ap
from oracle import bruteforce as bf
from oracle import pipeline
from synth.workloads import FULL, REINDEX, REUSE, DecodeWorkload

SCHEDULE = [FULL, REUSE, REINDEX, REUSE]


def _workload():
    return DecodeWorkload("tiny_pipeline", np.array([50, 3, 29], dtype=np.int64), schedule=list(SCHEDULE),
                          H=2, topk=5, n_keep=6, block=4, window=4, ring=8, seed=7)


def _token(wl, b, t, cos, sin):
    """Main KV row (128 floats) and indexer key (codes, scale) of position t, from the generator."""
    rows = synth.row_id(b, np.array([t]))
    kv = synth.normals_bf16(wl.seed, synth.Stream.KV, 0, rows, 128,
                            synth.outlier_channels(wl.seed, synth.Stream.KV_OUTLIER))
    ik = synth.normals_bf16(wl.seed, synth.Stream.IK, 0, rows, 64)
    kc, ks, ic, isc = ap.append_rows(kv, ik, cos[t:t + 1], sin[t:t + 1])
    return bf.fp4_row(kc[0].tolist(), ks[0].tolist()), ic[0].tolist(), float(isc[0])


def _window_row(wl, b, layer, t, cos, sin):
    rows = synth.row_id(b, np.array([t]))
    sw = synth.normals_bf16(wl.seed, synth.Stream.SWA, layer, rows, 128,
                            synth.outlier_channels(wl.seed, synth.Stream.SWA_OUTLIER))
    codes, scale = ap.swa_rows(sw, cos[t:t + 1], sin[t:t + 1])
    return bf.fp8_row(codes[0].tolist(), float(scale[0]))


def _layer_queries(wl, b, layer):
    """Attention queries (H x 128 floats), indexer queries (8 x 64), head weights (8) of one layer."""
    r = b                                              # one query row per sequence
    q = synth.normals_bf16(wl.seed, synth.Stream.Q, layer, synth.row_id(r, np.arange(wl.H)), 128)
    qi = synth.normals_bf16(wl.seed, synth.Stream.QIDX, layer, synth.row_id(r, np.arange(8)), 64)
    w = synth.head_weights(wl.seed, layer, r)
    f = lambda bits: ap.bf16_to_f32(bits).astype(np.float64).tolist()
    return f(q), f(qi), w.astype(np.float64).tolist()


def brute_chain(wl, b):
    """The step of sequence b from brute-force pieces: {'pool', 'topk' {l}, 'out' {l}, 'lse' {l}}."""
    L = int(wl.lengths[b])
    cos, sin = synth.rope_table(L)
    toks = [_token(wl, b, t, cos, sin) for t in range(L)]
    main = [x[0] for x in toks]
    codes = [x[1] for x in toks]
    scales = [x[2] for x in toks]
    res = {"topk": {}, "out": {}, "lse": {}}
    cur = pool = None
    for l, mode in enumerate(wl.schedule):
        q, qi, w = _layer_queries(wl, b, l)
        if mode == FULL:
            pool, cur, _ = bf.select(qi, w, codes, scales, wl.block, wl.n_keep, wl.topk)
            res["pool"] = pool
            res["topk"][l] = cur
        elif mode == REINDEX:
            cur = bf.reselect(qi, w, codes, scales, pool, wl.block, wl.topk)
            res["topk"][l] = cur
        rows = [main[t] for t in cur]
        rows += [_window_row(wl, b, l, t, cos, sin) for t in range(max(0, L - wl.window), L)]
        o, lse = bf.attend(q, rows, 1.0 / math.sqrt(128.0))
        res["out"][l] = np.array(o)
        res["lse"][l] = np.array(lse)
    return res


def compare(res, ref):
    """Raise AssertionError where the oracle's step differs from the brute-force chain."""
    ids = lambda a: [int(x) for x in np.asarray(a) if x >= 0]
    assert ids(res["pool"]) == ref["pool"], ("pool", ids(res["pool"]), ref["pool"])
    for l, top in ref["topk"].items():
        assert ids(res["topk"][l]) == top, ("topk", l, ids(res["topk"][l]), top)
    for l in ref["out"]:
        assert np.allclose(res["out"][l], ref["out"][l], rtol=1e-10, atol=1e-12), ("out", l)
        assert np.allclose(res["lse"][l], ref["lse"][l], rtol=1e-12, atol=1e-12), ("lse", l)


@pytest.fixture(scope="module")
def chains():
    wl = _workload()
    return wl, {b: brute_chain(wl, b) for b in range(wl.B)}


@pytest.mark.parametrize("b", [0, 1, 2])
def test_step_matches_brute_force_chain(chains, b):
    wl, ref = chains
    compare(pipeline.step(wl, b, pipeline.prepare(wl, b)), ref[b])


def test_planted_reindex_with_full_layer_queries_is_caught(chains):
    wl, ref = chains
    st = pipeline.prepare(wl, 0)
    q2, _, _ = st["inputs"][2]
    _, qi0, w0 = st["inputs"][0]
    st["inputs"][2] = (q2, qi0, w0)                   # the Reindex layer ranks with the Full layer's queries
    with pytest.raises(AssertionError):
        compare(pipeline.step(wl, 0, st), ref[0])


def test_planted_stale_list_in_attention_is_caught(chains, monkeypatch):
    wl, ref = chains
    real = pipeline.at.decode_row
    seen = []

    def stale(q, kc, ks, base, topk_row, *rest, **kw):
        seen.append(np.array(topk_row))
        if len(seen) == 3:                            # layer 2 (Reindex) attends over layer 0's list
            topk_row = seen[0]
        return real(q, kc, ks, base, topk_row, *rest, **kw)

    monkeypatch.setattr(pipeline.at, "decode_row", stale)
    with pytest.raises(AssertionError):
        compare(pipeline.step(wl, 0, pipeline.prepare(wl, 0)), ref[0])


def test_planted_ring_slot_shift_is_caught(chains, monkeypatch):
    wl, ref = chains
    real = pipeline.sequence_swa

    def shifted(*args, **kw):
        rc, rs = real(*args, **kw)
        return np.roll(rc, 1, axis=0), np.roll(rs, 1)

    monkeypatch.setattr(pipeline, "sequence_swa", shifted)
    with pytest.raises(AssertionError):
        compare(pipeline.step(wl, 0, pipeline.prepare(wl, 0)), ref[0])


def test_appended_token_rows_are_the_cache_and_ring_rows(chains):
    """The step's append quantises exactly the rows the prepared cache and rings hold for the
    new token (position L-1)."""
    wl, _ = chains
    for b in range(wl.B):
        st = pipeline.prepare(wl, b)
        (kc, ks, ic, isc), swa = pipeline.append_token(st["new"])
        L = int(wl.lengths[b])
        for got, cached in zip((kc, ks, ic, isc), st["cache"]):
            assert np.array_equal(got[0], cached[L - 1])
        for l, (codes, scale) in enumerate(swa):
            rc, rs = st["swa"][l]
            assert np.array_equal(codes[0], rc[(L - 1) % wl.ring]) and scale[0] == rs[(L - 1) % wl.ring]
