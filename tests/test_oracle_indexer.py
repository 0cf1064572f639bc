"""Pins for the oracle's indexer and selection (CPU only).

Against pure-Python brute force (``sorted`` with key (-score, id)) on tiny
contexts, special cases with a known answer, and the structural facts the
pages fix: the pool is 2,048 blocks of 8, Reindex picks only pool
positions, Reuse passes indices unchanged, and the Full top-k lies inside
the pool.
"""
import numpy as np
import pytest

import synth
from oracle import indexer, bruteforce
from oracle.append import quantize_fp8_token, bf16_to_f32


def _tiny_keys(rng, L, C=64):
    x = rng.standard_normal((L, C)).astype(np.float32)
    return quantize_fp8_token(x)


def _tiny_q(rng, H=8, C=64):
    q = synth.f32_to_bf16_bits(rng.standard_normal((H, C)).astype(np.float32))
    w = rng.uniform(0, 1, H).astype(np.float32)
    return q, w


@pytest.mark.parametrize("seed", range(12))
def test_full_select_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 65))
    block = int(rng.choice([1, 2, 4, 8]))
    n_keep = int(rng.integers(1, 9))
    topk = int(rng.integers(1, n_keep + 1))
    codes, scale = _tiny_keys(rng, L)
    q, w = _tiny_q(rng)
    pool, top, sig = indexer.full_select(q, w, codes, scale, block, n_keep, topk)
    qf = bf16_to_f32(q).astype(np.float64).tolist()
    bp, bt, bsig = bruteforce.select(qf, w.astype(np.float64).tolist(), codes.tolist(),
                                     scale.astype(np.float64).tolist(), block, n_keep, topk)
    assert np.allclose(sig, bsig, rtol=1e-12, atol=0)
    assert list(pool[pool >= 0]) == bp
    assert list(top[top >= 0]) == bt
    # Reindex over the pool against brute force
    q2, w2 = _tiny_q(rng)
    re, _, _ = indexer.reindex_select(q2, w2, codes, scale, pool, block, topk)
    br = bruteforce.reselect(bf16_to_f32(q2).astype(np.float64).tolist(), w2.astype(np.float64).tolist(),
                             codes.tolist(), scale.astype(np.float64).tolist(), list(pool), block, topk)
    assert list(re[re >= 0]) == br


def test_ties_break_to_lower_position_and_block():
    # identical keys everywhere: every score ties, so the lowest ids win
    rng = np.random.default_rng(5)
    codes, scale = _tiny_keys(rng, 1)
    codes = np.repeat(codes, 40, 0)
    scale = np.repeat(scale, 40, 0)
    q, w = _tiny_q(rng)
    pool, top, _ = indexer.full_select(q, w, codes, scale, block=4, n_keep=3, topk=5)
    assert list(pool) == [0, 1, 2] and list(top) == [0, 1, 2, 3, 4]


def test_single_head_weight_reduces_to_sorted_relu_scores():
    rng = np.random.default_rng(6)
    codes, scale = _tiny_keys(rng, 300)
    q, _ = _tiny_q(rng)
    w = np.zeros(8, dtype=np.float32)
    w[0] = 1.0
    _, top, sig = indexer.full_select(q, w, codes, scale, block=8, n_keep=40, topk=17)
    from oracle.formats import E4M3_TABLE
    d = E4M3_TABLE[codes] @ bf16_to_f32(q[0]).astype(np.float64)
    ref = scale.astype(np.float64) * np.maximum(d, 0)
    assert np.allclose(sig, ref, rtol=1e-13, atol=0)
    order = sorted(range(300), key=lambda t: (-ref[t], t))[:17]
    assert list(top) == sorted(order)


def test_short_context_returns_everything():
    rng = np.random.default_rng(8)
    codes, scale = _tiny_keys(rng, 37)
    q, w = _tiny_q(rng)
    pool, top, _ = indexer.full_select(q, w, codes, scale, block=8, n_keep=2048, topk=512)
    assert list(top[:37]) == list(range(37)) and np.all(top[37:] == -1)
    assert list(pool[:5]) == list(range(5)) and np.all(pool[5:] == -1)


@pytest.mark.parametrize("seed", range(4))
def test_full_topk_lies_inside_pool(seed):
    rng = np.random.default_rng(100 + seed)
    L = 3000
    codes, scale = _tiny_keys(rng, L)
    q, w = _tiny_q(rng)
    pool, top, sig = indexer.full_select(q, w, codes, scale, block=8, n_keep=64, topk=64)
    pos = set(indexer.pool_positions(pool, L, 8).tolist())
    assert set(top.tolist()) <= pos
    assert pool.shape == (64,) and np.all(np.diff(pool) > 0)


def test_reindex_picks_only_pool_positions_and_reuse_is_identity():
    rng = np.random.default_rng(9)
    L = 5000
    codes, scale = _tiny_keys(rng, L)
    q, w = _tiny_q(rng)
    pool, top, _ = indexer.full_select(q, w, codes, scale, block=8, n_keep=100, topk=50)
    q2, w2 = _tiny_q(rng)
    re, sig2, pos = indexer.reindex_select(q2, w2, codes, scale, pool, 8, 50)
    allowed = set(indexer.pool_positions(pool, L, 8).tolist())
    assert set(re.tolist()) <= allowed and len(set(re.tolist())) == 50
    assert indexer.reuse(re) is re
    # the pool positions beat every other pool position under the new scores
    full_sig = indexer.scores(q2, w2, codes, scale)
    chosen = full_sig[re]
    others = np.array(sorted(allowed - set(re.tolist())))
    assert chosen.min() >= full_sig[others].max()


def test_verify_rows_rank_the_pool_up_to_their_own_position():
    rng = np.random.default_rng(13)
    L = 4000
    codes, scale = _tiny_keys(rng, L)
    q, w = _tiny_q(rng)
    pool, _, _ = indexer.full_select(q, w, codes, scale, block=8, n_keep=120, topk=50)
    allowed_all = indexer.pool_positions(pool, L, 8)
    q2, w2 = _tiny_q(rng)
    # the last position of the context: the plain Reindex rule
    v, _, _ = indexer.verify_select(q2, w2, codes, scale, pool, L - 1, 8, 50)
    r, _, _ = indexer.reindex_select(q2, w2, codes, scale, pool, 8, 50)
    assert np.array_equal(v, r)
    full_sig = indexer.scores(q2, w2, codes, scale)
    for p in (int(allowed_all[40]), int(allowed_all[300]) - 1, 2500):
        v, _, _ = indexer.verify_select(q2, w2, codes, scale, pool, p, 8, 50)
        allowed = allowed_all[allowed_all <= p]
        got = v[v >= 0]
        # brute force: the min(50, |allowed|) best allowed positions, nothing after p
        assert got.shape[0] == min(50, allowed.shape[0]) and np.all(got <= p)
        assert set(got.tolist()) <= set(allowed.tolist()) and np.all(np.diff(got) > 0)
        rest = np.array(sorted(set(allowed.tolist()) - set(got.tolist())), np.int64)
        if rest.size:
            assert full_sig[got].min() >= full_sig[rest].max()
    # a position before the first pool block selects nothing
    v, _, _ = indexer.verify_select(q2, w2, codes, scale, pool, int(allowed_all[0]) - 1, 8, 50)
    assert np.all(v == -1)


def test_pool_is_2048_blocks_of_8_at_decoder_sizes():
    rng = np.random.default_rng(11)
    L = 20000
    codes, scale = _tiny_keys(rng, L)
    q, w = _tiny_q(rng)
    pool, top, _ = indexer.full_select(q, w, codes, scale)
    assert pool.shape == (2048,) and np.all(pool >= 0) and np.all(np.diff(pool) > 0)
    assert indexer.pool_positions(pool, L).shape == (16384,)
    assert top.shape == (512,) and np.all(np.diff(top) > 0)


@pytest.mark.parametrize("planted", ["no_relu", "ascending", "drop_scale"])
def test_planted_indexer_mistakes_are_caught(planted, monkeypatch):
    """Each plausible slip in the oracle's score or ranking fails the brute-force pin."""
    rng = np.random.default_rng(21)
    L = 48
    codes, scale = _tiny_keys(rng, L)
    q, w = _tiny_q(rng)
    good_scores = indexer.scores
    good_topk = indexer.top_k_ids

    def bad_scores(q_, w_, c_, s_):
        from oracle.formats import e4m3_decode
        qq = bf16_to_f32(q_).astype(np.float64)
        d = e4m3_decode(c_) @ qq.T
        if planted == "no_relu":
            return np.asarray(s_, np.float64) * (d @ np.asarray(w_, np.float64))
        if planted == "drop_scale":
            return np.maximum(d, 0) @ np.asarray(w_, np.float64)
        return good_scores(q_, w_, c_, s_)

    def bad_topk(v, ids, k):
        if planted == "ascending":
            return good_topk(-np.asarray(v), ids, k)
        return good_topk(v, ids, k)

    monkeypatch.setattr(indexer, "scores", bad_scores)
    monkeypatch.setattr(indexer, "top_k_ids", bad_topk)
    _, top, _ = indexer.full_select(q, w, codes, scale, 8, 4, 6)
    _, bt, _ = bruteforce.select(bf16_to_f32(q).astype(np.float64).tolist(), w.astype(np.float64).tolist(),
                                 codes.tolist(), scale.astype(np.float64).tolist(), 8, 4, 6)
    assert list(top[top >= 0]) != bt


def test_verify_step_last_row_of_the_full_layer_equals_its_full_top_k():
    """Containment: the last draft row sees the whole context, so its top-k from the shared pool
    equals the Full top-k over every position; earlier rows stay inside their own prefix."""
    from oracle import pipeline
    from synth.workloads import DecodeWorkload, FULL, REINDEX, REUSE
    wl = DecodeWorkload("tiny_verify", np.array([2000, 700], np.int64), schedule=[FULL, REUSE, REINDEX],
                        n_keep=40, topk=24, ring=256, drafts=4)
    for b in range(2):
        st = pipeline.prepare(wl, b, layers=[0, 2])
        res = pipeline.step(wl, b, st, with_attention=False)
        _, _, ic, isc = st["cache"]
        _, qi, w = st["inputs"][0]
        _, top, _ = indexer.full_select(qi, w, ic, isc, wl.block, wl.n_keep, wl.topk)
        assert np.array_equal(res["topk"][0][-1], top)
        L = int(wl.lengths[b])
        for l in (0, 2):
            assert res["topk"][l].shape == (4, wl.topk)
            for j in range(4):
                got = res["topk"][l][j]
                assert np.all(got[got >= 0] <= L - 4 + j)


@pytest.mark.parametrize("seed", range(6))
def test_chunked_rows_match_brute_force_on_their_prefix(seed):
    """A chunked-query row at position p: brute force over the first p + 1 positions only,
    and nothing at or after p + 1 may influence it (later keys are changed to check)."""
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(20, 70))
    block = int(rng.choice([1, 2, 4, 8]))
    n_keep = int(rng.integers(2, 9))
    topk = int(rng.integers(1, n_keep + 1))
    codes, scale = _tiny_keys(rng, L)
    q, w = _tiny_q(rng)
    qf = bf16_to_f32(q).astype(np.float64).tolist()
    for p in (0, int(rng.integers(1, L - 1)), L - 1):
        pool, top, _ = indexer.chunked_select(q, w, codes, scale, p, block, n_keep, topk)
        bp, bt, _ = bruteforce.select(qf, w.astype(np.float64).tolist(), codes[:p + 1].tolist(),
                                      scale[:p + 1].astype(np.float64).tolist(), block, n_keep, topk)
        assert list(pool[pool >= 0]) == bp and list(top[top >= 0]) == bt
        later = codes.copy()
        later[p + 1:] = rng.integers(0, 126, size=later[p + 1:].shape)      # finite E4M3 codes
        pool2, top2, _ = indexer.chunked_select(q, w, later, scale, p, block, n_keep, topk)
        assert np.array_equal(pool, pool2) and np.array_equal(top, top2)
