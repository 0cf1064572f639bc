"""End-to-end decode steps of the measured configurations against the oracle.

Each test builds the full-size cache on the GPU through kv_append_fp4, runs
one decode step exactly as the benchmark launches it (DecodeRunner.step:
append, Full select, Reindex/Reuse layers, attention per layer), and checks
sampled sequences against the oracle's own chain, computed from the seeded
inputs alone.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import pipeline
from oracle import attention as at
from oracle import indexer as ix
from oracle.append import swa_rows
from synth.workloads import DecodeWorkload, config, verify_workload, FULL, REINDEX
from tests.gpu_util import ATTN_TOL, attn_rel_err, check_index_set, csa2

pytestmark = pytest.mark.gpu


def _check_sequence(r, wl, b, layers=None):
    """Indices of sequence b against the oracle's chain, then every requested layer's attention.

    Attention is always checked: against the chain's own output where the layer's index list
    equals the oracle's, and otherwise (a tolerated boundary swap) against the oracle's
    attention recomputed from the GPU's own list, so both sides use the same indices.
    Returns (swapped pairs, worst attention error)."""
    st = pipeline.prepare(wl, b, layers)
    ref = pipeline.step(wl, b, st)
    L = int(wl.lengths[b])
    sig0 = ref["sigma"][0]
    bs = ix.block_scores(sig0, wl.block)
    swaps = check_index_set(r.pool[b].cpu().numpy(), ref["pool"], lambda j: bs[j], f"pool b={b}")
    layer_swaps = {}
    for l, otop in ref["topk"].items():
        g = r.topk[l][b].cpu().numpy()
        if wl.schedule[l] == FULL:
            score = sig0
        else:
            _, _, ic, isc = ref["cache"]
            qi = pipeline.layer_inputs(wl, b, l)
            score = ix.scores(qi[1], qi[2], ic, isc)
        layer_swaps[l] = check_index_set(g, otop, lambda p: score[p], f"topk layer {l} b={b}")
        swaps += layer_swaps[l]
    kc, ks, _, _ = ref["cache"]
    worst = 0.0
    for l, o in ref["out"].items():
        src = max(x for x in ref["topk"] if x <= l)            # the list layer l attends over
        exp_o, exp_lse = o, ref["lse"][l]
        if layer_swaps[src]:
            g = r.layer_topk(l)[b].cpu().numpy()
            rc, rs = st["swa"][l]
            exp_o, exp_lse = at.decode_row(st["inputs"][l][0], kc, ks, 0, g, rc, rs, L - 1, wl.window)
        e = attn_rel_err(r.out[l, b].cpu().numpy()[None], exp_o[None])
        le = float(np.max(np.abs(r.lse[l, b].cpu().numpy() - exp_lse)))
        assert e <= ATTN_TOL and le <= 1e-4, (l, e, le)
        worst = max(worst, e)
    print(f"b={b} swaps={swaps} max rel err {worst:.3e}")
    return swaps, worst


def _runner(cfg):
    from sparse_attention_fp4_02_b300.runner import DecodeRunner
    wl = config(cfg) if isinstance(cfg, int) else cfg
    r = DecodeRunner(wl)
    r.build_cache()
    r.step()
    torch.cuda.synchronize()
    r.check_device_errors()
    return wl, r


def test_config0_full_layer_ctx4096():
    wl, r = _runner(0)
    _check_sequence(r, wl, 0)


def test_config1_b32_ctx65536_full_and_reuse():
    wl, r = _runner(1)
    for b in (0, 13, 31):
        _check_sequence(r, wl, b)
    # Reuse layers attend over the Full layer's indices: one buffer for layers 0..3
    assert r.layer_topk(3) is r.topk[0]


def test_config2_b4_ctx1m_twenty_layers():
    wl, r = _runner(2)
    _check_sequence(r, wl, 2, layers=[0, 1, 4, 5, 12, 19])


def test_config4_ragged_b64_twenty_layers():
    wl, r = _runner(4)
    lens = wl.lengths
    for b in (int(np.argmin(lens)), 7):
        print("length", int(lens[b]))
        _check_sequence(r, wl, b, layers=[0, 3, 4, 8, 16, 19])


def test_config3_attention_on_seeded_causal_lists():
    from tests.test_gpu_attention import LSE_TOL_TC, World
    wl = config(3)
    w = World([wl.cache_len], ring=wl.ring)
    q_pos = np.arange(wl.cache_len - wl.n_query, wl.cache_len, dtype=np.int64)
    topk = synth.causal_topk(wl.seed, q_pos, wl.topk)
    q = synth.normals_bf16(wl.seed, synth.Stream.Q, 0, np.arange(wl.n_query * wl.H), 128).reshape(wl.n_query, wl.H, 128)
    out, lse, err = w.run(q, np.zeros(wl.n_query, np.int32), q_pos, topk, wl.window)
    assert err == 0
    rows = np.array([0, 1, 100, 2047, 3000, 4095])
    ref, rlse = w.oracle(q[rows], np.zeros(len(rows), np.int32), q_pos[rows], topk[rows], wl.window)
    e = attn_rel_err(out[rows], ref)
    assert e <= ATTN_TOL, e
    assert np.max(np.abs(lse[rows] - rlse)) <= LSE_TOL_TC      # many rows: the tensor-core path
    # every row's output is a convex combination: finite, and lse finite
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    print("max rel err", e)


def test_config3_chain_indexer_then_tensor_core_attention():
    """The chunked-query workload as the benchmark times it: ChunkedRunner's chunked-query
    indexer (every row's Full selection over its own prefix) feeding the tcgen05 attention.
    Sampled rows include the edges of every 16-row tensor-core group and 1,024-row indexer
    group the kernels use; each row's pool and top-k are compared with the oracle's Full
    selection over positions 0..p, then its attention with the oracle's on the same list."""
    from sparse_attention_fp4_02_b300.runner import ChunkedRunner
    from tests.test_gpu_attention import LSE_TOL_TC
    wl = config(3)
    r = ChunkedRunner(wl, use_indexer=True)
    r.step()
    torch.cuda.synchronize()
    r.check_device_errors()
    L, T, s = wl.cache_len, wl.n_query, wl.seed
    edges = [0, 1, 15, 16, 17, 31, 32, 127, 128, 1023, 1024, 1025, 2047, 2048, 3071, 3072, 4079, 4080, 4094, 4095]
    rng = np.random.default_rng(3)
    rows = sorted(set(edges) | set(rng.choice(T, 48, replace=False).tolist()))
    assert len(rows) >= 64
    kc, ks, ic, isc = pipeline.sequence_cache(DecodeWorkload("chunked_cache", np.array([L], np.int64), seed=s), 0)
    cos, sin = synth.rope_table(L)
    lo = L - T - wl.window + 1
    pos = np.arange(lo, L, dtype=np.int64)
    sw = synth.normals_bf16(s, synth.Stream.SWA, 0, synth.row_id(0, pos), 128,
                            synth.outlier_channels(s, synth.Stream.SWA_OUTLIER))
    rc = np.zeros((wl.ring, 128), np.uint8)
    rs = np.zeros(wl.ring, np.float32)
    rc[pos % wl.ring], rs[pos % wl.ring] = swa_rows(sw, cos[lo:L], sin[lo:L])
    pool, top = r.pool.cpu().numpy(), r.topk.cpu().numpy()
    out, lse = r.out.cpu().numpy(), r.lse.cpu().numpy()
    swaps, worst = 0, 0.0
    for t in rows:
        p = L - T + t
        qi = synth.normals_bf16(s, synth.Stream.QIDX, 0, synth.row_id(t, np.arange(8)), 64)
        w = synth.head_weights(s, 0, t)
        opool, otop, sig = ix.chunked_select(qi, w, ic, isc, p, 8, 2048, wl.topk)
        bs = ix.block_scores(sig, 8)
        swaps += check_index_set(pool[t], opool, lambda j: bs[j], f"pool row {t}")
        swaps += check_index_set(top[t], otop, lambda x: sig[x], f"top-k row {t}")
        q = synth.normals_bf16(s, synth.Stream.Q, 0, np.arange(t * wl.H, (t + 1) * wl.H), 128)
        o, l = at.decode_row(q, kc, ks, 0, top[t], rc, rs, p, wl.window)
        e = attn_rel_err(out[t], o)
        assert e <= ATTN_TOL, (t, e)
        assert np.max(np.abs(lse[t] - l)) <= LSE_TOL_TC, t
        worst = max(worst, e)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    print(f"{len(rows)} rows, swaps={swaps}, max rel err {worst:.3e}")


def test_verify_b32_ctx65536_five_drafts_twenty_layers():
    """Draft verification: 5 query rows per session, one shared pool, causal per-row top-k."""
    wl = verify_workload()
    wl, r = _runner(wl)
    D, L = wl.drafts, int(wl.lengths[0])
    for b in (0, 19, 31):
        layers = [0, 1, 4, 7, 19]
        st = pipeline.prepare(wl, b, layers)
        ref = pipeline.step(wl, b, st)
        kc, ks, ic, isc = ref["cache"]
        bs = ix.block_scores(ref["sigma"][0], wl.block)
        swaps = check_index_set(r.pool[b].cpu().numpy(), ref["pool"], lambda j: bs[j], f"pool b={b}")
        row_swaps = {}
        for l, otop in ref["topk"].items():
            for j in range(D):
                g = r.topk[l][b * D + j].cpu().numpy()
                qi = pipeline.layer_inputs(wl, b, l, j)
                p = L - D + j
                score = ix.scores(qi[1], qi[2], ic[:p + 1], isc[:p + 1])
                row_swaps[l, j] = check_index_set(g, otop[j], lambda t: score[t], f"topk layer {l} b={b} row {j}")
                swaps += row_swaps[l, j]
                assert np.all(g[g >= 0] <= p)
        worst = 0.0
        for l, o in ref["out"].items():
            src = max(x for x in ref["topk"] if x <= l)
            rc, rs = st["swa"][l]
            for j in range(D):
                exp_o, exp_lse = o[j], ref["lse"][l][j]
                if row_swaps[src, j]:                          # the oracle on the GPU's own list
                    g = r.layer_topk(l)[b * D + j].cpu().numpy()
                    exp_o, exp_lse = at.decode_row(st["rows"][l][j][0], kc, ks, 0, g, rc, rs, L - D + j, wl.window)
                e = attn_rel_err(r.out[l, b * D + j].cpu().numpy()[None], exp_o[None])
                le = float(np.max(np.abs(r.lse[l, b * D + j].cpu().numpy() - exp_lse)))
                assert e <= ATTN_TOL and le <= 1e-4, (l, j, e, le)
                worst = max(worst, e)
        print(f"b={b} swaps={swaps} max rel err {worst:.3e}")
