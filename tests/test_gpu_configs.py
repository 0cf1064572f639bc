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
from oracle import indexer as ix
from synth.workloads import config, verify_workload, FULL, REINDEX
from tests.gpu_util import ATTN_TOL, attn_rel_err, check_index_set, csa2

pytestmark = pytest.mark.gpu


def _check_sequence(r, wl, b, layers=None):
    ref = pipeline.decode_step(wl, b, layers=layers)
    L = int(wl.lengths[b])
    sig0 = ref["sigma"][0]
    bs = ix.block_scores(sig0, wl.block)
    swaps = check_index_set(r.pool[b].cpu().numpy(), ref["pool"], lambda j: bs[j], f"pool b={b}")
    for l, otop in ref["topk"].items():
        g = r.topk[l][b].cpu().numpy()
        if wl.schedule[l] == FULL:
            score = sig0
        else:
            _, _, ic, isc = ref["cache"]
            qi = pipeline.layer_inputs(wl, b, l)
            score = ix.scores(qi[1], qi[2], ic, isc)
        swaps += check_index_set(g, otop, lambda p: score[p], f"topk layer {l} b={b}")
    worst = 0.0
    if swaps == 0:       # identical indices: attention must match
        for l, o in ref["out"].items():
            e = attn_rel_err(r.out[l, b].cpu().numpy()[None], o[None])
            le = float(np.max(np.abs(r.lse[l, b].cpu().numpy() - ref["lse"][l])))
            assert e <= ATTN_TOL and le <= 1e-4, (l, e, le)
            worst = max(worst, e)
    return worst


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
    print("max rel err", _check_sequence(r, wl, 0))


def test_config1_b32_ctx65536_full_and_reuse():
    wl, r = _runner(1)
    for b in (0, 13, 31):
        print(b, "max rel err", _check_sequence(r, wl, b))
    # Reuse layers attend over the Full layer's indices: one buffer for layers 0..3
    assert r.layer_topk(3) is r.topk[0]


def test_config2_b4_ctx1m_twenty_layers():
    wl, r = _runner(2)
    print("max rel err", _check_sequence(r, wl, 2, layers=[0, 1, 4, 5, 12, 19]))


def test_config4_ragged_b64_twenty_layers():
    wl, r = _runner(4)
    lens = wl.lengths
    for b in (int(np.argmin(lens)), 7):
        print(b, int(lens[b]), "max rel err", _check_sequence(r, wl, b, layers=[0, 3, 4, 8, 16, 19]))


def test_config3_chunked_queries_h64_cache262144():
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


def test_verify_b32_ctx65536_five_drafts_twenty_layers():
    """Draft verification: 5 query rows per session, one shared pool, causal per-row top-k."""
    wl = verify_workload()
    wl, r = _runner(wl)
    D, L = wl.drafts, int(wl.lengths[0])
    for b in (0, 19, 31):
        ref = pipeline.decode_step(wl, b, layers=[0, 1, 4, 7, 19])
        _, _, ic, isc = ref["cache"]
        bs = ix.block_scores(ref["sigma"][0], wl.block)
        swaps = check_index_set(r.pool[b].cpu().numpy(), ref["pool"], lambda j: bs[j], f"pool b={b}")
        for l, otop in ref["topk"].items():
            for j in range(D):
                g = r.topk[l][b * D + j].cpu().numpy()
                qi = pipeline.layer_inputs(wl, b, l, j)
                p = L - D + j
                score = ix.scores(qi[1], qi[2], ic[:p + 1], isc[:p + 1])
                swaps += check_index_set(g, otop[j], lambda t: score[t], f"topk layer {l} b={b} row {j}")
                assert np.all(g[g >= 0] <= p)
        worst = 0.0
        if swaps == 0:
            for l, o in ref["out"].items():
                rows = slice(b * D, b * D + D)
                e = attn_rel_err(r.out[l, rows].cpu().numpy(), o)
                le = float(np.max(np.abs(r.lse[l, rows].cpu().numpy() - ref["lse"][l])))
                assert e <= ATTN_TOL and le <= 1e-4, (l, e, le)
                worst = max(worst, e)
        print(b, "swaps", swaps, "max rel err", worst)
