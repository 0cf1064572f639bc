"""GPU parity of indexer_full_select / indexer_reindex_select against the oracle.

Index sets must equal the oracle's; a boundary swap is tolerated only between
positions whose oracle scores differ by less than 1e-6 relative.  The oracle
computes from its own caches (regenerated from the seeded inputs), never from
GPU outputs.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import indexer as ix
from oracle.append import append_rows
from tests.gpu_util import check_index_set, csa2, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


def fill(lengths, seed=0, dup_rows=None):
    """GPU cache of sequences with the given lengths (positions 0..L-1) and the oracle's own copy."""
    lengths = [int(x) for x in lengths]
    B = len(lengths)
    padded = [((L + 15) // 16) * 16 for L in lengths]
    base = np.zeros(B, np.int64)
    base[1:] = np.cumsum(padded)[:-1]
    cache = csa2.Cache(max(1, sum(padded)), B)
    cache.seq_base.copy_(torch.from_numpy(base))
    cache.seq_len.copy_(torch.from_numpy(np.array(lengths, np.int32)))
    cos, sin = synth.rope_table(max(lengths) + 1)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    oc = synth.outlier_channels(seed, synth.Stream.KV_OUTLIER)
    ref = []
    for b, L in enumerate(lengths):
        if L == 0:
            ref.append(None)
            continue
        pos = np.arange(L, dtype=np.int64)
        rows = synth.row_id(b, pos)
        kv = synth.normals_bf16(seed, synth.Stream.KV, 0, rows, 128, oc)
        ik = synth.normals_bf16(seed, synth.Stream.IK, 0, rows, 64)
        if dup_rows is not None:
            ik = dup_rows(b, ik)
        csa2.kv_append_fp4(cache, None, dev_bf16(kv), dev_bf16(ik), None, dev(cos), dev(sin),
                           dev(np.full(L, b, np.int32)), dev(pos), d_err)
        ref.append(append_rows(kv, ik, cos[:L], sin[:L]))
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    return cache, ref


def queries(B, layer=0, seed=0):
    q = np.stack([synth.normals_bf16(seed, synth.Stream.QIDX, layer, synth.row_id(b, np.arange(8)), 64)
                  for b in range(B)])
    w = np.stack([synth.head_weights(seed, layer, b) for b in range(B)])
    return q, w


def run_full(cache, q, w, block, n_keep, topk, max_len):
    B = cache.B
    pool = torch.full((B, n_keep), -7, dtype=torch.int32, device="cuda")
    top = torch.full((B, topk), -7, dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_FULL_SELECT, B, max_len, block, n_keep, topk))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.indexer_full_select(cache, dev_bf16(q), dev(w), block, n_keep, topk, max_len, pool, top, ws, d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    return host(pool), host(top)


def run_reindex(cache, q, w, pool, block, n_keep, topk, max_len):
    B = cache.B
    top = torch.full((B, topk), -7, dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_REINDEX_SELECT, B, max_len, block, n_keep, topk))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.indexer_reindex_select(cache, dev_bf16(q), dev(w), dev(pool), block, n_keep, topk, max_len, top, ws, d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    return host(top)


def compare_full(lengths, block=8, n_keep=2048, topk=512, seed=0, reindex=True, dup_rows=None):
    cache, ref = fill(lengths, seed, dup_rows)
    B = len(lengths)
    max_len = max(lengths)
    q, w = queries(B, 0, seed)
    pool, top = run_full(cache, q, w, block, n_keep, topk, max_len)
    q2, w2 = queries(B, 5, seed)
    if reindex:
        # the oracle's own pools drive its reindex; the GPU reindex reads the GPU pool
        re = run_reindex(cache, q2, w2, pool, block, n_keep, topk, max_len)
    swaps = 0
    for b, L in enumerate(lengths):
        if L == 0:
            assert np.all(pool[b] == -1) and np.all(top[b] == -1)
            continue
        _, _, ic, isc = ref[b]
        opool, otop, sig = ix.full_select(q[b], w[b], ic, isc, block, n_keep, topk)
        bs = ix.block_scores(sig, block)
        swaps += check_index_set(pool[b], opool, lambda j: bs[j], f"pool b={b}")
        swaps += check_index_set(top[b], otop, lambda p: sig[p], f"top-k b={b}")
        if reindex:
            ore, sig2, pos2 = ix.reindex_select(q2[b], w2[b], ic, isc, opool, block, topk)
            full2 = ix.scores(q2[b], w2[b], ic, isc)
            swaps += check_index_set(re[b], ore, lambda p: full2[p], f"reindex b={b}")
            allowed = set(ix.pool_positions(pool[b], L, block).tolist())
            assert set(re[b][re[b] >= 0].tolist()) <= allowed
        # containment: the Full top-k lies inside the kept pool
        assert set(top[b][top[b] >= 0].tolist()) <= set(ix.pool_positions(pool[b], L, block).tolist())
    return swaps


def test_full_layer_context_4096():
    assert compare_full([4096]) == 0


def test_ragged_and_tiny_contexts():
    assert compare_full([1, 7, 8, 9, 127, 128, 129, 511, 512, 513, 4095, 20000, 0]) == 0


@pytest.mark.parametrize("block,n_keep,topk", [(1, 64, 64), (2, 3, 1), (4, 100, 17), (16, 40, 40), (8, 64, 3)])
def test_other_block_pool_topk_sizes(block, n_keep, topk):
    assert compare_full([50, 1000, 3333, 6000], block, n_keep, topk) == 0


def test_ties_break_to_lower_positions():
    # every key of sequence 1 repeats the same four rows: scores tie in groups
    def dup(b, ik):
        if b == 1:
            ik = ik.copy()
            ik[:] = ik[np.arange(ik.shape[0]) % 4]
        return ik
    assert compare_full([3000, 3000], block=8, n_keep=64, topk=40, dup_rows=dup) == 0


def test_many_sequences_and_long_context():
    assert compare_full([65536, 40000, 17, 90001], n_keep=2048, topk=512, reindex=True) == 0


def test_approximate_scores_obey_the_error_bound():
    lengths = [65536, 12345]
    cache, ref = fill(lengths, seed=1)
    q, w = queries(2, 0, seed=1)
    max_len = max(lengths)
    sigma = torch.full((2, max_len), -1.0, dtype=torch.float32, device="cuda")
    bound = torch.zeros(3, dtype=torch.float64, device="cuda")
    ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_FULL_SELECT, 2, max_len, 8, 1, 1))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.test_index_scores(cache, dev_bf16(q), dev(w), max_len, sigma, bound, ws, d_err)
    torch.cuda.synchronize()
    sg, bd = host(sigma).astype(np.float64), host(bound)
    r = bd[2]
    worst = 0.0
    for b, L in enumerate(lengths):
        _, _, ic, isc = ref[b]
        exact = ix.scores(q[b], w[b], ic, isc)
        err = np.abs(sg[b, :L] - exact)
        lim = bd[b] + r * sg[b, :L]
        assert np.all(err <= lim), f"bound violated: {np.max(err / lim)}"
        worst = max(worst, float(np.max(err / lim)))
    print(f"max |approx - exact| / bound = {worst:.3e}")


def test_invalid_lengths_and_pool_ids_flag_errors():
    cache, _ = fill([100, 50])
    q, w = queries(2)
    cache.seq_len[1] = 10_000_000                     # beyond max_len
    B, max_len = 2, 100
    pool = torch.full((B, 8), -1, dtype=torch.int32, device="cuda")
    top = torch.full((B, 4), -1, dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_FULL_SELECT, B, max_len, 8, 8, 4))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.indexer_full_select(cache, dev_bf16(q), dev(w), 8, 8, 4, max_len, pool, top, ws, d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) & csa2.DEVERR_LEN
    assert np.all(host(top)[1] == -1)
    cache.seq_len[1] = 50
    bad_pool = torch.tensor([[0, 1, 2, 99, -1, -1, -1, -1]] * 2, dtype=torch.int32, device="cuda")
    d_err.zero_()
    csa2.indexer_reindex_select(cache, dev_bf16(q), dev(w), bad_pool, 8, 8, 4, max_len, top, ws, d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) & csa2.DEVERR_POOL


def test_workspace_too_small_is_rejected():
    cache, _ = fill([64])
    q, w = queries(1)
    pool = torch.full((1, 8), -1, dtype=torch.int32, device="cuda")
    top = torch.full((1, 4), -1, dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(256)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.indexer_full_select(cache, dev_bf16(q), dev(w), 8, 8, 4, 64, pool, top, ws, d_err)
    assert e.value.status == csa2.ERR_WORKSPACE
