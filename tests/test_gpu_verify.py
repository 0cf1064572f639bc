"""GPU parity of indexer_verify_select (several query rows per session, causal limit) against the oracle.

Each row carries its own indexer queries, a session and a position; it ranks its
session's pool (a seeded synthetic block list, the same input on both sides)
up to its own position.  Index sets must equal the oracle's; a boundary swap is
tolerated only between positions whose oracle scores differ by < 1e-6 relative.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import indexer as ix
from tests.gpu_util import check_index_set, csa2, dev, dev_bf16, host
from tests.test_gpu_indexer import fill, run_reindex

pytestmark = pytest.mark.gpu


def pools(lengths, n_keep, block, seed):
    """Seeded pools: n_keep distinct blocks of each session, ascending, -1 padded when it has fewer."""
    rng = np.random.default_rng(seed)
    out = np.full((len(lengths), n_keep), -1, np.int32)
    for b, L in enumerate(lengths):
        nb = -(-L // block)
        ids = np.sort(rng.choice(nb, size=min(nb, n_keep), replace=False)).astype(np.int32)
        out[b, :ids.shape[0]] = ids
    return out


def row_queries(T, layer=7, seed=0):
    q = np.stack([synth.normals_bf16(seed, synth.Stream.QIDX, layer, synth.row_id(r, np.arange(8)), 64)
                  for r in range(T)])
    w = np.stack([synth.head_weights(seed, layer, r) for r in range(T)])
    return q, w


def run_verify(cache, q, w, q_seq, q_pos, pool, block, n_keep, topk, max_len):
    T = q_seq.shape[0]
    top = torch.full((T, topk), -7, dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_VERIFY_SELECT, block=block, n_keep_blocks=n_keep,
                                                   topk=topk, T=T))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.indexer_verify_select(cache, dev_bf16(q), dev(w), dev(q_seq), dev(q_pos), dev(pool), block, n_keep, topk,
                               max_len, top, ws, d_err)
    torch.cuda.synchronize()
    return host(top), int(d_err.item())


def compare(lengths, q_seq, q_pos, block=8, n_keep=2048, topk=512, seed=0):
    cache, ref = fill(lengths, seed)
    pool = pools(lengths, n_keep, block, seed + 100)
    q, w = row_queries(q_seq.shape[0], seed=seed)
    top, err = run_verify(cache, q, w, q_seq, q_pos, pool, block, n_keep, topk, max(lengths))
    assert err == 0
    swaps = 0
    for r in range(q_seq.shape[0]):
        b, p = int(q_seq[r]), int(q_pos[r])
        _, _, ic, isc = ref[b]
        ov, _, _ = ix.verify_select(q[r], w[r], ic, isc, pool[b], p, block, topk)
        full = ix.scores(q[r], w[r], ic[:p + 1], isc[:p + 1])
        swaps += check_index_set(top[r], ov, lambda t: full[t], f"verify row {r} (b={b}, p={p})")
        assert np.all(top[r][top[r] >= 0] <= p)
    return swaps


def test_five_draft_rows_per_session():
    lengths = [20000, 6000, 40000, 3000]
    q_seq = np.repeat(np.arange(4, dtype=np.int32), 5)
    q_pos = np.concatenate([np.arange(L - 5, L) for L in lengths]).astype(np.int64)
    assert compare(lengths, q_seq, q_pos) == 0


def test_rows_early_in_the_context_see_only_their_prefix():
    lengths = [30000, 9000]
    q_pos = np.array([0, 7, 100, 1000, 12345, 29999, 5, 4000, 8999], np.int64)
    q_seq = np.array([0, 0, 0, 0, 0, 0, 1, 1, 1], np.int32)
    assert compare(lengths, q_seq, q_pos, n_keep=512, topk=128) == 0


@pytest.mark.parametrize("block,n_keep,topk", [(4, 1024, 64), (16, 512, 256), (8, 4096, 512)])
def test_other_block_pool_topk_sizes(block, n_keep, topk):
    lengths = [50000, 2500]
    q_seq = np.array([0, 0, 0, 1, 1, 0], np.int32)
    q_pos = np.array([49999, 30000, 777, 2499, 1200, 49995], np.int64)
    assert compare(lengths, q_seq, q_pos, block, n_keep, topk) == 0


def test_last_position_rows_equal_the_reindex_entry():
    lengths = [12000, 700, 33000]
    cache, _ = fill(lengths)
    pool = pools(lengths, 2048, 8, 5)
    q, w = row_queries(3)
    top, err = run_verify(cache, q, w, np.arange(3, dtype=np.int32), np.array(lengths, np.int64) - 1, pool, 8, 2048,
                          512, max(lengths))
    assert err == 0
    re = run_reindex(cache, q, w, pool, 8, 2048, 512, max(lengths))
    assert np.array_equal(top, re)


def test_bad_rows_flag_errors_and_select_nothing():
    lengths = [500, 300]
    cache, _ = fill(lengths)
    pool = pools(lengths, 64, 8, 1)
    q_seq = np.array([0, 2, 1, -1, 1], np.int32)
    q_pos = np.array([499, 10, 300, 5, -3], np.int64)
    q, w = row_queries(5)
    top, err = run_verify(cache, q, w, q_seq, q_pos, pool, 8, 64, 32, 500)
    assert err & csa2.DEVERR_SEQ and err & csa2.DEVERR_POS
    assert np.all(top[1:] == -1) and np.all(top[0][:32] >= 0)
    bad = pool.copy()
    bad[1, 38] = 99                                    # block 99 starts at 792 > 300 (still ascending)
    top, err = run_verify(cache, q[:1], w[:1], np.array([1], np.int32), np.array([299], np.int64), bad, 8, 64, 32,
                          500)
    assert err & csa2.DEVERR_POOL


def test_zero_rows_and_small_workspace():
    cache, _ = fill([64])
    q, w = row_queries(1)
    pool = torch.full((1, 8), -1, dtype=torch.int32, device="cuda")
    top = torch.full((1, 4), -1, dtype=torch.int32, device="cuda")
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    empty_i32 = torch.zeros(0, dtype=torch.int32, device="cuda")
    empty_i64 = torch.zeros(0, dtype=torch.int64, device="cuda")
    ws = csa2.alloc_workspace(256)
    csa2.indexer_verify_select(cache, dev_bf16(q), dev(w), empty_i32, empty_i64, pool, 8, 8, 4, 64, top, ws, d_err)
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.indexer_verify_select(cache, dev_bf16(q), dev(w), dev(np.zeros(1, np.int32)),
                                   dev(np.array([63], np.int64)), pool, 8, 8, 4, 64, top, ws, d_err)
    assert e.value.status == csa2.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
