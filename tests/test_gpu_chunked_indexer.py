"""GPU parity of indexer_chunked_select (the Full selection per query row, causal) against the oracle.

Each row carries its own indexer queries, a session and a position; its pool and top-k
must equal the oracle's Full selection over the session's first position + 1 positions.
A boundary swap is tolerated only between items whose oracle scores differ by < 1e-6
relative.  The oracle computes from its own caches, regenerated from the seeded inputs.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import indexer as ix
from tests.gpu_util import check_index_set, csa2, dev, dev_bf16, host
from tests.test_gpu_indexer import fill
from tests.test_gpu_verify import row_queries

pytestmark = pytest.mark.gpu


def run_chunked(cache, q, w, q_seq, q_pos, block, n_keep, topk, max_len):
    T = q_seq.shape[0]
    pool = torch.full((T, n_keep), -7, dtype=torch.int32, device="cuda")
    top = torch.full((T, topk), -7, dtype=torch.int32, device="cuda")
    ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_CHUNKED_SELECT, max_len=max_len, block=block,
                                                   n_keep_blocks=n_keep, topk=topk, T=T))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.indexer_chunked_select(cache, dev_bf16(q), dev(w), dev(q_seq), dev(q_pos), block, n_keep, topk, max_len,
                                pool, top, ws, d_err)
    torch.cuda.synchronize()
    return host(pool), host(top), int(d_err.item())


def compare(lengths, q_seq, q_pos, block=8, n_keep=2048, topk=512, rows=None, seed=0):
    cache, ref = fill(lengths, seed)
    q, w = row_queries(q_seq.shape[0], layer=9, seed=seed)
    pool, top, err = run_chunked(cache, q, w, q_seq, q_pos, block, n_keep, topk, int(q_pos.max()) + 1)
    assert err == 0
    swaps = 0
    for r in (range(q_seq.shape[0]) if rows is None else rows):
        b, p = int(q_seq[r]), int(q_pos[r])
        _, _, ic, isc = ref[b]
        opool, otop, sig = ix.chunked_select(q[r], w[r], ic, isc, p, block, n_keep, topk)
        bs = ix.block_scores(sig, block)
        swaps += check_index_set(pool[r], opool, lambda j: bs[j], f"pool row {r} (b={b}, p={p})")
        swaps += check_index_set(top[r], otop, lambda t: sig[t], f"top-k row {r} (b={b}, p={p})")
        assert np.all(top[r][top[r] >= 0] <= p)
        assert set(top[r][top[r] >= 0].tolist()) <= set(ix.pool_positions(pool[r], p + 1, block).tolist())
    return swaps


def test_rows_at_many_positions():
    lengths = [9000, 3000]
    q_seq = np.array([0, 0, 0, 0, 0, 0, 1, 1], np.int32)
    q_pos = np.array([0, 5, 100, 2047, 4096, 8999, 2999, 1500], np.int64)
    assert compare(lengths, q_seq, q_pos, n_keep=256, topk=128) == 0


def test_decoder_sizes_rows_near_the_end():
    L = 20000
    q_pos = np.concatenate([np.arange(L - 40, L), [17, 3000, 16383, 16384]]).astype(np.int64)
    assert compare([L], np.zeros(q_pos.shape[0], np.int32), q_pos) == 0


@pytest.mark.parametrize("block,n_keep,topk", [(1, 64, 64), (2, 30, 9), (4, 100, 17), (16, 40, 40)])
def test_other_block_pool_topk_sizes(block, n_keep, topk):
    q_pos = np.array([0, 63, 700, 2222, 4999], np.int64)
    assert compare([5000], np.zeros(5, np.int32), q_pos, block, n_keep, topk) == 0


@pytest.mark.parametrize("block,n_keep,topk", [(1, 64, 64), (2, 300, 50), (4, 100, 17), (16, 40, 40)])
def test_other_block_sizes_on_whole_tiles(block, n_keep, topk):
    # 40 rows near the end of one session: the first group's rows all reach past most key
    # tiles (the scores' whole-tile path), the second group is mostly empty rows
    q_pos = np.arange(4960, 5000, dtype=np.int64)
    assert compare([5000], np.zeros(40, np.int32), q_pos, block, n_keep, topk) == 0


def test_more_rows_than_one_group():
    L = 3000
    T = 1100                                            # two groups of rows
    q_pos = np.arange(L - T, L, dtype=np.int64)
    assert compare([L], np.zeros(T, np.int32), q_pos, n_keep=64, topk=32, rows=[0, 1, 511, 1023, 1024, 1099]) == 0


def test_bad_rows_select_nothing_and_flag_errors():
    cache, _ = fill([500, 300])
    q_seq = np.array([0, 2, 1, -1], np.int32)
    q_pos = np.array([499, 10, 300, 5], np.int64)
    q, w = row_queries(4, layer=9)
    pool, top, err = run_chunked(cache, q, w, q_seq, q_pos, 8, 16, 8, 500)
    assert err & csa2.DEVERR_SEQ and err & csa2.DEVERR_POS
    assert np.all(pool[1:] == -1) and np.all(top[1:] == -1)
    assert np.all(top[0] >= 0) and np.all(pool[0] >= 0)


def test_chunk_of_4096_queries_over_a_262144_token_cache():
    """The chunked-query workload's own indices: 4,096 rows ending at the last position."""
    L, T = 262144, 4096
    q_pos = np.arange(L - T, L, dtype=np.int64)
    assert compare([L], np.zeros(T, np.int32), q_pos, rows=[0, 2047, 4095]) == 0


def test_tensor_core_scores_obey_the_error_bound():
    """The tcgen05 scores of 48 rows (three groups of 16) against the oracle's exact scores:
    |approx - exact| <= E_row + r * approx at every position up to the row's own; positions
    after it are left untouched."""
    L = 40000
    cache, ref = fill([L], seed=1)
    q_pos = np.concatenate([np.arange(L - 16, L), np.arange(100, 116), np.arange(20000, 20016)]).astype(np.int64)
    T = q_pos.shape[0]
    q, w = row_queries(T, layer=11, seed=1)
    sigma = torch.full((T, L), -1.0, dtype=torch.float32, device="cuda")
    bound = torch.zeros(T + 1, dtype=torch.float64, device="cuda")
    ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_CHUNKED_SELECT, max_len=L, block=8, n_keep_blocks=1,
                                                   topk=1, T=T))
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.test_chunk_scores(cache, dev_bf16(q), dev(w), dev(np.zeros(T, np.int32)), dev(q_pos), L, sigma, bound, ws,
                           d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    sg, bd = host(sigma).astype(np.float64), host(bound)
    rr = bd[T]
    _, _, ic, isc = ref[0]
    worst = 0.0
    for r in range(T):
        p = int(q_pos[r])
        exact = ix.scores(q[r], w[r], ic[:p + 1], isc[:p + 1])
        err = np.abs(sg[r, :p + 1] - exact)
        lim = bd[r] + rr * sg[r, :p + 1]
        assert np.all(err <= lim), f"row {r}: bound violated: {np.max(err / lim)}"
        assert np.all(sg[r, p + 1:] == -1.0)
        worst = max(worst, float(np.max(err / lim)))
    print(f"max |approx - exact| / bound = {worst:.3e}")
