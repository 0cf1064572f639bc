"""Hierarchical sparse indexer: Full, Reindex and Reuse selection (oracle side).

Follows origotech.dev deep dive, subsection "Compressed Sparse Attention
2(CSA2)": a Full layer computes its own indexer queries and keys and a fresh
top-k; a Reindex layer reuses the earlier layer's main KV and indexer keys
with its own indexer queries and recomputes top-k; a Reuse layer takes the
main KV and the top-k indices unchanged.  In the decoder the first Full
layer picks 2,048 blocks of 8 positions (a 16,384-position pool) and only
the Reindex layers score that pool; top-k is 512 (same subsection, and
trawling.dev "DeepSeek-V4.1-Flash 공개", section "CSA2와 FP4 KV 캐싱").

Readings where the pages are silent:

* score of position t for one layer: sigma_t = s_t * sum_h w_h *
  max(q_h . k_t, 0) over 8 indexer heads of dim 64, with k_t the E4M3 key
  values and s_t its float32 scale; evaluated in float64;
* block j covers positions [8j, min(8j+8, L)); its score is the maximum of
  its members' scores;
* ranking is by (score descending, position or block id ascending); outputs
  are sets written in ascending order and padded with -1;
* the Full layer's top-k ranges over every cached position; by the
  containment argument (a block holding a top-k position ranks among the
  top-k blocks) it always lies inside the kept pool;
* Reindex ranks only the pool's positions, using the Full layer's keys.
"""
from __future__ import annotations

import numpy as np

from .formats import e4m3_decode
from .append import bf16_to_f32


def scores(q_bf16, w, ik_codes, ik_scale) -> np.ndarray:
    """sigma_t for rows of one sequence, float64 [L].

    q_bf16: [8][64] bf16 bits; w: [8] float32; ik_codes: [L][64] u8;
    ik_scale: [L] float32.
    """
    q = bf16_to_f32(q_bf16).astype(np.float64)                 # [8][64]
    k = e4m3_decode(ik_codes)                                  # [L][64]
    d = k @ q.T                                                # [L][8] (library matmul)
    w64 = np.asarray(w, dtype=np.float32).astype(np.float64)
    return np.asarray(ik_scale, dtype=np.float32).astype(np.float64) * (np.maximum(d, 0.0) @ w64)


def block_scores(sigma: np.ndarray, block: int) -> np.ndarray:
    """Maximum over each block of ``block`` consecutive positions (last block may be short)."""
    L = sigma.shape[0]
    nb = -(-L // block)
    pad = np.full(nb * block, -np.inf)
    pad[:L] = sigma
    return pad.reshape(nb, block).max(axis=1)


def top_k_ids(values: np.ndarray, ids: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k best entries by (value descending, id ascending), returned ascending."""
    values = np.asarray(values, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    k = min(k, values.shape[0])
    order = np.lexsort((ids, -values))                         # primary key last
    return np.sort(ids[order[:k]])


def pad(ids: np.ndarray, n: int) -> np.ndarray:
    out = np.full(n, -1, dtype=np.int32)
    out[:ids.shape[0]] = ids
    return out


def full_select(q_bf16, w, ik_codes, ik_scale, block=8, n_keep=2048, topk=512):
    """Full layer of one sequence: (pool block ids [n_keep], top-k positions [topk]).

    ``ik_codes``/``ik_scale`` are the sequence's rows 0..L-1.
    """
    sigma = scores(q_bf16, w, ik_codes, ik_scale)
    L = sigma.shape[0]
    bs = block_scores(sigma, block)
    pool = top_k_ids(bs, np.arange(bs.shape[0]), n_keep)
    top = top_k_ids(sigma, np.arange(L), topk)
    return pad(pool, n_keep), pad(top, topk), sigma


def pool_positions(pool, L: int, block: int = 8) -> np.ndarray:
    """Positions covered by the pool's blocks, clipped to the context."""
    pool = np.asarray(pool, dtype=np.int64)
    pool = pool[pool >= 0]
    pos = (pool[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return pos[pos < L]


def reindex_select(q_bf16, w, ik_codes, ik_scale, pool, block=8, topk=512):
    """Reindex layer of one sequence: top-k over the pool's positions only."""
    L = ik_codes.shape[0]
    pos = pool_positions(pool, L, block)
    sigma = scores(q_bf16, w, ik_codes[pos], ik_scale[pos])
    return pad(top_k_ids(sigma, pos, topk), topk), sigma, pos


def chunked_select(q_bf16, w, ik_codes, ik_scale, p: int, block=8, n_keep=2048, topk=512):
    """One row of a chunk of prefill queries, at position p: the Full selection (pool +
    top-k) over positions 0..p only, a query seeing nothing after itself (origotech.dev deep
    dive, subsection "Compressed Sparse Attention 2(CSA2)")."""
    return full_select(q_bf16, w, ik_codes[:p + 1], ik_scale[:p + 1], block, n_keep, topk)


def verify_select(q_bf16, w, ik_codes, ik_scale, pool, p: int, block=8, topk=512):
    """One verify row at position p: top-k over the session's pool positions p' <= p.

    Speculative decoding (origotech.dev deep dive, section "아키텍처는 어떻게 KV 캐시를
    줄이나", the DSpark item) checks several drafted positions at once; each such row
    ranks the pool its session's Full layer kept, under the row's own indexer queries,
    and sees only the positions up to its own (the causal limit).
    """
    pos = pool_positions(pool, ik_codes.shape[0], block)
    pos = pos[pos <= p]
    sigma = scores(q_bf16, w, ik_codes[pos], ik_scale[pos])
    return pad(top_k_ids(sigma, pos, topk), topk), sigma, pos


def reuse(topk_idx):
    """Reuse layer: the indices are passed on unchanged."""
    return topk_idx
