"""Sparse attention over the selected global rows plus the sliding window (oracle side).

Follows ttj.kr "DeepSeek-V4.1-Flash, KV 캐시를 토큰당 890바이트까지 압축하다",
section "CSA2와 어텐션 재설계" (a 128-token local window combined with
global sparse retrieval), and origotech.dev deep dive, subsection
"Compressed Sparse Attention 2(CSA2)" (top-k 512, window 128).

Readings where the pages are silent:

* keys and values are the same dequantised vector (MQA, V = K);
* z_j = tau * <q_h, k_j> with tau = 1/sqrt(128) unless the caller passes
  another scale;
* one softmax over the concatenation of the valid selected rows (FP4 cache)
  and the window rows max(0, p-W+1)..p (this layer's FP8 SWA ring); a
  position can appear in both lists, they are different tensors, and it is
  not de-duplicated; no attention sink;
* lse = log sum_j exp(z_j); with no rows at all the output is 0 and lse is
  -inf.

Computed in float64 from the same dequantised values the GPU sees.
"""
from __future__ import annotations

import numpy as np

from .append import dequant_fp4, dequant_fp8, bf16_to_f32


def softmax_attention(q: np.ndarray, K: np.ndarray, tau: float):
    """q [H][D] float64, K [n][D] float64 (V = K) -> (o [H][D], lse [H])."""
    H, Dm = q.shape
    if K.shape[0] == 0:
        return np.zeros((H, Dm)), np.full(H, -np.inf)
    z = tau * (q @ K.T)                                   # [H][n]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e / l) @ K
    return o, (m + np.log(l))[:, 0]


def gather_rows(kv_codes, kv_scales, seq_base: int, topk_row, q_pos: int):
    """Dequantised global rows of the valid indices (-1 entries skipped)."""
    idx = np.asarray(topk_row, dtype=np.int64)
    idx = idx[idx >= 0]
    if np.any(idx > q_pos):
        raise ValueError("index beyond the query position")
    rows = seq_base + idx
    return dequant_fp4(kv_codes[rows], kv_scales[rows])


def window_rows(swa_codes_b, swa_scale_b, q_pos: int, window: int):
    """Dequantised SWA rows of positions max(0, p-W+1)..p from one sequence's ring."""
    ring = swa_codes_b.shape[0]
    pos = np.arange(max(0, q_pos - window + 1), q_pos + 1, dtype=np.int64)
    slot = pos % ring
    return dequant_fp8(swa_codes_b[slot], swa_scale_b[slot])


def decode_row(q_bf16, kv_codes, kv_scales, seq_base, topk_row, swa_codes_b, swa_scale_b,
               q_pos, window=128, tau=None):
    """Attention output of one query row: (o [H][128] float64, lse [H])."""
    q = bf16_to_f32(q_bf16).astype(np.float64)
    tau = 1.0 / np.sqrt(q.shape[1]) if tau is None else float(tau)
    K = np.concatenate([gather_rows(kv_codes, kv_scales, seq_base, topk_row, q_pos),
                        window_rows(swa_codes_b, swa_scale_b, q_pos, window)], axis=0)
    return softmax_attention(q, K, tau)
