"""Pins for the oracle's merged-softmax sparse attention (CPU only).

Against torch's scaled_dot_product_attention in float64 (dense case and
window-only case), the log-sum-exp merge of two partial attentions, index
permutation invariance and a pure-Python loop.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import attention, bruteforce
from oracle.append import append_rows, swa_rows, dequant_fp4, dequant_fp8, bf16_to_f32


def _cache(L, seed=0, ring=128, H=16):
    cos, sin = synth.rope_table(L)
    kv = synth.normals_bf16(seed, synth.Stream.KV, 0, synth.row_id(0, np.arange(L)), 128,
                            outliers=synth.outlier_channels(seed, synth.Stream.KV_OUTLIER))
    ik = synth.normals_bf16(seed, synth.Stream.IK, 0, synth.row_id(0, np.arange(L)), 64)
    kc, ks, _, _ = append_rows(kv, ik, cos, sin)
    lo = max(0, L - ring)
    swa = synth.normals_bf16(seed, synth.Stream.SWA, 0, synth.row_id(0, np.arange(lo, L)), 128)
    sc, ss = swa_rows(swa, cos[lo:], sin[lo:])
    ring_c = np.zeros((ring, 128), np.uint8)
    ring_s = np.zeros(ring, np.float32)
    ring_c[np.arange(lo, L) % ring] = sc
    ring_s[np.arange(lo, L) % ring] = ss
    q = synth.normals_bf16(seed, synth.Stream.Q, 0, np.arange(H), 128)
    return kc, ks, ring_c, ring_s, q


def _sdpa(q, K, tau):
    qt = torch.from_numpy(q)[None, :, None, :]                       # [1][H][1][D]
    kt = torch.from_numpy(K)[None, None].expand(1, q.shape[0], -1, -1)
    return F.scaled_dot_product_attention(qt, kt, kt, scale=tau)[0, :, 0, :].numpy()


def test_dense_when_topk_covers_context_and_no_window():
    L = 300
    kc, ks, rc, rs, q = _cache(L)
    topk = np.arange(L, dtype=np.int32)
    o, lse = attention.decode_row(q, kc, ks, 0, topk, rc, rs, L - 1, window=0)
    K = dequant_fp4(kc, ks)
    qf = bf16_to_f32(q).astype(np.float64)
    ref = _sdpa(qf, K, 1 / np.sqrt(128))
    assert np.allclose(o, ref, rtol=1e-10, atol=1e-12)
    z = qf @ K.T / np.sqrt(128)
    assert np.allclose(lse, np.log(np.exp(z).sum(1)), rtol=1e-12)


def test_window_only_when_topk_empty():
    L = 500
    kc, ks, rc, rs, q = _cache(L)
    topk = np.full(512, -1, dtype=np.int32)
    o, _ = attention.decode_row(q, kc, ks, 0, topk, rc, rs, L - 1, window=128)
    slots = np.arange(L - 128, L) % 128
    K = dequant_fp8(rc[slots], rs[slots])
    ref = _sdpa(bf16_to_f32(q).astype(np.float64), K, 1 / np.sqrt(128))
    assert np.allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_merged_softmax_is_lse_merge_of_parts_and_permutation_invariant():
    L = 2000
    kc, ks, rc, rs, q = _cache(L, seed=3)
    rng = np.random.default_rng(0)
    topk = np.sort(rng.choice(L, 512, replace=False)).astype(np.int32)
    o, lse = attention.decode_row(q, kc, ks, 0, topk, rc, rs, L - 1, window=128)
    qf = bf16_to_f32(q).astype(np.float64)
    tau = 1 / np.sqrt(128)
    og, lg = attention.softmax_attention(qf, dequant_fp4(kc[topk], ks[topk]), tau)
    slots = np.arange(L - 128, L) % 128
    ow, lw = attention.softmax_attention(qf, dequant_fp8(rc[slots], rs[slots]), tau)
    m = np.maximum(lg, lw)
    wg, ww = np.exp(lg - m), np.exp(lw - m)
    merged = (og * wg[:, None] + ow * ww[:, None]) / (wg + ww)[:, None]
    assert np.allclose(o, merged, rtol=1e-10, atol=1e-13)
    assert np.allclose(lse, m + np.log(wg + ww), rtol=1e-12)
    perm = topk[rng.permutation(512)]
    o2, lse2 = attention.decode_row(q, kc, ks, 0, perm, rc, rs, L - 1, window=128)
    assert np.allclose(o, o2, rtol=1e-12, atol=1e-14) and np.allclose(lse, lse2, rtol=1e-13)


def test_matches_pure_python_loop_on_tiny_case():
    L = 20
    kc, ks, rc, rs, q = _cache(L, seed=4, H=2)
    topk = np.array([1, 5, 7, 19, -1, -1], dtype=np.int32)
    o, lse = attention.decode_row(q, kc, ks, 0, topk, rc, rs, 19, window=4)
    rows = dequant_fp4(kc[[1, 5, 7, 19]], ks[[1, 5, 7, 19]]).tolist() + \
        dequant_fp8(rc[[16, 17, 18, 19]], rs[[16, 17, 18, 19]]).tolist()
    bo, bl = bruteforce.attend(bf16_to_f32(q).astype(np.float64).tolist(), rows, 1 / np.sqrt(128))
    assert np.allclose(o, bo, rtol=1e-12, atol=1e-14) and np.allclose(lse, bl, rtol=1e-13)


def test_no_rows_gives_zero_and_minus_inf():
    kc, ks, rc, rs, q = _cache(10)
    o, lse = attention.decode_row(q, kc, ks, 0, np.full(8, -1, np.int32), rc, rs, 9, window=0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_rejects_non_causal_index():
    kc, ks, rc, rs, q = _cache(10)
    with pytest.raises(ValueError):
        attention.decode_row(q, kc, ks, 0, np.array([3, 9], np.int32), rc, rs, 5, window=0)
