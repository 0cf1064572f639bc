"""GPU parity of sparse_attn_decode against the float64 oracle.

Both sides take the same (seeded) top-k index lists, so attention is checked
on its own; the oracle dequantises from its own caches.  Tolerance per
(row, head): max|o - r| / max|r| <= 2e-3.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as at
from oracle.append import append_rows, swa_rows
from tests.gpu_util import ATTN_TOL, attn_rel_err, csa2, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


class World:
    """A GPU cache + one SWA ring for sequences of given lengths, and the oracle's copies."""

    def __init__(self, lengths, ring=128, seed=0, layer=0):
        self.lengths = [int(x) for x in lengths]
        B = len(lengths)
        padded = [((L + 15) // 16) * 16 for L in self.lengths]
        self.base = np.zeros(B, np.int64)
        self.base[1:] = np.cumsum(padded)[:-1]
        self.cache = csa2.Cache(sum(padded), B)
        self.cache.seq_base.copy_(torch.from_numpy(self.base))
        self.cache.seq_len.copy_(torch.from_numpy(np.array(self.lengths, np.int32)))
        self.swa = csa2.SwaRing(B, ring)
        self.ring = ring
        cos, sin = synth.rope_table(max(self.lengths) + 1)
        d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
        oc = synth.outlier_channels(seed, synth.Stream.KV_OUTLIER)
        soc = synth.outlier_channels(seed, synth.Stream.SWA_OUTLIER)
        self.kc = np.zeros((sum(padded), 64), np.uint8)
        self.ks = np.zeros((sum(padded), 8), np.uint8)
        self.rc = np.zeros((B, ring, 128), np.uint8)
        self.rs = np.zeros((B, ring), np.float32)
        for b, L in enumerate(self.lengths):
            pos = np.arange(L, dtype=np.int64)
            rows = synth.row_id(b, pos)
            kv = synth.normals_bf16(seed, synth.Stream.KV, 0, rows, 128, oc)
            ik = synth.normals_bf16(seed, synth.Stream.IK, 0, rows, 64)
            lo = max(0, L - ring)
            sw = synth.normals_bf16(seed, synth.Stream.SWA, layer, rows[lo:], 128, soc)
            csa2.kv_append_fp4(self.cache, None, dev_bf16(kv), dev_bf16(ik), None, dev(cos), dev(sin),
                               dev(np.full(L, b, np.int32)), dev(pos), d_err)
            csa2.kv_append_fp4(self.cache, [self.swa], dev_bf16(kv[lo:]), None, dev_bf16(sw[None]), dev(cos),
                               dev(sin), dev(np.full(L - lo, b, np.int32)), dev(pos[lo:]), d_err)
            kc, ks, _, _ = append_rows(kv, ik, cos[:L], sin[:L])
            self.kc[self.base[b]:self.base[b] + L] = kc
            self.ks[self.base[b]:self.base[b] + L] = ks
            sc, ss = swa_rows(sw, cos[lo:L], sin[lo:L])
            self.rc[b, pos[lo:] % ring] = sc
            self.rs[b, pos[lo:] % ring] = ss
        torch.cuda.synchronize()
        assert int(d_err.item()) == 0

    def run(self, q, q_seq, q_pos, topk, window, tau=1 / math.sqrt(128), with_lse=True):
        T, H = q.shape[0], q.shape[1]
        out = torch.full((T, H, 128), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
        k = topk.shape[1]
        ws = csa2.alloc_workspace(csa2.workspace_bytes(csa2.OP_ATTN_DECODE, T=T, H=H, topk=k, window=window))
        d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
        csa2.sparse_attn_decode(self.cache, self.swa, dev_bf16(q), dev(q_seq), dev(q_pos), dev(topk), window, tau,
                                out, lse, ws, d_err)
        torch.cuda.synchronize()
        return host(out), (host(lse) if with_lse else None), int(d_err.item())

    def oracle(self, q, q_seq, q_pos, topk, window, tau=1 / math.sqrt(128)):
        outs, lses = [], []
        for t in range(q.shape[0]):
            b = int(q_seq[t])
            o, l = at.decode_row(q[t], self.kc, self.ks, int(self.base[b]), topk[t], self.rc[b], self.rs[b],
                                 int(q_pos[t]), window, tau)
            outs.append(o)
            lses.append(l)
        return np.stack(outs), np.stack(lses)


def _queries(T, H, seed=0, layer=0):
    return synth.normals_bf16(seed, synth.Stream.Q, layer, np.arange(T * H), 128).reshape(T, H, 128)


# lse tolerance of the tensor-core path: its row sums add the float32 P, while the P that
# multiplies V is rounded to f16 (each term within 2^-11 relative), and its exponentials come
# from ex2.approx; 6e-4 bounds both with room (the CUDA-core decode path: 1e-4).
LSE_TOL_TC = 6e-4


def _check(world, q, q_seq, q_pos, topk, window, lse_tol=1e-4):
    out, lse, err = world.run(q, q_seq, q_pos, topk, window)
    assert err == 0
    ref, rlse = world.oracle(q, q_seq, q_pos, topk, window)
    e = attn_rel_err(out, ref)
    fin = np.isfinite(rlse)
    assert np.array_equal(np.isfinite(lse), fin)
    le = np.max(np.abs(lse[fin] - rlse[fin])) if fin.any() else 0.0
    assert e <= ATTN_TOL, e
    assert le <= lse_tol, le
    return e


def test_decode_rows_topk512_window128():
    lengths = [4096, 65536 // 8, 700, 130]
    w = World(lengths)
    T = len(lengths)
    q_pos = np.array([L - 1 for L in lengths], np.int64)
    topk = synth.causal_topk(1, q_pos, 512)
    e = _check(w, _queries(T, 16), np.arange(T, dtype=np.int32), q_pos, topk, 128)
    print(f"max rel err {e:.3e}")


def test_dense_when_topk_covers_context_and_no_window():
    w = World([300])
    q_pos = np.array([299], np.int64)
    topk = np.arange(300, dtype=np.int32)[None, :]
    _check(w, _queries(1, 16), np.zeros(1, np.int32), q_pos, topk, 0)


def test_window_only_and_short_context():
    w = World([50, 500])
    q_pos = np.array([49, 499], np.int64)
    topk = np.full((2, 512), -1, np.int32)
    _check(w, _queries(2, 16), np.arange(2, dtype=np.int32), q_pos, topk, 128)


def test_sixty_four_heads_and_many_rows():
    w = World([262144 // 16], ring=8192)
    L = 262144 // 16
    q_pos = np.arange(L - 96, L, dtype=np.int64)
    topk = synth.causal_topk(3, q_pos, 512)
    e = _check(w, _queries(96, 64, layer=1), np.zeros(96, np.int32), q_pos, topk, 128)
    print(f"max rel err {e:.3e}")


def test_permuted_and_padded_indices_give_the_same_output():
    w = World([5000])
    q_pos = np.array([4999], np.int64)
    topk = synth.causal_topk(4, q_pos, 512)
    q = _queries(1, 16)
    out1, lse1, _ = w.run(q, np.zeros(1, np.int32), q_pos, topk, 128)
    rng = np.random.default_rng(0)
    shuffled = np.concatenate([topk[:, rng.permutation(512)], np.full((1, 64), -1, np.int32)], axis=1)
    shuffled = shuffled[:, rng.permutation(576)]
    out2, lse2, _ = w.run(q, np.zeros(1, np.int32), q_pos, shuffled, 128)
    # Only the summation order changes: f32 accumulation over <= 640 rows plus the f16 hi/lo split
    # of P (~2^-22 relative) moves an output by far less than 3e-5 of its row's largest value,
    # while a dropped or doubled row moves it by ~1e-3 (one of 640 weights).
    e = attn_rel_err(out2, out1)
    print(f"permutation rel diff {e:.3e}")
    assert e < 3e-5 and np.allclose(lse1, lse2, atol=1e-5)


def test_non_causal_index_is_flagged_and_skipped():
    w = World([200])
    q_pos = np.array([100], np.int64)
    topk = np.array([[5, 50, 150, -1]], np.int32)     # 150 > 100
    out, lse, err = w.run(_queries(1, 16), np.zeros(1, np.int32), q_pos, topk, 16)
    assert err & csa2.DEVERR_INDEX
    ref, rlse = w.oracle(_queries(1, 16), np.zeros(1, np.int32), q_pos, np.array([[5, 50, -1, -1]], np.int32), 16)
    assert attn_rel_err(out, ref) <= ATTN_TOL


def test_empty_row_gives_zero_and_minus_inf():
    w = World([64])
    out, lse, err = w.run(_queries(1, 16), np.zeros(1, np.int32), np.array([63], np.int64),
                          np.full((1, 16), -1, np.int32), 0)
    assert err == 0 and np.all(out == 0) and np.all(np.isneginf(lse))


# ---- the tensor-core (tcgen05) path: many query rows of one sequence, H <= 64 --------------

def test_tensor_core_path_many_rows_h64():
    L = 6000
    w = World([L], ring=512)
    q_pos = np.arange(L - 256, L, dtype=np.int64)              # 256 rows x 64 heads
    topk = synth.causal_topk(7, q_pos, 512)
    e = _check(w, _queries(256, 64, layer=3), np.zeros(256, np.int32), q_pos, topk, 128, LSE_TOL_TC)
    print(f"max rel err {e:.3e}")


def test_tensor_core_path_short_contexts_and_padding():
    # rows at the start of the sequence: fewer than 512 valid indices (-1 padded), clipped windows
    w = World([300], ring=512)
    q_pos = np.arange(0, 256, dtype=np.int64)
    topk = synth.causal_topk(8, q_pos, 512)
    e = _check(w, _queries(256, 64, layer=4), np.zeros(256, np.int32), q_pos, topk, 128, LSE_TOL_TC)
    print(f"max rel err {e:.3e}")


@pytest.mark.parametrize("H", [16, 32, 48])
def test_tensor_core_path_fewer_heads(H):
    L = 3000
    w = World([L], ring=2048)
    T = 16384 // H
    q_pos = np.arange(L - T, L, dtype=np.int64)
    topk = synth.causal_topk(9, q_pos, 512)
    e = _check(w, _queries(T, H, layer=5), np.zeros(T, np.int32), q_pos, topk, 128, LSE_TOL_TC)
    print(f"H={H} max rel err {e:.3e}")


def test_tensor_core_path_odd_topk_and_window():
    L = 5000
    w = World([L], ring=512)
    q_pos = np.arange(L - 256, L, dtype=np.int64)
    topk = synth.causal_topk(10, q_pos, 200)                    # partial chunks on both sides
    e = _check(w, _queries(256, 64, layer=6), np.zeros(256, np.int32), q_pos, topk, 50, LSE_TOL_TC)
    print(f"max rel err {e:.3e}")


def test_tensor_core_path_flags_non_causal_index():
    L = 3000
    w = World([L], ring=512)
    q_pos = np.arange(L - 256, L, dtype=np.int64)
    topk = synth.causal_topk(11, q_pos, 512)
    topk[5, 3] = int(q_pos[5]) + 1                              # in the cache but after the query
    out, lse, err = w.run(_queries(256, 64), np.zeros(256, np.int32), q_pos, topk, 128)
    assert err & csa2.DEVERR_INDEX
    assert np.all(np.isfinite(out))


def test_tensor_core_path_window_only():
    # no top-k lists: every step is a window step (per-key float32 scales, the general path)
    L = 4000
    w = World([L], ring=512)
    q_pos = np.arange(L - 256, L, dtype=np.int64)
    topk = np.zeros((256, 0), np.int32)
    e = _check(w, _queries(256, 64, layer=7), np.zeros(256, np.int32), q_pos, topk, 256, LSE_TOL_TC)
    print(f"max rel err {e:.3e}")


def test_tensor_core_path_topk_only():
    # no window: every step is a top-k step (the all-valid fast path)
    L = 4000
    w = World([L], ring=128)
    q_pos = np.arange(L - 256, L, dtype=np.int64)
    topk = synth.causal_topk(12, q_pos, 384)
    e = _check(w, _queries(256, 64, layer=8), np.zeros(256, np.int32), q_pos, topk, 0, LSE_TOL_TC)
    print(f"max rel err {e:.3e}")


def test_tensor_core_path_interleaved_sessions():
    # rows of three sessions interleaved: every row start loads a different sequence entry
    # (the producers prefetch them two rows ahead), some rows near their session's start
    lengths = [3000, 700, 1500]
    w = World(lengths, ring=512)
    T = 450
    q_seq = np.array([t % 3 for t in range(T)], np.int32)
    q_pos = np.array([(lengths[b] - 1 - 3 * (t // 3)) % lengths[b] for t, b in enumerate(q_seq)], np.int64)
    q_pos[3::47] = np.minimum(q_pos[3::47], 5)                 # a few rows with very short prefixes
    topk = synth.causal_topk(13, q_pos, 512)
    e = _check(w, _queries(T, 64, layer=9), q_seq, q_pos, topk, 128, LSE_TOL_TC)
    print(f"max rel err {e:.3e}")


def test_tensor_core_path_single_chunk_rows():
    # one step per row (top-k of at most 128, no window): row ends follow each other at every
    # step, so each row's read-out and the next rows' products interleave most tightly
    L = 3000
    w = World([L], ring=128)
    q_pos = np.arange(L - 300, L, dtype=np.int64)
    topk = synth.causal_topk(14, q_pos, 96)
    e = _check(w, _queries(300, 64, layer=10), np.zeros(300, np.int32), q_pos, topk, 0, LSE_TOL_TC)
    print(f"max rel err {e:.3e}")
