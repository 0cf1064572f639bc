"""GPU parity of kv_append_fp4 and its quantisers against the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import synth
from oracle import formats
from oracle.append import append_rows, swa_rows, quantize_fp4, quantize_fp8_token
from tests.gpu_util import dev, dev_bf16, host

pytestmark = pytest.mark.gpu

from tests.gpu_util import csa2


def test_fp4_quantiser_exhaustive_bf16_by_scale():
    # groups [6s, x1..x15]: amax exactly 6s, so the scale is exactly s; every bf16
    # magnitude up to 8s, both signs, for each of the 126 positive finite scales
    bits = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
    allx = synth.bf16_bits_to_f32(bits)
    groups = []
    for sc in range(1, 127):
        s = formats.E4M3_TABLE[sc]
        mag = allx[allx <= 8.0 * s]
        mag = np.concatenate([mag, -mag])
        n = -(-mag.shape[0] // 15)
        pad = np.zeros(n * 15, np.float32)
        pad[:mag.shape[0]] = mag
        g = np.empty((n, 16), np.float32)
        g[:, 0] = np.float32(6.0 * s)
        g[:, 1:] = pad.reshape(n, 15)
        groups.append(g)
    x = np.concatenate(groups)
    # the saturating elements (|x| > 6s) raise amax: keep them, the oracle sees the same groups
    codes = torch.empty((x.shape[0], 8), dtype=torch.uint8, device="cuda")
    scales = torch.empty((x.shape[0],), dtype=torch.uint8, device="cuda")
    csa2.test_quantize_fp4(dev(x), codes, scales)
    torch.cuda.synchronize()
    rows = np.zeros((x.shape[0], 128), np.float32)
    rows[:, :16] = x
    ref_c, ref_s = quantize_fp4(rows)
    assert np.array_equal(host(scales), ref_s[:, 0])
    assert np.array_equal(host(codes), ref_c[:, :8])
    assert x.shape[0] > 250_000


def test_fp4_quantiser_random_and_edge_groups():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((200000, 16)) * np.exp2(rng.integers(-14, 10, (200000, 1)))).astype(np.float32)
    x[:10] = 0.0
    x[10] = -0.0
    x[11, :] = 1e-30
    x[12, :] = 3e4
    x[13, 3] = -1e5
    codes = torch.empty((x.shape[0], 8), dtype=torch.uint8, device="cuda")
    scales = torch.empty((x.shape[0],), dtype=torch.uint8, device="cuda")
    csa2.test_quantize_fp4(dev(x), codes, scales)
    rows = np.zeros((x.shape[0], 128), np.float32)
    rows[:, :16] = x
    ref_c, ref_s = quantize_fp4(rows)
    assert np.array_equal(host(scales), ref_s[:, 0])
    assert np.array_equal(host(codes), ref_c[:, :8])


@pytest.mark.parametrize("C", [64, 128])
def test_fp8_token_quantiser(C):
    rng = np.random.default_rng(C)
    x = (rng.standard_normal((50000, C)) * np.exp2(rng.integers(-20, 12, (50000, 1)))).astype(np.float32)
    x[0] = 0.0
    x[1, :] = 7.0
    codes = torch.empty((x.shape[0], C), dtype=torch.uint8, device="cuda")
    scale = torch.empty((x.shape[0],), dtype=torch.float32, device="cuda")
    csa2.test_quantize_fp8(dev(x), codes, scale)
    rc, rs = quantize_fp8_token(x)
    assert np.array_equal(host(scale).view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(host(codes), rc)


def _small_cache(B, lengths, n_layers, ring, seed=0):
    T_cap = int(sum(((L + 15) // 16) * 16 for L in lengths))
    cache = csa2.Cache(T_cap, B)
    base = np.zeros(B, np.int64)
    base[1:] = np.cumsum([((L + 15) // 16) * 16 for L in lengths])[:-1]
    cache.seq_base.copy_(torch.from_numpy(base))
    cache.seq_len.copy_(torch.from_numpy(np.array(lengths, np.int32)))
    swa = [csa2.SwaRing(B, ring) for _ in range(n_layers)]
    return cache, swa, base


def test_append_bit_exact_with_rope_and_swa_layers():
    B, lengths, n_layers, ring = 3, [37, 300, 129], 3, 128
    cache, swa, base = _small_cache(B, lengths, n_layers, ring)
    for t in (cache.kv_codes, cache.kv_scales, cache.ik_codes):
        t.fill_(0xAB)
    rng = np.random.default_rng(3)
    # every token of every sequence in one shuffled batch
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lengths)])
    pos = np.concatenate([np.arange(L, dtype=np.int64) for L in lengths])
    perm = rng.permutation(seq.shape[0])
    seq, pos = seq[perm], pos[perm]
    rows = synth.row_id(seq, pos)
    oc = synth.outlier_channels(0, synth.Stream.KV_OUTLIER)
    kv = synth.normals_bf16(0, synth.Stream.KV, 0, rows, 128, oc)
    ik = synth.normals_bf16(0, synth.Stream.IK, 0, rows, 64)
    sw = np.stack([synth.normals_bf16(0, synth.Stream.SWA, l, rows, 128) for l in range(n_layers)])
    cos, sin = synth.rope_table(400)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the window rings only keep the last writes: append all tokens but SWA for the last ring positions only
    csa2.kv_append_fp4(cache, None, dev_bf16(kv), dev_bf16(ik), None, dev(cos), dev(sin), dev(seq), dev(pos), d_err)
    last = pos >= np.array(lengths)[seq] - ring
    csa2.kv_append_fp4(cache, swa, dev_bf16(kv[last]), None, dev_bf16(np.ascontiguousarray(sw[:, last])),
                       dev(cos), dev(sin), dev(seq[last]), dev(pos[last]), d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    kc, ks, ic, isc = append_rows(kv, ik, cos[pos], sin[pos])
    row = base[seq] + pos
    assert np.array_equal(host(cache.kv_codes)[row], kc)
    assert np.array_equal(host(cache.kv_scales)[row], ks)
    assert np.array_equal(host(cache.ik_codes)[row], ic)
    assert np.array_equal(host(cache.ik_scale)[row].view(np.uint32), isc.view(np.uint32))
    for l in range(n_layers):
        sc, ss = swa_rows(sw[l][last], cos[pos[last]], sin[pos[last]])
        b_, p_ = seq[last], pos[last]
        assert np.array_equal(host(swa[l].codes)[b_, p_ % ring], sc)
        assert np.array_equal(host(swa[l].scale)[b_, p_ % ring].view(np.uint32), ss.view(np.uint32))


def test_append_flags_bad_tokens_and_skips_them():
    cache, swa, base = _small_cache(2, [16, 16], 1, 16)
    cache.kv_codes.fill_(0x11)
    cos, sin = synth.rope_table(32)
    kv = synth.normals_bf16(0, synth.Stream.KV, 0, np.arange(3), 128)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seq = np.array([5, 0, 1], np.int32)        # bad sequence id
    pos = np.array([0, -1, 40], np.int64)      # negative, beyond the rope table
    csa2.kv_append_fp4(cache, None, dev_bf16(kv), None, None, dev(cos), dev(sin), dev(seq), dev(pos), d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == (csa2.DEVERR_SEQ | csa2.DEVERR_POS)
    assert torch.all(cache.kv_codes == 0x11)


def test_append_rejects_bad_arguments_before_launch():
    cache, swa, _ = _small_cache(1, [16], 1, 16)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cos, sin = synth.rope_table(16)
    kv = dev_bf16(synth.normals_bf16(0, synth.Stream.KV, 0, np.arange(2), 128))
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.kv_append_fp4(cache, None, kv.view(-1)[1:], None, None, dev(cos), dev(sin), dev(np.zeros(1, np.int32)),
                           dev(np.zeros(1, np.int64)), d_err)   # misaligned bf16 rows
    assert e.value.status == csa2.ERR_INVALID_ARG


def test_swa_refill_rebuilds_rings_bit_exact():
    # replay of the last window of each sequence into fresh rings; ring slots that no
    # replayed token maps to keep their old contents
    B, n_layers, ring = 3, 4, 128
    lengths = [37, 300, 1000]
    swa = [csa2.SwaRing(B, ring) for _ in range(n_layers)]
    for r in swa:
        r.codes.fill_(0x5A)
        r.scale.fill_(7.0)
    seq = np.concatenate([np.full(min(L, ring), b, np.int32) for b, L in enumerate(lengths)])
    pos = np.concatenate([np.arange(max(0, L - ring), L, dtype=np.int64) for L in lengths])
    rows = synth.row_id(seq, pos)
    soc = synth.outlier_channels(0, synth.Stream.SWA_OUTLIER)
    sw = np.stack([synth.normals_bf16(0, synth.Stream.SWA, l, rows, 128, soc) for l in range(n_layers)])
    cos, sin = synth.rope_table(1100)
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.swa_refill_fp8(swa, B, dev_bf16(sw), dev(cos), dev(sin), dev(seq), dev(pos), d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    for l in range(n_layers):
        sc, ss = swa_rows(sw[l], cos[pos], sin[pos])
        codes, scale = host(swa[l].codes), host(swa[l].scale)
        assert np.array_equal(codes[seq, pos % ring], sc)
        assert np.array_equal(scale[seq, pos % ring].view(np.uint32), ss.view(np.uint32))
        untouched = np.ones((B, ring), bool)
        untouched[seq, pos % ring] = False
        assert np.all(codes[untouched] == 0x5A) and np.all(scale[untouched] == 7.0)


def test_swa_refill_matches_the_append_window_bytes_and_flags_bad_tokens():
    B, n_layers, ring = 2, 2, 128
    cache, swa_a, _ = _small_cache(B, [200, 64], n_layers, ring)
    swa_r = [csa2.SwaRing(B, ring) for _ in range(n_layers)]
    seq = np.array([0, 1, 0, 1, 5], np.int32)          # the last token has a bad sequence id
    pos = np.array([199, 63, 150, 10, 3], np.int64)
    rows = synth.row_id(seq, pos)
    kv = synth.normals_bf16(1, synth.Stream.KV, 0, rows, 128)
    sw = np.stack([synth.normals_bf16(1, synth.Stream.SWA, l, rows, 128) for l in range(n_layers)])
    cos, sin = synth.rope_table(256)
    e1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    e2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.kv_append_fp4(cache, swa_a, dev_bf16(kv), None, dev_bf16(sw), dev(cos), dev(sin), dev(seq), dev(pos), e1)
    csa2.swa_refill_fp8(swa_r, B, dev_bf16(sw), dev(cos), dev(sin), dev(seq), dev(pos), e2)
    torch.cuda.synchronize()
    assert int(e1.item()) == csa2.DEVERR_SEQ and int(e2.item()) == csa2.DEVERR_SEQ
    for l in range(n_layers):
        assert torch.equal(swa_a[l].codes, swa_r[l].codes) and torch.equal(swa_a[l].scale, swa_r[l].scale)


def test_swa_refill_rejects_bad_arguments_before_launch():
    swa = [csa2.SwaRing(1, 128)]
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    cos = torch.zeros((4, 32), dtype=torch.float32, device="cuda")
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(csa2.Csa2Error):
        csa2.swa_refill_fp8([], 1, x, cos, cos, one, p, d_err)                    # no layers
    with pytest.raises(csa2.Csa2Error):
        csa2.swa_refill_fp8(swa, 0, x, cos, cos, one, p, d_err)                   # B < 1
