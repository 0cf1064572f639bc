"""Pins for the oracle's RoPE, FP8 quantiser and the input generator (CPU only)."""
import numpy as np

import synth
from oracle import formats
from oracle.append import (rope, quantize_fp8_token, append_rows, dequant_fp4,
                           dequant_fp8, bf16_to_f32)


def test_rope_position_zero_is_identity():
    cos, sin = synth.rope_table(1)
    assert np.all(cos == 1.0) and np.all(sin == 0.0)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    r = rope(x, np.repeat(cos, 4, 0), np.repeat(sin, 4, 0))
    assert np.array_equal(r, x)


def test_rope_matches_complex_rotation():
    # (x0 + i x1)(c + i s) in float64 agrees with the float32 rotation to a few ulps
    cos, sin = synth.rope_table(5000)
    rng = np.random.default_rng(1)
    pos = rng.integers(0, 5000, 256)
    x = rng.standard_normal((256, 128)).astype(np.float32)
    r = rope(x, cos[pos], sin[pos])
    z = (x[:, 64::2].astype(np.float64) + 1j * x[:, 65::2]) * (cos[pos] + 1j * sin[pos].astype(np.float64))
    assert np.allclose(r[:, 64::2], z.real, rtol=0, atol=4e-7 * np.abs(x).max() * 2)
    assert np.allclose(r[:, 65::2], z.imag, rtol=0, atol=4e-7 * np.abs(x).max() * 2)
    assert np.array_equal(r[:, :64], x[:, :64])
    # rotation keeps the norm of each pair to float32 rounding
    n0 = np.hypot(x[:, 64::2], x[:, 65::2])
    n1 = np.hypot(r[:, 64::2], r[:, 65::2])
    assert np.allclose(n0, n1, rtol=3e-7 * 4, atol=1e-30)


def test_rope_table_angles():
    cos, sin = synth.rope_table(70000)
    p, i = 65537, 5
    ang = p * 10000.0 ** (-2 * i / 64)
    assert cos[p, i] == np.float32(np.cos(ang)) and sin[p, i] == np.float32(np.sin(ang))


def test_fp8_token_quantiser_pins():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((500, 64)).astype(np.float32)
    x[7] = 0.0
    codes, s = quantize_fp8_token(x)
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(448)).astype(np.float32))
    assert np.all(codes[7] == 0) and s[7] == 0
    # the amax element always lands on +-448
    arg = np.abs(x).argmax(axis=1)
    top = codes[np.arange(500), arg]
    assert np.all((top[np.arange(500) != 7] & 0x7F) == 0x7E)
    # relative error of E4M3 normals is at most 2^-4
    deq = dequant_fp8(codes, s)
    big = np.abs(x) > 2 ** -6 * s[:, None] * 1.01
    assert np.all(np.abs(deq - x)[big] <= 2 ** -4 * np.abs(x)[big] + 1e-30)


def test_fp8_matches_torch_float8_on_scaled_rows():
    rng = np.random.default_rng(4)
    import torch
    x = rng.standard_normal((300, 128)).astype(np.float32)
    codes, s = quantize_fp8_token(x)
    y = x / s[:, None]
    ref = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_append_rows_position_zero_reduces_to_quantisers():
    cos, sin = synth.rope_table(1)
    kv = synth.normals_bf16(0, synth.Stream.KV, 0, np.arange(8), 128, outliers=(3, 99))
    ik = synth.normals_bf16(0, synth.Stream.IK, 0, np.arange(8), 64)
    kc, ks, ic, isc = append_rows(kv, ik, np.repeat(cos, 8, 0), np.repeat(sin, 8, 0))
    deq = dequant_fp4(kc, ks)
    x = bf16_to_f32(kv).astype(np.float64)
    s = np.repeat(formats.E4M3_TABLE[ks], 16, axis=1)
    assert np.all(np.abs(deq - x) <= s * 1.0 + 1e-30)
    assert kc.shape == (8, 64) and ks.shape == (8, 8) and ic.shape == (8, 64) and isc.shape == (8,)


def test_synth_determinism_and_distribution():
    a = synth.normals_bf16(0, synth.Stream.KV, 0, synth.row_id(3, np.arange(1000)), 128)
    b = synth.normals_bf16(0, synth.Stream.KV, 0, synth.row_id(3, np.arange(1000)), 128)
    c = synth.normals_bf16(1, synth.Stream.KV, 0, synth.row_id(3, np.arange(1000)), 128)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    # a row does not depend on which other rows are generated with it
    d = synth.normals_bf16(0, synth.Stream.KV, 0, synth.row_id(3, np.array([500, 17])), 128)
    assert np.array_equal(d, a[[500, 17]])
    v = bf16_to_f32(synth.normals_bf16(0, synth.Stream.IK, 0, np.arange(20000), 64)).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    oc = synth.outlier_channels(0, synth.Stream.KV_OUTLIER)
    big = bf16_to_f32(synth.normals_bf16(0, synth.Stream.KV, 0, np.arange(20000), 128, outliers=oc))
    stds = big.astype(np.float64).std(axis=0)
    assert len(oc) == 2 and np.all(np.abs(stds[list(oc)] - 8) < 0.3)
    assert np.all(np.abs(np.delete(stds, list(oc)) - 1) < 0.05)
    w = synth.head_weights(0, 0, 0)
    assert w.dtype == np.float32 and np.all((w > 0) & (w <= 1))


def test_ragged_lengths_and_causal_topk():
    L = synth.ragged_lengths(0, 64)
    assert L.min() >= 4096 and L.max() <= 1048576
    idx = synth.causal_topk(0, np.array([100, 5000, 262143]), 512)
    assert np.array_equal(idx[0, :101], np.arange(101)) and np.all(idx[0, 101:] == -1)
    for t, p in ((1, 5000), (2, 262143)):
        row = idx[t]
        assert row.shape == (512,) and np.all(np.diff(row) > 0) and row.max() <= p and row.min() >= 0
