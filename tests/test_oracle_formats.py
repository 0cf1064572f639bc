"""Pins for the oracle's FP4 / FP8 codecs (CPU only).

Each test checks the oracle against something other than itself: the
published OCP value tables, hand-worked quantisation examples, torch's own
float8 conversion, or an exhaustive brute-force nearest-value search.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats
from oracle.append import quantize_fp4, dequant_fp4
from synth import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_e2m1_table_matches_published_values():
    g = _load("format_tables.json")
    assert list(formats.E2M1_TABLE[:8]) == g["e2m1_magnitudes"]
    assert list(-formats.E2M1_TABLE[8:]) == g["e2m1_magnitudes"]


def test_e4m3_table_points():
    g = _load("format_tables.json")
    for code, val in g["e4m3_points"].items():
        got = formats.E4M3_TABLE[int(code)]
        assert got == val and np.signbit(got) == np.signbit(val), code
    for code in g["e4m3_nan_codes"]:
        assert np.isnan(formats.E4M3_TABLE[code])
    finite = formats.E4M3_TABLE[~np.isnan(formats.E4M3_TABLE)]
    assert finite.max() == 448.0 and finite.shape[0] == 254
    pos = formats.E4M3_TABLE[:127]
    assert np.all(np.diff(pos) > 0)


def test_e4m3_rne_hand_cases():
    g = _load("format_tables.json")
    for x, code in g["e4m3_rne_cases"]:
        assert int(formats.e4m3_encode(np.float32(x))) == code, x


def test_e4m3_encode_matches_torch_on_every_bf16_and_random_f32():
    # torch's CPU float -> float8_e4m3fn conversion rounds to nearest even;
    # within the finite range the oracle must agree code for code.
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    x = bf16_bits_to_f32(bits)
    rng = np.random.default_rng(1)
    y = (rng.standard_normal(400000) * np.exp2(rng.integers(-12, 9, 400000))).astype(np.float32)
    for v in (x, y):
        v = v[np.isfinite(v) & (np.abs(v) <= 448.0)]
        ours = formats.e4m3_encode(v)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ours, ref)


def test_e4m3_saturates():
    assert int(formats.e4m3_encode(np.float32(1e6))) == 0x7E
    assert int(formats.e4m3_encode(np.float32(-1e6))) == 0xFE


def test_fp4_worked_examples():
    g = _load("fp4_worked_examples.json")
    for ex in g["examples"]:
        x = np.array(ex["x"], dtype=np.float32)
        assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(x)), x)  # bf16-exact inputs
        row = np.zeros((1, 128), dtype=np.float32)
        row[0, 16:32] = x                                   # group 1 of a token
        codes, scales = quantize_fp4(row)
        assert scales[0, 1] == ex["scale_code"], ex["name"]
        assert formats.E4M3_TABLE[scales[0, 1]] == ex["scale"]
        nib = np.empty(16, dtype=np.uint8)
        nib[0::2] = codes[0, 8:16] & 0xF
        nib[1::2] = codes[0, 8:16] >> 4
        assert list(nib) == ex["codes"], ex["name"]
        assert np.all(scales[0, [0, 2, 3, 4, 5, 6, 7]] == 0)


def _brute_e2m1(mag, s):
    """Nearest of the 8 grid points by exact distance, ties to the even code."""
    grid = formats.E2M1_TABLE[:8][None, :] * s[:, None]
    dist = np.abs(mag[:, None] - grid)                          # exact in float64
    best = dist.min(axis=1, keepdims=True)
    tied = dist == best
    # prefer an even code among the tied ones, else the single nearest
    even = tied & (np.arange(8)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), tied.argmax(axis=1))
    return pick.astype(np.uint8)


def test_e2m1_exhaustive_against_brute_force():
    # every positive finite E4M3 scale x every bf16 magnitude up to 8s (saturation included)
    bits = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)      # non-negative finite bf16
    allx = bf16_bits_to_f32(bits).astype(np.float64)
    allx = allx[np.isfinite(allx)]
    n_checked = 0
    for sc in range(1, 127):
        s = formats.E4M3_TABLE[sc]
        mag = allx[allx <= 8.0 * s]
        svec = np.full(mag.shape, s)
        ours = formats.e2m1_code_of_magnitude(mag, svec)
        ref = _brute_e2m1(mag, svec)
        assert np.array_equal(ours, ref), sc
        n_checked += mag.shape[0]
    assert n_checked > 1_000_000


def test_fp4_group_path_with_exact_scales():
    # a group whose amax is exactly 6s has scale exactly s; every other
    # element must land on the brute-force nearest grid point
    rng = np.random.default_rng(7)
    for sc in range(1, 127):
        s = formats.E4M3_TABLE[sc]
        xs = rng.uniform(-6 * s, 6 * s, size=(64, 16)).astype(np.float32)
        xs = bf16_bits_to_f32(f32_to_bf16_bits(xs))
        xs = np.clip(xs, -6 * s, 6 * s).astype(np.float32)
        xs[:, 0] = np.float32(6 * s)
        row = np.zeros((64, 128), dtype=np.float32)
        row[:, :16] = xs
        codes, scales = quantize_fp4(row)
        assert np.all(scales[:, 0] == sc)
        nib = np.empty((64, 16), dtype=np.uint8)
        nib[:, 0::2] = codes[:, :8] & 0xF
        nib[:, 1::2] = codes[:, :8] >> 4
        ref = _brute_e2m1(np.abs(xs).astype(np.float64).ravel(), np.full(64 * 16, s)).reshape(64, 16)
        ref = ref | (np.signbit(xs).astype(np.uint8) << 3)
        assert np.array_equal(nib, ref), sc


def test_fp4_properties_roundtrip_error_monotone():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2000, 128)) * 2).astype(np.float32)
    codes, scales = quantize_fp4(x)
    deq = dequant_fp4(codes, scales)
    s = np.repeat(formats.E4M3_TABLE[scales], 16, axis=1)
    # half of the widest gap (between 4 and 6) bounds the error unless saturated at 6s
    err = np.abs(deq - x)
    sat = np.abs(x) > 6 * s
    assert np.all(err[~sat] <= 1.0 * s[~sat] + 1e-30)
    # grid points reproduce exactly
    grid = formats.E2M1_TABLE[:8]
    pts = np.zeros((1, 128), dtype=np.float32)
    pts[0, :8] = grid * 1.0
    pts[0, 8] = 6.0
    c, sc = quantize_fp4(pts)
    assert np.array_equal(dequant_fp4(c, sc)[0, :9], pts[0, :9])
    # monotone in |x| within a group of fixed scale
    mags = np.linspace(0, 6, 1001, dtype=np.float32)
    codes_m = formats.e2m1_code_of_magnitude(mags.astype(np.float64), np.ones_like(mags, dtype=np.float64))
    assert np.all(np.diff(formats.E2M1_TABLE[codes_m]) >= 0)


@pytest.mark.parametrize("planted", ["tie_up", "no_saturate"])
def test_planted_codec_mistakes_are_caught(planted, monkeypatch):
    """A plausible slip in the midpoint rule must fail the brute-force pin."""
    good = formats.e2m1_code_of_magnitude

    def bad(mag, s):
        c = good(mag, s).astype(np.int64)
        mag = np.asarray(mag, dtype=np.float64)
        s = np.asarray(s, dtype=np.float64)
        if planted == "tie_up":             # ties at 0.75 s go up-odd instead of even
            c = np.where(mag == 0.75 * s, 1, c)
        else:                               # values beyond 6 s wrap instead of saturating
            c = np.where(mag > 6 * s, 0, c)
        return c.astype(np.uint8)

    s = 1.0
    mag = np.array([0.75, 7.0, 0.1, 2.0])
    assert np.array_equal(good(mag, np.full(4, s)), _brute_e2m1(mag, np.full(4, s)))
    assert not np.array_equal(bad(mag, np.full(4, s)), _brute_e2m1(mag, np.full(4, s)))
