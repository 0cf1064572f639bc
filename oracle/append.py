"""Quantise-and-append of the decoder's global KV and SWA KV (oracle side).

Follows origotech.dev deep dive, subsection "FP4와 SWA Bounded Replay": the
main KV is stored in FP4 (E2M1, one E4M3 scale per 16 channels, quantised
after RoPE) and the SWA KV stays in FP8; trawling.dev "DeepSeek-V4.1-Flash
공개", section "CSA2와 FP4 KV 캐싱", gives the same format.

Readings where the pages are silent (each listed in the design notes):

* one 128-channel vector per token serves as both K and V (MQA); channels
  64..127 carry RoPE, rotated as interleaved pairs (64+2i, 65+2i) with the
  caller's cos/sin tables, in float32 without fused multiply-add;
* FP4 scale of a 16-channel group: s = E4M3(amax / 6) (IEEE float32 divide,
  round to nearest even, saturating), decoded back; each channel takes the
  nearest E2M1 magnitude of |r| / s (ties to even, saturating at 6) and the
  sign bit of r; s = 0 gives magnitude code 0;
* FP8 keys (indexer key, SWA KV): per-token float32 scale s = amax / 448 and
  codes E4M3(x / s) (IEEE float32 divide); s = 0 gives code 0;
* the indexer key carries no RoPE; the SWA vector gets the same RoPE as the
  main KV;
* nibble packing: byte j holds channel 2j in bits 0-3 and 2j+1 in bits 4-7.
"""
from __future__ import annotations

import numpy as np

from .formats import e4m3_encode, e4m3_decode, e2m1_code_of_magnitude

D = 128          # main KV channels
ROPE_LO = 64     # first rotated channel
D_IDX = 64       # indexer key channels
GROUP = 16       # channels per E4M3 scale


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate channels 64..127 of float32 rows x [n][128] by (cos, sin) [n][32].

    r0 = x0*c - x1*s and r1 = x0*s + x1*c, every product and sum rounded to
    float32 separately.
    """
    x = np.asarray(x, dtype=np.float32)
    r = x.copy()
    x0 = x[:, ROPE_LO::2]
    x1 = x[:, ROPE_LO + 1::2]
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    r[:, ROPE_LO::2] = np.subtract(np.multiply(x0, c, dtype=np.float32),
                                   np.multiply(x1, s, dtype=np.float32), dtype=np.float32)
    r[:, ROPE_LO + 1::2] = np.add(np.multiply(x0, s, dtype=np.float32),
                                  np.multiply(x1, c, dtype=np.float32), dtype=np.float32)
    return r


def quantize_fp4(r: np.ndarray):
    """float32 rows [n][128] -> (codes u8 [n][64], scales u8 [n][8])."""
    r = np.asarray(r, dtype=np.float32)
    n = r.shape[0]
    g = r.reshape(n, D // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=2)                                   # float32, exact
    s_code = e4m3_encode(np.divide(amax, np.float32(6.0), dtype=np.float32))
    s = e4m3_decode(s_code)                                            # scale round-trip
    mag = e2m1_code_of_magnitude(np.abs(g).astype(np.float64), s[:, :, None])
    code = mag | (np.signbit(g).astype(np.uint8) << 3)
    code = code.reshape(n, D)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_code.astype(np.uint8)


def quantize_fp8_token(x: np.ndarray):
    """float32 rows [n][C] -> (codes u8 [n][C], scale f32 [n]); scale = amax / 448."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=1)
    s = np.divide(amax, np.float32(448.0), dtype=np.float32)
    safe = np.where(s == 0, np.float32(1.0), s)
    y = np.divide(x, safe[:, None], dtype=np.float32)
    codes = e4m3_encode(y)
    codes = np.where((s == 0)[:, None], np.uint8(0), codes).astype(np.uint8)
    return codes, s.astype(np.float32)


def append_rows(kv_bf16, ik_bf16, cos, sin):
    """Main KV and indexer key of n tokens -> their cache rows.

    kv_bf16 [n][128] and ik_bf16 [n][64] are bf16 bit patterns; cos/sin are
    the rotation tables already indexed by each token's position ([n][32]).
    Returns (kv_codes [n][64], kv_scales [n][8], ik_codes [n][64], ik_scale [n]).
    """
    r = rope(bf16_to_f32(kv_bf16), cos, sin)
    kv_codes, kv_scales = quantize_fp4(r)
    ik_codes, ik_scale = quantize_fp8_token(bf16_to_f32(ik_bf16))
    return kv_codes, kv_scales, ik_codes, ik_scale


def swa_rows(swa_bf16, cos, sin):
    """SWA KV of n tokens (bf16 bits [n][128]) -> (codes u8 [n][128], scale f32 [n])."""
    return quantize_fp8_token(rope(bf16_to_f32(swa_bf16), cos, sin))


def dequant_fp4(codes, scales) -> np.ndarray:
    """Cache rows back to float64 [n][128]: E2M1 value times its group's scale (exact)."""
    from .formats import E2M1_TABLE
    codes = np.asarray(codes, dtype=np.uint8)
    n = codes.shape[0]
    nib = np.empty((n, D), dtype=np.uint8)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    vals = E2M1_TABLE[nib]
    s = e4m3_decode(scales)                                            # [n][8]
    return vals * np.repeat(s, GROUP, axis=1)


def dequant_fp8(codes, scale) -> np.ndarray:
    """FP8 rows back to float64: E4M3 value times the row's float32 scale."""
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[:, None]
