"""fp64 CPU oracle of a low-precision latent cache.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests may import
it; the library never does, and it shares no code with the CUDA path.

What it follows: the DeepSeek-V2 analysis page (section 1.3 and 6.2) says
the cache is further quantised at deployment, to about 6 bits per element,
which with MLA's 576 elements gives the quoted 93.3 % saving; it gives no
number format, scale axis or grouping, and warns (section 6) that scales
must be taken along an axis the absorbed product does not mix.

Reading (plainest one the rest supports): the 512-element latent c_kv of a
token is stored as FP8 E4M3 values with one fp32 scale per group of 128
consecutive latent elements of that token (four scales per token); the
64-element shared RoPE key stays bf16.  The scale runs along the latent axis
of ONE token, so it commutes with the per-token weights a_s of the
aggregation and with the per-token dot product q_nope . c_s.

E4M3 (the 8-bit float of the OCP FP8 format, "E4M3FN"): 1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds
subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN, so the largest
finite value is 1.75 * 2^8 = 448.  Encoding rounds to nearest, ties to even,
and saturates finite values beyond +-448 to +-448.

Group scale: s = amax / 448 (amax = largest |x| of the group; s = 1 for an
all-zero group), rounded to fp32; code = E4M3(x / s) with the quotient x / s
rounded to fp32 first (the precision in which the quantising kernel takes
the same decision: an fp32 division, correctly rounded, then one rounding to
E4M3); value = E4M3 * s.  (Rounding the float64 quotient of two fp32 numbers
to fp32 gives the correctly rounded fp32 quotient, since 53 >= 2 * 24 + 2.)
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
GROUP = 128


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of E4M3 codes (uint8); NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code (ties to even code), finite values saturated to
    +-448, NaN to 0x7F.  Works by comparing against the exact value table,
    not by bit manipulation of the input."""
    x = np.asarray(x, dtype=np.float64)
    pos_codes = np.arange(0, 0x7F, dtype=np.uint8)          # 0x00 .. 0x7E: all finite non-negative values
    pos_vals = e4m3_decode(pos_codes)                       # strictly increasing
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(pos_vals, a, side="left"), 0, len(pos_vals) - 1)
    lo = np.clip(hi - 1, 0, len(pos_vals) - 1)
    d_lo = np.abs(a - pos_vals[lo])
    d_hi = np.abs(pos_vals[hi] - a)
    tie = d_lo == d_hi
    pick = np.where(d_lo < d_hi, lo, hi)
    pick = np.where(tie, np.where(pos_codes[lo] % 2 == 0, lo, hi), pick)   # even mantissa code wins
    code = pos_codes[pick].astype(np.uint8)
    code = np.where(np.signbit(x) & (code != 0), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def _round_f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def quantize_latent(c, group: int = GROUP):
    """c [..., d_c] -> (codes uint8 [..., d_c], scales float64 [..., d_c // group])."""
    c = np.asarray(c, dtype=np.float64)
    d_c = c.shape[-1]
    assert d_c % group == 0
    g = c.reshape(*c.shape[:-1], d_c // group, group)
    amax = np.max(np.abs(g), axis=-1)
    scale = _round_f32(np.where(amax > 0, amax / E4M3_MAX, 1.0))
    codes = e4m3_encode(_round_f32(g / scale[..., None]))
    return codes.reshape(c.shape), scale


def dequantize_latent(codes, scales, group: int = GROUP) -> np.ndarray:
    """Inverse of quantize_latent up to the E4M3 rounding: value * group scale."""
    codes = np.asarray(codes, dtype=np.uint8)
    d_c = codes.shape[-1]
    v = e4m3_decode(codes).reshape(*codes.shape[:-1], d_c // group, group)
    return (v * np.asarray(scales, dtype=np.float64)[..., None]).reshape(codes.shape)


def quantize_cache_rows(rows, d_c: int, group: int = GROUP):
    """576-element cache rows [..., d_c + d_r] -> (latent codes, scales, RoPE
    part unchanged) in the reading above."""
    rows = np.asarray(rows, dtype=np.float64)
    codes, scales = quantize_latent(rows[..., :d_c], group)
    return codes, scales, rows[..., d_c:]


def cache_bytes_per_token(d_c: int, d_r: int, group: int = GROUP) -> int:
    """Stored bytes of one token's row: d_c E4M3 + fp32 scales + bf16 RoPE."""
    return d_c + 4 * (d_c // group) + 2 * d_r
