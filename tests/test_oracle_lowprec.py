"""Pins of the low-precision cache oracle (E4M3 latent with per-128-group
scales, bf16 RoPE key): the number format's defining values, round-to-
nearest-even against brute force over the whole code table, saturation,
the quantisation error bounds, and exactness on representable inputs."""
import numpy as np
import pytest

from oracle import lowprec_cache as L
import oracle as O


def test_e4m3_defining_values():
    d = L.e4m3_decode
    assert d(0x38) == 1.0 and d(0x30) == 0.5 and d(0x40) == 2.0
    assert d(0x7E) == 448.0                      # largest finite: 1.75 * 2^8
    assert d(0x77) == 240.0                      # 1.875 * 2^7
    assert d(0x08) == 2.0 ** -6                  # smallest normal
    assert d(0x01) == 2.0 ** -9                  # smallest subnormal: 1/8 * 2^-6
    assert d(0x07) == 7 / 8 * 2.0 ** -6          # largest subnormal
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x00) == 0.0 and d(0x80) == 0.0 and np.signbit(d(0x80))


def test_e4m3_table_is_monotone_and_symmetric():
    pos = L.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)              # 127 distinct non-negative finite values
    neg = L.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg[1:], -pos[1:])


def test_e4m3_round_trip_of_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    assert np.array_equal(L.e4m3_encode(L.e4m3_decode(codes)), codes)
    assert L.e4m3_encode(-0.0) == 0x00 and L.e4m3_encode(np.nan) == 0x7F


def test_e4m3_nearest_against_brute_force_and_ties_to_even():
    table = L.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(0, 448, 20000), np.exp2(rng.uniform(-12, 9, 20000))])
    x = np.minimum(x, 448.0)
    got = L.e4m3_decode(L.e4m3_encode(x))
    best = np.min(np.abs(table[None, :] - x[:, None]), axis=1)
    assert np.all(np.abs(got - x) == best)
    # every midpoint between neighbours goes to the code with an even mantissa
    mids = (table[:-1] + table[1:]) / 2
    codes = L.e4m3_encode(mids)
    assert np.all(codes % 2 == 0)
    assert np.all((codes == np.arange(0, 0x7E)) | (codes == np.arange(1, 0x7F)))
    # negative side mirrors the positive one (a value that rounds to zero
    # encodes as +0 either way)
    pos_code = L.e4m3_encode(x)
    assert np.array_equal(L.e4m3_encode(-x), np.where(pos_code != 0, pos_code | 0x80, 0))


def test_e4m3_saturates_finite_overflow():
    assert L.e4m3_encode(460.0) == 0x7E and L.e4m3_encode(1e9) == 0x7E
    assert L.e4m3_encode(-1e9) == 0xFE


@pytest.mark.parametrize("seed", [1, 2])
def test_quantize_latent_error_bounds(seed):
    rng = np.random.default_rng(seed)
    c = rng.standard_normal((16, 512)) * np.exp2(rng.uniform(-8, 8, (16, 1)))
    codes, scales = L.quantize_latent(c)
    assert codes.shape == (16, 512) and scales.shape == (16, 4)
    back = L.dequantize_latent(codes, scales)
    g = c.reshape(16, 4, 128)
    s = scales[..., None]
    err = np.abs(back.reshape(16, 4, 128) - g)
    normal = np.abs(g) / s >= 2.0 ** -6
    # normal range: half an ulp of 3 mantissa bits, relative to the value
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(g[normal]) * (1 + 1e-9))
    # subnormal range: half the subnormal step, in units of the group scale
    assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(s, g.shape)[~normal] * (1 + 1e-9))
    # each group's largest magnitude lands on +-448 * scale up to the fp32 scale rounding
    idx = np.argmax(np.abs(g), axis=-1)
    top = np.take_along_axis(back.reshape(16, 4, 128), idx[..., None], -1)[..., 0]
    amax = np.take_along_axis(g, idx[..., None], -1)[..., 0]
    assert np.all(np.abs(top - amax) <= 2.0 ** -4 * np.abs(amax))


def test_quantize_is_exact_on_representable_rows_and_zero_groups():
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 0x7F, (8, 512)).astype(np.uint8) | (rng.integers(0, 2, (8, 512)) * 0x80).astype(np.uint8)
    codes = np.where(codes == 0xFF, 0x7E, np.where(codes == 0x7F, 0x7E, codes)).astype(np.uint8)
    codes[:, ::128] = 0x7E                       # each group holds +448 once: its scale is exact
    k = np.exp2(rng.integers(-6, 6, (8, 4)))
    c = (L.e4m3_decode(codes).reshape(8, 4, 128) * k[..., None]).reshape(8, 512)
    c[3, 128:256] = 0.0                          # an all-zero group
    got_codes, got_scales = L.quantize_latent(c)
    back = L.dequantize_latent(got_codes, got_scales)
    assert np.array_equal(back, c)
    assert got_scales[3, 1] == 1.0 and np.all(got_codes[3, 128:256] == 0)


def test_decode_over_a_representable_quantized_cache_is_exact():
    # quantisation that loses nothing leaves the attention unchanged
    rng = np.random.default_rng(11)
    S, H = 40, 4
    codes = rng.integers(0, 0x70, (S, 512)).astype(np.uint8)
    codes[:, ::128] = 0x7E
    C = L.e4m3_decode(codes) * 2.0 ** -8          # group amax 1.75: scale exactly 2^-8
    R = rng.standard_normal((S, 64))
    qn, qr = rng.standard_normal((H, 512)), rng.standard_normal((H, 64))
    codes2, scales, rope = L.quantize_cache_rows(np.concatenate([C, R], 1), 512)
    Cq = L.dequantize_latent(codes2, scales)
    o1, l1, _ = O.decode_row(C, R, qn, qr, 0.07)
    o2, l2, _ = O.decode_row(Cq, rope, qn, qr, 0.07)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_bytes_per_token_of_the_reading():
    assert L.cache_bytes_per_token(512, 64) == 512 + 16 + 128 == 656
    # against 1,152 bytes in bf16: 43 % fewer bytes to stream per token
    assert abs(1 - 656 / 1152 - 0.4306) < 1e-3
