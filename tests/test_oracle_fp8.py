"""Pins of the FP8 (E4M3) oracle: the format's fixed points, a brute-force
nearest-code search, round trips, ties and saturation, and the fp8 branch of
the decode oracle."""

import numpy as np
import pytest

from oracle import fp8
from oracle.attention import paged_decode
from oracle.cache import bf16_to_f32, cache_append, cache_append_fp8, quantize_pool_fp8
from workloads import bf16_bits


def test_format_fixed_points():
    """Values the E4M3 format itself fixes (OCP 8-bit floating point
    specification): zero, smallest subnormal 2^-9, largest subnormal
    7·2^-9, smallest normal 2^-6, one, the largest finite 448, and the
    NaN codes; no infinities."""
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
            0x40: 2.0, 0x77: 240.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, val in want.items():
        assert fp8.decode(np.uint8(code)) == val, hex(code)
    assert np.isnan(fp8.decode(np.uint8(0x7F))) and np.isnan(fp8.decode(np.uint8(0xFF)))
    v = fp8.DECODE
    assert np.isfinite(v).sum() == 254 and np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    assert np.signbit(fp8.decode(np.uint8(0x80))) and fp8.decode(np.uint8(0x80)) == 0.0


def _nearest_code(x: float) -> int:
    """Brute force over all finite codes: the nearest value, ties to the
    code with an even mantissa; beyond ±448 the largest finite of that
    sign; NaN -> NaN code."""
    if np.isnan(x):
        return 0x7F
    sign = 0x80 if np.signbit(x) else 0
    a = abs(x)
    if a >= 448.0:
        return sign | 0x7E
    best, best_d = None, None
    for code in range(0x7F):  # non-negative finite codes
        d = abs(fp8.DECODE[code] - a)
        if best is None or d < best_d or (d == best_d and code % 2 == 0):
            best, best_d = code, d
    return sign | best


def test_encode_is_nearest_code_by_brute_force():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(30.0),
        rng.uniform(-0.03, 0.03, 1500).astype(np.float32),  # subnormal range and underflow
        rng.uniform(400, 500, 200).astype(np.float32),  # around saturation
        np.array([0.0, -0.0, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -10, 464.0, 480.0, 1e30, -1e30,
                  np.inf, -np.inf], dtype=np.float32),
    ])
    got = fp8.encode(xs)
    want = np.array([_nearest_code(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = fp8.decode(codes).astype(np.float32)  # every E4M3 value is exact in fp32
    assert np.array_equal(fp8.encode(vals), codes)


def test_midpoints_round_to_the_even_mantissa():
    pos = fp8.DECODE[:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # exact in fp32
    got = fp8.encode(mids)
    lo = np.arange(0x7E)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8))


def test_nan_and_saturation():
    got = fp8.encode(np.array([np.nan, 1e9, -1e9, 448.0, 447.9, -np.inf], dtype=np.float32))
    assert got[0] & 0x7F == 0x7F
    assert list(got[1:]) == [0x7E, 0xFE, 0x7E, 0x7E, 0xFE]


def test_quantize_divides_in_fp32():
    rng = np.random.default_rng(8)
    x = rng.standard_normal(500).astype(np.float32)
    for scale in (0.0173, 1.0 / 32, 3.0):
        q = fp8.quantize(x, scale)
        assert np.array_equal(q, fp8.encode(x / np.float32(scale)))
    # a power-of-two scale reproduces representable values exactly
    codes = np.arange(0x7F, dtype=np.uint8)
    assert np.array_equal(fp8.quantize(fp8.decode(codes).astype(np.float32) * np.float32(0.25), 0.25), codes)


def test_append_fp8_writes_codes_into_slots():
    rng = np.random.default_rng(9)
    k = bf16_bits(rng.standard_normal((5, 2, 16)).astype(np.float32))
    v = bf16_bits(rng.standard_normal((5, 2, 16)).astype(np.float32))
    slots = np.array([3, -1, 17, 0, 30], dtype=np.int64)
    kc = np.zeros((4, 2, 8, 16), dtype=np.uint8)
    vc = np.zeros_like(kc)
    k2, v2 = cache_append_fp8(kc, vc, k, v, slots, 0.05, 0.5)
    want_k, want_v = cache_append(kc, vc, fp8.quantize(bf16_to_f32(k), 0.05), fp8.quantize(bf16_to_f32(v), 0.5),
                                  slots)
    assert np.array_equal(k2, want_k) and np.array_equal(v2, want_v)
    assert k2[0, 1, 3, 5] == fp8.quantize(bf16_to_f32(k[0, 1, 5]), 0.05)
    pool = bf16_bits(rng.standard_normal((3, 2, 8, 16)).astype(np.float32))
    assert np.array_equal(quantize_pool_fp8(pool, 0.05), fp8.quantize(bf16_to_f32(pool), 0.05))


def test_decode_oracle_reads_codes_times_scale():
    """The fp8 branch equals the fp64 decode of the dequantized caches, and a
    single-token context returns that token's dequantized value."""
    rng = np.random.default_rng(10)
    n_blk, hkv, b, d, h = 6, 2, 4, 8, 4
    kc = rng.integers(0, 256, size=(n_blk, hkv, b, d)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(n_blk, hkv, b, d)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x11  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x22
    q = bf16_bits(rng.standard_normal((2, h, d)).astype(np.float32))
    tables = np.array([[5, 0, 3], [2, 4, 1]], dtype=np.int32)
    ctx = np.array([11, 1], dtype=np.int32)
    ks, vs = 0.03, 0.2
    got = paged_decode(q, kc, vc, tables, ctx, 0.7, "bf16", cache_dtype="fp8", k_scale=ks, v_scale=vs)
    qf = bf16_to_f32(q).astype(np.float64)
    want = paged_decode(qf, fp8.decode(kc) * ks, fp8.decode(vc) * vs, tables, ctx, 0.7, "f64")
    np.testing.assert_array_equal(got, want)
    for hh in range(h):
        assert np.array_equal(got[1, hh], fp8.decode(vc[2, hh // 2, 0]) * vs)


def _encode_ties_up(x):
    """Ties rounded away from zero instead of to the even mantissa."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    pos = fp8.DECODE[:0x7F]
    lo = np.clip(np.searchsorted(pos, a, side="right") - 1, 0, 0x7D)
    take_hi = (pos[lo + 1] - a) <= (a - pos[lo])
    mag = np.where(a >= 448.0, 0x7E, np.where(take_hi, lo + 1, lo)).astype(np.uint8)
    return mag | (np.signbit(x).astype(np.uint8) << np.uint8(7))


def _encode_no_saturation(x):
    """Quotients beyond 448 stored as NaN."""
    out = _orig_encode(x)
    out[np.abs(np.asarray(x, dtype=np.float64)) > 448.0] |= 0x7F
    return out


_orig_encode = fp8.encode
_PINS = [test_format_fixed_points, test_encode_is_nearest_code_by_brute_force, test_round_trip_of_every_finite_code,
         test_midpoints_round_to_the_even_mantissa, test_nan_and_saturation, test_quantize_divides_in_fp32,
         test_decode_oracle_reads_codes_times_scale]


@pytest.mark.parametrize("bad", ["bias", "subnormal_step", "ties_up", "no_saturation"])
def test_planted_codec_mistakes_are_caught(monkeypatch, bad):
    """The codec with a wrong exponent bias, a wrong subnormal step, ties
    rounded up, or no saturation fails at least one pin above."""
    if bad == "bias":
        monkeypatch.setattr(fp8, "DECODE", fp8.DECODE * 2.0)
    elif bad == "subnormal_step":
        table = fp8.DECODE.copy()
        table[1:8] *= 2.0
        table[0x81:0x88] *= 2.0
        monkeypatch.setattr(fp8, "DECODE", table)
    elif bad == "ties_up":
        monkeypatch.setattr(fp8, "encode", _encode_ties_up)
    else:
        monkeypatch.setattr(fp8, "encode", _encode_no_saturation)
    failed = 0
    for pin in _PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1


def test_fp8_serving_loop_equals_attention_over_dequantized_history():
    """Serving steps with an E4M3 cache: every output equals dense attention
    (scipy softmax) over each sequence's token history, each token read back
    as decode(quantize(x)) · scale and kept contiguously by the test."""
    import scipy.special

    from oracle.serving import ServingOracle, initial_state

    rng = np.random.default_rng(24)
    b, hkv, d, h, s = 4, 2, 8, 4, 3
    ctx = np.array([5, 9, 2], dtype=np.int32)
    nblk, ks, vs = 20, 0.02, 0.3
    alloc, pairs = initial_state(s, b, ctx, nblk, rng.permutation(nblk))
    kc = fp8.quantize(rng.standard_normal((nblk, hkv, b, d)).astype(np.float32), ks)
    vc = fp8.quantize(rng.standard_normal((nblk, hkv, b, d)).astype(np.float32), vs)
    hist_k, hist_v = [], []
    for i in range(s):
        t = alloc.block_table(i)
        n = alloc.num_tokens(i)
        hist_k.append(fp8.decode(kc[t]).transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :n] * ks)
        hist_v.append(fp8.decode(vc[t]).transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :n] * vs)
    srv = ServingOracle(alloc, kc, vc, s, "bf16", 0.4, fp8_scales=(ks, vs))
    for step in range(5):
        q = bf16_bits(rng.standard_normal((s, h, d)).astype(np.float32))
        kn = bf16_bits(rng.standard_normal((s, hkv, d)).astype(np.float32))
        vn = bf16_bits(rng.standard_normal((s, hkv, d)).astype(np.float32))
        _, _, out = srv.step(q, kn, vn, width=8)
        qf = bf16_to_f32(q).astype(np.float64)
        for i in range(s):
            hist_k[i] = np.concatenate([hist_k[i], (fp8.decode(fp8.quantize(bf16_to_f32(kn[i]), ks)) * ks)[:, None]],
                                       axis=1)
            hist_v[i] = np.concatenate([hist_v[i], (fp8.decode(fp8.quantize(bf16_to_f32(vn[i]), vs)) * vs)[:, None]],
                                       axis=1)
            for hh in range(h):
                p = scipy.special.softmax(0.4 * hist_k[i][hh // 2] @ qf[i, hh])
                np.testing.assert_allclose(out[i, hh], hist_v[i][hh // 2].T @ p, rtol=0, atol=1e-12)
