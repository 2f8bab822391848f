"""Pins for the FP8 oracle (oracle/fp8.py): the e4m3 format against its
definition and a brute-force nearest-code search, and the quantisers against
closed forms.  CPU only."""
import numpy as np
import pytest

from oracle import fp8

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def test_named_codes_decode():
    named = {0x00: 0.0, 0x38: 1.0, 0x39: 1.125, 0x3C: 1.5, 0x40: 2.0, 0x30: 0.5, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x80: -0.0}
    for c, val in named.items():
        assert fp8.e4m3_decode(np.array([c]))[0] == val, hex(c)
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_round_trip_every_finite_code():
    vals = fp8.e4m3_decode(FINITE)
    back = fp8.e4m3_encode(vals.astype(np.float32))
    # -0 encodes as 0x80, +0 as 0x00: compare values, and codes for the nonzero ones
    assert np.array_equal(fp8.e4m3_decode(back), vals)
    nz = vals != 0
    assert np.array_equal(back[nz], FINITE[nz])


def _brute(y):
    """nearest finite code, ties to the even mantissa, saturating"""
    vals = fp8.e4m3_decode(FINITE)
    out = []
    for t in y:
        t = float(np.clip(t, -448.0, 448.0))
        d = np.abs(vals - t)
        best = np.flatnonzero(d == d.min())
        cand = [c for c in FINITE[best] if (fp8.e4m3_decode(np.array([c]))[0] != 0 or np.signbit(t) == bool(c & 0x80))]
        if len(cand) > 1:
            cand = [c for c in cand if (c & 1) == 0]
        out.append(cand[0])
    return np.array(out, dtype=np.uint8)


def test_encode_matches_brute_force():
    rng = np.random.default_rng(0)
    y = np.concatenate([rng.standard_normal(2000) * 50, rng.standard_normal(500) * 0.01,
                        rng.uniform(-500, 500, 500), rng.standard_normal(300) * 1e-3]).astype(np.float32)
    got = fp8.e4m3_encode(y)
    want = _brute(y.astype(np.float64))
    assert np.array_equal(fp8.e4m3_decode(got), fp8.e4m3_decode(want))


def test_ties_go_to_even_and_saturation():
    mid = lambda a, b: (fp8.e4m3_decode(np.array([a]))[0] + fp8.e4m3_decode(np.array([b]))[0]) / 2
    assert fp8.e4m3_encode(np.array([mid(0x38, 0x39)], np.float32))[0] == 0x38
    assert fp8.e4m3_encode(np.array([mid(0x39, 0x3A)], np.float32))[0] == 0x3A
    assert fp8.e4m3_encode(np.array([mid(0x00, 0x01)], np.float32))[0] == 0x00     # 2^-10 -> 0
    assert fp8.e4m3_encode(np.array([mid(0x07, 0x08)], np.float32))[0] == 0x08     # subnormal/normal tie
    assert fp8.e4m3_encode(np.array([464.0, 1e9, -1e9], np.float32)).tolist() == [0x7E, 0x7E, 0xFE]


def test_quantisers_closed_forms():
    rng = np.random.default_rng(3)
    S, H, D = 300, 2, 128
    x = rng.standard_normal((S, H, D)).astype(np.float32)
    codes, s = fp8.quantize_rows(x)
    # every row's largest magnitude maps to (nearly) 448, scales are amax / 448 in fp32
    assert np.array_equal(s, (np.abs(x).max(axis=2) / np.float32(448)).T)
    top = np.abs(fp8.e4m3_decode(codes)).max(axis=2)
    assert np.all(np.abs(top - 448) <= 16)
    # every dequantised value within half a quantum (relative 2^-4, or 2^-10 s in
    # the subnormal range) of its input, up to the fp32 roundings of r, s and x * r
    deq = fp8.e4m3_decode(codes) * s.T[:, :, None]
    err = np.abs(deq - x)
    assert np.all(err <= (2.0 ** -4 + 2.0 ** -20) * np.abs(x) + 2.0 ** -10 * s.T[:, :, None] + 1e-12)
    # key tiles follow document boundaries; channels span all tokens
    cu = np.array([0, 130, 131, 300])
    assert fp8.key_tiles(cu) == [(0, 128), (128, 130), (130, 131), (131, 259), (259, 300)]
    k8, sk = fp8.quantize_key_tiles(x, cu)
    assert np.array_equal(sk[:, 128], sk[:, 129]) and sk[0, 128] == np.float32(np.abs(x[128:130, 0]).max()) / np.float32(448)
    v8, sv = fp8.quantize_channels(x)
    assert sv.shape == (H, D) and np.array_equal(sv, np.abs(x).max(axis=0) / np.float32(448))
    # an all-zero row takes scale 1 and zero codes
    z = x.copy(); z[5, 1] = 0
    c2, s2 = fp8.quantize_rows(z)
    assert s2[1, 5] == 1.0 and not c2[5, 1].any()


def _clear_of_boundaries(y):
    """Elements whose magnitude is more than one fp32 ulp away from every
    e4m3 rounding boundary (the midpoints between neighbouring finite
    magnitudes): there fp32 rounding of the product cannot change the code."""
    mags = np.unique(np.abs(fp8.e4m3_decode(FINITE)))
    mids = (mags[:-1] + mags[1:]) / 2
    a = np.abs(y)
    i = np.searchsorted(mids, a)
    lo = mids[np.clip(i - 1, 0, mids.size - 1)]
    hi = mids[np.clip(i, 0, mids.size - 1)]
    dist = np.minimum(np.abs(a - lo), np.abs(a - hi))
    return dist > np.spacing(a.astype(np.float32)).astype(np.float64)


def test_row_codes_are_the_nearest_codes_of_the_exact_product():
    # Fixed by the format alone, not by the oracle's formula: with amax the
    # row's largest magnitude, each code is the e4m3 value nearest to the
    # exact product x * 448 / amax (brute-force search over all finite codes),
    # wherever that product is more than one fp32 ulp from a rounding
    # boundary; there the dequantised value is within half a quantum of x:
    # 2^-4 |x| (normal codes) or 2^-10 s (subnormal codes), without widening.
    rng = np.random.default_rng(11)
    S, H, D = 96, 2, 128
    x = (rng.standard_normal((S, H, D)) * np.exp(rng.uniform(-3, 3, (S, H, 1)))).astype(np.float32)
    x[3, 0, 7] = 0.0
    codes, s = fp8.quantize_rows(x)
    amax = np.abs(x).astype(np.float64).max(axis=2)
    y = x.astype(np.float64) * (448.0 / amax)[:, :, None]
    clear = _clear_of_boundaries(y)
    assert clear.mean() > 0.99
    want = _brute(y[clear])
    assert np.array_equal(fp8.e4m3_decode(codes[clear]), fp8.e4m3_decode(want))
    deq = fp8.e4m3_decode(codes) * s.T[:, :, None].astype(np.float64)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s.T[:, :, None])
    assert np.all(np.abs(deq - x)[clear] <= bound[clear])


def test_key_tile_and_channel_codes_are_the_nearest_codes_of_the_exact_product():
    # the same pin for the per-key-tile and per-channel quantisers
    rng = np.random.default_rng(12)
    S, H, D = 300, 2, 32
    x = rng.standard_normal((S, H, D)).astype(np.float32) * np.float32(3.0)
    cu = np.array([0, 130, 131, 300])
    k8, sk = fp8.quantize_key_tiles(x, cu)
    y = np.zeros(x.shape)
    for a, b in fp8.key_tiles(cu):
        amax = np.abs(x[a:b]).astype(np.float64).max(axis=(0, 2))
        y[a:b] = x[a:b].astype(np.float64) * (448.0 / amax)[None, :, None]
    clear = _clear_of_boundaries(y)
    assert np.array_equal(fp8.e4m3_decode(k8[clear]), fp8.e4m3_decode(_brute(y[clear])))
    v8, sv = fp8.quantize_channels(x)
    yv = x.astype(np.float64) * (448.0 / np.abs(x).astype(np.float64).max(axis=0))[None]
    clear = _clear_of_boundaries(yv)
    assert np.array_equal(fp8.e4m3_decode(v8[clear]), fp8.e4m3_decode(_brute(yv[clear])))


def test_row_pin_catches_a_truncating_encoder(monkeypatch):
    # a plausible mistake -- rounding the product toward zero instead of to
    # nearest -- fails the nearest-code pin
    real = fp8.e4m3_encode

    def truncating(y):
        y = np.asarray(y, dtype=np.float64)
        c = real(y)
        v = fp8.e4m3_decode(c)
        over = np.abs(v) > np.abs(y)
        down = np.where(c & 0x7F, c - 1, c).astype(np.uint8)
        return np.where(over, down, c).astype(np.uint8)

    monkeypatch.setattr(fp8, "e4m3_encode", truncating)
    with pytest.raises(AssertionError):
        test_row_codes_are_the_nearest_codes_of_the_exact_product()


def test_error_bound_covers_p_rounding():
    # a brute-force emulation of P rounding on a small case stays inside the bound
    rng = np.random.default_rng(9)
    L, D = 200, 128
    q = rng.standard_normal((L, 1, D)); k = rng.standard_normal((L, 1, D)) * 0.3; v = rng.standard_normal((L, 1, D))
    cu = np.array([0, L]); scale = 1 / np.sqrt(D)
    s = (q[:, 0] @ k[:, 0].T) * scale
    p = np.exp2(s * np.log2(np.e) - (s * np.log2(np.e)).max(axis=1, keepdims=True) + rng.uniform(0, 8, (L, 1)))
    p8 = fp8.e4m3_decode(fp8.e4m3_encode(p.astype(np.float32)))
    o_k = (p8 @ v[:, 0]) / p.sum(axis=1, keepdims=True)
    o_x = (p @ v[:, 0]) / p.sum(axis=1, keepdims=True)
    bound = fp8.error_bound(q, k, v, cu, scale, [0], np.arange(L))[:, 0]
    assert np.all(np.abs(o_k - o_x) <= bound)
