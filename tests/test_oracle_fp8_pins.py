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
    # codes are e4m3(x * (448 / amax)) in fp32; dequantised values within half a quantum
    # (relative 2^-4) of the input, or 2^-10 s absolute, up to the fp32 roundings of r and s
    r = np.float32(448) / np.abs(x).max(axis=2)
    assert np.array_equal(codes, fp8.e4m3_encode((x * r[:, :, None]).astype(np.float32)))
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
