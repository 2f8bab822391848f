"""Oracle: the FP8 (e4m3) variant of the attention step.  Test infrastructure
only (imported by tests/, smoke() and bench.py's CPU legs, never by the
product path).

Pages: vllm.cpp PR #26 "feat(minimax-h3)" and the "h3-spark" model card,
"What this config does", name a SageAttention2++-style low-precision
attention (INT8/FP8 QK and PV) without giving its scheme.  Reading taken here,
the plainest scheme that uses sm_103's FP8 tensor cores for both products:

  quantisation (scales and codes decided in fp32, as the kernel does):
    q-hat: one scale per (token, head) row     s_q = amax_d |q| / 448
    k-hat: one scale per (head, 128-key tile of a document: tokens
           [a + 128 j, min(a + 128 j + 128, b)) of document [a, b))
           s_k = amax over the tile's tokens and dims / 448
    v:     one scale per (head, channel) over all S tokens
           s_v = amax_t |v| / 448
    code = e4m3(x * r) with r = 448 / amax (one fp32 division per row, tile
    or channel), x * r one fp32 product (round to nearest even), and e4m3
    round-to-nearest-even with saturation to +-448; an all-zero row, tile or
    channel takes s = r = 1.  Dequantisation multiplies the code by s.
  the attention it approximates: exact softmax attention (two-pass, fp64) on
    the dequantised values q~ = code_q s_q, k~ = code_k s_k, v~ = code_v s_v.
    The kernel additionally rounds the probabilities P to e4m3 for the PV
    product (|P| <= 2^8, no scale), so it is held to a per-element bound
    derived from that rounding (``error_bound``).

e4m3 (the "FN" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
exponent field 0 holds subnormals m/8 * 2^-6; the largest finite value is
1.75 * 2^8 = 448 (exponent 15, mantissa 6); exponent 15 with mantissa 7 is
NaN; there is no infinity.

Parity: pinned (decode of named codes, encode/decode round trip over every
finite code, ties to even, saturation, and encode against a brute-force
nearest-code search).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Exact values (fp64) of e4m3 codes (uint8); NaN for the NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Round fp32 values to e4m3 codes: nearest, ties to even mantissa,
    magnitudes above 448 saturate to 448.  Inputs are finite."""
    y = np.asarray(y, dtype=np.float64)
    neg = np.signbit(y)
    a = np.minimum(np.abs(y), E4M3_MAX)
    # exponent of the binade (subnormals share the quantum of the lowest binade)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))
    n = a / quantum                      # exact: quantum is a power of two
    r = np.floor(n)
    frac = n - r
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2) == 1))
    r = r + up
    # r counts quanta within the binade: 8..16 for normals (16 = next binade), 0..8 for subnormals
    val = r * quantum
    e2 = np.floor(np.log2(np.where(val > 0, val, 1.0)))
    e2 = np.maximum(e2, -6.0)
    is_sub = val < 2.0 ** -6
    mant = np.where(is_sub, np.round(val / 2.0 ** -9), np.round(val / np.ldexp(1.0, (e2 - 3).astype(np.int64))) - 8)
    exp_field = np.where(is_sub, 0, e2 + 7)
    code = (exp_field.astype(np.int64) << 3) | mant.astype(np.int64)
    code = np.where(val == 0, 0, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def _scale(amax: np.ndarray) -> np.ndarray:
    """dequantisation scale s = amax / 448 (fp32; 1 for amax = 0)"""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = amax / np.float32(E4M3_MAX)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def _recip(amax: np.ndarray) -> np.ndarray:
    """quantisation factor r = 448 / amax (fp32; 1 for amax = 0)"""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.float32(E4M3_MAX) / amax
    return np.where(amax > 0, r, np.float32(1.0)).astype(np.float32)


def _codes(x: np.ndarray, r: np.ndarray) -> np.ndarray:
    y = np.asarray(x, dtype=np.float32) * np.asarray(r, dtype=np.float32)  # one fp32 product
    return e4m3_encode(y.astype(np.float32))


def quantize_rows(x: np.ndarray):
    """Per (token, head) rows.  x: [S, H, D] (values of bf16).  Returns
    codes [S, H, D] uint8 and scales [H, S] fp32."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=2)                     # [S, H]
    return _codes(x, _recip(amax)[:, :, None]), np.ascontiguousarray(_scale(amax).T)


def key_tiles(cu: np.ndarray, tile: int = 128):
    """(begin, end) token ranges of every document's 128-key tiles."""
    out = []
    for d in range(len(cu) - 1):
        a, b = int(cu[d]), int(cu[d + 1])
        for t0 in range(a, b, tile):
            out.append((t0, min(t0 + tile, b)))
    return out


def quantize_key_tiles(x: np.ndarray, cu: np.ndarray):
    """Per (head, 128-key tile of a document).  Returns codes [S, H, D] uint8
    and scales [H, S] fp32 (every token carries its tile's scale)."""
    x = np.asarray(x, dtype=np.float32)
    S, H, D = x.shape
    codes = np.zeros((S, H, D), dtype=np.uint8)
    scales = np.zeros((H, S), dtype=np.float32)
    for a, b in key_tiles(cu):
        amax = np.abs(x[a:b]).max(axis=(0, 2))       # [H]
        codes[a:b] = _codes(x[a:b], _recip(amax)[None, :, None])
        scales[:, a:b] = _scale(amax)[:, None]
    return codes, scales


def quantize_channels(x: np.ndarray):
    """Per (head, channel) over all tokens.  Returns codes [S, H, D] uint8 and
    scales [H, D] fp32."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=0)                     # [H, D]
    return _codes(x, _recip(amax)[None, :, :]), _scale(amax)


def quantize(q_hat: np.ndarray, k_hat: np.ndarray, v: np.ndarray, cu: np.ndarray):
    """The three quantisations of the FP8 step (fp64 arrays of bf16 values in)."""
    q8, sq = quantize_rows(q_hat)
    k8, sk = quantize_key_tiles(k_hat, cu)
    v8, sv = quantize_channels(v)
    return q8, sq, k8, sk, v8, sv


def dequantize(q8, sq, k8, sk, v8, sv):
    """fp64 values q~, k~, v~ ([S, H, D] each)."""
    q = e4m3_decode(q8) * sq.T.astype(np.float64)[:, :, None]
    k = e4m3_decode(k8) * sk.T.astype(np.float64)[:, :, None]
    v = e4m3_decode(v8) * sv.astype(np.float64)[None, :, :]
    return q, k, v


def error_bound(q, k, v, cu, scale, heads, rows):
    """Per-element bound on |o_kernel - o_exact| for the given query rows,
    from the kernel's rounding of P to e4m3: each probability p_j (<= 2^8 after
    division by 2^m, m the kernel's reference max) is off by at most 2^-4 p_j
    (normal range) or 2^-10 (subnormals), so with w_j = p_j / l
        |delta o_c| <= 2^-4 sum_j w_j |v~_jc| + 2^-10 sum_j |v~_jc| / l
    where l = sum_j p_j >= 1 because the reference max is at most 2^8 below
    the row max.  The final bf16 rounding (2^-9 |o|) and fp32 arithmetic
    (< 1e-5 here) are added by the caller."""
    heads = np.asarray(list(heads), dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    D = k.shape[2]
    out = np.zeros((rows.size, heads.size, D), dtype=np.float64)
    docs = np.searchsorted(cu, rows, side="right") - 1
    for d in np.unique(docs):
        a, b = int(cu[d]), int(cu[d + 1])
        sel = np.nonzero(docs == d)[0]
        for hi, h in enumerate(heads):
            s = (q[rows[sel], h, :] @ k[a:b, h, :].T) * scale
            w = np.exp(s - s.max(axis=1, keepdims=True))
            w /= w.sum(axis=1, keepdims=True)
            av = np.abs(v[a:b, h, :])
            out[sel, hi, :] = 2.0 ** -4 * (w @ av) + 2.0 ** -10 * av.sum(axis=0)[None, :]
    return out
