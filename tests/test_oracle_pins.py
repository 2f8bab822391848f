"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-type the oracle's formulas: they use closed forms, exact
rational arithmetic, invariants, brute force on tiny inputs and library
routines.  The ``test_planted_*`` cases plant a plausible mistake in a copy
of an oracle function and check that a pin catches it.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import attention as oatt
from oracle import plan as oplan
from oracle import prologue as opro

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------- plan ----

def test_cu_seqlens_tiny_closed_form():
    w = synth.config(1)
    cu = oplan.cu_seqlens(synth.spans_to_tuples(w.docs))
    assert cu.dtype == np.int32
    assert cu.tolist() == [0, 2 * 4 * 8, 2 * 4 * 8 + 1 * 8 * 10]


def test_ref2va_token_count_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "ref2va_token_count.json")))
    w = synth.config(3)
    cu = oplan.cu_seqlens(synth.spans_to_tuples(w.docs))
    assert int(cu[-1]) == g["S"] == 20423
    assert len(w.docs[0]) == 1 + g["references"] + 1


@pytest.mark.parametrize("n,S", [(1, 144), (2, 4096), (3, 20423), (4, 21353), (5, 32768)])
def test_workload_lengths(n, S):
    w = synth.config(n)
    cu = oplan.cu_seqlens(synth.spans_to_tuples(w.docs))
    assert int(cu[-1]) == S
    assert np.all(np.diff(cu) > 0)


def test_config5_documents():
    w = synth.config(5)
    assert len(w.docs) == 16
    assert all(L % 8 == 0 for L in w.doc_lengths)
    # lengths are the rescaled U[512, 4096] draws, so they stay within the rescaled range
    assert min(w.doc_lengths) >= 8 and max(w.doc_lengths) <= 4096 * 32768 // (16 * 512)


def _brute_positions(docs):
    out = []
    for d in docs:
        for (n_t, n_h, n_w, start, step) in d:
            for it, ih, iw in itertools.product(range(n_t), range(n_h), range(n_w)):
                out.append((it, ih, iw, start, step))
    return out


def test_integer_grid_positions_are_indices():
    # start 0 and step 1: the position of each token is exactly its index tuple
    docs = [[(2, 3, 4, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))], [(5, 1, 1, (0.0, 0.0, 0.0), (1.0, 0.0, 0.0))]]
    pos = oplan.positions(docs)
    brute = _brute_positions(docs)
    assert pos.shape == (len(brute), 3)
    for row, (it, ih, iw, _s, _st) in zip(pos, brute):
        assert row.tolist() == [float(it), float(ih), float(iw)]


def test_reference_images_sit_at_negative_t():
    w = synth.config(3)
    pos = oplan.positions(synth.spans_to_tuples(w.docs))
    video = 32 * 15 * 27
    for i in range(6):
        blk = pos[video + i * 405: video + (i + 1) * 405]
        assert np.all(blk[:, 0] == -(i + 1))
        assert blk[:, 1].max() == 14 and blk[:, 2].max() == 26
    audio = pos[video + 6 * 405:]
    assert audio[:, 0].tolist() == list(range(5033))
    assert np.all(audio[:, 1:] == 0)


def _round_exact(x: Fraction) -> float:
    """Nearest double (ties to even) of an exact rational."""
    return float(x)  # Fraction.__float__ rounds correctly


def test_fractional_positions_are_two_roundings_not_one():
    # i*step + start with one rounding after the product and one after the sum
    # (a linspace without endpoint), as opposed to a single fused rounding.
    start = (-0.7, 0.1, 1.0 / 3.0)
    step = (1.0 / 3.0, 0.1, 2.0 / 7.0)
    n = 64
    docs = [[(n, 1, 1, start, (step[0], 0.0, 0.0))], [(1, n, 1, start, (0.0, step[1], 0.0))],
            [(1, 1, n, start, (0.0, 0.0, step[2]))]]
    pos = oplan.positions(docs)
    fused_differs = 0
    for a in range(3):
        col = pos[a * n:(a + 1) * n, a]
        for i in range(n):
            prod = _round_exact(Fraction(i) * Fraction(step[a]))
            want = _round_exact(Fraction(prod) + Fraction(start[a]))
            fused = _round_exact(Fraction(i) * Fraction(step[a]) + Fraction(start[a]))
            assert col[i] == want, (a, i)
            fused_differs += fused != want
    # the inputs are chosen so that the order matters somewhere
    assert fused_differs > 0


# ----------------------------------------------------------- prologue ----

def _rand_x(S, H, D=128, scale=1.0):
    return RNG.standard_normal((S, H, D)) * scale


def _rand_pos(S):
    return np.stack([RNG.integers(-8, 40, S), RNG.integers(0, 30, S), RNG.integers(0, 30, S)],
                    axis=1).astype(np.float64)


def test_rope_preserves_norm():
    x = _rand_x(40, 3)
    g = 1.0 + 0.1 * RNG.standard_normal(128)
    pos = _rand_pos(40)
    y = opro.rms_norm(x, g, 1e-6)
    yr = opro.qk_prologue(x, g, pos)
    np.testing.assert_allclose(np.linalg.norm(yr, axis=-1), np.linalg.norm(y, axis=-1), rtol=1e-13)


def check_plain_rmsnorm_closed_form(fn):
    """gain 1 and position 0: ||y||^2 = 128 m / (m + eps), m = mean x^2, and y is parallel to x."""
    x = _rand_x(16, 2, scale=0.05)
    eps = 1e-6
    y = fn(x, np.ones(128), np.zeros((16, 3)), eps)
    m = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.sum(y * y, axis=-1), 128 * m / (m + eps), rtol=1e-12)
    cosang = np.sum(x * y, axis=-1) / (np.linalg.norm(x, axis=-1) * np.linalg.norm(y, axis=-1))
    np.testing.assert_allclose(cosang, 1.0, rtol=1e-12)


def test_plain_rmsnorm_closed_form():
    check_plain_rmsnorm_closed_form(opro.qk_prologue)


def test_gain_scales_each_dim():
    x = _rand_x(8, 2)
    g = 1.0 + 0.1 * RNG.standard_normal(128)
    pos = np.zeros((8, 3))
    y1 = opro.qk_prologue(x, np.ones(128), pos)
    yg = opro.qk_prologue(x, g, pos)
    np.testing.assert_allclose(yg, y1 * g, rtol=1e-13)
    # a per-head gain array with identical rows equals the shared gain
    yh = opro.qk_prologue(x, np.tile(g, (2, 1)), pos)
    np.testing.assert_array_equal(yh, yg)


def test_tail_dims_do_not_rotate():
    x = _rand_x(10, 2)
    g = np.ones(128)
    y0 = opro.qk_prologue(x, g, np.zeros((10, 3)))
    y1 = opro.qk_prologue(x, g, _rand_pos(10) + 1.0)
    np.testing.assert_array_equal(y0[..., 96:], y1[..., 96:])
    assert np.max(np.abs(y0[..., :96] - y1[..., :96])) > 1e-3


# Closed-form rotations of unit inputs.  The pages state NeoX rotate-half with
# a cos/sin cache repeated over the two halves and three axes off the grid;
# the 16/16/16 angle blocks and omega_k = 10000^(-k/16) are the reading taken
# where the pages print no formula.  For x = e_j (j < 48), eps = 0 and gain 1
# the norm gives y = sqrt(128) e_j; the rotation then puts sqrt(128) cos(theta)
# on dim j and sqrt(128) sin(theta) on dim j + 48.
UNIT_CASES = [
    # (dim j, position (t, h, w), theta)
    (0, (1.0, 0.0, 0.0), 1.0),                          # t axis, k = 0, omega = 1
    (16, (0.0, 2.0, 0.0), 2.0),                         # h axis, k = 0
    (32, (0.0, 0.0, -3.0), -3.0),                       # w axis, k = 0
    (8, (5.0, 0.0, 0.0), 5.0 * 0.01),                   # t axis, k = 8: 10000^(-1/2) = 0.01
    (24, (0.0, 7.0, 9.0), 7.0 * 0.01),                  # h axis, k = 8
    (44, (1.0, 1.0, 100.0), 100.0 * 10.0 ** (-3.0)),    # w axis, k = 12: 10000^(-3/4)
    (4, (2.0, 3.0, 4.0), 2.0 * 0.1),                    # t axis, k = 4: 10000^(-1/4) = 0.1
]


def check_unit_rotations(fn):
    r = math.sqrt(128.0)
    for j, p, theta in UNIT_CASES:
        x = np.zeros((1, 1, 128))
        x[0, 0, j] = 1.0
        y = fn(x, np.ones(128), np.asarray([p], dtype=np.float64), 0.0)[0, 0]
        want = np.zeros(128)
        want[j] = r * math.cos(theta)
        want[j + 48] = r * math.sin(theta)
        np.testing.assert_allclose(y, want, atol=1e-12, err_msg=f"e_{j} at {p}")
        # the partner dim rotates the other way: e_{j+48} -> (-sin, cos)
        x = np.zeros((1, 1, 128))
        x[0, 0, j + 48] = 1.0
        y = fn(x, np.ones(128), np.asarray([p], dtype=np.float64), 0.0)[0, 0]
        want = np.zeros(128)
        want[j] = -r * math.sin(theta)
        want[j + 48] = r * math.cos(theta)
        np.testing.assert_allclose(y, want, atol=1e-12, err_msg=f"e_{j + 48} at {p}")
    # dims 96..127 pass through: e_100 stays e_100 at any position
    x = np.zeros((1, 1, 128))
    x[0, 0, 100] = 1.0
    y = fn(x, np.ones(128), np.asarray([[3.0, 4.0, 5.0]]), 0.0)[0, 0]
    want = np.zeros(128)
    want[100] = r
    np.testing.assert_allclose(y, want, atol=1e-12)


def test_unit_rotations():
    check_unit_rotations(opro.qk_prologue)


def check_relative_position(fn):
    """<R(q, p), R(k, p')> depends only on p - p': shifting every position of a
    document by one offset leaves all scores unchanged; changing one relative
    offset changes them."""
    S = 24
    xq, xk = _rand_x(S, 2), _rand_x(S, 2)
    g = 1.0 + 0.1 * RNG.standard_normal(128)
    pos = _rand_pos(S)

    def scores(p):
        q = fn(xq, g, p, 1e-6)
        k = fn(xk, g, p, 1e-6)
        return np.einsum("ihd,jhd->hij", q, k)

    s0 = scores(pos)
    s1 = scores(pos + np.array([3.0, -5.0, 11.0]))
    np.testing.assert_allclose(s1, s0, atol=1e-10, rtol=0)
    p2 = pos.copy()
    p2[0] += np.array([1.0, 0.0, 0.0])
    assert np.max(np.abs(scores(p2) - s0)) > 1e-3


def test_relative_position():
    check_relative_position(opro.qk_prologue)


# ---------------------------------------------------------- attention ----

def _tiny_case(lengths, H=2, D=128, seed=7):
    rng = np.random.default_rng(seed)
    S = sum(lengths)
    q, k, v = (rng.standard_normal((S, H, D)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, cu


def test_softmax_rows_sum_to_one():
    q, k, v, cu = _tiny_case([5, 37, 64])
    sums = oatt.softmax_row_sums(q * 3, k, cu, 1 / math.sqrt(128), head=1, rows=range(106))
    np.testing.assert_allclose(sums, 1.0, atol=1e-12)


def check_segment_isolation(fn):
    q, k, v, cu = _tiny_case([40, 50, 30])
    o, lse = fn(q, k, v, cu, 0.1)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[60] += 1.0
    k2[45] -= 2.0
    v2[70] *= 3.0
    o2, lse2 = fn(q2, k2, v2, cu, 0.1)
    np.testing.assert_array_equal(o2[:40], o[:40])
    np.testing.assert_array_equal(o2[90:], o[90:])
    np.testing.assert_array_equal(lse2[:, :40], lse[:, :40])
    assert np.max(np.abs(o2[40:90] - o[40:90])) > 1e-3


def test_segment_isolation():
    check_segment_isolation(oatt.attention)


def test_single_token_documents_return_v():
    q, k, v, cu = _tiny_case([1, 1, 3, 1])
    o, lse = oatt.attention(q, k, v, cu, 0.3)
    for i in (0, 1, 5):
        np.testing.assert_array_equal(o[i], v[i])
        np.testing.assert_allclose(lse[:, i], 0.3 * np.einsum("hd,hd->h", q[i], k[i]), rtol=1e-14)


def test_zero_queries_give_document_mean():
    q, k, v, cu = _tiny_case([17, 29])
    q[:] = 0.0
    o, lse = oatt.attention(q, k, v, cu, 0.2)
    np.testing.assert_allclose(o[:17], np.broadcast_to(v[:17].mean(axis=0), (17, 2, 128)), atol=1e-13)
    np.testing.assert_allclose(o[17:], np.broadcast_to(v[17:].mean(axis=0), (29, 2, 128)), atol=1e-13)
    np.testing.assert_allclose(lse[:, :17], math.log(17), atol=1e-13)


def test_identical_keys_give_document_mean():
    q, k, v, cu = _tiny_case([23])
    k[:] = k[0]
    o, _ = oatt.attention(q, k, v, cu, 0.2)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), atol=1e-13)


def test_permutation_equivariance_full_path():
    # permuting a document's tokens together with their positions permutes the output
    w = synth.config(1)
    docs = synth.spans_to_tuples(w.docs)
    pos = oplan.positions(docs)
    cu = oplan.cu_seqlens(docs)
    rng = np.random.default_rng(3)
    x = [rng.standard_normal((144, 2, 128)) for _ in range(3)]
    g = 1.0 + 0.1 * rng.standard_normal(128)
    perm = np.concatenate([rng.permutation(64), 64 + rng.permutation(80)])

    def run(xq, xk, v, p):
        return oatt.attention(opro.qk_prologue(xq, g, p), opro.qk_prologue(xk, g, p), v, cu,
                              1 / math.sqrt(128))[0]

    o = run(*x, pos)
    op = run(x[0][perm], x[1][perm], x[2][perm], pos[perm])
    np.testing.assert_allclose(op, o[perm], atol=1e-12)


def _python_attention_one(qr, K, V, scale):
    """Pure-Python softmax attention of one query row (brute force)."""
    s = [scale * sum(a * b for a, b in zip(qr, kr)) for kr in K]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    return [sum(e[j] * V[j][d] for j in range(len(K))) / z for d in range(len(V[0]))], m + math.log(z)


def test_brute_force_python_tiny():
    q, k, v, cu = _tiny_case([3, 5], H=1, D=6)
    o, lse = oatt.attention(q, k, v, cu, 0.7)
    for i in range(8):
        a, b = (0, 3) if i < 3 else (3, 8)
        want, wl = _python_attention_one(q[i, 0].tolist(), k[a:b, 0].tolist(), v[a:b, 0].tolist(), 0.7)
        np.testing.assert_allclose(o[i, 0], want, rtol=1e-13, atol=1e-14)
        assert abs(lse[0, i] - wl) < 1e-13


def test_brute_force_torch_sdpa_tiny_config():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    from scipy.special import logsumexp
    w = synth.config(1)
    t = synth.make_tensors(w)
    docs = synth.spans_to_tuples(w.docs)
    pos = oplan.positions(docs)
    cu = oplan.cu_seqlens(docs)
    q = opro.qk_prologue(synth.bf16_bits_to_f64(t.q), t.gain_q.astype(np.float64), pos)
    k = opro.qk_prologue(synth.bf16_bits_to_f64(t.k), t.gain_k.astype(np.float64), pos)
    v = synth.bf16_bits_to_f64(t.v)
    o, lse = oatt.attention(q, k, v, cu, w.softmax_scale)
    for d in range(2):
        a, b = int(cu[d]), int(cu[d + 1])
        tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x[a:b].transpose(1, 0, 2))) for x in (q, k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv, scale=w.softmax_scale).numpy().transpose(1, 0, 2)
        np.testing.assert_allclose(o[a:b], ref, atol=1e-12)
        s = np.einsum("ihd,jhd->hij", q[a:b], k[a:b]) * w.softmax_scale
        np.testing.assert_allclose(lse[:, a:b], logsumexp(s, axis=-1), atol=1e-12)


def test_sampled_rows_equal_full():
    q, k, v, cu = _tiny_case([30, 41, 9], H=3)
    o, lse = oatt.attention(q, k, v, cu, 0.2)
    rows = np.array([79, 0, 35, 70, 29, 30])
    os_, ls = oatt.attention_rows(q[rows], k, v, cu, 0.2, [2, 0], rows)
    # same arithmetic per row; BLAS may order the dot products differently per shape
    np.testing.assert_allclose(os_[:, 0], o[rows, 2], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ls[1], lse[0, rows], rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------- flops ----

def test_flop_convention_reproduces_page_figure():
    g = json.load(open(os.path.join(GOLDEN, "flop_convention.json")))
    w = synth.Workload("thor", 0, g["heads"], [[synth.run1d(g["seq_len"])]], head_dim=g["head_dim"])
    gflops = w.flops() * g["layers"] / g["attention_seconds"] / 1e9
    assert abs(gflops - g["printed_gflops"]) <= g["printed_gflops_rounding"], gflops


# ------------------------------------------------- planted mistakes ----

def _rope_wrong_sign(y, theta, rope_dims=96):
    half = rope_dims // 2
    c, s = np.cos(theta)[:, None, :], np.sin(theta)[:, None, :]
    a, b = y[..., :half], y[..., half:rope_dims]
    out = y.copy()
    out[..., :half] = a * c + b * s          # planted: sign flipped
    out[..., half:rope_dims] = b * c - a * s
    return out


def _rope_pairs_adjacent(y, theta, rope_dims=96):
    out = y.copy()                            # planted: GPT-J style adjacent pairs
    c, s = np.cos(theta)[:, None, :], np.sin(theta)[:, None, :]
    a, b = y[..., 0:rope_dims:2], y[..., 1:rope_dims:2]
    out[..., 0:rope_dims:2] = a * c - b * s
    out[..., 1:rope_dims:2] = b * c + a * s
    return out


def _make_prologue(rope=None, eps_outside=False, freq_div=32):
    def fn(x, gain, pos, eps=1e-6, base=10000.0, rope_dims=96):
        if eps_outside:
            ms = np.mean(x * x, axis=-1, keepdims=True)
            y = x / (np.sqrt(ms) + eps) * gain
        else:
            y = opro.rms_norm(x, gain, eps)
        k = np.arange(16, dtype=np.float64)
        w = base ** (-(2.0 * k) / freq_div)
        theta = np.concatenate([pos[:, a:a + 1] * w[None, :] for a in range(3)], axis=1)
        return (rope or opro.apply_rope)(y, theta, rope_dims)
    return fn


@pytest.mark.parametrize("mutant", ["wrong_sign", "adjacent_pairs", "freq_over_64"])
def test_planted_rope_mistakes_are_caught(mutant):
    fn = {"wrong_sign": _make_prologue(rope=_rope_wrong_sign),
          "adjacent_pairs": _make_prologue(rope=_rope_pairs_adjacent),
          "freq_over_64": _make_prologue(freq_div=64)}[mutant]
    # the unmutated reconstruction passes
    check_unit_rotations(_make_prologue())
    with pytest.raises(AssertionError):
        check_unit_rotations(fn)


def test_planted_eps_placement_is_caught():
    check_plain_rmsnorm_closed_form(_make_prologue())
    with pytest.raises(AssertionError):
        check_plain_rmsnorm_closed_form(_make_prologue(eps_outside=True))


def test_planted_cross_document_leak_is_caught():
    def leaky(q, k, v, cu, scale):
        # planted: the whole packed sequence treated as one document
        S = q.shape[0]
        return oatt.attention(q, k, v, np.array([0, S], dtype=np.int32), scale)
    with pytest.raises(AssertionError):
        check_segment_isolation(leaky)


def test_planted_absolute_position_is_caught():
    def absolute(x, gain, pos, eps=1e-6):
        # planted: angles from a position-dependent offset that breaks relativity
        return opro.qk_prologue(x, gain, pos * pos, eps)
    check_relative_position(opro.qk_prologue)
    with pytest.raises(AssertionError):
        check_relative_position(absolute)
