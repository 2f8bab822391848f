"""Plan parity: cu_seqlens and the fp64 position grid from the library are
bit-identical to the oracle's independent planner; the cos/sin table matches
the fp64 angles to fp32 rounding."""
import numpy as np
import pytest

import synth
from oracle import plan as oplan
from oracle import prologue as opro
from packed_varlen_non_gb300 import h3attn as H

pytestmark = pytest.mark.gpu


def _check(docs, num_heads=2):
    with H.Plan(docs, num_heads) as p:
        cu = H.h3attn_plan_copy_cu_seqlens(p.handle)
        pos = H.h3attn_plan_copy_positions(p.handle)
        rope = H.h3attn_plan_copy_rope_table(p.handle)
        info = p.info
    want_cu = oplan.cu_seqlens(docs)
    want_pos = oplan.positions(docs)
    np.testing.assert_array_equal(cu, want_cu)
    assert pos.tobytes() == want_pos.tobytes(), "position grid is not bit-identical"
    th = opro.rope_angles(want_pos)
    np.testing.assert_allclose(rope[..., 0], np.cos(th), rtol=0, atol=1.2e-7)
    np.testing.assert_allclose(rope[..., 1], np.sin(th), rtol=0, atol=1.2e-7)
    lens = np.diff(want_cu)
    assert info["S"] == int(want_cu[-1]) and info["n_docs"] == len(docs)
    assert info["max_seqlen"] == int(lens.max())


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_plan_bit_exact_on_workloads(lib, n):
    w = synth.config(n)
    _check(synth.spans_to_tuples(w.docs), w.num_heads)


def test_plan_bit_exact_fractional_spans(lib):
    # steps and starts that are not exactly representable: the grid must be
    # one rounded product then one rounded sum, never a fused multiply-add
    docs = [
        [(5, 7, 9, (-0.7, 0.1, 1.0 / 3.0), (1.0 / 3.0, 0.1, 2.0 / 7.0))],
        [(64, 1, 1, (0.3, 0.0, 0.0), (0.1, 0.0, 0.0)),
         (3, 4, 5, (-1.0 / 7.0, 2.5, -3.25), (0.7, 1.0 / 9.0, 0.01))],
        [(1, 1, 1, (1e-300, -0.0, 1e10), (1.0, 1.0, 1.0))],
    ]
    _check(docs)


def test_plan_many_small_documents(lib):
    rng = np.random.default_rng(5)
    docs = [[(int(L), 1, 1, (float(-i), 0.0, 0.0), (1.0, 0.0, 0.0))]
            for i, L in enumerate(rng.integers(1, 40, 300))]
    _check(docs, 3)
