"""The forward with the Q prologue fused in (h3attn_forward_fused_q, with the
k-only prologue): the same bits as prologue + forward, and parity with the
oracle.  Pages: "h3-spark" model card, "What this config does" (Q RMSNorm +
rot96 RoPE fused into one kernel)."""
import numpy as np
import pytest

import synth
from tests.gpu_cases import (check_attention, docs_1d, oracle_reference, random_tensors,
                             run_product, sample_rows)

pytestmark = pytest.mark.gpu

LAYOUTS = {
    "ragged_docs": ([1000, 3, 513, 129, 1], 3),
    "tile_edges": ([255, 256, 257, 383, 384, 385, 640], 2),
    "many_tiny": ([int(x) for x in np.random.default_rng(5).integers(1, 60, 50)], 2),
    "one_long": ([3000], 4),
}


@pytest.mark.parametrize("name", sorted(LAYOUTS))
def test_fused_q_bit_identical(lib, name):
    lens, Hh = LAYOUTS[name]
    docs = docs_1d(lens)
    t = random_tensors(sum(lens), Hh, seed=len(name) * 13)
    r0 = run_product(docs, Hh, t)
    r1 = run_product(docs, Hh, t, fused_q=True)
    assert np.array_equal(r1.k_bits, r0.k_bits), "k-only prologue differs from the q+k prologue's k"
    assert np.array_equal(r1.o_bits, r0.o_bits), "fused-Q forward differs from prologue + forward"
    assert np.array_equal(r1.lse, r0.lse)


def test_fused_q_workload_grid_positions(lib):
    # the 4,096-token video grid: real (t, h, w) angles, 21 heads
    w = synth.config(2)
    t = synth.make_tensors(w)
    docs = synth.spans_to_tuples(w.docs)
    r0 = run_product(docs, w.num_heads, t)
    r1 = run_product(docs, w.num_heads, t, fused_q=True)
    assert np.array_equal(r1.o_bits, r0.o_bits)
    cu = np.concatenate([[0], np.cumsum(w.doc_lengths)])
    rows = sample_rows(cu, seed=2)
    _, o, lse, _ = oracle_reference(docs, t, rows=rows)
    check_attention(r1.o[rows], o, r1.lse[:, rows], lse, "config 2, fused Q, end to end")


def test_fused_q_dit_geometry_fused_qkv(lib):
    # 56 heads read out of one fused-qkv buffer: the forward reads raw q from
    # the buffer (never writing it), k-hat is written in place
    lens = [700, 450]
    docs = docs_1d(lens)
    t = random_tensors(sum(lens), 56, seed=77)
    r0 = run_product(docs, 56, t, fused=True)
    r1 = run_product(docs, 56, t, fused=True, fused_q=True)
    assert np.array_equal(r1.o_bits, r0.o_bits)
