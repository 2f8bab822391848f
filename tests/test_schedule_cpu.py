"""The forward's work list (segment-aware scheduling), built on the host
through h3attn_work_list_host: no GPU is needed.

Checked on the five workloads and on edge layouts, for the 76 CTA pairs of a
GB300 and for other pair counts:
  - every (document, head, 512-row query block) is covered exactly once, its
    key tiles [0, ceil(L / 128)) partitioned by its segments; only tiles of
    the query block's own document are ever visited;
  - a unit split along the keys gives each piece its own partial slot, and
    the slots are 0 .. n_parts - 1;
  - the pairs with work are the leading ones and each has at least one segment;
  - each pair runs the whole units of the full rounds in list order (longest
    document first, then head, then query rows);
  - the placement meets the list-scheduling bound: no pair's estimated load
    exceeds the mean load by more than the largest segment.
"""
import math

import numpy as np
import pytest

import synth
from packed_varlen_non_gb300 import h3attn as H

UNIT_ROWS, KEY_TILE = 512, 128


def cost(seg):
    """The placement's load estimate, as the header states it."""
    return int(seg[5]) - int(seg[4]) + 1


def list_key(lengths):
    """(document rank, head, first row) order of the whole units."""
    order = sorted(range(len(lengths)), key=lambda d: -lengths[d])  # stable: ties keep the index order
    return {d: r for r, d in enumerate(order)}


def check_work_list(lengths, heads, pairs):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    units, off = H.h3attn_work_list_host(cu, heads, pairs)
    n = units.shape[0]
    used = off.size - 1
    # offsets: leading pairs, each with work
    assert off[0] == 0 and off[-1] == n
    assert np.all(np.diff(off) >= 1)
    assert used == min(n, pairs)
    doc_of = {int(cu[d]): d for d in range(len(lengths))}
    # coverage of every (document, head, query block)
    pieces = {}
    for seg in units:
        q0, b, e, h, lo, hi, part, voff = (int(x) for x in seg)
        d = doc_of[b]
        assert e == cu[d + 1] and 0 <= h < heads
        assert b <= q0 < e and (q0 - b) % UNIT_ROWS == 0
        assert 0 <= lo < hi <= math.ceil((e - b) / KEY_TILE)
        assert voff == sum((l + 15) // 16 * 16 for l in lengths[:d])
        pieces.setdefault((d, h, q0), []).append((lo, hi, part))
    expected = {(d, h, q0) for d, L in enumerate(lengths) for h in range(heads)
                for q0 in range(int(cu[d]), int(cu[d + 1]), UNIT_ROWS)}
    assert set(pieces) == expected
    parts = []
    for (d, h, q0), ps in pieces.items():
        ps.sort()
        n_kv = math.ceil(lengths[d] / KEY_TILE)
        assert ps[0][0] == 0 and ps[-1][1] == n_kv
        assert all(ps[i][1] == ps[i + 1][0] for i in range(len(ps) - 1))
        if len(ps) == 1:
            assert ps[0][2] == -1
        else:
            assert all(p >= 0 for _, _, p in ps)
            slots = sorted(p for _, _, p in ps)
            assert slots == list(range(slots[0], slots[0] + len(ps)))
            parts += slots
    assert sorted(parts) == list(range(len(parts)))
    # whole units of the full rounds: list order within each pair
    rank = list_key(lengths)
    n_whole = len(expected) // pairs * pairs
    full_keys = sorted((rank[d], h, q0) for d, h, q0 in expected)[:n_whole]
    full_set = set(full_keys)
    for p in range(used):
        keys = [(rank[doc_of[int(s[1])]], int(s[3]), int(s[0])) for s in units[off[p]:off[p + 1]]]
        keys = [k for k in keys if k in full_set]
        assert keys == sorted(keys)
    # list-scheduling bound on the estimated loads
    loads = np.array([sum(cost(s) for s in units[off[p]:off[p + 1]]) for p in range(used)], dtype=np.int64)
    total = sum(cost(s) for s in units)
    assert loads.max() <= total / pairs + max(cost(s) for s in units)
    return units, off, loads


WORKLOADS = [1, 2, 3, 4, 5]


@pytest.mark.parametrize("cfg", WORKLOADS)
@pytest.mark.parametrize("pairs", [76, 7])
def test_work_list_on_the_workloads(lib, cfg, pairs):
    w = synth.config(cfg)
    check_work_list(list(w.doc_lengths), w.num_heads, pairs)


@pytest.mark.parametrize("lengths,heads,pairs", [
    ([1], 1, 76),                        # one row, one unit: split impossible
    ([128], 1, 76),                      # one key tile
    ([129, 1, 511, 512, 513], 3, 76),    # tile and block edges
    ([4096] * 19, 4, 76),                # 76 units x 8 blocks: full rounds only
    ([300] * 500, 2, 76),                # many one-tile-block units
    ([20423], 56, 76),                   # 56 heads, one long document
    ([16320, 5033], 21, 1),              # one pair takes everything
    ([777, 5, 3000, 64], 5, 1024),       # more pairs than units
])
def test_work_list_edge_layouts(lib, lengths, heads, pairs):
    check_work_list(lengths, heads, pairs)


def test_lpt_spread_on_mixed_documents_beats_rounds(lib):
    # two documents of very different lengths (the 21,353-token two-document
    # layout): the spread of estimated loads stays within one segment, and is
    # smaller than that of dealing the same units out in rounds
    w = synth.config(4)
    units, off, loads = check_work_list(list(w.doc_lengths), w.num_heads, 76)
    assert loads.max() - loads.min() <= max(cost(s) for s in units)
    whole = [(math.ceil(L / KEY_TILE), q0) for L in sorted(w.doc_lengths, reverse=True)
             for _ in range(w.num_heads) for q0 in range(0, L, UNIT_ROWS)]
    rounds = np.zeros(76, dtype=np.int64)
    for i, (n_kv, _) in enumerate(whole[:len(whole) // 76 * 76]):
        rounds[i % 76] += n_kv + 1
    assert rounds.max() - rounds.min() > loads.max() - loads.min()


def test_work_list_rejects_bad_arguments(lib):
    def status(fn):
        with pytest.raises(H.H3AttnError) as e:
            fn()
        return e.value.status
    assert status(lambda: H.h3attn_work_list_host([0, 10], 2, 0)) == H.H3ATTN_EINVAL
    assert status(lambda: H.h3attn_work_list_host([0, 10], 2, 1025)) == H.H3ATTN_EINVAL
    assert status(lambda: H.h3attn_work_list_host([0, 10], 0, 4)) == H.H3ATTN_EINVAL
    assert status(lambda: H.h3attn_work_list_host([0, 10, 10], 2, 4)) == H.H3ATTN_EINVAL
    assert status(lambda: H.h3attn_work_list_host([1, 10], 2, 4)) == H.H3ATTN_EINVAL
    assert status(lambda: H.h3attn_work_list_host([0], 2, 4)) == H.H3ATTN_EINVAL
