"""Oracle: packed layout -- cu_seqlens and the fp64 position grid.

Follows [PR26], PR description ("How this is gated" and the first commit
message): documents are packed back to back and delimited by cu_seqlens, and
the fp64 grid that feeds the rotary embedding is gated bit-exact, which means
keeping upstream's arithmetic order -- a linspace without endpoint evaluates
``i*step + start`` (one rounded product, then one rounded sum; never a fused
multiply-add).

A span is ``(n_t, n_h, n_w, start(3), step(3))``; its tokens run t-major,
then h, with w fastest, and the position of token (i_t, i_h, i_w) on axis a
is ``i_a*step[a] + start[a]``.  A document is the concatenation of its spans.

Parity: pinned (closed forms for integer grids, exact-rational rounding for
fractional steps, token counts of the pages' workloads).
"""
from __future__ import annotations

import numpy as np


def cu_seqlens(docs) -> np.ndarray:
    """int32 [n_docs + 1]: prefix sums of document lengths, starting at 0."""
    out = [0]
    for d in docs:
        n = 0
        for (n_t, n_h, n_w, _start, _step) in d:
            n += n_t * n_h * n_w
        out.append(out[-1] + n)
    return np.asarray(out, dtype=np.int32)


def span_positions(n_t, n_h, n_w, start, step) -> np.ndarray:
    """fp64 [n_t*n_h*n_w, 3] positions of one span, t-major order."""
    it, ih, iw = np.meshgrid(np.arange(n_t, dtype=np.float64),
                             np.arange(n_h, dtype=np.float64),
                             np.arange(n_w, dtype=np.float64), indexing="ij")
    idx = [it.ravel(), ih.ravel(), iw.ravel()]
    cols = []
    for a in range(3):
        prod = idx[a] * np.float64(step[a])      # rounded product
        cols.append(prod + np.float64(start[a]))  # rounded sum
    return np.stack(cols, axis=1)


def positions(docs) -> np.ndarray:
    """fp64 [S, 3]: every document's spans concatenated, documents in order."""
    parts = [span_positions(*s) for d in docs for s in d]
    if not parts:
        return np.zeros((0, 3), dtype=np.float64)
    return np.concatenate(parts, axis=0)
