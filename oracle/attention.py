"""Oracle: packed varlen non-causal attention.

Follows [PR26], PR description: attention over the packed sequence is
bidirectional inside each cu_seqlens document and never crosses a document
boundary -- the contract of a cu_seqlens varlen flash-attention call with
causal=false.  For a query row i of document [a, b):

    s_ij  = scale * <q_i, k_j>            for j in [a, b)
    m_i   = max_j s_ij
    l_i   = sum_j exp(s_ij - m_i)
    o_i   = sum_j (exp(s_ij - m_i) / l_i) * v_j
    lse_i = m_i + ln(l_i)

The softmax is evaluated in two passes (the row maximum first, then the
exponentials), not with the online recurrence the GPU kernel uses, so the two
sides do not share an algorithm.  Query rows are independent, so rows may be
processed in chunks or as a sample without changing any row's arithmetic.

Parity: pinned (rows of the softmax sum to one, segment isolation, one-token
documents return v, zero queries return the document mean of v, permutation
equivariance, and agreement with a library fp64 softmax attention on tiny
inputs).
"""
from __future__ import annotations

import numpy as np


def doc_of_rows(cu: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Index of the document holding each token row."""
    return np.searchsorted(cu, rows, side="right") - 1


def attention_rows(q_sel: np.ndarray, k: np.ndarray, v: np.ndarray, cu: np.ndarray,
                   scale: float, heads, rows, chunk: int = 1024):
    """o [len(rows), len(heads), D] and lse [len(heads), len(rows)] for the
    given query rows and heads.  q_sel: fp64 [len(rows), H, D], the queries of
    tokens ``rows``; k, v: fp64 [S, H, D]."""
    heads = np.asarray(list(heads), dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    D = k.shape[2]
    o = np.zeros((rows.size, heads.size, D), dtype=np.float64)
    lse = np.zeros((heads.size, rows.size), dtype=np.float64)
    docs = doc_of_rows(cu, rows)
    for d in np.unique(docs):
        a, b = int(cu[d]), int(cu[d + 1])
        sel = np.nonzero(docs == d)[0]
        for hi, h in enumerate(heads):
            kd = k[a:b, h, :]
            vd = v[a:b, h, :]
            for c0 in range(0, sel.size, chunk):
                ii = sel[c0:c0 + chunk]
                s = scale * (q_sel[ii, h, :] @ kd.T)            # [n, L]
                m = np.max(s, axis=1, keepdims=True)            # pass 1: row max
                e = np.exp(s - m)                               # pass 2: exponentials
                l = np.sum(e, axis=1, keepdims=True)
                o[ii, hi, :] = (e / l) @ vd
                lse[hi, ii] = m[:, 0] + np.log(l[:, 0])
    return o, lse


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu: np.ndarray, scale: float):
    """Full output: o fp64 [S, H, D], lse fp64 [H, S]."""
    S, H, _ = q.shape
    return attention_rows(q, k, v, cu, scale, range(H), np.arange(S))


def softmax_row_sums(q: np.ndarray, k: np.ndarray, cu: np.ndarray, scale: float, head: int,
                     rows) -> np.ndarray:
    """sum_j p_ij for the given rows of one head (an internal check: each is 1)."""
    rows = np.asarray(rows, dtype=np.int64)
    docs = doc_of_rows(cu, rows)
    out = np.zeros(rows.size)
    for n, (i, d) in enumerate(zip(rows, docs)):
        a, b = int(cu[d]), int(cu[d + 1])
        s = scale * (k[a:b, head, :] @ q[i, head, :])
        e = np.exp(s - s.max())
        out[n] = np.sum(e / e.sum())
    return out
