"""Tiled float64 attention with an online softmax (test infrastructure).

Only the test suite may use this module; it exists to check the oracle's
materialised result against the block-by-block formulation, which the pages
say must agree for every block size.

Follows "Tiled attention with an online softmax", section "Task", and the
same recurrence in "The Hidden Recurrence in Softmax Attention", section
"Chunk-wise Mode with Online Softmax Re-scale" (there the stored scale
m is exp(row max); here m is the row max itself).

The step's formulas are missing from the page text (the sentence that
introduces them ends without them). The reading used here, which reproduces
all three printed examples, is, for query row i and one key block:

    m_i'  = max(m_i, max_j s_ij)
    c_i   = exp(m_i - m_i')
    l_i'  = c_i * l_i + sum_j exp(s_ij - m_i')
    a_i'  = c_i * a_i + sum_j exp(s_ij - m_i') * v_j

with 0 used in place of m_i' inside both exponentials when m_i' = -inf (the
page's rule for a row that has no allowed key yet).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["online_softmax_step", "flash_attention"]


def online_softmax_step(m, l, acc, scores, v_block):
    """Add one block of keys to the running state of each query row.

    m, l: [n]; acc: [n, dv]; scores: [n, bs] (-inf = blocked key);
    v_block: [bs, dv]. Returns new (m, l, acc) with the same shapes; the
    inputs are not modified.
    """
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    acc = np.asarray(acc, dtype=np.float64)
    scores = np.asarray(scores, dtype=np.float64)
    v_block = np.asarray(v_block, dtype=np.float64)
    blk_max = scores.max(axis=1) if scores.shape[1] else np.full(m.shape, -np.inf)
    m_new = np.maximum(m, blk_max)
    ref = np.where(np.isneginf(m_new), 0.0, m_new)   # the -inf rule
    c = np.exp(m - ref)                              # 0 when m = -inf
    p = np.exp(scores - ref[:, None])                # 0 on blocked keys
    l_new = c * l + p.sum(axis=1)
    acc_new = c[:, None] * acc + p @ v_block
    return m_new, l_new, acc_new


def flash_attention(Q, K, V, block_size, causal=False, scale=None):
    """Single head: Q [Tq,d], K [Tk,d], V [Tk,dv] -> (output [Tq,dv], lse [Tq]).

    Scores of a block are scale * Q K_b^T with scale = 1/sqrt(d) unless given
    (d = last axis of Q). Blocks start at 0, block_size, 2*block_size, ...;
    the last may be shorter, and block_size may exceed Tk. With causal, key j
    is blocked for query i when j > i (global indices). The output row is
    a_i / l_i and the log-sum-exp is m_i + log l_i; a row with no allowed
    key (l_i = 0) gives output 0 and lse -inf.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Tq, d = Q.shape
    Tk, dv = K.shape[0], V.shape[1]
    if block_size < 1:
        raise ValueError("block_size must be >= 1")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    m = np.full(Tq, -np.inf)
    l = np.zeros(Tq)
    acc = np.zeros((Tq, dv))
    rows = np.arange(Tq)[:, None]
    for start in range(0, Tk, block_size):
        stop = min(Tk, start + block_size)
        s = scale * (Q @ K[start:stop].T)
        if causal:
            cols = np.arange(start, stop)[None, :]
            s = np.where(cols > rows, -np.inf, s)
        m, l, acc = online_softmax_step(m, l, acc, s, V[start:stop])
    live = l > 0
    out = np.where(live[:, None], acc / np.where(live, l, 1.0)[:, None], 0.0)
    lse = np.where(live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    return out, lse
