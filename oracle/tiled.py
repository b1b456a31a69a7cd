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

__all__ = ["online_softmax_step", "flash_attention", "merge_states", "chunked_attention"]


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


def merge_states(states):
    """Combine the running states (m, l, acc) that the step builds for the
    same query rows over disjoint key chunks into the state over all of them.

    Each chunk's state is rescaled to the common maximum and added, the same
    rescale the step applies to the running state when a block raises the
    maximum ("The Hidden Recurrence in Softmax Attention", section "Chunk-wise
    Mode with Online Softmax Re-scale"), here applied to a second chunk's
    state in place of a block of raw scores:
        m = max_c m_c,  w_c = exp(m_c - m),  l = sum_c w_c l_c,  acc = sum_c w_c acc_c
    with 0 in place of m inside the exponentials when m = -inf (no chunk has
    an allowed key for the row).
    """
    ms = [np.asarray(st[0], dtype=np.float64) for st in states]
    m = ms[0]
    for mc in ms[1:]:
        m = np.maximum(m, mc)
    ref = np.where(np.isneginf(m), 0.0, m)
    l = np.zeros_like(m)
    acc = np.zeros_like(np.asarray(states[0][2], dtype=np.float64))
    for (mc, lc, ac) in states:
        w = np.exp(np.asarray(mc, dtype=np.float64) - ref)   # 0 for a chunk with no allowed key
        l = l + w * np.asarray(lc, dtype=np.float64)
        acc = acc + w[:, None] * np.asarray(ac, dtype=np.float64)
    return m, l, acc


def chunked_attention(Q, K, V, chunk_bounds, block_size=64, causal=False, scale=None):
    """Single head, keys split at chunk_bounds (e.g. [0, 300, 301, Tk]): each
    chunk runs the block-by-block step from the empty state on its own keys,
    the chunk states are merged with merge_states, and the output is
    acc / l (0 where l = 0) with lse = m + log l (-inf where l = 0).
    Returns (output [Tq, dv], lse [Tq]).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Tq, d = Q.shape
    dv = V.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    states = []
    for c0, c1 in zip(chunk_bounds[:-1], chunk_bounds[1:]):
        m = np.full(Tq, -np.inf)
        l = np.zeros(Tq)
        acc = np.zeros((Tq, dv))
        for b0 in range(c0, c1, block_size):
            b1 = min(b0 + block_size, c1)
            s = scale * (Q @ K[b0:b1].T)
            if causal:
                s = np.where(np.arange(b0, b1)[None, :] > np.arange(Tq)[:, None], -np.inf, s)
            m, l, acc = online_softmax_step(m, l, acc, s, V[b0:b1])
        states.append((m, l, acc))
    m, l, acc = merge_states(states)
    out = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
    lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse

