"""Materialised float64 attention: the plain definition (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
use this module; the product never does.

Forward ("The Hidden Recurrence in Softmax Attention", section "Standard
Attention / Forward Pass"; "attention_backprop", section "Forward Pass")::

    S   = scale * Q K^T            (blocked entries set to -inf)
    P   = softmax(S) row by row
    O   = P V
    LSE = log sum_j exp(S_ij)      (natural log, in units of scale*QK^T)

The mask M is either "none" or causal ("Chunk-wise Mode": M is the causal
mask or no mask). Causal blocks key j for query i when j > i, with global
row indices ("Tiled attention with an online softmax", section "Task").

Backward ("attention_backprop", sections "Gradient of V and P", "Gradient of
S", "Gradient of Q and K"; the same result in matrix form in "The Hidden
Recurrence in Softmax Attention", section "Backward Pass")::

    dV = P^T dO
    dP = dO V^T
    D  = rowsum(dO o O)
    dS = P o (dP - D)
    dQ = scale * dS K
    dK = scale * dS^T Q

The pages drop the softmax scale from S; differentiating S = scale * Q K^T
by the chain rule puts the factor ``scale`` on dQ and dK.

Readings where the pages are silent:

* a query row whose keys are all blocked (possible only with Tq > Tk or an
  empty key set) returns O = 0, LSE = -inf and zero gradients;
* the row maximum is subtracted before ``exp``; softmax is invariant to it,
  and without it float64 ``exp`` overflows once logits pass about 709.

Each query row's softmax runs over all Tk keys at once. Rows are processed
``row_chunk`` at a time only to bound host memory; rows are independent, so
this changes no value, only the summation order of dK and dV over rows.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "forward_head",
    "backward_head",
    "forward",
    "backward",
    "backward_head_matrix_form",
]


def _as64(x):
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _scores(q_rows, k, scale, causal, row_ids):
    """scale * q k^T for the given global query rows, blocked keys at -inf."""
    s = scale * (q_rows @ k.T)
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > row_ids[:, None], -np.inf, s)
    return s


def _softmax_rows(s):
    """Row softmax of s and its log-sum-exp; all-blocked rows give P = 0, LSE = -inf."""
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 on blocked keys
    l = e.sum(axis=1)
    p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
    lse = np.where(live, m_safe + np.log(np.where(live, l, 1.0)), -np.inf)
    return p, lse


def forward_head(q, k, v, scale, causal=False, rows=None, row_chunk=512):
    """One head: q [Tq,d], k [Tk,d], v [Tk,dv] -> (o [n,dv], lse [n]) in float64.

    ``rows`` selects global query rows (default: all Tq rows).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.zeros((rows.size, v.shape[1]))
    lse = np.full(rows.size, -np.inf)
    for c0 in range(0, rows.size, row_chunk):
        r = rows[c0:c0 + row_chunk]
        p, lse[c0:c0 + r.size] = _softmax_rows(_scores(q[r], k, scale, causal, r))
        o[c0:c0 + r.size] = p @ v
    return o, lse


def backward_head(q, k, v, do, scale, causal=False, row_chunk=512, rows=None):
    """One head: closed-form gradients in float64.

    Returns dict with dq [Tq,d], dk [Tk,d], dv [Tk,dv], and the forward
    o, lse and D = rowsum(dO o O) that the gradients use.

    ``rows`` restricts the work to those global query rows (a sample): their
    dq, o, lse and D are filled (other rows stay 0 / -inf), and dk, dv hold
    the contributions of those rows only.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    Tq = q.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros((Tq, v.shape[1]))
    lse = np.full(Tq, -np.inf)
    D = np.zeros(Tq)
    rows = np.arange(Tq) if rows is None else np.asarray(rows, dtype=np.int64)
    for c0 in range(0, rows.size, row_chunk):
        r = rows[c0:c0 + row_chunk]
        p, lse[r] = _softmax_rows(_scores(q[r], k, scale, causal, r))
        o[r] = p @ v
        D[r] = np.sum(do[r] * o[r], axis=1)           # ROW_SUM(dL/dO o O)
        dv += p.T @ do[r]                             # dL/dV = P^T dL/dO
        dp = do[r] @ v.T                              # dL/dP = dL/dO V^T
        ds = p * (dp - D[r][:, None])                 # dL/dS = dP o P - D o P
        dq[r] = scale * (ds @ k)                      # dL/dQ = dS K (times scale)
        dk += scale * (ds.T @ q[r])                   # dL/dK = dS^T Q (times scale)
    return {"dq": dq, "dk": dk, "dv": dv, "o": o, "lse": lse, "D": D}


def backward_head_matrix_form(q, k, v, do, scale, causal=False):
    """The matrix-form gradients of "The Hidden Recurrence in Softmax Attention"
    (section "Backward Pass"), written with E = exp(S) o M and l = E 1:

        dE = Diag(l)^-1 (dO V^T - diag(dO O^T) 1^T)
        dV = E^T Diag(l)^-1 dO
        dQ = (dE o E) K,  dK = (dE o E)^T Q      (times scale for S = scale*QK^T)

    E is formed with the row maximum taken out (E' = E exp(-max)), which
    leaves dE o E and E^T Diag(l)^-1 unchanged. Small sizes only: no chunking.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    r = np.arange(q.shape[0])
    s = _scores(q, k, scale, causal, r)
    m = s.max(axis=1)
    live = np.isfinite(m)
    e = np.exp(s - np.where(live, m, 0.0)[:, None])
    l = e.sum(axis=1)
    inv_l = np.where(live, 1.0 / np.where(live, l, 1.0), 0.0)
    o = (inv_l[:, None] * e) @ v
    de = inv_l[:, None] * (do @ v.T - np.sum(do * o, axis=1)[:, None])
    g = de * e
    return {
        "dq": scale * (g @ k),
        "dk": scale * (g.T @ q),
        "dv": e.T @ (inv_l[:, None] * do),
        "o": o,
    }


def _heads(x):
    B, H = x.shape[0], x.shape[1]
    for b in range(B):
        for h in range(H):
            yield b, h


def forward(Q, K, V, scale, causal=False, heads=None, row_chunk=512):
    """[B,H,Tq,d] inputs -> (O [B,H,Tq,dv], LSE [B,H,Tq]) float64.

    ``heads`` optionally restricts the work to a list of (b, h) pairs; the
    other heads are left as NaN.
    """
    Q, K, V = _as64(Q), _as64(K), _as64(V)
    B, H, Tq, _ = Q.shape
    O = np.full((B, H, Tq, V.shape[-1]), np.nan)
    LSE = np.full((B, H, Tq), np.nan)
    for b, h in (heads if heads is not None else _heads(Q)):
        O[b, h], LSE[b, h] = forward_head(Q[b, h], K[b, h], V[b, h], scale, causal,
                                          row_chunk=row_chunk)
    return O, LSE


def backward(Q, K, V, dO, scale, causal=False, heads=None, row_chunk=512):
    """[B,H,T,*] inputs -> dict of float64 dQ, dK, dV, O, LSE, D (NaN off ``heads``)."""
    Q, K, V, dO = _as64(Q), _as64(K), _as64(V), _as64(dO)
    B, H, Tq, d = Q.shape
    Tk, dv = K.shape[2], V.shape[3]
    out = {
        "dQ": np.full((B, H, Tq, d), np.nan),
        "dK": np.full((B, H, Tk, d), np.nan),
        "dV": np.full((B, H, Tk, dv), np.nan),
        "O": np.full((B, H, Tq, dv), np.nan),
        "LSE": np.full((B, H, Tq), np.nan),
        "D": np.full((B, H, Tq), np.nan),
    }
    for b, h in (heads if heads is not None else _heads(Q)):
        r = backward_head(Q[b, h], K[b, h], V[b, h], dO[b, h], scale, causal, row_chunk)
        out["dQ"][b, h], out["dK"][b, h], out["dV"][b, h] = r["dq"], r["dk"], r["dv"]
        out["O"][b, h], out["LSE"][b, h], out["D"][b, h] = r["o"], r["lse"], r["D"]
    return out
