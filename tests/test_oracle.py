"""Pins for the CPU float64 oracle (no GPU).

Each check ties the oracle to something other than its own formula: the
worked examples printed on "Tiled attention with an online softmax"
(section "Examples"), closed forms, brute-force scalar loops, central finite
differences of the forward, and CPU float64 torch.autograd. The mutation
tests at the end plant plausible mistakes in the oracle's source and show
that these pins reject each of them.
"""
import inspect
import math
import types

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A
from oracle import tiled as T

PRINT_TOL = 1e-8  # the examples print 8 decimals


# --------------------------------------------------------------------------
# worked examples printed on the page
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["example1_no_mask.json", "example2_causal.json"])
def test_printed_examples_materialised_and_tiled(golden, name):
    g = golden(name)
    Q, K, V = (np.array(g[k]) for k in ("Q", "K", "V"))
    scale = 1.0 / math.sqrt(Q.shape[1])
    o, lse = A.forward_head(Q, K, V, scale, g["causal"])
    np.testing.assert_allclose(o, g["output"], atol=PRINT_TOL, rtol=0)
    np.testing.assert_allclose(lse, g["lse"], atol=PRINT_TOL, rtol=0)
    for bs in g["block_sizes"] + [1, 2, 3, 4, 128]:
        o2, lse2 = T.flash_attention(Q, K, V, bs, causal=g["causal"])
        np.testing.assert_allclose(o2, g["output"], atol=PRINT_TOL, rtol=0)
        np.testing.assert_allclose(lse2, g["lse"], atol=PRINT_TOL, rtol=0)


def test_printed_example_step(golden):
    g = golden("example3_step.json")
    args = [np.array(g[k]) for k in ("m", "l", "acc", "scores", "v_block")]
    copies = [a.copy() for a in args]
    m, l, acc = T.online_softmax_step(*args)
    np.testing.assert_allclose(m, g["m_new"], atol=PRINT_TOL, rtol=0)
    np.testing.assert_allclose(l, g["l_new"], atol=PRINT_TOL, rtol=0)
    np.testing.assert_allclose(acc, g["acc_new"], atol=PRINT_TOL, rtol=0)
    for a, c in zip(args, copies):  # "Do not change the input arrays."
        np.testing.assert_array_equal(a, c)


def test_step_all_blocked_row_keeps_empty_state():
    # the -inf rule: a row with no allowed key yet returns (-inf, 0, 0)
    m, l, acc = T.online_softmax_step(np.array([-np.inf]), np.array([0.0]),
                                      np.zeros((1, 3)), np.array([[-np.inf, -np.inf]]),
                                      np.ones((2, 3)))
    assert np.isneginf(m[0]) and l[0] == 0.0 and np.all(acc == 0.0)
    assert np.all(np.isfinite(acc))


# --------------------------------------------------------------------------
# block-size invariance (the page: equal to standard attention for every
# block size, to about 1e-9; block size may exceed Tk; last block ragged)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(5, 7, 3, 2), (17, 33, 8, 5), (64, 64, 64, 64), (1, 1, 1, 1),
                                   (40, 9, 6, 6)])
def test_block_size_invariance(shape, causal):
    Tq, Tk, d, dv = shape
    rng = np.random.default_rng(Tq * 1000 + Tk)
    Q, K, V = rng.standard_normal((Tq, d)), rng.standard_normal((Tk, d)), rng.standard_normal((Tk, dv))
    Qc, Kc, Vc = Q.copy(), K.copy(), V.copy()
    o_ref, lse_ref = A.forward_head(Q, K, V, 1.0 / math.sqrt(d), causal)
    for bs in sorted({1, 2, 3, 7, 64, 128, Tk, Tk + 5}):
        o, lse = T.flash_attention(Q, K, V, bs, causal=causal)
        np.testing.assert_allclose(o, o_ref, atol=1e-9, rtol=1e-9)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-9, rtol=1e-9)
    for a, c in ((Q, Qc), (K, Kc), (V, Vc)):
        np.testing.assert_array_equal(a, c)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape,bounds", [
    ((9, 40, 5, 3), [0, 13, 40]),
    ((9, 40, 5, 3), [0, 1, 2, 39, 40]),        # one-key chunks
    ((50, 70, 8, 6), [0, 20, 20, 45, 70]),     # an empty chunk
    ((30, 10, 4, 4), [0, 3, 6, 10]),           # causal: rows 0-2 see no key of the later chunks
])
def test_merged_key_chunks_equal_whole_softmax(shape, bounds, causal):
    """Keys split into chunks, each chunk's state built from the empty state,
    states merged by rescaling to the common maximum: the whole-row softmax."""
    Tq, Tk, d, dv = shape
    rng = np.random.default_rng(Tq + 7 * Tk)
    Q, K, V = rng.standard_normal((Tq, d)), 3 * rng.standard_normal((Tk, d)), rng.standard_normal((Tk, dv))
    o_ref, lse_ref = A.forward_head(Q, K, V, 1.0 / math.sqrt(d), causal)
    for bs in (1, 4, 64):
        o, lse = T.chunked_attention(Q, K, V, bounds, block_size=bs, causal=causal)
        np.testing.assert_allclose(o, o_ref, atol=1e-12, rtol=1e-11)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-12, rtol=1e-12)


def test_merging_states_with_no_key_keeps_the_empty_state():
    empty = (np.full(2, -np.inf), np.zeros(2), np.zeros((2, 3)))
    m, l, acc = T.merge_states([empty, empty])
    assert np.all(np.isneginf(m)) and np.all(l == 0) and np.all(acc == 0)
    one = (np.array([0.5, -1.0]), np.array([2.0, 3.0]), np.ones((2, 3)))
    m, l, acc = T.merge_states([empty, one, empty])
    np.testing.assert_array_equal(m, one[0])
    np.testing.assert_array_equal(l, one[1])
    np.testing.assert_array_equal(acc, one[2])


MERGE_MUTANTS = [
    ("w = np.exp(np.asarray(mc, dtype=np.float64) - ref)", "w = np.exp(ref - np.asarray(mc, dtype=np.float64))"),
    ("l = l + w * np.asarray(lc, dtype=np.float64)", "l = l + np.asarray(lc, dtype=np.float64)"),   # unscaled sums
    ("acc = acc + w[:, None] * np.asarray(ac, dtype=np.float64)", "acc = acc + np.asarray(ac, dtype=np.float64)"),
]


@pytest.mark.parametrize("old,new", MERGE_MUTANTS)
def test_planted_merge_mistakes_are_caught(old, new):
    bad, _ = _mutant(T, "merge_states", old, new)
    ns = dict(vars(T))
    ns["merge_states"] = bad
    src = inspect.getsource(T.chunked_attention)
    exec(compile(src, "<chunked with mutant merge>", "exec"), ns)
    rng = np.random.default_rng(3)
    Q, K, V = rng.standard_normal((6, 4)), 3 * rng.standard_normal((20, 4)), rng.standard_normal((20, 2))
    o_ref, lse_ref = A.forward_head(Q, K, V, 0.5)
    with np.errstate(all="ignore"):
        o, lse = ns["chunked_attention"](Q, K, V, [0, 7, 20], block_size=4, scale=0.5)
    assert not (np.allclose(o, o_ref, atol=1e-6) and np.allclose(lse, lse_ref, atol=1e-6))


def test_huge_scores_across_blocks_stay_finite_and_exact():
    # scores > 1000 in one block and < -1000 in the next (and the reverse)
    d = 4
    Q = np.ones((3, d))
    K = np.concatenate([np.full((4, d), 800.0), np.full((4, d), -800.0), np.full((4, d), 800.0)])
    K[1, 0] += 0.25          # break the tie inside the first block
    V = np.arange(36.0).reshape(12, 3)
    scale = 1.0 / math.sqrt(d)  # scores +-1600
    o_ref, lse_ref = A.forward_head(Q, K, V, scale)
    # closed form: only the +1600 keys count; their exps relative to the max
    s_pos = scale * (K[[0, 1, 2, 3, 8, 9, 10, 11]] @ Q[0])
    w = np.exp(s_pos - s_pos.max())
    o_cf = (w / w.sum()) @ V[[0, 1, 2, 3, 8, 9, 10, 11]]
    lse_cf = s_pos.max() + math.log(w.sum())
    np.testing.assert_allclose(o_ref[0], o_cf, rtol=1e-12)
    assert abs(lse_ref[0] - lse_cf) < 1e-9
    for bs in (1, 3, 4, 5, 8, 12, 20):
        for causal in (False, True):
            o, lse = T.flash_attention(Q, K, V, bs, causal=causal, scale=scale)
            o2, lse2 = A.forward_head(Q, K, V, scale, causal)
            assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
            np.testing.assert_allclose(o, o2, rtol=1e-9, atol=1e-9)
            np.testing.assert_allclose(lse, lse2, rtol=1e-12, atol=1e-9)


# --------------------------------------------------------------------------
# closed forms and special cases
# --------------------------------------------------------------------------

def test_single_key_gives_its_value_and_score():
    rng = np.random.default_rng(1)
    Q, K, V = rng.standard_normal((6, 3)), rng.standard_normal((1, 3)), rng.standard_normal((1, 4))
    o, lse = A.forward_head(Q, K, V, 0.7)
    np.testing.assert_allclose(o, np.repeat(V, 6, axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.7 * (Q @ K[0]), rtol=1e-15, atol=1e-15)


def test_equal_scores_give_mean_value():
    rng = np.random.default_rng(2)
    k = rng.standard_normal(5)
    Q, K, V = rng.standard_normal((4, 5)), np.tile(k, (9, 1)), rng.standard_normal((9, 3))
    o, lse = A.forward_head(Q, K, V, 0.3)
    np.testing.assert_allclose(o, np.tile(V.mean(axis=0), (4, 1)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, 0.3 * (Q @ k) + math.log(9), rtol=1e-13)


def test_causal_first_row_is_first_value_and_top_left_alignment():
    rng = np.random.default_rng(3)
    Q, K, V = rng.standard_normal((5, 4)), rng.standard_normal((3, 4)), rng.standard_normal((3, 2))
    o, lse = A.forward_head(Q, K, V, 0.5, causal=True)
    np.testing.assert_allclose(o[0], V[0], atol=1e-15)
    np.testing.assert_allclose(lse[0], 0.5 * Q[0] @ K[0], rtol=1e-15)
    # rows 2.. see all 3 keys (top-left alignment: key j blocked when j > i)
    o_full, _ = A.forward_head(Q, K, V, 0.5, causal=False)
    np.testing.assert_allclose(o[2:], o_full[2:], rtol=1e-14)


def test_no_keys_gives_zero_output_and_neg_inf_lse():
    o, lse = A.forward_head(np.ones((2, 3)), np.zeros((0, 3)), np.zeros((0, 4)), 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    o, lse = T.flash_attention(np.ones((2, 3)), np.zeros((0, 3)), np.zeros((0, 4)), 4)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def _brute_force_forward(Q, K, V, scale, causal):
    """Scalar loops straight from softmax's definition exp(s_j)/sum_k exp(s_k)."""
    Tq, Tk, dv = len(Q), len(K), len(V[0])
    O = [[0.0] * dv for _ in range(Tq)]
    L = [0.0] * Tq
    for i in range(Tq):
        keys = [j for j in range(Tk) if not (causal and j > i)]
        e = {j: math.exp(scale * math.fsum(Q[i][c] * K[j][c] for c in range(len(Q[i])))) for j in keys}
        z = math.fsum(e.values())
        for c in range(dv):
            O[i][c] = math.fsum(e[j] * V[j][c] for j in keys) / z
        L[i] = math.log(z)
    return np.array(O), np.array(L)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_brute_force_loops(causal):
    rng = np.random.default_rng(4)
    Q, K, V = rng.standard_normal((4, 3)), rng.standard_normal((6, 3)), rng.standard_normal((6, 2))
    o_bf, l_bf = _brute_force_forward(Q.tolist(), K.tolist(), V.tolist(), 0.6, causal)
    o, lse = A.forward_head(Q, K, V, 0.6, causal)
    np.testing.assert_allclose(o, o_bf, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, l_bf, rtol=1e-13, atol=1e-14)


def test_batched_forward_matches_per_head():
    rng = np.random.default_rng(5)
    Q, K, V = rng.standard_normal((2, 3, 7, 4)), rng.standard_normal((2, 3, 9, 4)), rng.standard_normal((2, 3, 9, 5))
    O, L = A.forward(Q, K, V, 0.5, causal=True)
    for b in range(2):
        for h in range(3):
            o, l = _brute_force_forward(Q[b, h].tolist(), K[b, h].tolist(), V[b, h].tolist(), 0.5, True)
            np.testing.assert_allclose(O[b, h], o, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(L[b, h], l, rtol=1e-13)


# --------------------------------------------------------------------------
# backward: central finite differences of the forward, torch.autograd,
# and agreement of the two pages' derivations
# --------------------------------------------------------------------------

def _loss(Q, K, V, dO, scale, causal):
    o, _ = _brute_force_forward(Q.tolist(), K.tolist(), V.tolist(), scale, causal)
    return float(np.sum(o * dO))


def _finite_diff(Q, K, V, dO, scale, causal, h=1e-6):
    grads = []
    for X in (Q, K, V):
        g = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            fp = _loss(Q, K, V, dO, scale, causal)
            X[idx] = old - h
            fm = _loss(Q, K, V, dO, scale, causal)
            X[idx] = old
            g[idx] = (fp - fm) / (2 * h)
        grads.append(g)
    return grads


FD_CASES = [(3, 4, 2, 2, 1.0, False), (3, 4, 2, 2, 1.0, True), (4, 4, 3, 2, 0.37, True),
            (5, 3, 2, 3, 0.8, True), (3, 5, 2, 2, 1 / math.sqrt(2), False)]


@pytest.mark.parametrize("Tq,Tk,d,dv,scale,causal", FD_CASES)
def test_backward_matches_finite_differences(Tq, Tk, d, dv, scale, causal):
    rng = np.random.default_rng(Tq * 7 + Tk)
    Q, K, V = rng.standard_normal((Tq, d)), rng.standard_normal((Tk, d)), rng.standard_normal((Tk, dv))
    dO = rng.standard_normal((Tq, dv))
    r = A.backward_head(Q, K, V, dO, scale, causal)
    fq, fk, fv = _finite_diff(Q, K, V, dO, scale, causal)
    for got, want in ((r["dq"], fq), (r["dk"], fk), (r["dv"], fv)):
        np.testing.assert_allclose(got, want, atol=2e-7, rtol=1e-6)


def _torch_grads(Q, K, V, dO, scale, causal):
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        i = torch.arange(q.shape[-2])[:, None]
        j = torch.arange(k.shape[-2])[None, :]
        s = s.masked_fill(j > i, float("-inf"))
    o = torch.softmax(s, dim=-1) @ v
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return o.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    rng = np.random.default_rng(11)
    Q, K, V = rng.standard_normal((2, 2, 37, 16)), rng.standard_normal((2, 2, 37, 16)), rng.standard_normal((2, 2, 37, 8))
    dO = rng.standard_normal((2, 2, 37, 8))
    r = A.backward(Q, K, V, dO, 0.25, causal, row_chunk=10)
    o, gq, gk, gv = _torch_grads(Q, K, V, dO, 0.25, causal)
    np.testing.assert_allclose(r["O"], o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dQ"], gq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["dK"], gk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["dV"], gv, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["D"], np.sum(o * dO, axis=-1), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_two_pages_backward_derivations_agree(causal):
    rng = np.random.default_rng(12)
    Q, K, V = rng.standard_normal((9, 5)), rng.standard_normal((9, 5)), rng.standard_normal((9, 4))
    dO = rng.standard_normal((9, 4))
    a = A.backward_head(Q, K, V, dO, 0.9, causal)
    b = A.backward_head_matrix_form(Q, K, V, dO, 0.9, causal)
    for k in ("dq", "dk", "dv", "o"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-11, atol=1e-12)


def test_huge_logits_backward_is_finite():
    rng = np.random.default_rng(13)
    Q = rng.standard_normal((6, 4))
    K = rng.standard_normal((10, 4)) * np.where(np.arange(10) // 5 % 2 == 0, 400.0, -400.0)[:, None]
    V, dO = rng.standard_normal((10, 3)), rng.standard_normal((6, 3))
    r = A.backward_head(Q, K, V, dO, 1.0, False)
    for k in ("dq", "dk", "dv", "o", "lse"):
        assert np.all(np.isfinite(r[k]))
    o, gq, gk, gv = _torch_grads(Q, K, V, dO, 1.0, False)
    np.testing.assert_allclose(r["dv"], gv, rtol=1e-9, atol=1e-9)


def test_chunked_rows_equal_unchunked():
    rng = np.random.default_rng(14)
    Q, K, V, dO = (rng.standard_normal(s) for s in ((33, 8), (47, 8), (47, 6), (33, 6)))
    a = A.backward_head(Q, K, V, dO, 0.3, True, row_chunk=5)
    b = A.backward_head(Q, K, V, dO, 0.3, True, row_chunk=4096)
    for k in ("dq", "dk", "dv", "o", "lse", "D"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-12, atol=1e-13)


def test_backward_row_samples_add_up_to_the_full_result():
    rng = np.random.default_rng(16)
    Q, K, V, dO = (rng.standard_normal(s) for s in ((40, 6), (40, 6), (40, 5), (40, 5)))
    full = A.backward_head(Q, K, V, dO, 0.4, True)
    a = A.backward_head(Q, K, V, dO, 0.4, True, row_chunk=7, rows=np.arange(0, 40, 2))
    b = A.backward_head(Q, K, V, dO, 0.4, True, row_chunk=7, rows=np.arange(1, 40, 2))
    np.testing.assert_allclose(a["dk"] + b["dk"], full["dk"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a["dv"] + b["dv"], full["dv"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a["dq"][::2], full["dq"][::2], rtol=1e-12, atol=1e-13)
    assert np.all(a["dq"][1::2] == 0)


def test_sampled_rows_equal_full_rows():
    rng = np.random.default_rng(15)
    Q, K, V = rng.standard_normal((50, 8)), rng.standard_normal((50, 8)), rng.standard_normal((50, 3))
    rows = np.array([0, 7, 8, 49])
    o, l = A.forward_head(Q, K, V, 0.3, True, rows=rows)
    of, lf = A.forward_head(Q, K, V, 0.3, True)
    np.testing.assert_allclose(o, of[rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l, lf[rows], rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# planted mistakes: each plausible slip in the oracle's source must be caught
# --------------------------------------------------------------------------

def _mutant(module, func_name, old, new):
    src = inspect.getsource(getattr(module, func_name))
    assert old in src, (func_name, old)
    ns = dict(vars(module))
    exec(compile(src.replace(old, new, 1), f"<mutant {func_name}>", "exec"), ns)
    return ns[func_name], ns


BWD_MUTANTS = [
    ("scale * (ds @ k)", "(ds @ k)"),                 # dropped scale on dQ
    ("scale * (ds.T @ q[r])", "(ds.T @ q[r])"),       # dropped scale on dK
    ("dp - D[r][:, None]", "dp + D[r][:, None]"),     # wrong sign of D
    ("p.T @ do[r]", "p @ do[r]"),                     # transposed operand
    ("ds.T @ q[r]", "ds @ q[r]"),                     # transposed operand
    ("do[r] @ v.T", "do[r] @ v.T * 0.5"),             # lost factor
]


@pytest.mark.parametrize("old,new", BWD_MUTANTS)
def test_planted_backward_mistakes_are_caught(old, new):
    bad, _ = _mutant(A, "backward_head", old, new)
    Tq, Tk, d, dv, scale, causal = 4, 4, 3, 2, 0.37, True
    rng = np.random.default_rng(Tq * 7 + Tk)
    Q, K, V = rng.standard_normal((Tq, d)), rng.standard_normal((Tk, d)), rng.standard_normal((Tk, dv))
    dO = rng.standard_normal((Tq, dv))
    r = bad(Q, K, V, dO, scale, causal)
    fq, fk, fv = _finite_diff(Q, K, V, dO, scale, causal)
    ok = all(np.allclose(g, w, atol=2e-7, rtol=1e-6) for g, w in ((r["dq"], fq), (r["dk"], fk), (r["dv"], fv)))
    assert not ok


FWD_MUTANTS = [
    ("_scores", "j > row_ids[:, None]", "j >= row_ids[:, None]"),  # off-by-one mask
    ("_scores", "s = scale * (q_rows @ k.T)", "s = (q_rows @ k.T)"),  # dropped scale
    ("_softmax_rows", "m_safe + np.log(", "np.log("),                 # lse missing max
]


@pytest.mark.parametrize("func,old,new", FWD_MUTANTS)
def test_planted_forward_mistakes_are_caught(golden, monkeypatch, func, old, new):
    bad, _ = _mutant(A, func, old, new)
    monkeypatch.setattr(A, func, bad)
    caught = False
    for name in ("example1_no_mask.json", "example2_causal.json"):
        g = golden(name)
        Q, K, V = (np.array(g[k]) for k in ("Q", "K", "V"))
        o, lse = A.forward_head(Q, K, V, 1 / math.sqrt(2), g["causal"])
        caught |= not (np.allclose(o, g["output"], atol=PRINT_TOL) and np.allclose(lse, g["lse"], atol=PRINT_TOL))
    assert caught


STEP_MUTANTS = [
    ("c * l + p.sum(axis=1)", "l + p.sum(axis=1)"),           # no rescale of l
    ("c[:, None] * acc + p @ v_block", "acc + p @ v_block"),  # no rescale of acc
    ("np.exp(m - ref)", "np.exp(ref - m)"),                   # inverted correction
]


@pytest.mark.parametrize("old,new", STEP_MUTANTS)
def test_planted_step_mistakes_are_caught(golden, old, new):
    bad, _ = _mutant(T, "online_softmax_step", old, new)
    g = golden("example3_step.json")
    args = [np.array(g[k]) for k in ("m", "l", "acc", "scores", "v_block")]
    with np.errstate(all="ignore"):
        m, l, acc = bad(*args)
    ok = (np.allclose(l, g["l_new"], atol=PRINT_TOL) and np.allclose(acc, g["acc_new"], atol=PRINT_TOL))
    assert not ok


def test_zero_columns_change_nothing():
    """Zero columns appended to Q and K (d -> dp) and to V and dO (dv -> dvp)
    leave S = scale QK^T, P, LSE and D = rowsum(dO o O) as they were: O and
    the gradients gain zero columns and keep their first d / dv columns. The
    bf16 paths for widths below a tile width rely on exactly this."""
    rng = np.random.default_rng(3)
    Tq, Tk, d, dv, dp, dvp = 37, 53, 40, 24, 64, 128
    q, k = rng.standard_normal((Tq, d)), rng.standard_normal((Tk, d))
    v, do = rng.standard_normal((Tk, dv)), rng.standard_normal((Tq, dv))

    def pad(a, w):
        return np.concatenate([a, np.zeros((a.shape[0], w - a.shape[1]))], axis=1)

    for causal in (False, True):
        r = A.backward_head(q, k, v, do, 0.3, causal)
        rp = A.backward_head(pad(q, dp), pad(k, dp), pad(v, dvp), pad(do, dvp), 0.3, causal)
        np.testing.assert_allclose(rp["lse"], r["lse"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(rp["D"], r["D"], rtol=0, atol=1e-12)
        for key, w in (("o", dv), ("dq", d), ("dk", d), ("dv", dv)):
            np.testing.assert_allclose(rp[key][:, :w], r[key], rtol=0, atol=1e-12)
            assert np.all(rp[key][:, w:] == 0.0)
