"""The device-side online-softmax step against the oracle's step (and the
page's printed step example), through the C ABI."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_softmax_attn_gb300 as pkg
from exact_tiled_softmax_attn_gb300.workloads import make_random
from oracle import attention as ref
from oracle import tiled as T

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 1e-5   # fp32 state: max |x - ref| / max |ref|


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg.load_library()
    yield
    assert pkg.attn_device_status() == pkg.ATTN_OK


def dev(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(DEV).contiguous()


def step(m, l, acc, scores, v):
    m, l, acc = dev(m), dev(l), dev(acc)
    n, bs = np.shape(scores)
    pkg.attn_online_softmax_step(m, l, acc, dev(scores), dev(v), n, bs, acc.shape[1])
    torch.cuda.synchronize()
    return m.cpu().double().numpy(), l.cpu().double().numpy(), acc.cpu().double().numpy()


def rel(x, r):
    x, r = np.asarray(x, np.float64), np.asarray(r, np.float64)
    fin = np.isfinite(r)
    assert np.array_equal(np.isneginf(x), np.isneginf(r))
    den = max(np.abs(r[fin]).max(), 1e-30) if fin.any() else 1.0
    return np.abs(x[fin] - r[fin]).max() / den if fin.any() else 0.0


def test_page_example(golden):
    g = golden("example3_step.json")
    m, l, acc = step(g["m"], g["l"], g["acc"], g["scores"], g["v_block"])
    tol = 0.5 * 10.0 ** -g["printed_decimals"] + 1e-7
    np.testing.assert_allclose(m, g["m_new"], atol=tol, rtol=0)
    np.testing.assert_allclose(l, g["l_new"], atol=tol, rtol=0)
    np.testing.assert_allclose(acc, g["acc_new"], atol=tol, rtol=0)


@pytest.mark.parametrize("n,bs,dv", [(1, 1, 1), (37, 0, 5), (200, 129, 64), (64, 1500, 128), (5, 3000, 512)])
def test_random_blocks_with_blocked_keys(n, bs, dv):
    rng = np.random.default_rng(n * 7 + bs)
    m = rng.normal(size=n) * 3
    m[::4] = -np.inf                                  # rows with no key so far
    l = np.where(np.isneginf(m), 0.0, rng.uniform(0.5, 3.0, size=n))
    acc = np.where(np.isneginf(m)[:, None], 0.0, rng.normal(size=(n, dv)))
    s = rng.normal(size=(n, bs)) * 4
    s[rng.random((n, bs)) < 0.3] = -np.inf           # blocked keys
    if n > 2 and bs:
        s[1] = -np.inf                                # a row whose block is all blocked
    v = rng.normal(size=(bs, dv))
    m32, l32, a32, s32, v32 = (np.asarray(t, np.float32) for t in (m, l, acc, s, v))
    got = step(m32, l32, a32, s32, v32)
    want = T.online_softmax_step(m32, l32, a32, s32, v32)
    for g_, w_, name in zip(got, want, ("m", "l", "acc")):
        assert rel(g_, w_) <= TOL, name


@pytest.mark.parametrize("block", [1, 48, 128, 1000])
def test_chained_steps_give_attention(block):
    # fold a whole causal head block by block, then O = acc / l, LSE = m + log l
    x = make_random((1, 1, 150, 32), (1, 1, 300, 32), (1, 1, 300, 24), seed=12, dtype=torch.float32, device="cpu")
    Q, K, V = (x[k][0, 0].double().numpy() for k in ("Q", "K", "V"))
    scale = 0.3
    n, Tk, dv = Q.shape[0], K.shape[0], V.shape[1]
    m = dev(np.full(n, -np.inf)); l = dev(np.zeros(n)); acc = dev(np.zeros((n, dv)))
    for b0 in range(0, Tk, block):
        b1 = min(Tk, b0 + block)
        s = scale * Q @ K[b0:b1].T
        s[np.arange(b0, b1)[None, :] > np.arange(n)[:, None]] = -np.inf
        pkg.attn_online_softmax_step(m, l, acc, dev(s), dev(V[b0:b1]), n, b1 - b0, dv)
    torch.cuda.synchronize()
    O_ref, L_ref = ref.forward_head(Q, K, V, scale, True)
    mm, ll, aa = (t.cpu().double().numpy() for t in (m, l, acc))
    assert rel(aa / ll[:, None], O_ref) <= TOL
    assert rel(mm + np.log(ll), L_ref) <= TOL
