"""GPU forward vs the CPU float64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_softmax_attn_gb300 as pkg
from exact_tiled_softmax_attn_gb300.workloads import WORKLOADS, make_inputs, make_random
from oracle import attention as ref

from parity import check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg.load_library()
    yield
    assert pkg.attn_device_status() == pkg.ATTN_OK


def run_fwd(x, causal, scale):
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse


def oracle_fwd(x, causal, scale, heads=None):
    return ref.forward(x["Q"], x["K"], x["V"], scale, causal, heads=heads)


# ------------------------------------------------------------------ fp32

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block_n", [32, 64, 128])
def test_f32_c1_every_tile_size(causal, block_n):
    w = WORKLOADS["c1_causal" if causal else "c1"]
    x = make_inputs(w, DEV)
    B, H, Tq, Tk, d, dv = w.B, w.H, w.Tq, w.Tk, w.d, w.dv
    o = torch.empty(B, H, Tq, dv, device=DEV)
    lse = torch.empty(B, H, Tq, device=DEV)
    pkg.attn_fwd_f32_blocked(x["Q"], x["K"], x["V"], o, lse, B, H, Tq, Tk, d, dv, w.softmax_scale, causal,
                             block_n)
    torch.cuda.synchronize()
    O, L = oracle_fwd(x, causal, w.softmax_scale)
    check_o(o, O, torch.float32)
    check_lse(lse, L, torch.float32)


F32_SHAPES = [  # B, H, Tq, Tk, d, dv
    (1, 1, 1, 1, 1, 1),
    (2, 3, 77, 133, 40, 24),
    (1, 2, 200, 65, 128, 128),
    (1, 1, 33, 300, 7, 128),
    (3, 1, 64, 64, 64, 64),
    (1, 2, 100, 150, 256, 256),   # head sizes above 128
    (1, 1, 70, 90, 200, 136),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", F32_SHAPES)
def test_f32_ragged_shapes(shape, causal):
    B, H, Tq, Tk, d, dv = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + Tk, device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(x, causal, scale)
    O, L = oracle_fwd(x, causal, scale)
    check_o(o, O, torch.float32)
    check_lse(lse, L, torch.float32)


@pytest.mark.parametrize("name", ["c4", "c4_scale1"])
def test_f32_c4_banded_keys_full_size(name):
    w = WORKLOADS[name]
    x = make_inputs(w, DEV)
    o, lse = run_fwd(x, w.causal, w.softmax_scale)
    O, L = oracle_fwd(x, w.causal, w.softmax_scale)
    if name == "c4_scale1":
        assert np.abs(L).max() > 1000      # the logits really pass +-1000
    check_o(o, O, torch.float32)
    check_lse(lse, L, torch.float32)


# ------------------------------------------------------------------ bf16

BF16_SHAPES = [  # B, H, Tq, Tk, d
    (1, 1, 1, 1, 64),
    (2, 3, 300, 300, 64),
    (1, 2, 257, 129, 128),
    (1, 1, 128, 1000, 128),
    (2, 2, 512, 512, 128),
    (1, 1, 700, 70, 64),
]


MIXED_DV_SHAPES = [  # B, H, Tq, Tk, d, dv
    (1, 2, 300, 257, 64, 128),
    (2, 1, 200, 700, 128, 64),
    (1, 1, 1024, 1024, 64, 128),
    (1, 1, 129, 4000, 128, 64),
]


D256_SHAPES = [  # B, H, Tq, Tk, dv: d = 256, 128-key tiles; dv > 64 on CTA pairs (two query tiles per unit)
    (1, 2, 300, 257, 256),    # three query tiles: the second pair's second CTA has no rows
    (1, 3, 77, 300, 256),     # one query tile: no pair has a second tile
    (2, 1, 129, 700, 128),
    (1, 1, 1, 1, 64),
    (1, 2, 512, 512, 256),
    (3, 60, 200, 200, 256),   # several units per CTA
    (1, 1, 1000, 64, 128),    # the second 64-key half of the only V tile lies past Tk
    (1, 2, 130, 100, 256),    # a partial second half
    (1, 1, 640, 1000, 64),    # causal units of 1 to 5 key tiles, ragged last tile
]


PAD_SHAPES = [  # B, H, Tq, Tk, d, dv: widths below the tile width they run on (zero columns)
    (1, 2, 200, 300, 96, 96),      # the d <= 128 kernel at 128 / 128
    (2, 1, 130, 257, 40, 72),      # 64 / 128
    (1, 1, 300, 500, 120, 8),      # dv = 8: one 16-byte store per row
    (1, 2, 129, 200, 200, 136),    # the wide-row kernel, V tile 256
    (1, 1, 257, 300, 64, 256),     # d = 64 on the wide-row kernel (dv = 256)
    (1, 1, 100, 140, 248, 24),     # V tile 64 on the wide-row kernel
    (3, 40, 200, 200, 96, 40),     # several units per CTA
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("split", [None, 3])
@pytest.mark.parametrize("shape", PAD_SHAPES)
def test_bf16_padded_widths(shape, split, causal):
    """d, dv multiples of 8 below 64 / 128 / 256 run on the next tile width:
    the same result as the oracle, and nothing is written past O's last row
    (O lies at the start of a larger buffer filled with a sentinel)."""
    B, H, Tq, Tk, d, dv = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + Tk + d + dv, dtype=torch.bfloat16,
                    device=DEV)
    scale = 1 / math.sqrt(d)
    n = B * H * Tq * dv
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device=DEV)
    o = buf[:n].view(B, H, Tq, dv)
    lse = torch.empty(B, H, Tq, dtype=torch.float32, device=DEV)
    if split is None:
        pkg.attn_fwd(x["Q"], x["K"], x["V"], o, lse, B, H, Tq, Tk, d, dv, scale, causal, pkg.ATTN_BF16)
    else:
        nbytes = pkg.attn_fwd_splitkv_workspace_size(B, H, Tq, Tk, d, dv, pkg.ATTN_BF16, split)
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=DEV)
        pkg.attn_fwd_splitkv(x["Q"], x["K"], x["V"], o, lse, B, H, Tq, Tk, d, dv, scale, causal, pkg.ATTN_BF16,
                             split, ws, ws.numel())
    torch.cuda.synchronize()
    assert pkg.attn_device_status() == pkg.ATTN_OK
    assert torch.all(buf[n:] == 7.0)
    O, L = oracle_fwd(x, causal, scale)
    check_o(o, O, torch.bfloat16)
    check_lse(lse, L, torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", D256_SHAPES)
def test_bf16_d256_forward(shape, causal):
    B, H, Tq, Tk, dv = shape
    d = 256
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + 3 * Tk + dv, dtype=torch.bfloat16,
                    device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(x, causal, scale)
    assert o.shape == (B, H, Tq, dv)
    heads = [(0, 0), (B - 1, H - 1)]
    O, L = oracle_fwd(x, causal, scale, heads=heads)
    check_o(torch.stack([o[b, h] for b, h in heads]), np.stack([np.asarray(O)[b, h] for b, h in heads]),
            torch.bfloat16)
    check_lse(torch.stack([lse[b, h] for b, h in heads]), np.stack([np.asarray(L)[b, h] for b, h in heads]),
              torch.bfloat16)


def test_bf16_d256_large_logits():
    # scores beyond +-1000 across 64-key tiles stay finite and exact
    B, H, T, d = 1, 1, 384, 256
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=6, dtype=torch.float32, device="cpu")
    sign = torch.where((torch.arange(T) // 64) % 2 == 0, 30.0, -30.0).view(1, 1, T, 1)
    x = {k: (v * sign if k == "K" else v).to(torch.bfloat16).to(DEV) for k, v in x.items()}
    for causal in (False, True):
        o, lse = run_fwd(x, causal, 1.0)
        O, L = oracle_fwd(x, causal, 1.0)
        assert np.abs(L).max() > 1000
        check_o(o, O, torch.bfloat16)
        check_lse(lse, L, torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", MIXED_DV_SHAPES)
def test_bf16_d_neq_dv(shape, causal):
    B, H, Tq, Tk, d, dv = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + 5 * Tk + d, dtype=torch.bfloat16,
                    device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(x, causal, scale)
    assert o.shape == (B, H, Tq, dv)
    O, L = oracle_fwd(x, causal, scale)
    check_o(o, O, torch.bfloat16)
    check_lse(lse, L, torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", BF16_SHAPES)
def test_bf16_ragged_shapes(shape, causal):
    B, H, Tq, Tk, d = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, d), seed=Tq * 3 + Tk, dtype=torch.bfloat16,
                    device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(x, causal, scale)
    O, L = oracle_fwd(x, causal, scale)
    check_o(o, O, torch.bfloat16)
    check_lse(lse, L, torch.bfloat16)


def test_bf16_large_logits_across_tiles():
    # scores beyond +-1000 in alternating 128-key bands stay finite and exact
    B, H, T, d = 1, 2, 640, 128
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=5, dtype=torch.float32, device="cpu")
    sign = torch.where((torch.arange(T) // 128) % 2 == 0, 40.0, -40.0).view(1, 1, T, 1)
    x = {k: (v * sign if k == "K" else v).to(torch.bfloat16).to(DEV) for k, v in x.items()}
    for causal in (False, True):
        o, lse = run_fwd(x, causal, 1.0)
        O, L = oracle_fwd(x, causal, 1.0)
        assert np.abs(L).max() > 1000
        check_o(o, O, torch.bfloat16)
        check_lse(lse, L, torch.bfloat16)


def test_bf16_c2_full_size():
    w = WORKLOADS["c2"]
    x = make_inputs(w, DEV)
    o, lse = run_fwd(x, w.causal, w.softmax_scale)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    O, L = oracle_fwd(x, w.causal, w.softmax_scale, heads=heads)
    check_o(o, O, torch.bfloat16)
    check_lse(lse, L, torch.bfloat16)


@pytest.mark.parametrize("name,heads", [("c3", [(0, 0), (1, 15)]), ("c5", [(0, 7)]), ("m1", [(1, 3)]),
                                        ("w256", [(0, 0), (1, 15)])])
def test_bf16_full_size_sampled_heads(name, heads):
    w = WORKLOADS[name]
    x = make_inputs(w, DEV, with_dO=False)
    o, lse = run_fwd(x, w.causal, w.softmax_scale)
    rows = np.unique(np.concatenate([np.arange(0, 200), np.arange(w.Tq - 200, w.Tq),
                                     np.random.default_rng(0).integers(0, w.Tq, 600)]))
    for b, h in heads:
        O, L = ref.forward_head(x["Q"][b, h], x["K"][b, h], x["V"][b, h], w.softmax_scale, w.causal, rows=rows)
        check_o(o[b, h, rows], O, torch.bfloat16)
        check_lse(lse[b, h, rows], L, torch.bfloat16)


# ------------------------------------------------------------------ edge cases and invariants

@pytest.mark.parametrize("dt,d", [(torch.float32, 32), (torch.bfloat16, 64)])
def test_no_keys_gives_zero_and_neg_inf(dt, d):
    x = make_random((2, 2, 5, d), (2, 2, 0, d), (2, 2, 0, d), seed=1, dtype=dt, device=DEV)
    o, lse = run_fwd(x, False, 0.3)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_inputs_unchanged_and_repeatable(dt):
    x = make_random((1, 2, 200, 64), (1, 2, 300, 64), (1, 2, 300, 64), seed=3, dtype=dt, device=DEV)
    keep = {k: v.clone() for k, v in x.items()}
    o1, l1 = run_fwd(x, True, 0.125)
    o2, l2 = run_fwd(x, True, 0.125)
    for k in x:
        assert torch.equal(x[k], keep[k]), k
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
