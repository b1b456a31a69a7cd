"""Split-KV forward: host-side split arithmetic and validation (CPU), and
parity of the split forward with the float64 oracle and with the plain
forward on the GPU.

The split forward divides each query tile's (bf16: each query-tile pair's)
key tiles into ranges whose partial softmax states are merged by the
associative rescale of "The Hidden Recurrence in Softmax Attention", section
"Chunk-wise Mode with Online Softmax Re-scale"; its result is the same
attention ("Tiled attention with an online softmax", section "Task"), so the
oracle and the tolerances are those of the plain forward of each dtype.
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_softmax_attn_gb300 as B
from exact_tiled_softmax_attn_gb300.workloads import make_random
from oracle import attention as ref

from parity import check_lse, check_o


# ------------------------------------------------------------------ CPU

@pytest.mark.parametrize("Tk,req,want", [
    (128, 4, 1),        # one key tile: no split
    (1000, 3, 3),       # 8 tiles -> 3, 3, 2
    (1000, 5, 4),       # 8 tiles in ranges of 2 -> 4 splits
    (1000, 100, 8),     # clamped to the key tiles
    (65536, 100, 64),   # clamped to 64
    (8192, 1, 1),
])
def test_split_counts(Tk, req, want):
    assert B.attn_fwd_splitkv_splits(1, 1, 128, Tk, 128, 128, B.ATTN_BF16, req) == want


def test_split_count_invalid_and_fp32():
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 128, 128, B.ATTN_BF16, -1) == -1
    # fp32 counts 64-key tiles: 1024 keys are 16 tiles
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 128, 128, B.ATTN_F32, 2) == 2
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 128, 128, B.ATTN_F32, 5) == 4   # ranges of 4 tiles
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 128, 128, B.ATTN_F32, 100) == 16
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 64, 128, 128, B.ATTN_F32, 4) == 1     # one key tile
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 300, 128, B.ATTN_F32, 2) == -1  # beyond 256 columns
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 100, 100, B.ATTN_BF16, 2) == -1
    # padded widths split like the tile width they run on
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 96, 40, B.ATTN_BF16, 2) == 2
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 1024, 72, 200, B.ATTN_BF16, 3) == 3


def test_workspace_size_formula():
    Bn, H, Tq, Tk, d = 2, 3, 300, 1000, 64
    S = B.attn_fwd_splitkv_splits(Bn, H, Tq, Tk, d, d, B.ATTN_BF16, 3)
    rows = Bn * H * Tq
    r256 = lambda x: (x + 255) // 256 * 256
    assert B.attn_fwd_splitkv_workspace_size(Bn, H, Tq, Tk, d, d, B.ATTN_BF16, 3) == \
        r256(S * rows * d * 4) + r256(S * rows * 4)
    assert B.attn_fwd_splitkv_workspace_size(Bn, H, Tq, Tk, d, d, B.ATTN_BF16, 1) == 0
    S = B.attn_fwd_splitkv_splits(Bn, H, Tq, Tk, 7, 13, B.ATTN_F32, 5)
    # fp32: the partial log-sum-exps are fp64
    assert S == 4 and B.attn_fwd_splitkv_workspace_size(Bn, H, Tq, Tk, 7, 13, B.ATTN_F32, 5) == \
        r256(S * rows * 13 * 4) + r256(S * rows * 8)


@pytest.mark.parametrize("kw,status", [
    (dict(num_splits=-1), B.ATTN_ERR_INVALID_ARG),
    (dict(dtype=B.ATTN_F32, num_splits=2, workspace_bytes=1024), B.ATTN_ERR_WORKSPACE),
    (dict(workspace=0, workspace_bytes=0), B.ATTN_ERR_WORKSPACE),
    (dict(workspace_bytes=1024), B.ATTN_ERR_WORKSPACE),
    (dict(workspace=0x9000010), B.ATTN_ERR_WORKSPACE),                  # misaligned
    (dict(workspace=0x100000 - 4096), B.ATTN_ERR_WORKSPACE),            # overlaps Q
])
def test_splitkv_host_validation(kw, status):
    Bn, H, Tq, Tk, d = 1, 1, 128, 1024, 128
    a = dict(Q=0x100000, K=0x200000, V=0x300000, O=0x400000, LSE=0x500000, B=Bn, H=H, Tq=Tq, Tk=Tk, d=d, dv=d,
             scale=0.1, causal=0, dtype=B.ATTN_BF16, num_splits=4, workspace=0x9000000, workspace_bytes=1 << 30)
    a.update(kw)
    assert B.attn_fwd_splitkv(**a, stream=0, check=False) == status


# ------------------------------------------------------------------ GPU

SHAPES = [  # B, H, Tq, Tk, d, num_splits
    (1, 1, 128, 8192, 128, 0),
    (1, 2, 128, 4096, 128, 5),
    (2, 1, 300, 1000, 64, 3),
    (1, 1, 257, 129, 128, 2),
    (1, 1, 700, 70, 64, 2),      # one key tile: no split
    (1, 3, 1, 5000, 64, 7),
    (1, 1, 1000, 3000, 128, 64),
    (1, 2, 1300, 700, 64, 3),    # Tq > Tk: under the causal mask the last query tiles see every key
    (4, 40, 256, 1024, 64, 3),   # 480 units: several split units per CTA
    (8, 40, 256, 256, 64, 2),    # causal: the second range holds no key tile for the first query tile
]


def _x(Bn, H, Tq, Tk, d, seed):
    return make_random((Bn, H, Tq, d), (Bn, H, Tk, d), (Bn, H, Tk, d), seed=seed, dtype=torch.bfloat16,
                       device="cuda")


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_splitkv_matches_oracle(shape, causal):
    Bn, H, Tq, Tk, d, ns = shape
    x = _x(Bn, H, Tq, Tk, d, Tq + 7 * Tk)
    scale = 1.0 / math.sqrt(d)
    o, lse = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale, num_splits=ns)
    torch.cuda.synchronize()
    assert B.attn_device_status() == B.ATTN_OK
    O, L = ref.forward(x["Q"], x["K"], x["V"], scale, causal)
    check_o(o, O, torch.bfloat16)
    check_lse(lse, L, torch.bfloat16)
    # the same attention as the plain forward, up to fp32 rounding order and
    # one bf16 rounding step of the output
    o1, lse1 = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert (lse - lse1).abs().max().item() <= 1e-4
    assert (o.float() - o1.float()).abs().max().item() <= 2.0 ** -7 * max(1.0, o1.float().abs().max().item())


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 200, 3000, 64, 128, 5), (1, 1, 128, 5000, 128, 64, 0)])
def test_splitkv_d_neq_dv(shape, causal):
    Bn, H, Tq, Tk, d, dv, ns = shape
    x = make_random((Bn, H, Tq, d), (Bn, H, Tk, d), (Bn, H, Tk, dv), seed=Tk + dv, dtype=torch.bfloat16,
                    device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale, num_splits=ns)
    torch.cuda.synchronize()
    assert B.attn_device_status() == B.ATTN_OK
    O, L = ref.forward(x["Q"], x["K"], x["V"], scale, causal)
    check_o(o, O, torch.bfloat16)
    check_lse(lse, L, torch.bfloat16)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [
    (1, 2, 128, 3000, 256, 5),    # dv = 256: the merge's second column half
    (1, 1, 300, 1000, 128, 3),    # causal: the last range holds no key tile for the first query tile
    (1, 1, 130, 2000, 64, 0),     # automatic split count
    (2, 3, 1, 700, 256, 64),      # more splits asked for than key tiles
])
def test_splitkv_d256(shape, causal):
    Bn, H, Tq, Tk, dv, ns = shape
    d = 256
    x = make_random((Bn, H, Tq, d), (Bn, H, Tk, d), (Bn, H, Tk, dv), seed=Tq + Tk + dv, dtype=torch.bfloat16,
                    device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale, num_splits=ns)
    torch.cuda.synchronize()
    assert B.attn_device_status() == B.ATTN_OK
    O, L = ref.forward(x["Q"], x["K"], x["V"], scale, causal)
    check_o(o, O, torch.bfloat16)
    check_lse(lse, L, torch.bfloat16)
    o1, lse1 = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert (lse - lse1).abs().max().item() <= 1e-4
    assert (o.float() - o1.float()).abs().max().item() <= 2.0 ** -7 * max(1.0, o1.float().abs().max().item())


F32_SHAPES = [  # B, H, Tq, Tk, d, dv, num_splits
    (1, 2, 70, 300, 48, 40, 2),
    (1, 2, 70, 300, 48, 40, 0),      # automatic: few query tiles, so it splits
    (1, 1, 128, 4000, 128, 128, 0),
    (2, 3, 1, 5000, 64, 64, 7),      # one query row per head
    (1, 1, 200, 1000, 7, 13, 5),     # odd widths
    (1, 2, 300, 700, 128, 128, 64),  # clamped to the key tiles
    (1, 1, 1000, 300, 200, 136, 3),  # Tq > Tk; rows above 128 columns (compensated scores)
    (1, 1, 100, 64, 64, 64, 4),      # one key tile: no split
]


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", F32_SHAPES)
def test_splitkv_fp32_matches_oracle(shape, causal):
    """fp32 split-KV forward (64-row query tiles, 64-key tiles, ranges merged
    in fp32): the oracle at the fp32 bounds, and the plain fp32 forward up to
    fp32 rounding order."""
    Bn, H, Tq, Tk, d, dv, ns = shape
    x = make_random((Bn, H, Tq, d), (Bn, H, Tk, d), (Bn, H, Tk, dv), seed=Tq + 3 * Tk + d, dtype=torch.float32,
                    device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale, num_splits=ns)
    torch.cuda.synchronize()
    assert B.attn_device_status() == B.ATTN_OK
    O, L = ref.forward(x["Q"], x["K"], x["V"], scale, causal)
    check_o(o, O, torch.float32)
    check_lse(lse, L, torch.float32)
    o1, lse1 = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert (lse - lse1).abs().max().item() <= 1e-5 * max(1.0, lse1.abs().max().item())
    assert (o - o1).abs().max().item() <= 1e-5 * max(1.0, o1.abs().max().item())


@pytest.mark.gpu
@pytest.mark.parametrize("scale", [1.0 / math.sqrt(128), 1.0])
def test_splitkv_fp32_banded_keys(scale):
    """The c4 key bands (rows of K scaled by +-40 in alternating 128-key
    bands; logits beyond 1000 at scale 1) through the fp32 split forward: the
    merge weights exp(LSE_s - max) span many orders of magnitude."""
    from exact_tiled_softmax_attn_gb300.workloads import band_signs
    Bn, H, Tq, Tk, d = 1, 2, 100, 4000, 128
    x = make_random((Bn, H, Tq, d), (Bn, H, Tk, d), (Bn, H, Tk, d), seed=41, dtype=torch.float32, device="cpu")
    x["K"] = x["K"] * (40.0 * band_signs(Tk)).view(1, 1, Tk, 1)
    xg = {k: v.cuda() for k, v in x.items()}
    o, lse = B.forward(xg["Q"], xg["K"], xg["V"], causal=False, scale=scale, num_splits=6)
    torch.cuda.synchronize()
    O, L = ref.forward(x["Q"], x["K"], x["V"], scale, False)
    check_o(o, O, torch.float32)
    check_lse(lse, L, torch.float32)


@pytest.mark.gpu
def test_splitkv_long_keys_sampled_rows():
    """B=1 H=4 Tq=256 Tk=65536, automatic split count: sampled query rows of
    two heads against the oracle, with and without the causal mask."""
    Bn, H, Tq, Tk, d = 1, 4, 256, 65536, 128
    x = _x(Bn, H, Tq, Tk, d, 12)
    scale = 1.0 / math.sqrt(d)
    assert B.attn_fwd_splitkv_splits(Bn, H, Tq, Tk, d, d, B.ATTN_BF16, 0) > 1
    rows = [0, 1, 127, 128, 200, 255]
    for causal in (False, True):
        o, lse = B.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale, num_splits=0)
        torch.cuda.synchronize()
        assert B.attn_device_status() == B.ATTN_OK
        for h in (0, 3):
            O, L = ref.forward_head(x["Q"][0, h], x["K"][0, h], x["V"][0, h], scale, causal, rows=rows)
            check_o(o[0, h, rows], O, torch.bfloat16)
            check_lse(lse[0, h, rows], L, torch.bfloat16)
