"""GPU backward vs the CPU float64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_softmax_attn_gb300 as pkg
from exact_tiled_softmax_attn_gb300.workloads import WORKLOADS, make_inputs, make_random
from oracle import attention as ref

from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg.load_library()
    yield
    assert pkg.attn_device_status() == pkg.ATTN_OK


def run(x, causal, scale, deterministic):
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    dq, dk, dv = pkg.backward(x["Q"], x["K"], x["V"], o, lse, x["dO"], causal=causal, scale=scale,
                              deterministic=deterministic)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def check_all(x, causal, scale, dt, deterministic, heads=None):
    o, lse, dq, dk, dv = run(x, causal, scale, deterministic)
    r = ref.backward(x["Q"], x["K"], x["V"], x["dO"], scale, causal, heads=heads)
    sel = (lambda t: t) if heads is None else (lambda t: np.stack([np.asarray(t)[b, h] for b, h in heads]))
    tsel = (lambda t: t) if heads is None else (lambda t: torch.stack([t[b, h] for b, h in heads]))
    check_o(tsel(o), sel(r["O"]), dt)
    check_lse(tsel(lse), sel(r["LSE"]), dt)
    check_grad(tsel(dq), sel(r["dQ"]), dt, "dQ")
    check_grad(tsel(dk), sel(r["dK"]), dt, "dK")
    check_grad(tsel(dv), sel(r["dV"]), dt, "dV")


# ------------------------------------------------------------------ fp32

@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("name", ["c1", "c1_causal"])
def test_f32_c1(name, deterministic):
    w = WORKLOADS[name]
    check_all(make_inputs(w, DEV), w.causal, w.softmax_scale, torch.float32, deterministic)


F32_SHAPES = [(1, 1, 1, 1, 1, 1), (2, 3, 77, 133, 40, 24), (1, 2, 200, 65, 128, 128), (1, 1, 33, 300, 7, 128),
              (1, 2, 100, 150, 256, 256), (1, 1, 70, 90, 200, 136),   # head sizes above 128
              (2, 3, 150, 64, 128, 128)]   # one 64-key tile: the deterministic dK/dV kernel writes dQ itself


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", F32_SHAPES)
def test_f32_ragged(shape, causal, deterministic):
    B, H, Tq, Tk, d, dv = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + 2 * Tk, device=DEV)
    check_all(x, causal, 1 / math.sqrt(d), torch.float32, deterministic)


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("name", ["c4", "c4_scale1"])
def test_f32_c4_full_size(name, deterministic):
    w = WORKLOADS[name]
    check_all(make_inputs(w, DEV), w.causal, w.softmax_scale, torch.float32, deterministic)


def _split_edge_rows(rng, n, d, scaled=False):
    """n fp32 rows of d entries from patterns aimed at the exact row split of
    the fp32 score products: zero rows; one entry of 3 among entries 2^20
    smaller; every entry on a rounding tie of the split grid; subnormal rows;
    a largest entry that is an exact power of two, with entries of +-that
    size; a largest entry that rounds to the end of the grid (256 steps);
    plain normals; with `scaled`, also normals scaled by 40. (With the dense
    +-2 rows those give logits in the thousands, where an fp32 backward with
    exact logits already misses the 1e-4 gradient bound: the backward cases
    leave them to the c4 workloads.)"""
    x = rng.standard_normal((n, d)).astype(np.float32)
    for i, kind in enumerate(rng.integers(0, 8 if scaled else 7, n)):
        if kind == 0:
            x[i] = 0.0
        elif kind == 1:
            x[i] *= np.float32(2.0 ** -20)
            x[i, rng.integers(d)] = 3.0
        elif kind == 2:
            x[i] = (rng.integers(-255, 255, d) + 0.5) / 128.0   # largest entry in [1, 2): grid step 2^-7
            x[i, 0] = 1.0
        elif kind == 3:
            x[i] = (x[i].astype(np.float64) * 1e-40).astype(np.float32)
        elif kind == 4:
            x[i] = np.where(rng.random(d) < 0.5, -2.0, 2.0) * (rng.random(d) < 0.7)
            x[i, 0] = 2.0
        elif kind == 5:
            x[i] = rng.uniform(-1.0, 1.0, d)
            x[i, 0] = np.float32(1.9999999)
        elif kind == 7:
            x[i] *= 40.0
    return x


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (120, 72)])
def test_f32_split_edge_rows(d, dv, causal, deterministic):
    B, H, Tq, Tk = 1, 2, 77, 150
    rng = np.random.default_rng(1000 + d + dv)
    Q = _split_edge_rows(rng, B * H * Tq, d).reshape(B, H, Tq, d)
    K = _split_edge_rows(rng, B * H * Tk, d).reshape(B, H, Tk, d)
    V = rng.standard_normal((B, H, Tk, dv)).astype(np.float32)
    dO = rng.standard_normal((B, H, Tq, dv)).astype(np.float32)
    x = {k: torch.from_numpy(v).to(DEV) for k, v in (("Q", Q), ("K", K), ("V", V), ("dO", dO))}
    check_all(x, causal, 1 / math.sqrt(d), torch.float32, deterministic)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (120, 72)])
def test_f32_split_edge_rows_forward_large_logits(d, dv, causal):
    B, H, Tq, Tk = 1, 2, 77, 150
    rng = np.random.default_rng(2000 + d + dv)
    Q = _split_edge_rows(rng, B * H * Tq, d, scaled=True).reshape(B, H, Tq, d)
    K = _split_edge_rows(rng, B * H * Tk, d, scaled=True).reshape(B, H, Tk, d)
    V = rng.standard_normal((B, H, Tk, dv)).astype(np.float32)
    x = {k: torch.from_numpy(v).to(DEV) for k, v in (("Q", Q), ("K", K), ("V", V))}
    scale = 1 / math.sqrt(d)
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    torch.cuda.synchronize()
    O, L = ref.forward(x["Q"], x["K"], x["V"], scale, causal)
    assert np.abs(np.asarray(L)[np.isfinite(L)]).max() > 1000   # logits in the thousands
    check_o(o, O, torch.float32)
    check_lse(lse, L, torch.float32)


def test_f32_deterministic_is_bitwise_repeatable():
    w = WORKLOADS["c1_causal"]
    x = make_inputs(w.with_(H=3, Tq=300, Tk=300), DEV)
    a = run(x, True, w.softmax_scale, 1)
    b = run(x, True, w.softmax_scale, 1)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("dt,d", [(torch.float32, 16), (torch.bfloat16, 64)])
@pytest.mark.parametrize("Tq,Tk", [(0, 5), (5, 0)])
def test_empty_sides_give_zero_gradients(dt, d, Tq, Tk):
    x = make_random((1, 2, Tq, d), (1, 2, Tk, d), (1, 2, Tk, d), seed=2, dtype=dt, device=DEV)
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=False, scale=0.2)
    dq, dk, dv = [torch.full_like(t, 7.0) for t in (x["Q"], x["K"], x["V"])]
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)
    pkg.attn_bwd(x["Q"], x["K"], x["V"], o, lse, x["dO"], dq, dk, dv, 1, 2, Tq, Tk, d, d, 0.2, 0,
                 pkg.ATTN_F32 if dt == torch.float32 else pkg.ATTN_BF16, 0, ws, ws.numel())
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.all(t == 0)


# ------------------------------------------------------------------ bf16

BF16_SHAPES = [  # B, H, Tq, Tk, d
    (1, 1, 1, 1, 64),
    (2, 3, 300, 300, 64),
    (1, 2, 257, 129, 128),
    (1, 1, 130, 700, 128),
    (2, 2, 512, 512, 128),
    (1, 1, 700, 70, 64),
]


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", BF16_SHAPES)
def test_bf16_ragged(shape, causal, deterministic):
    B, H, Tq, Tk, d = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, d), seed=Tq * 5 + Tk, dtype=torch.bfloat16,
                    device=DEV)
    check_all(x, causal, 1 / math.sqrt(d), torch.bfloat16, deterministic)


MIXED_DV_SHAPES = [  # B, H, Tq, Tk, d, dv
    (1, 2, 300, 257, 64, 128),
    (2, 1, 200, 700, 128, 64),
    (1, 1, 640, 640, 64, 128),
    (1, 1, 257, 1000, 128, 64),
]


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", MIXED_DV_SHAPES)
def test_bf16_d_neq_dv(shape, causal, deterministic):
    B, H, Tq, Tk, d, dv = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq * 3 + Tk + dv, dtype=torch.bfloat16,
                    device=DEV)
    check_all(x, causal, 1 / math.sqrt(d), torch.bfloat16, deterministic)


PAD_BWD_SHAPES = [  # B, H, Tq, Tk, d, dv: bf16 widths other than 64 / 128 (zero-padded copies)
    (1, 2, 200, 300, 96, 96),
    (2, 1, 130, 257, 40, 72),
    (1, 1, 300, 500, 120, 8),
]


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", PAD_BWD_SHAPES)
def test_bf16_padded_widths_backward(shape, causal, deterministic):
    B, H, Tq, Tk, d, dv = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + Tk + d + 5 * dv, dtype=torch.bfloat16,
                    device=DEV)
    check_all(x, causal, 1 / math.sqrt(d), torch.bfloat16, deterministic)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_padded_widths_split_dq(causal):
    """Few query tiles against many keys at a padded width: the deterministic
    dQ pass of the padded problem splits its key ranges."""
    B, H, Tq, Tk, d, dv = 1, 1, 128, 4096, 96, 96
    assert pkg.attn_bwd_dq_splits(B, H, Tq, Tk, d, dv, pkg.ATTN_BF16, 1) > 1
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=23, dtype=torch.bfloat16, device=DEV)
    check_all(x, causal, 1 / math.sqrt(d), torch.bfloat16, 1)


def test_bf16_padded_backward_writes_only_its_gradients():
    """The cropped gradients land in place: a sentinel after each of dQ, dK,
    dV is untouched."""
    B, H, Tq, Tk, d, dv = 1, 2, 150, 200, 40, 24
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=11, dtype=torch.bfloat16, device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=True, scale=scale)
    outs = []
    for shape in ((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv)):
        n = math.prod(shape)
        buf = torch.full((n + 2048,), 5.0, dtype=torch.bfloat16, device=DEV)
        outs.append((buf, n, buf[:n].view(shape)))
    ws_bytes = pkg.attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, pkg.ATTN_BF16, 1)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    pkg.attn_bwd(x["Q"], x["K"], x["V"], o, lse, x["dO"], outs[0][2], outs[1][2], outs[2][2], B, H, Tq, Tk, d, dv,
                 scale, 1, pkg.ATTN_BF16, 1, ws, ws.numel())
    torch.cuda.synchronize()
    assert pkg.attn_device_status() == pkg.ATTN_OK
    for buf, n, _ in outs:
        assert torch.all(buf[n:] == 5.0)
    r = ref.backward(x["Q"], x["K"], x["V"], x["dO"], scale, True)
    for (_, _, g), name in zip(outs, ("dQ", "dK", "dV")):
        check_grad(g, r[name], torch.bfloat16, name)


SPLIT_DQ_SHAPES = [  # B, H, Tq, Tk, d, dv: few query tiles, many key tiles
    (1, 1, 1, 5000, 128, 128),     # one query row: 9 key ranges
    (1, 2, 128, 4096, 128, 128),
    (1, 1, 256, 3000, 64, 128),
    (2, 1, 200, 2500, 128, 64),
    (1, 1, 1300, 1100, 128, 128),  # Tq > Tk: causal query tiles see 1 ... all 9 key tiles
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SPLIT_DQ_SHAPES)
def test_bf16_split_dq_deterministic(shape, causal):
    """The deterministic backward with dQ split over key ranges (partials
    added in split order): parity with the oracle, bitwise equal across two
    runs, and close to the atomic mode."""
    B, H, Tq, Tk, d, dv = shape
    assert pkg.attn_bwd_dq_splits(B, H, Tq, Tk, d, dv, pkg.ATTN_BF16, 1) > 1
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + Tk, dtype=torch.bfloat16, device=DEV)
    scale = 1 / math.sqrt(d)
    check_all(x, causal, scale, torch.bfloat16, 1)
    o, lse, dq1, dk1, dv1 = run(x, causal, scale, 1)
    _, _, dq2, dk2, dv2 = run(x, causal, scale, 1)
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    # the atomic mode forms dS from S^T in its own kernel (other fp32 rounding
    # before the bf16 dS): the two agree to about twice one mode's error
    # (absolute floor: one causal query row has dQ = 0 exactly, both modes give rounding noise)
    _, _, dqa, _, _ = run(x, causal, scale, 0)
    assert (dq1.float() - dqa.float()).norm() <= 1e-2 * dqa.float().norm() + 1e-5


F32_SPLIT_DQ_SHAPES = [  # B, H, Tq, Tk, d, dv: a dQ partial per 64-key tile from the dK/dV kernel
    (1, 1, 1, 5000, 128, 128),     # one query row, 79 key tiles
    (1, 2, 128, 8192, 128, 128),   # 128 key tiles
    (1, 1, 256, 3000, 64, 64),     # 64-key steps (rows of 64 columns)
    (2, 1, 200, 2500, 40, 24),     # odd widths (scalar partial stores)
    (1, 1, 1300, 1100, 128, 128),  # Tq > Tk: causal query tiles see 1 ... all 18 key tiles
    (1, 1, 100, 900, 200, 136),    # rows above 128 columns (compensated scores, K whole in shared memory)
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", F32_SPLIT_DQ_SHAPES)
def test_f32_split_dq_deterministic(shape, causal):
    """The fp32 deterministic backward with a dQ partial per 64-key tile,
    written by the dK/dV kernel and added in key-tile order: parity with the
    oracle at the fp32 bounds, bitwise equal across two runs, dK and dV
    bitwise equal to the atomic mode's (the same kernel; only where the dQ
    share goes differs), and dQ equal to it up to fp32 rounding order."""
    B, H, Tq, Tk, d, dv = shape
    assert pkg.attn_bwd_dq_splits(B, H, Tq, Tk, d, dv, pkg.ATTN_F32, 1) > 1
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + Tk + d, device=DEV)
    scale = 1 / math.sqrt(d)
    check_all(x, causal, scale, torch.float32, 1)
    _, _, dq1, dk1, dv1 = run(x, causal, scale, 1)
    _, _, dq2, dk2, dv2 = run(x, causal, scale, 1)
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    _, _, dqa, dka, dva = run(x, causal, scale, 0)
    assert torch.equal(dk1, dka) and torch.equal(dv1, dva)
    assert (dq1 - dqa).abs().max().item() <= 1e-5 * max(dqa.abs().max().item(), 1e-30) + 1e-7


@pytest.mark.parametrize("causal", [False, True])
def test_f32_dq_kernel_ranges_above_the_partials_cap(causal):
    """Above 1 GiB of per-key-tile partials the fp32 deterministic backward
    runs the dQ kernel over key ranges (7 ranges of 147 key tiles here, 2 GiB
    of partials otherwise). The shape is too large for the oracle, so the
    path is held to the ones the oracle pins: bitwise equal across two runs,
    dK and dV bitwise equal to the atomic mode's (the same dK/dV kernel and
    order), dQ equal to the atomic mode's up to fp32 rounding order. The dQ
    kernel's ranges themselves met the oracle before the partials moved into
    the dK/dV kernel, and their code has not changed since."""
    B, H, Tq, Tk, d = 1, 8, 512, 65536, 128
    assert pkg.attn_bwd_dq_splits(B, H, Tq, Tk, d, d, pkg.ATTN_F32, 1) == 7
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, d), seed=11 + causal, device=DEV)
    scale = 1 / math.sqrt(d)
    _, _, dq1, dk1, dv1 = run(x, causal, scale, 1)
    _, _, dq2, dk2, dv2 = run(x, causal, scale, 1)
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    _, _, dqa, dka, dva = run(x, causal, scale, 0)
    assert torch.equal(dk1, dka) and torch.equal(dv1, dva)
    assert torch.isfinite(dq1).all()
    assert (dq1 - dqa).abs().max().item() <= 1e-5 * max(dqa.abs().max().item(), 1e-30) + 1e-7


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(20, 16, 130, 128), (40, 8, 256, 64), (75, 4, 70, 128), (3, 100, 1, 64)])
def test_bf16_many_short_units(shape, causal, deterministic):
    """More units than SMs, each of one or two tiles: every kernel walks
    several short units per CTA, so tile loads for the next unit overlap the
    last steps of the previous one."""
    B, H, T, d = shape
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=B * H + T, dtype=torch.bfloat16, device=DEV)
    check_all(x, causal, 1 / math.sqrt(d), torch.bfloat16, deterministic,
              heads=[(0, 0), (B // 2, H // 2), (B - 1, H - 1)])


@pytest.mark.parametrize("deterministic", [0, 1])
def test_bf16_many_small_heads(deterministic):
    """256 heads of 200 rows: far more units than SMs, every unit ragged."""
    B, H, T, d = 16, 16, 200, 64
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=21, dtype=torch.bfloat16, device=DEV)
    check_all(x, True, 1 / math.sqrt(d), torch.bfloat16, deterministic, heads=[(0, 0), (7, 9), (15, 15)])


@pytest.mark.parametrize("deterministic", [0, 1])
def test_bf16_c2_full_size(deterministic):
    w = WORKLOADS["c2"]
    check_all(make_inputs(w, DEV), w.causal, w.softmax_scale, torch.bfloat16, deterministic)


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("name,heads", [("c3", [(0, 3), (1, 12)]), ("c5", [(0, 31)])])
def test_bf16_full_size_sampled_heads(name, heads, deterministic):
    w = WORKLOADS[name]
    check_all(make_inputs(w, DEV), w.causal, w.softmax_scale, torch.bfloat16, deterministic, heads=heads)


def test_bf16_large_logits_across_tiles():
    B, H, T, d = 1, 2, 640, 128
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=9, device="cpu")
    sign = torch.where((torch.arange(T) // 128) % 2 == 0, 40.0, -40.0).view(1, 1, T, 1)
    x = {k: (v * sign if k == "K" else v).to(torch.bfloat16).to(DEV) for k, v in x.items()}
    for causal in (False, True):
        for det in (0, 1):
            check_all(x, causal, 1.0 / math.sqrt(d), torch.bfloat16, det)


def test_bf16_deterministic_is_bitwise_repeatable():
    x = make_random((2, 3, 700, 128), (2, 3, 700, 128), (2, 3, 700, 128), seed=4, dtype=torch.bfloat16,
                    device=DEV)
    a = run(x, True, 0.088, 1)
    b = run(x, True, 0.088, 1)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_bf16_atomic_and_deterministic_agree():
    x = make_random((1, 4, 1024, 64), (1, 4, 1024, 64), (1, 4, 1024, 64), seed=6, dtype=torch.bfloat16,
                    device=DEV)
    a = run(x, True, 0.125, 0)
    b = run(x, True, 0.125, 1)
    for u, v, name in zip(a[2:], b[2:], ("dQ", "dK", "dV")):
        check_grad(u, v, torch.bfloat16, name)
    # dK and dV differ only through D, which the two modes sum in a
    # different order (the deterministic dQ kernel forms it itself)
    for u, v, name in zip(a[3:], b[3:], ("dK", "dV")):
        err = (u.float() - v.float()).norm() / v.float().norm()
        assert err <= 2e-3, f"{name} differs between dQ modes by {err:.2e}"


def test_bf16_inputs_unchanged():
    x = make_random((1, 2, 300, 64), (1, 2, 200, 64), (1, 2, 200, 64), seed=8, dtype=torch.bfloat16, device=DEV)
    keep = {k: v.clone() for k, v in x.items()}
    o, lse, *_ = run(x, False, 0.1, 0)
    o2, lse2 = o.clone(), lse.clone()
    pkg.backward(x["Q"], x["K"], x["V"], o, lse, x["dO"], causal=False, scale=0.1, deterministic=1)
    torch.cuda.synchronize()
    for k in x:
        assert torch.equal(x[k], keep[k]), k
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("dt,d,Tq,Tk", [(torch.float32, 64, 515, 515), (torch.bfloat16, 128, 515, 515),
                                        (torch.bfloat16, 128, 128, 4096),    # split dQ when deterministic
                                        (torch.bfloat16, 256, 300, 333)])    # rows of 256: D formed in phase 5
@pytest.mark.parametrize("deterministic", [0, 1])
def test_phases_equal_one_call(dt, d, Tq, Tk, deterministic):
    # preprocess, dQ kernel, dK/dV kernel, dQ conversion / split reduction
    # launched one by one (phases 1, 5, 4, 3) give what one attn_bwd call gives
    B, H = 1, 3
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, d), seed=11, dtype=dt, device=DEV)
    code = pkg.ATTN_BF16 if dt == torch.bfloat16 else pkg.ATTN_F32
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=True, scale=0.09)
    ws = torch.empty(max(pkg.attn_bwd_workspace_size(B, H, Tq, Tk, d, d, code, deterministic), 256),
                     dtype=torch.uint8, device=DEV)
    outs = []
    for phases in ((0,), (1, 5, 4, 3)):
        g = [torch.full_like(t, float("nan")) for t in (x["Q"], x["K"], x["V"])]
        for ph in phases:
            pkg.attn_bwd_phase(x["Q"], x["K"], x["V"], o, lse, x["dO"], g[0], g[1], g[2], B, H, Tq, Tk, d, d, 0.09,
                               True, code, deterministic, ws, ws.numel(), ph)
        torch.cuda.synchronize()
        outs.append(g)
    (dq0, dk0, dv0), (dq1, dk1, dv1) = outs
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    if deterministic:
        assert torch.equal(dq0, dq1)
    else:
        check_grad(dq1, dq0, dt, "dQ")


# ------------------------------------------------------------------ dQ on CTA pairs (phase 6)

def _backward_by_phases(x, o, lse, causal, scale, phases, dv=None):
    B, H, Tq, d = x["Q"].shape
    Tk = x["K"].shape[2]
    dv = x["V"].shape[3]
    code = pkg.ATTN_BF16
    ws = torch.empty(max(pkg.attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, code, 1), 256), dtype=torch.uint8,
                     device=DEV)
    g = [torch.full_like(t, float("nan")) for t in (x["Q"], x["K"], x["V"])]
    for ph in phases:
        pkg.attn_bwd_phase(x["Q"], x["K"], x["V"], o, lse, x["dO"], g[0], g[1], g[2], B, H, Tq, Tk, d, dv, scale,
                           causal, code, 1, ws, ws.numel(), ph)
    torch.cuda.synchronize()
    return g


PAIR_SHAPES = [  # B, H, Tq, Tk, dv: odd query-tile counts leave the last pair's second CTA without rows
    (1, 2, 300, 300, 128),
    (2, 1, 640, 640, 128),
    (1, 3, 129, 513, 128),
    (1, 1, 1000, 200, 64),
    (1, 2, 128, 4096, 128),   # few query tiles: split dQ (partials added in split order)
    (1, 1, 384, 1000, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", PAIR_SHAPES)
def test_bf16_dq_on_cta_pairs(shape, causal):
    """Phases 1, 6, 4, 3 (the dQ pass on CTA pairs) against the oracle; dK and
    dV bitwise those of attn_bwd (the same dK/dV kernel on the same D)."""
    B, H, Tq, Tk, dv = shape
    d = 128
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + 3 * Tk + dv, dtype=torch.bfloat16,
                    device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    dq, dk, dvv = _backward_by_phases(x, o, lse, causal, scale, (1, 6, 4, 3))
    r = ref.backward(x["Q"], x["K"], x["V"], x["dO"], scale, causal)
    check_grad(dq, r["dQ"], torch.bfloat16, "dQ")
    check_grad(dk, r["dK"], torch.bfloat16, "dK")
    check_grad(dvv, r["dV"], torch.bfloat16, "dV")
    dq1, dk1, dv1 = _backward_by_phases(x, o, lse, causal, scale, (1, 5, 4, 3))
    assert torch.equal(dk, dk1) and torch.equal(dvv, dv1)
    check_grad(dq, dq1.double().cpu().numpy(), torch.bfloat16, "dQ vs the one-CTA pass")
    # fixed key order: the same bits on every run
    dq2, _, _ = _backward_by_phases(x, o, lse, causal, scale, (1, 6, 4, 3))
    assert torch.equal(dq, dq2)


@pytest.mark.parametrize("dt,d,det", [(torch.bfloat16, 64, 1), (torch.float32, 128, 1), (torch.bfloat16, 128, 0)])
def test_dq_on_cta_pairs_outside_its_domain_is_refused(dt, d, det):
    B, H, T = 1, 1, 256
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=3, dtype=dt, device=DEV)
    code = pkg.ATTN_BF16 if dt == torch.bfloat16 else pkg.ATTN_F32
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=True, scale=0.1)
    ws = torch.empty(max(pkg.attn_bwd_workspace_size(B, H, T, T, d, d, code, det), 256), dtype=torch.uint8,
                     device=DEV)
    g = [torch.empty_like(t) for t in (x["Q"], x["K"], x["V"])]
    st = pkg.attn_bwd_phase(x["Q"], x["K"], x["V"], o, lse, x["dO"], g[0], g[1], g[2], B, H, T, T, d, d, 0.1, True,
                            code, det, ws, ws.numel(), 6, check=False)
    assert st == pkg.ATTN_ERR_UNSUPPORTED


# ------------------------------------------------------------------ bf16 rows of 256 columns

D256_SHAPES = [  # B, H, Tq, Tk, d, dv (64-row steps with ragged tails; Tq != Tk both ways)
    (1, 2, 300, 300, 256, 256),
    (2, 1, 129, 700, 256, 128),
    (1, 1, 700, 129, 256, 64),
    (1, 3, 64, 64, 256, 256),
    (1, 1, 513, 1000, 256, 256),
    (1, 2, 200, 300, 200, 136),   # padded to 256 / 256
    (1, 1, 130, 250, 64, 200),    # value rows above 128: both pad to 256
    (1, 1, 190, 190, 248, 24),    # padded to 256 / 64
]


@pytest.mark.parametrize("deterministic", [0, 1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", D256_SHAPES)
def test_bf16_d256_backward(shape, causal, deterministic):
    B, H, Tq, Tk, d, dv = shape
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq + Tk + d + dv, dtype=torch.bfloat16,
                    device=DEV)
    check_all(x, causal, 1 / math.sqrt(d), torch.bfloat16, deterministic)


def test_bf16_d256_large_logits_across_tiles():
    B, H, T, d = 1, 1, 520, 256
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=19, device="cpu")
    sign = torch.where((torch.arange(T) // 128) % 2 == 0, 20.0, -20.0).view(1, 1, T, 1)
    x = {k: (v * sign if k == "K" else v).to(torch.bfloat16).to(DEV) for k, v in x.items()}
    for causal in (False, True):
        check_all(x, causal, 1.0 / math.sqrt(d), torch.bfloat16, 1)


def test_bf16_d256_bitwise_repeatable_and_flag_independent():
    """Every d = 256 accumulation runs in a fixed order: the same bits on
    every call, whichever value `deterministic` has."""
    B, H, T, d = 1, 2, 400, 256
    x = make_random((B, H, T, d), (B, H, T, d), (B, H, T, d), seed=23, dtype=torch.bfloat16, device=DEV)
    a = run(x, True, 0.0625, 1)
    b = run(x, True, 0.0625, 1)
    c = run(x, True, 0.0625, 0)
    for u, v, w in zip(a[2:], b[2:], c[2:]):
        assert torch.equal(u, v) and torch.equal(u, w)


@pytest.mark.parametrize("deterministic", [1])
def test_bf16_w256_full_size_sampled_heads(deterministic):
    w = WORKLOADS["w256"]
    check_all(make_inputs(w, DEV), w.causal, w.softmax_scale, torch.bfloat16, deterministic,
              heads=[(0, 0), (1, 15)])
