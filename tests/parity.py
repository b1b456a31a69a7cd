"""Tolerances and comparisons between the CUDA path and the CPU oracle.

Bounds (the same for every GPU test):
  fp32: max|x - ref| / max|ref| <= 1e-5 for O and LSE, <= 1e-4 for dQ, dK, dV
  bf16: O: for every query row, rms(O - O_ref) <= 1e-2 * rms(O_ref) over the
        row's dv entries; max|LSE - ref| <= 1e-2;
        ||x - ref||_F / ||ref||_F <= 2e-2 for dQ, dK, dV
A row with no allowed key must give O = 0 and LSE = -inf exactly.

The bf16 O bound is the stated "max abs error on O <= 1e-2 * rms(O)" read
per query row with the rms of the error in place of its max. Read literally
(max over all of O against the rms of all of O) it is below the rounding step
of a bf16 output: the oracle's exact O rounded to bf16 already breaks it on
the causal workloads (test_tolerance_reading.py shows this), because rows
that average few keys have |O| of order 1 while the global rms is ~0.1.
The literal ratio is still computed and reported (``literal_o_ratio``).
"""
import numpy as np
import torch

F32_FWD = 1e-5
F32_BWD = 1e-4
BF16_O = 1e-2
BF16_LSE = 1e-2
BF16_GRAD = 2e-2


def np64(t):
    return t.detach().double().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def max_rel(x, ref):
    x, ref = np64(x), np64(ref)
    den = np.abs(ref).max()
    return float(np.abs(x - ref).max() / den) if den > 0 else float(np.abs(x - ref).max())


def frob_rel(x, ref):
    x, ref = np64(x), np64(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x - ref))


def row_rms_ratio(o, ref):
    """max over query rows of rms(o - ref) / rms(ref), rows along the last axis."""
    o, ref = np64(o), np64(ref)
    num = np.sqrt(np.mean((o - ref) ** 2, axis=-1))
    den = np.sqrt(np.mean(ref ** 2, axis=-1))
    live = den > 0
    if not live.all():
        assert np.all(num[~live] == 0)
    return float((num[live] / den[live]).max()) if live.any() else 0.0


def literal_o_ratio(o, ref):
    """max|o - ref| / rms(ref) over the whole tensor (the bound read literally)."""
    o, ref = np64(o), np64(ref)
    return float(np.abs(o - ref).max() / np.sqrt(np.mean(ref ** 2)))


def check_lse(lse, ref, dtype):
    lse, ref = np64(lse), np64(ref)
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(lse), inf), "rows with no allowed key must give LSE = -inf"
    assert np.all(np.isfinite(lse[~inf]))
    if (~inf).any():
        a, b = lse[~inf], ref[~inf]
        if dtype == torch.float32:
            err = np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)
            assert err <= F32_FWD, f"LSE rel err {err:.3e}"
        else:
            err = np.abs(a - b).max()
            assert err <= BF16_LSE, f"LSE abs err {err:.3e}"


def check_o(o, ref, dtype):
    o, ref = np64(o), np64(ref)
    assert np.all(np.isfinite(o))
    if dtype == torch.float32:
        err = max_rel(o, ref)
        assert err <= F32_FWD, f"O rel err {err:.3e}"
    else:
        err = row_rms_ratio(o, ref)
        assert err <= BF16_O, f"O worst row rms-error / row rms {err:.3e} (literal ratio {literal_o_ratio(o, ref):.3e})"


def check_grad(g, ref, dtype, name):
    g, ref = np64(g), np64(ref)
    assert np.all(np.isfinite(g)), name
    if dtype == torch.float32:
        err = max_rel(g, ref)
        assert err <= F32_BWD, f"{name} rel err {err:.3e}"
    else:
        err = frob_rel(g, ref)
        assert err <= BF16_GRAD, f"{name} Frobenius rel err {err:.3e}"
