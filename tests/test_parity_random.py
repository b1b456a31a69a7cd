"""GPU forward and backward vs the CPU float64 oracle on seeded random
problems: shapes, widths, masks, scales and dQ modes drawn together, so that
combinations the hand-picked cases do not list are checked as well. Examples
are the CTA-pair forward with a ragged last key tile, padded widths with
split dQ, and Tq != Tk under the causal mask. Each case also draws whether
the forward runs through the split-KV forward (automatic or a fixed count
of key ranges), from a stream of its own so that the problems themselves
stay the same. The draw is fixed by the seed, and every case is small
enough for the oracle to finish in about a second."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_softmax_attn_gb300 as pkg
from exact_tiled_softmax_attn_gb300.workloads import make_random
from oracle import attention as ref

from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _width(rng, bf16):
    # bf16: multiples of 8 up to 256, often at or next to a tile width; fp32: any width up to 256
    if not bf16:
        return int(rng.integers(1, 257))
    if rng.random() < 0.5:
        return int(rng.choice([64, 128, 256]))
    return int(8 * rng.integers(1, 33))


def _cases(n=24, seed=20261203):
    rng = np.random.default_rng(seed)
    rng_split = np.random.default_rng(seed + 1)
    out = []
    for _ in range(n):
        bf16 = rng.random() < 0.8
        d, dv = _width(rng, bf16), _width(rng, bf16)
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        Tq, Tk = int(rng.integers(1, 701)), int(rng.integers(1, 901))
        # keep the oracle's work bounded
        while B * H * Tq * Tk * (d + dv) > 1.2e9:
            Tq, Tk = max(1, Tq // 2), max(1, Tk // 2)
        causal = bool(rng.random() < 0.5)
        det = int(rng.random() < 0.6)
        scale = float(rng.uniform(0.5, 2.0) / math.sqrt(d))
        # forward: plain (None), split-KV with the automatic count (0), or 2 .. 9 key ranges
        pick = int(rng_split.integers(0, 3))
        splits = None if pick == 0 else 0 if pick == 1 else int(rng_split.integers(2, 10))
        out.append((B, H, Tq, Tk, d, dv, "bf16" if bf16 else "f32", causal, det, scale, splits))
    return out


CASES = _cases()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg.load_library()
    yield
    assert pkg.attn_device_status() == pkg.ATTN_OK


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_random_problem(case):
    B, H, Tq, Tk, d, dv, dts, causal, det, scale, splits = case
    dt = torch.bfloat16 if dts == "bf16" else torch.float32
    x = make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, dv), seed=Tq * 7 + Tk * 3 + d + dv, dtype=dt,
                    device=DEV)
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale, num_splits=splits)
    dq, dk, dvv = pkg.backward(x["Q"], x["K"], x["V"], o, lse, x["dO"], causal=causal, scale=scale,
                               deterministic=det)
    torch.cuda.synchronize()
    r = ref.backward(x["Q"], x["K"], x["V"], x["dO"], scale, causal)
    check_o(o, r["O"], dt)
    check_lse(lse, r["LSE"], dt)
    check_grad(dq, r["dQ"], dt, "dQ")
    check_grad(dk, r["dK"], dt, "dK")
    check_grad(dvv, r["dV"], dt, "dV")
