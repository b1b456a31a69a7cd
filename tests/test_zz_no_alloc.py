"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (no CUDA allocator of their own, or not allowed to grow the device
footprint at run time). Its workspace is the library's static scratch
buffer, shared by every call on a device.

Each case calls it on the target problem, then on a larger problem with other
inputs (so the shared buffer holds different D, -LSE*log2(e), accumulator and
padded-copy contents, written further into it), then on the target again, and
checks both target calls against attn_bwd with a workspace of the caller's
own: bitwise equal in deterministic mode (the same kernels on the same
inputs), within the parity tolerance with fp32 atomics (whose order of
addition varies from run to run). This file sorts last so a
stop-at-first-failure run has already run every other test."""
import math

import pytest
import torch

import exact_tiled_softmax_attn_gb300 as pkg
from exact_tiled_softmax_attn_gb300.workloads import make_random

from parity import check_grad

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [  # B, H, Tq, Tk, d, dtype, causal, deterministic
    (1, 4, 1000, 1000, 128, torch.bfloat16, True, 0),
    (2, 2, 300, 700, 64, torch.bfloat16, False, 0),
    (1, 3, 513, 513, 128, torch.bfloat16, True, 1),
    (1, 2, 128, 4096, 128, torch.bfloat16, False, 1),   # deterministic with split dQ partials
    (2, 2, 77, 133, 40, torch.float32, True, 0),
    (2, 2, 77, 133, 40, torch.float32, True, 1),
    (1, 2, 300, 400, 96, torch.bfloat16, True, 1),      # bf16 width 96: padded copies in the scratch
]


def _inputs(B, H, Tq, Tk, d, dt, seed):
    return make_random((B, H, Tq, d), (B, H, Tk, d), (B, H, Tk, d), seed=seed, dtype=dt, device=DEV)


def _noalloc(x, o, lse, B, H, Tq, Tk, d, scale, causal, code, det):
    got = [torch.full_like(t, float("nan")) for t in (x["Q"], x["K"], x["V"])]
    pkg.attn_bwd_noalloc(x["Q"], x["K"], x["V"], o, lse, x["dO"], *got, B, H, Tq, Tk, d, d, scale, causal, code,
                         det)
    return got


@pytest.mark.parametrize("case", CASES)
def test_noalloc_matches_workspace_backward(case):
    B, H, Tq, Tk, d, dt, causal, det = case
    code = pkg.ATTN_BF16 if dt == torch.bfloat16 else pkg.ATTN_F32
    scale = 1.0 / math.sqrt(d)
    # the problem run between the two checked calls: twice the heads, other draws
    H2 = 2 * H
    assert pkg.attn_bwd_workspace_size(B, H2, Tq, Tk, d, d, code, det) <= pkg.ATTN_NOALLOC_SCRATCH_BYTES
    assert pkg.attn_bwd_workspace_size(B, H2, Tq, Tk, d, d, code, det) > \
        pkg.attn_bwd_workspace_size(B, H, Tq, Tk, d, d, code, det)
    x = _inputs(B, H, Tq, Tk, d, dt, seed=Tq + Tk + d)
    y = _inputs(B, H2, Tq, Tk, d, dt, seed=Tq + Tk + d + 1)
    o, lse = pkg.forward(x["Q"], x["K"], x["V"], causal=causal, scale=scale)
    o2, lse2 = pkg.forward(y["Q"], y["K"], y["V"], causal=causal, scale=scale)
    want = pkg.backward(x["Q"], x["K"], x["V"], o, lse, x["dO"], causal=causal, scale=scale, deterministic=det)
    for call in range(2):
        if call == 1:
            _noalloc(y, o2, lse2, B, H2, Tq, Tk, d, scale, causal, code, det)
        got = _noalloc(x, o, lse, B, H, Tq, Tk, d, scale, causal, code, det)
        torch.cuda.synchronize()
        for g, w, name in zip(got, want, ("dQ", "dK", "dV")):
            if det:
                assert torch.equal(g, w), f"{name}: call {call} differs from attn_bwd"
            else:
                check_grad(g, w, dt, name)
    assert pkg.attn_device_status() == pkg.ATTN_OK


def test_noalloc_rejects_problems_beyond_its_buffer():
    # bf16 with the fp32 dQ accumulator: about B*H*Tq*(d+2)*4 bytes > 64 MiB
    B, H, T, d = 4, 16, 2048, 128
    assert pkg.attn_bwd_workspace_size(B, H, T, T, d, d, pkg.ATTN_BF16, 0) > pkg.ATTN_NOALLOC_SCRATCH_BYTES
    st = pkg.attn_bwd_noalloc(0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000, 0x700000,
                              0x800000, 0x900000, B, H, T, T, d, d, 0.088, 1, pkg.ATTN_BF16, 0, check=False)
    assert st == pkg.ATTN_ERR_WORKSPACE
