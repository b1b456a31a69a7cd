"""Seeded synthetic workloads for exact tiled softmax attention.

This module only draws and shapes random inputs. It holds none of the
method's arithmetic (no scores, no softmax, no gradients), so both the CUDA
path and the CPU oracle may consume what it produces.

Layout of every tensor is [batch, heads, seq_len, head_dim], contiguous
("attention_backprop", section "Forward Pass": Q, K, V are
[batch_size, num_heads, seq_len, head_dim]).

The named workloads:

=====  ===========================================  =====  ======  ==========  ====
name   shape                                        dtype  mask    scale       seed
=====  ===========================================  =====  ======  ==========  ====
c1     B1  H1  Tq=Tk=128   d=dv=64                  f32    none    1/sqrt(64)  0
       (run both with no mask and with causal)
c2     B4  H16 Tq=Tk=2048  d=dv=64                  bf16   causal  1/sqrt(64)  1
c3     B2  H16 Tq=Tk=8192  d=dv=128                 bf16   causal  1/sqrt(128) 2
c4     B2  H8  Tq=1000 Tk=4000 d=dv=128             f32    none    1/sqrt(128) 3
       K rows scaled by +40 / -40 in alternating 128-key bands
       (also run at scale 1.0, where the logits pass +-1000)
c5     B1  H32 Tq=Tk=32768 d=dv=128                 bf16   causal  1/sqrt(128) 4
s1     B1  H8  Tq=256 Tk=65536 d=dv=128             bf16   none    1/sqrt(128) 5
       (few query tiles, many keys: the split-KV forward's case)
s1f    the same shape and seed                      f32    none    1/sqrt(128) 5
m1     B2  H16 Tq=Tk=4096  d=64 dv=128              bf16   causal  1/sqrt(64)  6
=====  ===========================================  =====  ======  ==========  ====

Draw order: one CPU ``torch.Generator`` seeded with the workload's seed
draws fp32 standard normals for Q, K, V, dO in that order; then the c4 band
rule is applied to K; then every tensor is rounded to the workload dtype.
Consumers that need float64 upcast the rounded values exactly.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "band_signs"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Tq: int
    Tk: int
    d: int
    dv: int
    dtype: str          # "f32" or "bf16"
    causal: bool
    seed: int
    scale: Optional[float] = None   # None -> 1/sqrt(d)
    k_bands: float = 0.0            # 0 -> plain; else alternating +-k_bands per 128 keys

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "bf16": torch.bfloat16}[self.dtype]

    def pair_flop(self) -> float:
        """2 * B*H*Tq*Tk, halved under causal: a contraction of depth k over all
        allowed (query, key) pairs costs pair_flop() * k."""
        f = 2.0 * self.B * self.H * self.Tq * self.Tk
        return f * 0.5 if self.causal else f

    def fwd_flop(self) -> float:
        """Useful attention FLOPs of one forward: S = Q K^T (depth d) and P V
        (depth dv); 4*B*H*Tq*Tk*d when d = dv, halved under causal."""
        return self.pair_flop() * (self.d + self.dv)

    def bwd_flop(self) -> float:
        """Useful attention FLOPs of one backward: S (d), dP = dO V^T (dv),
        dV = P^T dO (dv), dQ = dS K (d), dK = dS^T Q (d); 2.5 x the forward
        count when d = dv."""
        return self.pair_flop() * (3 * self.d + 2 * self.dv)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "c1": Workload("c1", 1, 1, 128, 128, 64, 64, "f32", False, 0),
    "c1_causal": Workload("c1_causal", 1, 1, 128, 128, 64, 64, "f32", True, 0),
    "c2": Workload("c2", 4, 16, 2048, 2048, 64, 64, "bf16", True, 1),
    "c3": Workload("c3", 2, 16, 8192, 8192, 128, 128, "bf16", True, 2),
    "c4": Workload("c4", 2, 8, 1000, 4000, 128, 128, "f32", False, 3, k_bands=40.0),
    "c4_scale1": Workload("c4_scale1", 2, 8, 1000, 4000, 128, 128, "f32", False, 3,
                          scale=1.0, k_bands=40.0),
    "c5": Workload("c5", 1, 32, 32768, 32768, 128, 128, "bf16", True, 4),
    # few query tiles against many keys (8 query-tile pairs for 152 SMs): the
    # split-KV forward's case
    "s1": Workload("s1", 1, 8, 256, 65536, 128, 128, "bf16", False, 5),
    # the same in fp32 (32 query tiles of 64 rows: the fp32 split-KV forward's case)
    "s1f": Workload("s1f", 1, 8, 256, 65536, 128, 128, "f32", False, 5),
    # V with its own head dimension (d = 64, dv = 128)
    "m1": Workload("m1", 2, 16, 4096, 4096, 64, 128, "bf16", True, 6),
    # head size 256 (forward and backward on the tensor cores)
    "w256": Workload("w256", 2, 16, 4096, 4096, 256, 256, "bf16", True, 7),
}


def band_signs(Tk: int, band: int = 128) -> torch.Tensor:
    """+1 for keys in even 128-key bands, -1 for odd bands (shape [Tk])."""
    j = torch.arange(Tk)
    return torch.where((j // band) % 2 == 0, 1.0, -1.0)


def make_inputs(w: Workload, device: str = "cpu", with_dO: bool = True):
    """Draw (Q, K, V, dO) for workload ``w`` on the CPU, then move them.

    Returns a dict of contiguous tensors in the workload dtype.
    """
    g = torch.Generator().manual_seed(w.seed)
    Q = torch.randn(w.B, w.H, w.Tq, w.d, generator=g, dtype=torch.float32)
    K = torch.randn(w.B, w.H, w.Tk, w.d, generator=g, dtype=torch.float32)
    V = torch.randn(w.B, w.H, w.Tk, w.dv, generator=g, dtype=torch.float32)
    dO = torch.randn(w.B, w.H, w.Tq, w.dv, generator=g, dtype=torch.float32) if with_dO else None
    if w.k_bands:
        K = K * (w.k_bands * band_signs(w.Tk)).view(1, 1, w.Tk, 1)
    out = {"Q": Q, "K": K, "V": V}
    if dO is not None:
        out["dO"] = dO
    dt = w.torch_dtype
    return {k: v.to(dt).contiguous().to(device) for k, v in out.items()}


def make_random(shape_q, shape_k, shape_v, seed: int, dtype=torch.float32, device="cpu",
                with_dO: bool = True):
    """Small ad-hoc draws (ragged shapes for tests), same draw order as ``make_inputs``."""
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn(*shape_q, generator=g)
    K = torch.randn(*shape_k, generator=g)
    V = torch.randn(*shape_v, generator=g)
    out = {"Q": Q, "K": K, "V": V}
    if with_dO:
        out["dO"] = torch.randn(*shape_q[:-1], shape_v[-1], generator=g)
    return {k: v.to(dtype).contiguous().to(device) for k, v in out.items()}
