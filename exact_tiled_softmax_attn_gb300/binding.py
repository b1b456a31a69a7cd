"""ctypes binding of libattn.so (include/attn.h), argument marshalling only.

The functions named like the C entry points (``attn_fwd``, ``attn_bwd``, ...)
take torch tensors (or raw device addresses as ints) and pass their data
pointers, sizes and the CUDA stream straight through; every step of the
computation runs in the library's CUDA kernels. ``forward``/``backward``
additionally allocate the outputs (and the backward workspace) with torch.

There is no fallback: if libattn.so is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

__all__ = [
    "LIB_PATH", "EXPORTED_SYMBOLS", "AttnError", "load_library",
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_MISALIGNED", "ATTN_ERR_CUDA",
    "ATTN_ERR_TIMEOUT", "ATTN_ERR_WORKSPACE", "ATTN_F32", "ATTN_BF16",
    "attn_fwd", "attn_fwd_f32_blocked", "attn_fwd_splitkv", "attn_fwd_splitkv_splits",
    "attn_fwd_splitkv_workspace_size", "attn_bwd", "attn_bwd_phase", "attn_bwd_workspace_size", "attn_bwd_dq_splits",
    "attn_bwd_noalloc", "ATTN_NOALLOC_SCRATCH_BYTES", "attn_online_softmax_step", "attn_device_status",
    "attn_selftest_wait_timeout", "attn_strerror", "attn_last_cuda_error", "attn_version",
    "forward", "backward",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_MISALIGNED = 0, 1, 2, 3
ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT, ATTN_ERR_WORKSPACE = 4, 5, 6
ATTN_F32, ATTN_BF16 = 0, 1

_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes); must list every function of include/attn.h
_SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "attn_fwd_f32_blocked": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "attn_fwd_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _SZ, _P]),
    "attn_fwd_splitkv_splits": (_I, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "attn_fwd_splitkv_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "attn_bwd_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "attn_bwd_dq_splits": (_I, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _SZ, _P]),
    "attn_bwd_phase": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _SZ,
                            _I, _P]),
    "attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "attn_online_softmax_step": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "attn_device_status": (_I, [_P]),
    "attn_selftest_wait_timeout": (_I, [_I, _P]),
    "attn_strerror": (ctypes.c_char_p, [_I]),
    "attn_last_cuda_error": (_I, []),
    "attn_version": (_I, []),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib: Optional[ctypes.CDLL] = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = attn_strerror(status) if _lib is not None else str(status)
        extra = ""
        if status == ATTN_ERR_CUDA and _lib is not None:
            extra = f" (cuda error {_lib.attn_last_cuda_error()})"
        super().__init__(f"{where}: {msg}{extra} [status {status}]")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libattn.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m exact_tiled_softmax_attn_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    if isinstance(t, int):
        return t
    if t.dtype == torch.float32:
        return ATTN_F32
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def attn_strerror(status: int) -> str:
    return load_library().attn_strerror(status).decode()


def attn_last_cuda_error() -> int:
    return load_library().attn_last_cuda_error()


def attn_version() -> int:
    return load_library().attn_version()


def attn_fwd(Q, K, V, O, LSE, B, H, Tq, Tk, d, dv, scale, causal, dtype, stream=None, check=True) -> int:
    st = load_library().attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, Tq, Tk, d, dv,
                                 float(scale), int(causal), int(dtype), _stream(stream))
    if check:
        _check(st, "attn_fwd")
    return st


def attn_fwd_f32_blocked(Q, K, V, O, LSE, B, H, Tq, Tk, d, dv, scale, causal, block_n, stream=None,
                         check=True) -> int:
    st = load_library().attn_fwd_f32_blocked(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, Tq, Tk, d, dv,
                                             float(scale), int(causal), int(block_n), _stream(stream))
    if check:
        _check(st, "attn_fwd_f32_blocked")
    return st


def attn_fwd_splitkv(Q, K, V, O, LSE, B, H, Tq, Tk, d, dv, scale, causal, dtype, num_splits, workspace,
                     workspace_bytes, stream=None, check=True) -> int:
    st = load_library().attn_fwd_splitkv(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, Tq, Tk, d, dv,
                                         float(scale), int(causal), int(dtype), int(num_splits), _ptr(workspace),
                                         int(workspace_bytes), _stream(stream))
    if check:
        _check(st, "attn_fwd_splitkv")
    return st


def attn_fwd_splitkv_splits(B, H, Tq, Tk, d, dv, dtype, num_splits) -> int:
    return load_library().attn_fwd_splitkv_splits(B, H, Tq, Tk, d, dv, int(dtype), int(num_splits))


def attn_fwd_splitkv_workspace_size(B, H, Tq, Tk, d, dv, dtype, num_splits) -> int:
    return load_library().attn_fwd_splitkv_workspace_size(B, H, Tq, Tk, d, dv, int(dtype), int(num_splits))


def attn_online_softmax_step(m, l, acc, scores, v_block, n, bs, dv, stream=None, check=True) -> int:
    st = load_library().attn_online_softmax_step(_ptr(m), _ptr(l), _ptr(acc), _ptr(scores), _ptr(v_block), int(n),
                                                 int(bs), int(dv), _stream(stream))
    if check:
        _check(st, "attn_online_softmax_step")
    return st


def attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, dtype, deterministic) -> int:
    return load_library().attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, int(dtype), int(deterministic))


def attn_bwd_dq_splits(B, H, Tq, Tk, d, dv, dtype, deterministic) -> int:
    return load_library().attn_bwd_dq_splits(B, H, Tq, Tk, d, dv, int(dtype), int(deterministic))


def attn_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, Tq, Tk, d, dv, scale, causal, dtype, deterministic,
             workspace, workspace_bytes, stream=None, check=True) -> int:
    st = load_library().attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dO), _ptr(dQ), _ptr(dK),
                                 _ptr(dV), B, H, Tq, Tk, d, dv, float(scale), int(causal), int(dtype),
                                 int(deterministic), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(st, "attn_bwd")
    return st


def attn_bwd_phase(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, Tq, Tk, d, dv, scale, causal, dtype, deterministic,
                   workspace, workspace_bytes, phase, stream=None, check=True) -> int:
    st = load_library().attn_bwd_phase(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dO), _ptr(dQ),
                                       _ptr(dK), _ptr(dV), B, H, Tq, Tk, d, dv, float(scale), int(causal),
                                       int(dtype), int(deterministic), _ptr(workspace), int(workspace_bytes),
                                       int(phase), _stream(stream))
    if check:
        _check(st, "attn_bwd_phase")
    return st


def attn_bwd_noalloc(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, Tq, Tk, d, dv, scale, causal, dtype, deterministic,
                     stream=None, check=True) -> int:
    """attn_bwd with the library's static scratch buffer instead of a workspace."""
    st = load_library().attn_bwd_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dO), _ptr(dQ),
                                         _ptr(dK), _ptr(dV), B, H, Tq, Tk, d, dv, float(scale), int(causal),
                                         int(dtype), int(deterministic), _stream(stream))
    if check:
        _check(st, "attn_bwd_noalloc")
    return st


ATTN_NOALLOC_SCRATCH_BYTES = 64 << 20


def attn_device_status(stream=None) -> int:
    return load_library().attn_device_status(_stream(stream))


def attn_selftest_wait_timeout(limit_ms: int, stream=None) -> int:
    return load_library().attn_selftest_wait_timeout(int(limit_ms), _stream(stream))


# ------------------------------------------------------------------ helpers

def _shape(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [B, H, T, d] tensors")
    B, H, Tq, d = q.shape
    Tk, dv = k.shape[2], v.shape[3]
    if tuple(k.shape) != (B, H, Tk, d) or tuple(v.shape) != (B, H, Tk, dv):
        raise ValueError("Q, K, V shapes disagree")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    return B, H, Tq, Tk, d, dv


def forward(q, k, v, causal: bool = False, scale: Optional[float] = None, stream=None,
            num_splits: Optional[int] = None):
    """O, LSE = attention(q, k, v). Allocates O (q.dtype) and LSE (fp32) with torch.

    num_splits selects the split-KV forward (0 = automatic, n >= 1 = that many
    key splits); None is the plain forward."""
    B, H, Tq, Tk, d, dv = _shape(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty(B, H, Tq, dv, dtype=q.dtype, device=q.device)
    lse = torch.empty(B, H, Tq, dtype=torch.float32, device=q.device)
    dt = _dtype_code(q)
    if num_splits is None:
        attn_fwd(q, k, v, o, lse, B, H, Tq, Tk, d, dv, scale, causal, dt, stream)
    else:
        nbytes = attn_fwd_splitkv_workspace_size(B, H, Tq, Tk, d, dv, dt, num_splits)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        attn_fwd_splitkv(q, k, v, o, lse, B, H, Tq, Tk, d, dv, scale, causal, dt, num_splits, ws, ws.numel(),
                         stream)
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool = False, scale: Optional[float] = None,
             deterministic: bool = False, stream=None, workspace=None):
    """dQ, dK, dV. Allocates the gradients and (unless given) the workspace with torch."""
    B, H, Tq, Tk, d, dv = _shape(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dt = _dtype_code(q)
    ws_bytes = attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, dt, int(deterministic))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    attn_bwd(q, k, v, o, lse, do, dq, dk, dvv, B, H, Tq, Tk, d, dv, scale, causal, dt, int(deterministic),
             workspace, workspace.numel(), stream)
    return dq, dk, dvv
