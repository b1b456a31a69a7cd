"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/attn.h, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import exact_tiled_softmax_attn_gb300 as pkg
from exact_tiled_softmax_attn_gb300 import binding as B
from exact_tiled_softmax_attn_gb300 import build as build_mod

HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return pkg.load_library()


def header_functions():
    text = open(HEADER).read()
    return set(re.findall(r"ATTN_API\s+[\w\s\*]*?\b(attn_\w+)\s*\(", text))


def test_header_declares_the_binding_functions():
    assert header_functions() == set(B.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    # nothing but the C ABI is visible
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert header_functions() <= exported
    assert {s for s in exported if s.startswith("attn_")} == header_functions()


def test_version_and_strerror(lib):
    assert pkg.attn_version() >> 16 == 1
    for s in range(7):
        assert pkg.attn_strerror(s)
    assert pkg.attn_strerror(99) == "unknown status"


def _fwd(**kw):
    a = dict(Q=0x10000, K=0x20000, V=0x30000, O=0x40000, LSE=0x50000, B=1, H=1, Tq=8, Tk=8, d=64, dv=64,
             scale=0.125, causal=0, dtype=B.ATTN_BF16, stream=0, check=False)
    a.update(kw)
    return B.attn_fwd(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), B.ATTN_ERR_INVALID_ARG),
    (dict(Tq=-3), B.ATTN_ERR_INVALID_ARG),
    (dict(d=0), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), B.ATTN_ERR_INVALID_ARG),
    (dict(scale=-1.0), B.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), B.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), B.ATTN_ERR_INVALID_ARG),
    (dict(d=100, dv=100), B.ATTN_ERR_UNSUPPORTED),   # bf16 rows are whole 16-byte units: d % 8 == 0
    (dict(d=64, dv=60), B.ATTN_ERR_UNSUPPORTED),
    (dict(d=128, dv=264), B.ATTN_ERR_UNSUPPORTED),   # at most 256 columns
    (dict(d=512, dv=128), B.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=B.ATTN_F32, d=257), B.ATTN_ERR_UNSUPPORTED),
    (dict(Q=None), B.ATTN_ERR_INVALID_ARG),
    (dict(LSE=None), B.ATTN_ERR_INVALID_ARG),
    (dict(Q=0x10008), B.ATTN_ERR_MISALIGNED),
    (dict(dtype=B.ATTN_F32, V=0x30002), B.ATTN_ERR_MISALIGNED),
    (dict(O=0x10000), B.ATTN_ERR_INVALID_ARG),             # output overlaps Q
    (dict(LSE=0x40010), B.ATTN_ERR_INVALID_ARG),           # LSE overlaps O
])
def test_forward_host_validation(lib, kw, status):
    assert _fwd(**kw) == status


def test_empty_problems_need_no_device(lib):
    # nothing to compute: accepted without any CUDA call (no GPU here)
    assert _fwd(B=0) == B.ATTN_OK
    assert _fwd(Tq=0) == B.ATTN_OK
    assert _fwd(B=0, Q=None, K=None, V=None, O=None, LSE=None) == B.ATTN_OK


def test_blocked_forward_key_tile_must_fit_shared_memory(lib):
    # d = dv = 256 with 128-key tiles needs ~330 KB of shared memory per CTA
    st = B.attn_fwd_f32_blocked(0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 1, 1, 8, 8, 256, 256, 0.1, 0,
                                128, stream=0, check=False)
    assert st == B.ATTN_ERR_UNSUPPORTED


def test_blocked_forward_validates_block(lib):
    st = B.attn_fwd_f32_blocked(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 1, 8, 8, 64, 64, 0.1, 0, 48,
                                stream=0, check=False)
    assert st == B.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,det,want", [
    ((2, 16, 8192, 8192, 128), 1, 1),    # 2048 query tiles: no split
    ((1, 2, 128, 4096, 128), 1, 8),      # 2 query tiles, 32 key tiles: 8 splits of 4
    ((1, 2, 128, 4096, 128), 0, 1),      # atomic dQ never splits
    ((1, 8, 256, 65536, 128), 1, 9),     # 16 query tiles: 144 units, one wave
    ((1, 1, 256, 3000, 64), 1, 6),       # 24 key tiles: at least 4 per split
    ((1, 1, 128, 700, 128), 1, 1),       # 6 key tiles: too few to split
])
def test_dq_split_rule(lib, shape, det, want):
    B_, H, Tq, Tk, d = shape
    assert B.attn_bwd_dq_splits(B_, H, Tq, Tk, d, d, B.ATTN_BF16, det) == want
    part = (B_ * H * ((Tq + 127) // 128 * 128) * 4 + 255) // 256 * 256
    acc = B_ * H * Tq * d * 4
    ws = B.attn_bwd_workspace_size(B_, H, Tq, Tk, d, d, B.ATTN_BF16, det)
    r256 = lambda x: (x + 255) // 256 * 256
    # + 256 bytes for the unit counters of the bf16 dQ and dK/dV kernels
    assert ws == r256(2 * part + (acc if det == 0 else (want * acc if want > 1 else 0))) + 256


@pytest.mark.parametrize("shape,det,want", [
    ((2, 8, 1000, 4000, 128), 1, 63),    # c4: 63 key tiles, 516 MB of partials: one per key tile (dK/dV kernel)
    ((2, 8, 1000, 4000, 128), 0, 1),     # atomic dQ never splits
    ((1, 8, 256, 65536, 128), 1, 1024),  # s1f: 1024 key tiles, exactly 1 GiB of partials
    ((1, 1, 128, 200, 64), 1, 4),        # 4 key tiles: one partial each
    ((1, 1, 128, 192, 64), 1, 3),
    ((1, 1, 100, 50, 64), 1, 1),         # one key tile: the dK/dV kernel writes dQ itself
    ((1, 2, 128, 8192, 128), 1, 128),
    ((2, 16, 8192, 8192, 128), 1, 1),    # 16 GiB of partials: the dQ kernel; 4096 query tiles fill the SMs
    ((4, 16, 8192, 4096, 128), 1, 1),
    ((1, 8, 512, 65536, 128), 1, 7),     # 2 GiB of partials, 64 query tiles: the dQ kernel, 7 ranges
])
def test_dq_split_rule_fp32(lib, shape, det, want):
    """fp32 deterministic dQ. With at most 1 GiB of partials (one per 64-key
    tile), every key tile is its own range: the dK/dV kernel writes its
    partial dQ, and the partials are added in key-tile order.
    Otherwise the dQ kernel splits its 64-row query tiles over ranges of
    64-key tiles: the smallest count whose waves of units x ranges on 152
    SMs, times the key tiles of a range, come within 5 % of the best count."""
    B_, H, Tq, Tk, d = shape
    S = B.attn_bwd_dq_splits(B_, H, Tq, Tk, d, d, B.ATTN_F32, det)
    assert S == want
    r256 = lambda x: (x + 255) // 256 * 256
    part = r256(B_ * H * ((Tq + 127) // 128 * 128) * 4)
    partials = B_ * H * Tq * d * 4 * S if S > 1 else 0
    assert B.attn_bwd_workspace_size(B_, H, Tq, Tk, d, d, B.ATTN_F32, det) == 2 * part + partials


def test_noalloc_refuses_fp32_partials_beyond_its_buffer(lib):
    """The fp32 deterministic backward of c4 keeps 63 dQ partials (516 MB) in
    its workspace, beyond the no-allocation entry point's fixed 64 MiB: it
    refuses the call on the host, before any device work, as it does for any
    problem beyond its buffer."""
    args = (0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000, 0x700000, 0x800000, 0x900000,
            2, 8, 1000, 4000, 128, 128, 0.088, 0, B.ATTN_F32)
    assert B.attn_bwd_workspace_size(2, 8, 1000, 4000, 128, 128, B.ATTN_F32, 1) > B.ATTN_NOALLOC_SCRATCH_BYTES
    assert B.attn_bwd_noalloc(*args, 1, stream=0, check=False) == B.ATTN_ERR_WORKSPACE


def test_workspace_size(lib):
    # -LSE*log2(e) and D, each [B*H, Tq rounded up to 128] fp32 and 256-byte
    # aligned, then (bf16 with fp32 dQ accumulation) the [B*H*Tq, d]
    # accumulator, then (bf16) 256 bytes of unit counters
    r256 = lambda x: (x + 255) // 256 * 256
    part = r256(2 * 3 * 128 * 4)
    assert B.attn_bwd_workspace_size(2, 3, 100, 50, 64, 64, B.ATTN_F32, 0) == 2 * part
    assert B.attn_bwd_workspace_size(2, 3, 100, 50, 64, 64, B.ATTN_BF16, 1) == 2 * part + 256
    assert B.attn_bwd_workspace_size(2, 3, 100, 50, 64, 64, B.ATTN_BF16, 0) == \
        r256(2 * part + 2 * 3 * 100 * 64 * 4) + 256
    assert B.attn_bwd_workspace_size(2, 3, 0, 50, 64, 64, B.ATTN_BF16, 0) == 0
    assert B.attn_bwd_workspace_size(-1, 3, 100, 50, 64, 64, B.ATTN_BF16, 0) == 0


def _bwd(**kw):
    a = dict(Q=0x100000, K=0x200000, V=0x300000, O=0x400000, LSE=0x500000, dO=0x600000, dQ=0x700000,
             dK=0x800000, dV=0x900000, B=1, H=1, Tq=8, Tk=8, d=64, dv=64, scale=0.125, causal=0,
             dtype=B.ATTN_BF16, deterministic=0, workspace=0xA00000, workspace_bytes=1 << 20, stream=0,
             check=False)
    a.update(kw)
    return B.attn_bwd(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(deterministic=3), B.ATTN_ERR_INVALID_ARG),
    (dict(workspace=None), B.ATTN_ERR_WORKSPACE),
    (dict(workspace_bytes=16), B.ATTN_ERR_WORKSPACE),
    (dict(workspace=0xA00010), B.ATTN_ERR_WORKSPACE),
    (dict(workspace=0x100000), B.ATTN_ERR_WORKSPACE),     # workspace overlaps Q
    (dict(dK=0x700000), B.ATTN_ERR_INVALID_ARG),          # two outputs overlap
    (dict(dQ=0x600000), B.ATTN_ERR_INVALID_ARG),          # output overlaps dO
    (dict(dO=None), B.ATTN_ERR_INVALID_ARG),
    (dict(dV=0x900008), B.ATTN_ERR_MISALIGNED),
    (dict(d=264, dv=64), B.ATTN_ERR_UNSUPPORTED),    # the bf16 backward takes d, dv <= 256
    (dict(d=100, dv=64), B.ATTN_ERR_UNSUPPORTED),    # a multiple of 8
    (dict(d=256, dv=264), B.ATTN_ERR_UNSUPPORTED),
])
def test_backward_host_validation(lib, kw, status):
    assert _bwd(**kw) == status


def test_backward_phase_range(lib):
    args = dict(Q=0x100000, K=0x200000, V=0x300000, O=0x400000, LSE=0x500000, dO=0x600000, dQ=0x700000,
                dK=0x800000, dV=0x900000, B=1, H=1, Tq=8, Tk=8, d=64, dv=64, scale=0.125, causal=0,
                dtype=B.ATTN_BF16, deterministic=0, workspace=0xA00000, workspace_bytes=1 << 20)
    for ph in (-1, 7):
        assert B.attn_bwd_phase(**args, phase=ph, stream=0, check=False) == B.ATTN_ERR_INVALID_ARG
    # phase 6 (the dQ pass on CTA pairs) takes bf16, d = 128, deterministic dQ only; refused on the host
    assert B.attn_bwd_phase(**args, phase=6, stream=0, check=False) == B.ATTN_ERR_UNSUPPORTED
    assert B.attn_bwd_phase(**dict(args, deterministic=1), phase=6, stream=0, check=False) == B.ATTN_ERR_UNSUPPORTED
    assert B.attn_bwd_phase(**dict(args, d=128, dv=128, dtype=B.ATTN_F32, deterministic=1), phase=6, stream=0,
                            check=False) == B.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), B.ATTN_ERR_INVALID_ARG),
    (dict(bs=-2), B.ATTN_ERR_INVALID_ARG),
    (dict(dv=0), B.ATTN_ERR_INVALID_ARG),
    (dict(dv=513), B.ATTN_ERR_INVALID_ARG),
    (dict(m=None), B.ATTN_ERR_INVALID_ARG),
    (dict(scores=0x400002), B.ATTN_ERR_MISALIGNED),
    (dict(l=0x100000), B.ATTN_ERR_INVALID_ARG),            # l overlaps m
    (dict(acc=0x400000), B.ATTN_ERR_INVALID_ARG),          # acc overlaps scores
    (dict(n=0, m=None, l=None, acc=None, scores=None), B.ATTN_OK),
])
def test_step_host_validation(lib, kw, status):
    a = dict(m=0x100000, l=0x200000, acc=0x300000, scores=0x400000, v_block=0x500000, n=8, bs=16, dv=32)
    a.update(kw)
    assert B.attn_online_softmax_step(**a, stream=0, check=False) == status


def test_error_text_carries_status(lib):
    with pytest.raises(B.AttnError) as e:
        B.attn_fwd(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 1, 8, 8, 100, 100, 0.1, 0, B.ATTN_BF16,
                   stream=0)
    assert "unsupported" in str(e.value)


def test_d256_bf16_backward_workspace_and_splits(lib):
    """d = 256: the workspace holds -LSE*log2(e) and D only (dQ is written in
    one fixed-order pass for either value of `deterministic`, no splits); other
    widths above 128 pad to 256 columns (and dv to 64, 128 or 256)."""
    r256 = lambda x: (x + 255) // 256 * 256
    B_, H, Tq, Tk = 2, 3, 300, 500
    rows_pad = B_ * H * 384
    for det in (0, 1):
        for dv in (64, 128, 256):
            assert B.attn_bwd_workspace_size(B_, H, Tq, Tk, 256, dv, B.ATTN_BF16, det) == 2 * r256(rows_pad * 4)
            assert B.attn_bwd_dq_splits(B_, H, 128, 65536, 256, dv, B.ATTN_BF16, det) == 1
        # d = 200, dv = 136: copies padded to 256 and 256 columns, then the d = 256 workspace
        bh = B_ * H
        pads = [bh * Tq * 256, bh * Tk * 256, bh * Tk * 256, bh * Tq * 256, bh * Tq * 256, bh * Tq * 256,
                bh * Tk * 256, bh * Tk * 256]
        assert B.attn_bwd_workspace_size(B_, H, Tq, Tk, 200, 136, B.ATTN_BF16, det) == \
            sum(r256(2 * n) for n in pads) + 2 * r256(rows_pad * 4)
        # d = 64, dv = 200: the value rows are wider than 128, so d pads to 256 as well
        pads = [bh * Tq * 256, bh * Tk * 256, bh * Tk * 256, bh * Tq * 256, bh * Tq * 256, bh * Tq * 256,
                bh * Tk * 256, bh * Tk * 256]
        assert B.attn_bwd_workspace_size(B_, H, Tq, Tk, 64, 200, B.ATTN_BF16, det) == \
            sum(r256(2 * n) for n in pads) + 2 * r256(rows_pad * 4)


def test_d256_bf16_forward_splits(lib):
    # the forward splits at d = 256 as at d <= 128: 64 key tiles in 8 ranges of 8
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 8192, 256, 256, B.ATTN_BF16, 8) == 8
    assert B.attn_fwd_splitkv_splits(1, 1, 128, 8192, 256, 64, B.ATTN_BF16, 100) == 64
    rows = 1 * 1 * 128
    r256 = lambda x: (x + 255) // 256 * 256
    assert B.attn_fwd_splitkv_workspace_size(1, 1, 128, 8192, 256, 256, B.ATTN_BF16, 8) == \
        r256(8 * rows * 256 * 4) + r256(8 * rows * 4)



def test_plain_c_program_uses_the_header_and_library(lib, tmp_path):
    """The boundary needs no Python or torch: a C99 program that includes
    attn.h (with -Wall -Werror -pedantic) links libattn.so and calls the
    host-only entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_attn.c"
    src.write_text(r'''
#include <stdio.h>
#include "attn.h"
int main(void) {
  size_t ws = attn_bwd_workspace_size(1, 2, 300, 300, 64, 64, ATTN_BF16, 0);
  int s1 = attn_fwd_splitkv_splits(1, 1, 128, 8192, 128, 128, ATTN_BF16, 8);
  attn_status_t st = attn_fwd(0, 0, 0, 0, 0, 1, 1, 8, 8, 100, 100, 0.1f, 0, ATTN_BF16, 0);
  printf("%d %zu %d %d %s\n", attn_version(), ws, s1, (int)st, attn_strerror(st));
  return 0;
}
''')
    exe = tmp_path / "use_attn"
    libdir = os.path.dirname(B.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-lattn", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr
    version, ws, s1, st, text = r.stdout.split(maxsplit=4)
    assert int(version) == B.attn_version()
    assert int(ws) == B.attn_bwd_workspace_size(1, 2, 300, 300, 64, 64, B.ATTN_BF16, 0)
    assert int(s1) == 8 and int(st) == B.ATTN_ERR_UNSUPPORTED and "unsupported" in text


def test_padded_bf16_backward_workspace_and_phases(lib):
    """bf16 widths other than 64 / 128 (multiples of 8 up to 128) run the
    backward on zero-padded copies held in the workspace, as one call."""
    r256 = lambda x: (x + 255) // 256 * 256
    for det in (0, 1):
        B_, H, Tq, Tk, d, dv = 1, 2, 300, 500, 96, 40
        dp, dvp = 128, 64
        bh = B_ * H
        pads = [bh * Tq * dp, bh * Tk * dp, bh * Tk * dvp, bh * Tq * dvp, bh * Tq * dvp, bh * Tq * dp, bh * Tk * dp,
                bh * Tk * dvp]
        inner = B.attn_bwd_workspace_size(B_, H, Tq, Tk, dp, dvp, B.ATTN_BF16, det)
        assert B.attn_bwd_workspace_size(B_, H, Tq, Tk, d, dv, B.ATTN_BF16, det) == sum(r256(2 * n) for n in pads) + inner
        assert B.attn_bwd_dq_splits(B_, H, Tq, Tk, d, dv, B.ATTN_BF16, det) == \
            B.attn_bwd_dq_splits(B_, H, Tq, Tk, dp, dvp, B.ATTN_BF16, det)
    args = dict(Q=0x100000, K=0x200000, V=0x300000, O=0x400000, LSE=0x500000, dO=0x600000, dQ=0x700000,
                dK=0x800000, dV=0x900000, B=1, H=1, Tq=8, Tk=8, d=96, dv=96, scale=0.125, causal=0,
                dtype=B.ATTN_BF16, deterministic=1, workspace=0xA00000, workspace_bytes=1 << 20)
    for ph in (1, 2, 3, 4, 5, 6):
        assert B.attn_bwd_phase(**args, phase=ph, stream=0, check=False) == B.ATTN_ERR_UNSUPPORTED
