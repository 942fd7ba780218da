"""C-ABI checks that need no GPU: the library builds, loads, exports what the header
declares, and rejects bad arguments on the host before touching CUDA."""
from __future__ import annotations

import ctypes
import subprocess

import pytest

from bit_exact_attention_gb300 import _build, _lib

FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: the checks fail first


@pytest.fixture(scope="module")
def lib():
    return _lib.lib()


def test_library_exports_every_header_function(lib):
    names = _lib.header_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(lib, n)


def test_built_for_sm103a_only():
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.sage2_status_str(code)
    assert lib.sage2_version() == 100


def test_workspace_size_and_layout(lib):
    n = lib.sage2_workspace_size(2, 32, 8, 4096, 4096, 128, 8192, 8192)
    assert n > 0
    L = _lib.WsLayout()
    assert lib.sage2_workspace_layout(2, 32, 8, 4096, 4096, 128, 8192, 8192, ctypes.byref(L)) == 0
    assert L.total_bytes == n and L.Dp == 128
    offs = sorted([L.status, L.qcode, L.kcode, L.vcodeT, L.qscale, L.kscale, L.qmean, L.kmean,
                   L.vscale, L.vinv, L.dsc, L.kpart, L.vpart])
    assert all(o % 1024 == 0 for o in offs)
    assert len(set(offs)) == len(offs) and offs[-1] < n
    # padded rows hold every sequence with its tail: total + 128 per sequence
    assert L.Tq >= 8192 + 2 * 128 and L.Tq % 128 == 0
    assert L.nkv_pad == 4096
    # D <= 64 computes in 64 channels
    assert lib.sage2_workspace_layout(1, 2, 2, 256, 256, 64, 256, 256, ctypes.byref(L)) == 0
    assert L.Dp == 64
    # invalid sizes
    assert lib.sage2_workspace_size(1, 3, 2, 16, 16, 64, 16, 16) == 0      # Hq % Hkv
    assert lib.sage2_workspace_size(1, 2, 2, 16, 16, 256, 16, 16) == 0     # D > 128
    assert lib.sage2_workspace_size(1, 2, 2, 16, 16, 60, 16, 16) == 0      # D % 8


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, in_dt=1, out_dt=1, B=1, Hq=2, Hkv=2, Nq=16,
             Nkv=16, D=64, causal=0, scale=0.0, ws=FAKE, wsb=1 << 40, stream=None)
    a.update(kw)
    return lib.sage2_attn_fwd(a["q"], a["k"], a["v"], a["out"], a["in_dt"], a["out_dt"], a["B"],
                              a["Hq"], a["Hkv"], a["Nq"], a["Nkv"], a["D"], a["causal"],
                              a["scale"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(D=256), _lib.EUNSUPPORTED),
    (dict(D=136), _lib.EUNSUPPORTED),
    (dict(D=60), _lib.EUNSUPPORTED),
    (dict(D=0), _lib.EINVAL),
    (dict(Hq=3, Hkv=2), _lib.EINVAL),
    (dict(B=0), _lib.EINVAL),
    (dict(Nq=-1), _lib.EINVAL),
    (dict(q=None), _lib.EINVAL),
    (dict(k=ctypes.c_void_p(0x10008)), _lib.EINVAL),   # not 16-byte aligned
    (dict(in_dt=2), _lib.EINVAL),                      # fp32 inputs are not accepted
    (dict(out_dt=0), _lib.EINVAL),                     # bf16 in, fp16 out
    (dict(causal=2), _lib.EINVAL),
    (dict(wsb=1024), _lib.EWORKSPACE),
    (dict(ws=None), _lib.EWORKSPACE),
])
def test_host_side_argument_errors(lib, kw, code):
    assert _fwd(lib, **kw) == code


def test_varlen_requires_cu_seqlens(lib):
    rc = lib.sage2_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, 1, 1, None, None, 2, 4, 2, 64, 64,
                                   100, 100, 128, 0, 0.0, FAKE, 1 << 40, None)
    assert rc == _lib.EINVAL
    # totals larger than B * max are impossible
    rc = lib.sage2_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, 1, 1, FAKE, FAKE, 2, 4, 2, 10, 64,
                                   100, 100, 128, 0, 0.0, FAKE, 1 << 40, None)
    assert rc == _lib.EINVAL


def test_workspace_size_per_code_format(lib):
    """The INT8 (v1) path stores two-byte Q and K codes: its workspace is larger by exactly the
    extra code bytes (rounded to the 1 KB granule); invalid switch words give 0."""
    args = (1, 8, 2, 1000, 1500, 128, 1000, 1500)
    n4 = lib.sage2_workspace_size(*args)
    assert n4 > 0 and lib.sage2_workspace_size_ex(*args, 0) == n4
    assert lib.sage2_workspace_size_ex(*args, 1 | 2 | 4) == n4  # ablations: same layout
    n8 = lib.sage2_workspace_size_ex(*args, 8)
    L4, L8 = _lib.WsLayout(), _lib.WsLayout()
    assert lib.sage2_workspace_layout_ex(*args, 0, ctypes.byref(L4)) == 0
    assert lib.sage2_workspace_layout_ex(*args, 8, ctypes.byref(L8)) == 0
    assert (L4.code_bytes, L8.code_bytes) == (1, 2)
    extra = (L8.kcode - L8.qcode) - (L4.kcode - L4.qcode)  # the Q code region doubled
    assert extra >= 8 * L4.Tq * 128 - 1024
    assert n8 > n4
    for bad in (16, 8 | 4, -1):
        assert lib.sage2_workspace_size_ex(*args, bad) == 0
        assert lib.sage2_workspace_layout_ex(*args, bad, ctypes.byref(L8)) == _lib.EINVAL


def test_ex_entry_points_reject_bad_switches_before_cuda(lib):
    cu = FAKE
    rc = lib.sage2_prepass_varlen_ex(FAKE, FAKE, FAKE, 1, cu, cu, 1, 2, 2, 128, 128, 128, 128, 64,
                                     0, 0.0, 8 | 1, FAKE, 1 << 30, None)
    assert rc == _lib.EINVAL
    rc = lib.sage2_attention_varlen_ex(FAKE, 2, cu, cu, 1, 2, 2, 128, 128, 128, 128, 64, 0, 0.0,
                                       32, FAKE, 1 << 30, None)
    assert rc == _lib.EINVAL


def test_host_forward_scratch_size(lib):
    """Two slots, each holding one chunk's inputs, output and workspace: more chunks need less
    scratch; chunk sizes that do not divide Hkv (or bad types) give 0 / SAGE2_EINVAL."""
    B, Hq, Hkv, N, D = 1, 32, 8, 4096, 128
    sizes = [lib.sage2_host_scratch_size(B, Hq, Hkv, N, N, D, 1, c, 0) for c in (8, 4, 2, 1)]
    assert all(s > 0 for s in sizes) and sizes == sorted(sizes, reverse=True)
    one_chunk_inputs = B * N * (Hq + 2 * Hkv) * D * 2
    assert sizes[0] >= 2 * one_chunk_inputs  # two slots of the whole problem
    assert lib.sage2_host_scratch_size(B, Hq, Hkv, N, N, D, 1, 3, 0) == 0
    assert lib.sage2_host_scratch_size(B, Hq, Hkv, N, N, D, 7, 1, 0) == 0
    assert lib.sage2_host_scratch_size(B, Hq, Hkv, N, N, D, 1, 1, 8) > sizes[3]  # 2-byte codes
    out = ctypes.c_void_p(0x20000)
    rc = lib.sage2_attn_fwd_host(FAKE, FAKE, FAKE, out, 1, 1, B, Hq, Hkv, N, N, D, 0, 0.0, 0, 3,
                                 FAKE, 1 << 40, None)
    assert rc == _lib.EINVAL
    rc = lib.sage2_attn_fwd_host(FAKE, FAKE, FAKE, out, 1, 1, B, Hq, Hkv, N, N, D, 0, 0.0, 0, 1,
                                 FAKE, 16, None)
    assert rc == _lib.EWORKSPACE
