"""The allocation-free forward entry point (sage2_attn_fwd_noalloc) against the regular one.

Some callers cannot allocate device memory -- runtimes that own every device allocation and
forbid allocation calls from libraries they host, or allocation-free latency-critical loops --
so the library offers a forward that uses its own fixed scratch array instead of a caller
workspace. This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import bit_exact_attention_gb300 as S
from bit_exact_attention_gb300 import _lib
from bit_exact_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

REL_L1, MAX_ABS = 1e-3, 2e-3


def _dense(w):
    x = W.make_inputs(w)
    B, nq, nkv = w.batch, w.nq[0], w.nkv[0]
    q = x["q"].view(B, nq, w.hq, w.d).cuda()
    k = x["k"].view(B, nkv, w.hkv, w.d).cuda()
    v = x["v"].view(B, nkv, w.hkv, w.d).cuda()
    return q, k, v


def _noalloc_via_abi(q, k, v, out, causal):
    lib = _lib.lib()
    B, Nq, Hq, D = q.shape
    _, Nkv, Hkv, _ = k.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sage2_attn_fwd_noalloc(p(q), p(k), p(v), p(out), code[q.dtype], code[out.dtype],
                                      B, Hq, Hkv, Nq, Nkv, D, int(causal), 0.0, stream)


def _close(a, r):
    a = a.double().cpu().numpy()
    r = r.double().cpu().numpy()
    rel = np.abs(a - r).sum() / np.abs(r).sum()
    return rel <= REL_L1 and np.abs(a - r).max() <= MAX_ABS, (rel, np.abs(a - r).max())


def test_noalloc_matches_regular_entry_on_two_calls_in_a_row():
    assert torch.cuda.is_available()
    cases = [
        (W.scaled(W.PREFILL, (384, 384), (384, 384), hq=4, hkv=2, name="na_a"), True),
        (W.TINY, False),  # smaller second call: stale scratch contents must not matter
    ]
    for w, causal in cases:
        q, k, v = _dense(w)
        ref = S.attn_fwd(q, k, v, causal=causal, out_dtype=torch.float32)
        out = torch.empty_like(ref)
        assert _noalloc_via_abi(q, k, v, out, causal) == 0
        assert S.noalloc_status() == (0, 0)  # synchronizes, then reads the scratch status word
        ok, info = _close(out, ref)
        assert ok, (w.name, info)


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.lib()
    need = lib.sage2_workspace_size(1, 32, 8, 32768, 32768, 128, 32768, 32768)
    assert need > S.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check fails first
    rc = lib.sage2_attn_fwd_noalloc(fake, fake, fake, fake, 1, 1, 1, 32, 8, 32768, 32768, 128, 1,
                                    0.0, None)
    assert rc == _lib.EWORKSPACE
