"""The forward from host memory (sage2_attn_fwd_host): chunked over kv-head groups with the
copies overlapped; its result must equal the device forward on the whole problem bit for bit,
for every chunk size, both code formats and both output types."""
from __future__ import annotations

import pytest
import torch

import bit_exact_attention_gb300 as S
from bit_exact_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    S.load_library()


CASES = [
    (W.TINY, (1, 2)),
    (W.scaled(W.PREFILL, (384, 384), (384, 384), hq=4, hkv=2, name="prefill_d"), (1, 2)),
    (W.scaled(W.GQA_LONG, (1000,), (1000,), hq=8, hkv=4, name="gqa_d"), (1, 2, 4)),
    (W.scaled(W.VIDEO_DIT, (333, 333), (333, 333), hq=3, hkv=3, name="dit_d"), (1, 3)),
    # causal with Nq != Nkv (bottom-right aligned), both ways, GQA groups of 3
    (W.scaled(W.GQA_LONG, (300,), (700,), hq=6, hkv=2, name="gqa_q_lt_kv"), (1, 2)),
    (W.scaled(W.GQA_LONG, (650,), (260,), hq=6, hkv=2, name="gqa_q_gt_kv"), (1, 2)),
]


@pytest.mark.parametrize("quant", [0, S.QUANT_SAGE1], ids=["sage2", "sage1"])
@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_host_forward_equals_device_forward(case, quant):
    w, chunk_sizes = case
    x = W.make_inputs(w)
    B, nq, nkv = w.batch, w.nq[0], w.nkv[0]
    q = x["q"].view(B, nq, w.hq, w.d)
    k = x["k"].view(B, nkv, w.hkv, w.d)
    v = x["v"].view(B, nkv, w.hkv, w.d)
    for out_dtype in (torch.float32, q.dtype):
        want = S.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, out_dtype=out_dtype,
                          quant_flags=quant).cpu()
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        for c in chunk_sizes:
            out = torch.full((B, nq, w.hq, w.d), float("nan"), dtype=out_dtype).pin_memory()
            scratch = S.attn_fwd_host(qh, kh, vh, out, causal=w.causal, quant_flags=quant,
                                      kv_heads_per_chunk=c)
            assert S.host_status(scratch) == (0, 0)
            assert torch.equal(out, want), (w.name, c, out_dtype)


def test_host_forward_pageable_memory_and_bad_chunking():
    w = W.TINY
    x = W.make_inputs(w)
    q = x["q"].view(1, 256, 2, 64)
    k = x["k"].view(1, 256, 2, 64)
    v = x["v"].view(1, 256, 2, 64)
    out = torch.empty(1, 256, 2, 64, dtype=torch.float32)
    s = S.attn_fwd_host(q, k, v, out, kv_heads_per_chunk=2)  # pageable: correct, not overlapped
    torch.cuda.synchronize()
    assert S.host_status(s) == (0, 0)
    want = S.attn_fwd(q.cuda(), k.cuda(), v.cuda(), out_dtype=torch.float32).cpu()
    assert torch.equal(out, want)
    with pytest.raises((S.Sage2Error, ValueError)):
        S.attn_fwd_host(q, k, v, out, kv_heads_per_chunk=3)  # does not divide Hkv = 2
