"""The forward's stream behaviour: the prepass runs its Q codes and its V and K codes on
library-owned side streams forked from the caller's stream and joined back into it (events), so
the pair prepass + attention must stay ordered on any caller stream, and must be capturable in a
CUDA graph whose replays give the same bits as direct calls."""
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


def _problem(name):
    w = W.scaled(W.GQA_LONG, (1200,), (1500,), hq=8, hkv=2, name=name)
    x = W.make_inputs(w)
    dev = torch.device("cuda", 0)
    q, k, v = (x[n].to(dev) for n in "qkv")
    cu_q = torch.tensor(x["cu_q"], dtype=torch.int32, device=dev)
    cu_kv = torch.tensor(x["cu_kv"], dtype=torch.int32, device=dev)
    return w, q, k, v, cu_q, cu_kv


def _forward(w, q, k, v, cu_q, cu_kv, out, ws, stream):
    nq, nkv = max(w.nq), max(w.nkv)
    S.prepass_varlen(q, k, v, cu_q, cu_kv, nq, nkv, ws, causal=w.causal, stream=stream)
    S.attention_varlen(out, ws, cu_q, cu_kv, w.hkv, nq, nkv, sum(w.nkv), causal=w.causal,
                       stream=stream)


def _workspace(w, dev):
    return S.alloc_workspace(S.workspace_size(w.batch, w.hq, w.hkv, max(w.nq), max(w.nkv), w.d,
                                              sum(w.nq), sum(w.nkv)), dev)


def test_forward_on_a_side_stream_matches_the_default_stream():
    w, q, k, v, cu_q, cu_kv = _problem("streams_a")
    dev = q.device
    ref = torch.empty(sum(w.nq), w.hq, w.d, dtype=q.dtype, device=dev)
    ws0 = _workspace(w, dev)
    _forward(w, q, k, v, cu_q, cu_kv, ref, ws0, None)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = torch.full_like(ref, float("nan"))
    ws1 = _workspace(w, dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):  # back-to-back calls reuse the side streams' events
            _forward(w, q, k, v, cu_q, cu_kv, out, ws1, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert S.device_status(ws1) == (0, 0)
    assert torch.equal(out, ref)


def test_forward_captured_in_a_cuda_graph_replays_bit_identically():
    w, q, k, v, cu_q, cu_kv = _problem("streams_b")
    dev = q.device
    ref = torch.empty(sum(w.nq), w.hq, w.d, dtype=q.dtype, device=dev)
    ws = _workspace(w, dev)
    _forward(w, q, k, v, cu_q, cu_kv, ref, ws, None)  # first calls outside any capture
    torch.cuda.synchronize()
    out = torch.full_like(ref, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _forward(w, q, k, v, cu_q, cu_kv, out, ws, torch.cuda.current_stream())
    torch.cuda.synchronize()
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert S.device_status(ws) == (0, 0)
        assert torch.equal(out, ref)
