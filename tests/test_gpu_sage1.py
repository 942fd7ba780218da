"""GPU parity of the SageAttention (v1) path (SAGE2_QUANT_SAGE1), through the C ABI.

The SageAttention2 research note contrasts the method with SageAttention's INT8 path (its
opening paragraph and the comparison of the two versions): Q and K on the INT8 grid with
per-block scales, K smoothed, Q not; P~ and V as in the method. Here Q K^T runs on 16-bit
tensor-core operands that hold the integer codes exactly. Gates, against the oracle run with
the same switches (oracle.SAGE1):
  * prepass results bit-exact (INT8 codes, scales, K means, V codes);
  * the raw Q K^T accumulators bit-exact (integers up to 127^2 * 128 < 2^24: exact in FP32);
  * P~ codes equal except one-step flips at exponential rounding midpoints;
  * the output within relative L1 1e-3 of the emulation and every element within 2e-3,
    except rows proven to differ only through located P~ midpoint flips
    (parity_util.check_forward_proven);
  * a workspace of one code format is refused by the other format's attention kernel.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import bit_exact_attention_gb300 as S
from bit_exact_attention_gb300 import workloads as W
from parity_util import (GpuCase, bits, check_forward_proven, compare_p_codes, kv_tiles,
                         metrics, unit_rows, units_sample)

pytestmark = pytest.mark.gpu

F = S.QUANT_SAGE1
KW = oracle.SAGE1

CASES = {
    "tiny": W.TINY,
    "prefill": W.scaled(W.PREFILL, (700, 300), (700, 300), hq=4, hkv=4, name="prefill_s"),
    "gqa": W.scaled(W.GQA_LONG, (1000,), (1000,), hq=8, hkv=2, name="gqa_s"),
    "dit": W.scaled(W.VIDEO_DIT, (600, 333), (600, 333), hq=3, hkv=3, name="dit_s"),
    "varlen": W.scaled(W.VARLEN, (300, 77, 129), (500, 129, 1000), hq=8, hkv=2, name="varlen_s"),
}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    assert torch.cuda.get_device_capability() == (10, 3), "expected an sm_103 GPU"
    oracle.build()
    S.load_library()


_inputs = {}


def _case(name):
    if name not in _inputs:
        w = CASES[name]
        _inputs[name] = (w, W.make_inputs(w))
    return _inputs[name]


def _args(w, x):
    return (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)


@pytest.mark.parametrize("name", ["tiny", "prefill", "dit", "varlen"])
def test_prepass_bit_exact(name):
    w, x = _case(name)
    g = GpuCase(w, x, quant_flags=F)
    assert g.L.code_bytes == 2
    g.prepass()
    assert g.status() == (0, 0)
    got = g.gathered()
    dt = W.dtype_code(w)
    kmean, vamax = oracle.kv_stats(bits(x["k"]), bits(x["v"]), dt, x["cu_kv"], w.hkv, w.d)
    qmean, qc, sq = oracle.quant_q(bits(x["q"]), dt, x["cu_q"], w.hq, w.d, smooth_q=False,
                                   per_block=True, qk_bits=8)
    kc, sk = oracle.quant_k(bits(x["k"]), dt, x["cu_kv"], w.hkv, w.d, kmean=kmean, gk=128,
                            qk_bits=8)
    vc, sv = oracle.quant_v(bits(x["v"]), dt, x["cu_kv"], w.hkv, w.d, vamax)
    assert np.abs(qc).max() == 127 and np.abs(kc).max() == 127
    np.testing.assert_array_equal(got["kmean"], kmean)
    np.testing.assert_array_equal(got["vscale"], sv)
    assert int((got["qcode"] != qc).sum()) == 0, "Q code mismatches"
    np.testing.assert_array_equal(got["qscale"], sq)
    assert int((got["kcode"] != kc).sum()) == 0, "K code mismatches"
    np.testing.assert_array_equal(got["kscale"], sk)
    np.testing.assert_array_equal(got["vcode"], oracle.e4m3_decode(vc))


@pytest.mark.parametrize("name", ["tiny", "prefill", "dit", "varlen"])
def test_qk_accumulators_bit_exact(name):
    w, x = _case(name)
    g = GpuCase(w, x, quant_flags=F)
    g.prepass()
    dt = W.dtype_code(w)
    kmean, _ = oracle.kv_stats(bits(x["k"]), bits(x["v"]), dt, x["cu_kv"], w.hkv, w.d)
    _, qc, _ = oracle.quant_q(bits(x["q"]), dt, x["cu_q"], w.hq, w.d, smooth_q=False,
                              per_block=True, qk_bits=8)
    kc, _ = oracle.quant_k(bits(x["k"]), dt, x["cu_kv"], w.hkv, w.d, kmean=kmean, gk=128,
                           qk_bits=8)
    Dp = g.L.Dp
    checked = 0
    for b in range(w.batch):
        nqb = (w.nq[b] + 127) // 128
        for (h, qt) in {(0, 0), (w.hq - 1, nqb - 1), (w.hq // 2, nqb // 2)}:
            if nqb == 0:
                continue
            T = kv_tiles(qt, w.nq[b], w.nkv[b], w.causal)
            for kt in sorted({0, T - 1}):
                if kt < 0:
                    continue
                s_out, _, _ = g.debug_tile(b, h, qt, kt)
                A = np.zeros((128, Dp), np.int64)
                rows = np.arange(qt * 128, min(w.nq[b], qt * 128 + 128))
                A[: len(rows)] = qc[x["cu_q"][b] + rows, h]
                Kt = np.zeros((128, Dp), np.int64)
                keys = np.arange(kt * 128, min(w.nkv[b], kt * 128 + 128))
                Kt[: len(keys)] = kc[x["cu_kv"][b] + keys, h // (w.hq // w.hkv)]
                want = A @ Kt.T
                assert np.abs(want).max() > 7 * 7 * 128, "codes beyond the INT4 range expected"
                got = s_out.cpu().numpy()
                assert np.array_equal(got, want.astype(np.float64)), (
                    f"{name} b{b} h{h} qt{qt} kt{kt}: {(got != want).sum()} accumulator mismatches")
                checked += 1
    assert checked >= 2


@pytest.mark.parametrize("name", ["prefill", "dit", "varlen"])
def test_p_codes_agree_except_at_exp2_rounding_midpoints(name):
    w, x = _case(name)
    g = GpuCase(w, x, quant_flags=F)
    g.prepass()
    n_diff, n_cmp = compare_p_codes(g, w, x, KW)
    assert n_diff <= 1e-3 * n_cmp, (n_diff, n_cmp)


@pytest.mark.parametrize("name", list(CASES))
def test_forward_matches_emulation(name):
    w, x = _case(name)
    g = GpuCase(w, x, quant_flags=F)
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    check_forward_proven(g, w, x, out, oracle.attention_emulated(*_args(w, x), **KW), KW)


@pytest.mark.parametrize("name", ["prefill", "gqa", "dit", "varlen"])
def test_int8_path_is_more_accurate_than_int4(name):
    """Against exact attention the INT8 path meets cosine >= 0.99 and relative L1 <= 0.06 on
    these distributions, and errs less than the INT4 method (as in the emulation)."""
    w, x = _case(name)
    ex = oracle.attention_exact(*_args(w, x))
    o1 = GpuCase(w, x, quant_flags=F).forward(out_dtype=torch.float32).cpu().numpy()
    o2 = GpuCase(w, x).forward(out_dtype=torch.float32).cpu().numpy()
    m1, m2 = metrics(o1, ex), metrics(o2, ex)
    assert m1["cos"] >= 0.99 and m1["relL1"] <= 0.06, m1
    assert m1["relL1"] < m2["relL1"], (m1, m2)


EDGE = [
    # (nq, nkv, hq, hkv, d, causal, dtype)
    ((1,), (1,), 1, 1, 64, False, "fp16"),
    ((300,), (100,), 2, 2, 128, True, "bf16"),     # rows with no visible key output 0
    ((100,), (300,), 2, 2, 64, True, "fp16"),
    ((129, 0, 5), (0, 64, 257), 4, 2, 128, False, "bf16"),  # empty sequences
    ((200,), (333,), 2, 2, 80, False, "fp16"),     # D0 = 80
    ((150,), (150,), 2, 2, 112, True, "bf16"),
]


@pytest.mark.parametrize("case", EDGE, ids=[f"e{i}" for i in range(len(EDGE))])
def test_edge_cases(case):
    nq, nkv, hq, hkv, d, causal, dt = case
    w = W.Workload("edge", nq, nkv, hq, hkv, d, dt, causal, "kbias9", 31, varlen=True)
    x = W.make_inputs(w)
    g = GpuCase(w, x, quant_flags=F)
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    emu = oracle.attention_emulated(*_args(w, x), **KW)
    if np.abs(emu).sum() == 0:
        assert np.all(out == 0)
    else:
        check_forward_proven(g, w, x, out, emu, KW)
    for b in range(w.batch):
        for i in range(w.nq[b]):
            if w.nkv[b] == 0 or (causal and i + w.nkv[b] - w.nq[b] < 0):
                assert np.all(out[x["cu_q"][b] + i] == 0)


def test_dense_entry_equals_varlen():
    w = W.scaled(W.PREFILL, (384, 384), (384, 384), hq=4, hkv=2, name="dense_eq")
    x = W.make_inputs(w)
    a = GpuCase(w, x, quant_flags=F).forward(out_dtype=torch.float32)
    q = x["q"].view(2, 384, 4, 128).cuda()
    k = x["k"].view(2, 384, 2, 128).cuda()
    v = x["v"].view(2, 384, 2, 128).cuda()
    b = S.attn_fwd(q, k, v, causal=True, out_dtype=torch.float32, quant_flags=F)
    assert torch.equal(a.view(2, 384, 4, 128), b)


def test_format_mismatch_is_refused_on_the_device():
    """An attention call whose code format differs from the one its prepass recorded writes
    nothing and reports SAGE2_EINVAL through the device status; the context stays usable."""
    w, x = _case("tiny")
    # INT8 workspace, INT4 kernel: the workspace is large enough for either
    g = GpuCase(w, x, quant_flags=F)
    g.prepass()
    out = torch.full((g.tq, w.hq, w.d), 7.0, dtype=torch.float32, device="cuda")
    S.attention_varlen(out, g.ws, g.cu_q, g.cu_kv, w.hkv, g.max_nq, g.max_nkv, g.tkv,
                       causal=w.causal, quant_flags=S.QUANT_PER_BLOCK)
    code, raw = g.status()
    assert code == -1 and raw == 0x300, (code, hex(raw))
    assert torch.all(out == 7.0)
    # INT4 workspace, INT8 kernel
    g2 = GpuCase(w, x)
    g2.prepass()
    ws_big = torch.zeros(S.workspace_size(w.batch, w.hq, w.hkv, g2.max_nq, g2.max_nkv, w.d,
                                          g2.tq, g2.tkv, quant_flags=F), dtype=torch.uint8,
                         device="cuda")
    # the status area (error word, then the code format) sits at the 1024-aligned base
    off = (-ws_big.data_ptr()) % 1024
    ws_big[off: off + 256].copy_(g2.ws[g2.off0: g2.off0 + 256])
    S.attention_varlen(out, ws_big, g2.cu_q, g2.cu_kv, w.hkv, g2.max_nq, g2.max_nkv, g2.tkv,
                       causal=w.causal, quant_flags=F)
    code, raw = S.device_status(ws_big)
    assert code == -1 and raw == 0x300, (code, hex(raw))
    assert torch.all(out == 7.0)
    # and a correct call afterwards works
    ok = GpuCase(w, x, quant_flags=F).forward(out_dtype=torch.float32).cpu().numpy()
    assert metrics(ok, oracle.attention_emulated(*_args(w, x), **KW))["relL1"] <= 1e-3


@pytest.mark.parametrize("wl", [W.GQA_LONG, W.PREFILL], ids=["gqa_long", "prefill"])
def test_full_size_sampled_units(wl):
    """Full-size workloads, as the benchmark launches them with the INT8 switch; the oracle
    computes >= 32 seeded (sequence, head, Q block) units including the last partial block,
    the first block and a causal-diagonal block."""
    x = W.make_inputs(wl)
    g = GpuCase(wl, x, quant_flags=F)
    out = g.forward(out_dtype=torch.float32)
    assert g.status() == (0, 0)
    units = units_sample(wl, 32, seed=wl.seed)
    emu = oracle.attention_emulated(*_args(wl, x), units=units, **KW)
    toks, heads = unit_rows(wl, x["cu_q"], units)
    got = out[torch.from_numpy(toks).cuda(), torch.from_numpy(heads).cuda()].cpu().numpy()
    want = emu[toks, heads]
    m = metrics(got, want)
    assert m["relL1"] <= 1e-3, m
