"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties an oracle function to a library routine, a closed form, a
hand-worked fixture under ``tests/golden/``, an invariant of the mathematics or an
independent brute-force restatement, chosen so that a dropped term, a wrong sign
or index, or a transposed operand fails at least one of them.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from bit_exact_attention_gb300 import workloads as W
import np_restatement as NR

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F16, BF16 = 0, 1


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def relL1(a, r):
    return float(np.abs(a - r).sum() / np.abs(r).sum())


def cosine(a, r):
    a, r = a.ravel(), r.ravel()
    return float(a @ r / math.sqrt((a @ a) * (r @ r)))


# ----------------------------------------------------------------- number formats
def test_f16_decode_matches_numpy(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = oracle_mod.f16_to_f64(allbits)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_bf16_decode_matches_torch(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_mod.bf16_to_f64(allbits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])


def _e4m3_probe_values():
    """Every finite e4m3 value, every midpoint between neighbours, and the fp32
    neighbours of both, plus random values in range."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = codes.to(torch.float64).numpy()
    finite = np.unique(vals[np.isfinite(vals)])
    mids = (finite[1:] + finite[:-1]) / 2
    base = np.concatenate([finite, mids]).astype(np.float32)
    up = np.nextafter(base, np.float32(np.inf))
    dn = np.nextafter(base, np.float32(-np.inf))
    rng = np.random.default_rng(7)
    rnd = (rng.standard_normal(20000) * rng.choice([1e-3, 0.1, 3, 60, 200], 20000)).astype(np.float32)
    allv = np.concatenate([base, up, dn, rnd])
    return allv[np.abs(allv) < 464.0]  # above this torch returns NaN, ours saturates


def test_e4m3_encode_matches_torch_cast(oracle_mod):
    x = _e4m3_probe_values()
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


def test_e4m3_decode_matches_torch(oracle_mod):
    allc = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(allc).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle_mod.e4m3_decode(allc)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_saturation_closed_form(oracle_mod):
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e4, 1e30, np.inf])
    assert list(oracle_mod.e4m3_encode(x)) == [0x7E] * len(x)
    assert list(oracle_mod.e4m3_encode(-x)) == [0xFE] * len(x)


def test_e4m3_golden_boundaries(oracle_mod):
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_boundaries.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                parts = line.split()
                rows.append((float(parts[0]), int(parts[1], 16)))
    got = oracle_mod.e4m3_encode(np.array([r[0] for r in rows]))
    for (x, want), g in zip(rows, got):
        assert g == want, (x, hex(g), hex(want))


def test_round_output_fp16_matches_numpy(oracle_mod):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.uniform(-8, 4, 50000),
                        [0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e6, -1e6, 2 ** -25, 2 ** -24 * 1.5]])
    got = oracle_mod.round_output(x, F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_round_output_bf16_matches_torch(oracle_mod):
    rng = np.random.default_rng(2)
    x32 = (rng.standard_normal(50000) * 10.0 ** rng.uniform(-30, 30, 50000)).astype(np.float32)
    got = oracle_mod.round_output(x32.astype(np.float64), BF16)
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------- Mode E
def _sdpa_ref(q, k, v, cu_q, cu_kv, hq, hkv, causal, scale):
    """torch SDPA in float64 per sequence with an explicit bottom-right mask."""
    out = np.zeros((cu_q[-1], hq, q.shape[-1]))
    g = hq // hkv
    for b in range(len(cu_q) - 1):
        Q = torch.from_numpy(q[cu_q[b]:cu_q[b + 1]]).permute(1, 0, 2)
        K = torch.from_numpy(k[cu_kv[b]:cu_kv[b + 1]]).permute(1, 0, 2).repeat_interleave(g, 0)
        V = torch.from_numpy(v[cu_kv[b]:cu_kv[b + 1]]).permute(1, 0, 2).repeat_interleave(g, 0)
        nq, nkv = Q.shape[1], K.shape[1]
        mask = None
        if causal:
            i = torch.arange(nq)[:, None]
            j = torch.arange(nkv)[None, :]
            mask = j <= i + (nkv - nq)
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        o = o.permute(1, 0, 2).numpy()
        if causal:  # rows with no visible key: the method outputs 0
            empty = ~mask.any(dim=1).numpy()
            o[empty] = 0.0
        out[cu_q[b]:cu_q[b + 1]] = o
    return out


@pytest.mark.parametrize("dtype,causal,nq,nkv,hq,hkv,d0", [
    ("fp16", False, (37, 5), (40, 129), 4, 2, 64),
    ("bf16", True, (70, 9), (70, 3), 2, 1, 128),
    ("bf16", True, (20,), (45,), 3, 3, 80),
])
def test_exact_matches_sdpa(oracle_mod, dtype, causal, nq, nkv, hq, hkv, d0):
    w = W.Workload("t", nq, nkv, hq, hkv, d0, dtype, causal, "kbias9", 11, varlen=True)
    x = W.make_inputs(w)
    q64, k64, v64 = (x[n].to(torch.float64).numpy() for n in "qkv")
    scale = 1.0 / math.sqrt(d0)
    got = oracle_mod.attention_exact(bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w),
                                     x["cu_q"], x["cu_kv"], hq, hkv, d0, causal, scale)
    ref = _sdpa_ref(q64, k64, v64, x["cu_q"], x["cu_kv"], hq, hkv, causal, float(np.float32(scale)))
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_exact_closed_forms(oracle_mod):
    # K == 0: every visible key has the same logit -> mean of the visible V rows.
    nq = nkv = 6
    q = torch.randn(nq, 1, 64, generator=torch.Generator().manual_seed(3)).half()
    k = torch.zeros(nkv, 1, 64).half()
    v = torch.randn(nkv, 1, 64, generator=torch.Generator().manual_seed(4)).half()
    out = oracle_mod.attention_exact(bits(q), bits(k), bits(v), F16, [0, nq], [0, nkv], 1, 1, 64, True)
    v64 = v.double().numpy()[:, 0]
    for i in range(nq):
        np.testing.assert_allclose(out[i, 0], v64[: i + 1].mean(axis=0), rtol=1e-12, atol=1e-14)
    # causal with nq > nkv: the first nq - nkv rows see nothing -> 0; the next sees one key.
    out = oracle_mod.attention_exact(bits(q), bits(k[:2]), bits(v[:2]), F16, [0, nq], [0, 2], 1, 1, 64, True)
    assert np.all(out[:4] == 0.0)
    np.testing.assert_allclose(out[4, 0], v64[0], rtol=1e-12)


def test_exact_units_subset_matches_full(oracle_mod):
    w = W.scaled(W.PREFILL, (300,), (300,), hq=2, hkv=2)
    x = W.make_inputs(w)
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), BF16, x["cu_q"], x["cu_kv"], 2, 2, 128, True)
    full = oracle_mod.attention_exact(*args)
    units = [(0, 1, 2), (0, 0, 0)]
    part = oracle_mod.attention_exact(*args, units=units)
    np.testing.assert_array_equal(part[256:300, 1], full[256:300, 1])
    np.testing.assert_array_equal(part[0:128, 0], full[0:128, 0])
    assert np.all(part[0:128, 1] == 0)


# ----------------------------------------------------------------- Mode Q steps
def test_kv_stats_vs_numpy(oracle_mod):
    w = W.scaled(W.VARLEN, (5, 5), (100, 37), hq=4, hkv=2, d=80)
    x = W.make_inputs(w)
    km, va = oracle_mod.kv_stats(bits(x["k"]), bits(x["v"]), BF16, x["cu_kv"], 2, 80)
    k64, v64 = x["k"].double().numpy(), x["v"].double().numpy()
    for b in range(2):
        s, e = x["cu_kv"][b], x["cu_kv"][b + 1]
        np.testing.assert_array_equal(km[b, :, :80], k64[s:e].mean(axis=0).astype(np.float32))
        np.testing.assert_array_equal(va[b, :, :80], np.abs(v64[s:e]).max(axis=0).astype(np.float32))
        assert np.all(km[b, :, 80:] == 0) and np.all(va[b, :, 80:] == 0)


def test_quant_golden_rows(oracle_mod):
    with open(os.path.join(GOLDEN, "int4_rows.txt")) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    vals, codes, scales = [], [], []
    for ln in lines:
        a, b, c = ln.split("|")
        vals.append([float(t) for t in a.split()])
        codes.append([int(t) for t in b.split()])
        scales.append(float(c))
    # rows of one head, one token each; smoothing off so Q~ = Q exactly
    q = torch.zeros(len(vals), 1, 8)
    q[:, 0, :] = torch.tensor(vals)
    qm, qc, sq = oracle_mod.quant_q(bits(q.half()), F16, [0, len(vals)], 1, 8, smooth_q=False)
    for r in range(len(vals)):
        assert list(qc[r, 0, :8]) == codes[r], r
        assert np.all(qc[r, 0, 8:] == 0)
        assert sq[r, 0] == np.float32(scales[r]), r


def _check_codes(xt, codes, scale):
    """Invariants of the INT4-grid quantizer for one group."""
    assert codes.min() >= -7 and codes.max() <= 7
    if scale == 0:
        assert np.all(codes == 0) and np.all(xt == 0)
        return
    assert np.abs(codes).max() == 7
    err = np.abs(xt.astype(np.float64) - codes * float(scale))
    assert err.max() <= 0.5 * float(scale) * (1 + 1e-5) + 1e-30


def test_quant_q_means_and_invariants(oracle_mod):
    w = W.scaled(W.PREFILL, (300,), (300,), hq=2, hkv=2)
    x = W.make_inputs(w)
    qm, qc, sq = oracle_mod.quant_q(bits(x["q"]), BF16, x["cu_q"], 2, 128)
    q64 = x["q"].double().numpy()
    for h in range(2):
        for qb in range(3):
            rows = slice(qb * 128, min(300, qb * 128 + 128))
            np.testing.assert_array_equal(qm[0, h, qb], q64[rows, h].mean(axis=0).astype(np.float32))
            xt = (q64[rows, h].astype(np.float32) - qm[0, h, qb]).astype(np.float32)
            for r in range(xt.shape[0]):
                _check_codes(xt[r], qc[rows, h][r], sq[rows, h][r])


def test_quant_k_groups_and_ragged_tail(oracle_mod):
    w = W.scaled(W.VARLEN, (3, 3), (70, 33), hq=2, hkv=1)
    x = W.make_inputs(w)
    km, _ = oracle_mod.kv_stats(bits(x["k"]), bits(x["v"]), BF16, x["cu_kv"], 1, 128)
    kc, sk = oracle_mod.quant_k(bits(x["k"]), BF16, x["cu_kv"], 1, 128, kmean=km)
    k64 = x["k"].double().numpy()
    for b in range(2):
        s, e = x["cu_kv"][b], x["cu_kv"][b + 1]
        kt = (k64[s:e, 0].astype(np.float32) - km[b, 0]).astype(np.float32)
        for t0 in range(0, e - s, 32):           # groups restart at each sequence start
            grp = slice(t0, min(t0 + 32, e - s))
            assert len(set(sk[s:e, 0][grp].tolist())) == 1
            _check_codes(kt[grp], kc[s:e, 0][grp], sk[s:e, 0][grp][0])
            assert sk[s:e, 0][grp][0] == np.float32(np.abs(kt[grp]).max() / np.float32(7))


def test_quant_v_per_channel(oracle_mod):
    w = W.scaled(W.TINY, (4,), (50,), hq=1, hkv=1)
    x = W.make_inputs(w)
    _, va = oracle_mod.kv_stats(bits(x["k"]), bits(x["v"]), F16, x["cu_kv"], 1, 64)
    vc, sv = oracle_mod.quant_v(bits(x["v"]), F16, x["cu_kv"], 1, 64, va)
    v64 = x["v"].double().numpy()[:, 0]
    dec = oracle_mod.e4m3_decode(vc[:, 0])
    # the channel maximum maps to +-448 exactly; every value within e4m3 rounding
    for d in range(64):
        j = int(np.argmax(np.abs(v64[:, d])))
        assert abs(dec[j, d]) == 448.0
    recon = dec * sv[0, 0][None, :].astype(np.float64)
    rel = np.abs(recon - v64) / np.maximum(np.abs(v64), 2 ** -6 * va[0, 0][None, :] / 448)
    assert rel.max() <= 1 / 16 + 1e-6


def _f32_nearest(fr: Fraction) -> np.float32:
    """The FP32 value nearest to a rational, ties to even (checked among the neighbours of its
    FP64 rounding)."""
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr),
                                     int(np.array(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_delta_s_is_the_correctly_rounded_dot_product(oracle_mod):
    """Delta-S = qbar . K~ with K~ = fl32(K - kmean): on 96 keys the oracle's value is the exact
    rational dot product of the FP32 operands rounded to the nearest FP32 value."""
    w = W.scaled(W.PREFILL, (200,), (300,), hq=1, hkv=1)
    x = W.make_inputs(w)
    km, _ = oracle_mod.kv_stats(bits(x["k"]), bits(x["v"]), BF16, x["cu_kv"], 1, 128)
    qm, _, _ = oracle_mod.quant_q(bits(x["q"]), BF16, x["cu_q"], 1, 128)
    qbar = qm[0, 0, 1]
    ds = oracle_mod.delta_s(bits(x["k"]), BF16, x["cu_kv"], 0, 1, 0, 128, km, qbar)
    kt = (x["k"].float().numpy()[:, 0] - km[0, 0]).astype(np.float32)  # fl32(K - kmean)
    rng = np.random.default_rng(5)
    for j in sorted(rng.choice(300, 96, replace=False)):
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qbar, kt[j]))
        assert ds[j] == _f32_nearest(exact), (j, ds[j], float(exact))
    # sign and term: the correction is + qbar . K~ (not minus, not qbar . K)
    assert np.corrcoef(ds, kt.astype(np.float64) @ qbar.astype(np.float64))[0, 1] > 0.999999


# ----------------------------------------------------------------- Mode Q pins
def _golden_example():
    data = {}
    with open(os.path.join(GOLDEN, "worked_example_smoothing.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            p = line.split()
            if p[0] == "SM_SCALE":
                data["sm"] = float(p[1])
            else:
                r, c = int(p[1]), int(p[2])
                vals = [float(Fraction(t)) for t in p[3:]]
                data[p[0]] = np.array(vals).reshape(r, c)
    return data


def test_worked_example_both_modes(oracle_mod):
    g = _golden_example()
    q = torch.tensor(g["Q"])[:, None, :].half()
    k = torch.tensor(g["K"])[:, None, :].half()
    v = torch.tensor(g["V"])[:, None, :].half()
    assert np.float32(1.4426950408889634 * g["sm"]) == np.float32(1.0)
    args = (bits(q), bits(k), bits(v), F16, [0, 2], [0, 2], 1, 1, 4, False, g["sm"])
    emu = oracle_mod.attention_emulated(*args)[:, 0]
    ex = oracle_mod.attention_exact(*args)[:, 0]
    np.testing.assert_allclose(emu, g["O"], rtol=2e-6)
    np.testing.assert_allclose(ex, g["O"], rtol=1e-7)


def _sm_scale_for_unit_c():
    s = np.float32(math.log(2.0))
    assert np.float32(1.4426950408889634 * float(s)) == np.float32(1.0)
    return float(s)


def _zero_error_inputs(seed, nq=24, nkv=40, d0=64, with_means=True, g=7, qmean=True):
    """Inputs on which every quantization step is exact ([R] pin of the pipeline):
    Q~ rows come in adjacent +-pairs (so every Q block of even size has mean exactly
    qbar) and K~ rows in +-pairs (channel mean exactly kmean); both sit on the INT4
    grid with a 7 in a channel the other side leaves zero, so every scale is 1; V is on
    the e4m3 grid with 448 in every channel; every logit gap is an integer <= 12, so
    448 P stays on the normal e4m3 grid."""
    rng = np.random.default_rng(seed)
    qt = np.zeros((nq, d0))
    kt = np.zeros((nkv, d0))
    qt[0::2, :2] = rng.integers(-1, 2, size=(nq // 2, 2))
    qt[0::2, d0 - 2] = g
    qt[1::2] = -qt[0::2]
    half_k = nkv // 2
    kt[:half_k, :2] = rng.integers(-1, 2, size=(half_k, 2))
    kt[:half_k, 2] = 2 * rng.integers(-1, 2, size=half_k)
    kt[:half_k, d0 - 1] = g
    kt[half_k:] = -kt[:half_k]
    kt = kt[rng.permutation(nkv)]
    qbar = np.zeros(d0)
    kmean = np.zeros(d0)
    if with_means:
        # |A| <= 2 and |dS| <= 3; the 0.5 in channel 2 meets even K~ values only, so dS
        # stays an integer, while an unsmoothed Q would round that 0.5 away
        if qmean:
            qbar[:2] = rng.integers(-1, 2, size=2)
            qbar[2] = 0.5
        kmean[4:8] = rng.integers(-3, 4, size=4)
    q = qt + qbar
    k = kt + kmean
    e4 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    grid = e4[np.isfinite(e4)]
    v = rng.choice(grid, size=(nkv, d0))
    v[0, :] = 448.0
    return q, k, v


@pytest.mark.parametrize("with_means", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_zero_rounding_error_reduces_to_exact(oracle_mod, with_means, causal):
    q, k, v = _zero_error_inputs(5, with_means=with_means)
    T = lambda a: torch.tensor(a)[:, None, :].half()
    args = (bits(T(q)), bits(T(k)), bits(T(v)), F16, [0, len(q)], [0, len(k)], 1, 1, 64, causal,
            _sm_scale_for_unit_c())
    emu = oracle_mod.attention_emulated(*args, bq=8, bkv=16, gk=32)
    ex = oracle_mod.attention_exact(*args)
    # only FP32 rounding of the partials (|R| ~ 1e5) remains: ~1e-7 of max|V| = 448
    np.testing.assert_allclose(emu, ex, rtol=2e-6, atol=448 * 1e-7)
    # and a broken smoothing would not: drop the Delta-S correction
    if with_means:
        bad = oracle_mod.attention_emulated(*args, bq=8, bkv=16, gk=32, smooth_q=False)
        assert not np.allclose(bad, ex, rtol=1e-3)


@pytest.mark.parametrize("causal", [False, True])
def test_int8_path_with_zero_rounding_error_reduces_to_exact(oracle_mod, causal):
    """The SageAttention (v1) switches (INT8 per-block Q and K codes, K smoothed, Q not):
    inputs on the INT8 grid with a 127 in every row (every scale 1) and a K channel mean
    pass through exactly; a quantizer still on the INT4 grid would not."""
    q, k, v = _zero_error_inputs(7, g=127, qmean=False)
    T = lambda a: torch.tensor(a)[:, None, :].half()
    args = (bits(T(q)), bits(T(k)), bits(T(v)), F16, [0, len(q)], [0, len(k)], 1, 1, 64, causal,
            _sm_scale_for_unit_c())
    emu = oracle_mod.attention_emulated(*args, bq=8, bkv=16, **oracle_mod.SAGE1)
    ex = oracle_mod.attention_exact(*args)
    np.testing.assert_allclose(emu, ex, rtol=2e-6, atol=448 * 1e-7)
    bad = oracle_mod.attention_emulated(*args, bq=8, bkv=16, per_block=True, smooth_q=False)
    assert not np.allclose(bad, ex, rtol=1e-3)


def test_int8_quantizer_invariants(oracle_mod):
    """INT8 grid: codes in [-127, 127], 127 reached in every non-zero group, rounding within
    half a step, scale = amax / 127; per-block Q blocks share one scale."""
    w = W.scaled(W.PREFILL, (300,), (300,), hq=2, hkv=2)
    x = W.make_inputs(w)
    km, _ = oracle_mod.kv_stats(bits(x["k"]), bits(x["v"]), BF16, x["cu_kv"], 2, 128)
    kc, sk = oracle_mod.quant_k(bits(x["k"]), BF16, x["cu_kv"], 2, 128, kmean=km, gk=128,
                                qk_bits=8)
    qm, qc, sq = oracle_mod.quant_q(bits(x["q"]), BF16, x["cu_q"], 2, 128, smooth_q=False,
                                    per_block=True, qk_bits=8)
    assert np.all(qm == 0)
    k64, q64 = x["k"].double().numpy(), x["q"].double().numpy()
    for h in range(2):
        kt = (k64[:, h].astype(np.float32) - km[0, h]).astype(np.float32)
        for t0 in range(0, 300, 128):
            grp = slice(t0, min(300, t0 + 128))
            assert len(set(sk[grp, h].tolist())) == 1
            s = sk[grp, h][0]
            assert s == np.float32(np.abs(kt[grp]).max() / np.float32(127))
            c = kc[grp, h]
            assert c.min() >= -127 and c.max() <= 127 and np.abs(c).max() == 127
            assert np.abs(kt[grp] - c * float(s)).max() <= 0.5 * float(s) * (1 + 1e-5)
            qb = q64[grp, h].astype(np.float32)
            assert len(set(sq[grp, h].tolist())) == 1
            assert np.abs(qc[grp, h]).max() == 127
            assert np.abs(qb - qc[grp, h] * float(sq[grp, h][0])).max() <= 0.5 * float(sq[grp, h][0]) * (1 + 1e-5)


def test_k_channel_shift_leaves_softmax_rows_unchanged(oracle_mod):
    """Adding the same vector c to every key of a (sequence, kv head) adds q . c to every logit
    of a row, which softmax ignores: exact attention is unchanged up to FP64 rounding. With K
    smoothing the quantized pipeline subtracts the shifted mean again, so on inputs whose means
    are exact (keys in +-pairs) and an exactly representable shift its output is bit-identical;
    without K smoothing the shift reaches the INT4 codes and changes it."""
    q, k, v = _zero_error_inputs(11, with_means=False)
    shift = np.zeros(k.shape[1])
    shift[[3, 17, 62]] = [4.0, 2.5, 16.0]  # channel 62 is one Q uses (its 7s); 16 > every |K~|
    assert np.abs(q[:, 62]).min() > 0
    T = lambda a: torch.tensor(a)[:, None, :].half()
    for causal in (False, True):
        base = (bits(T(q)), bits(T(k)), bits(T(v)), F16, [0, len(q)], [0, len(k)], 1, 1, 64, causal)
        moved = (bits(T(q)), bits(T(k + shift)), bits(T(v)), F16, [0, len(q)], [0, len(k)], 1, 1,
                 64, causal)
        np.testing.assert_allclose(oracle_mod.attention_exact(*moved),
                                   oracle_mod.attention_exact(*base), rtol=1e-12, atol=1e-9)
        np.testing.assert_array_equal(oracle_mod.attention_emulated(*moved, bq=8, bkv=16),
                                      oracle_mod.attention_emulated(*base, bq=8, bkv=16))
        a = oracle_mod.attention_emulated(*moved, bq=8, bkv=16, smooth_k=False)
        b = oracle_mod.attention_emulated(*base, bq=8, bkv=16, smooth_k=False)
        assert not np.array_equal(a, b)


ABLATION_FLAGS = [dict(), dict(smooth_q=False), dict(smooth_k=False), dict(per_block=True),
                  dict(smooth_q=False, smooth_k=False, per_block=True),
                  dict(qk_bits=8, per_block=True, smooth_q=False), dict(qk_bits=8)]


@pytest.mark.parametrize("flags", ABLATION_FLAGS,
                         ids=["method", "noQs", "noKs", "block", "naive", "sage1", "int8thread"])
@pytest.mark.parametrize("case", [
    dict(nq=(5,), nkv=(7,), hq=2, hkv=1, d0=4, causal=False, dtype="fp16", dist="tiny"),
    dict(nq=(6, 3), nkv=(4, 8), hq=2, hkv=2, d0=8, causal=True, dtype="bf16", dist="outlier"),
    dict(nq=(8,), nkv=(5,), hq=1, hkv=1, d0=8, causal=True, dtype="bf16", dist="dit"),
])
def test_brute_force_tiny_vs_restatement(oracle_mod, case, flags):
    w = W.Workload("bf", case["nq"], case["nkv"], case["hq"], case["hkv"], case["d0"],
                   case["dtype"], case["causal"], case["dist"], 21, varlen=True)
    x = W.make_inputs(w)
    dt = W.dtype_code(w)
    got = oracle_mod.attention_emulated(bits(x["q"]), bits(x["k"]), bits(x["v"]), dt, x["cu_q"],
                                        x["cu_kv"], w.hq, w.hkv, w.d, w.causal, bq=4, bkv=4, gk=2,
                                        **flags)
    ref = NR.mode_q(x["q"].double().numpy(), x["k"].double().numpy(), x["v"].double().numpy(),
                    x["cu_q"], x["cu_kv"], w.hq, w.hkv, w.d, w.causal, bq=4, bkv=4, gk=2, **flags)
    np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-9)


def test_quant_q_per_block_invariants(oracle_mod):
    """Per-block Q granularity: every valid row of a block carries the block's one scale,
    which is the largest of the block's per-row scales (so some row reaches code +-7 and no
    row's scale exceeds it); rounding stays within half a step; padding channels stay 0."""
    w = W.scaled(W.PREFILL, (300,), (300,), hq=2, hkv=2)
    x = W.make_inputs(w)
    qm, qc_row, sq_row = oracle_mod.quant_q(bits(x["q"]), BF16, x["cu_q"], 2, 128)
    qm_b, qc_blk, sq_blk = oracle_mod.quant_q(bits(x["q"]), BF16, x["cu_q"], 2, 128,
                                              per_block=True)
    np.testing.assert_array_equal(qm, qm_b)            # the smoothing does not depend on it
    q64 = x["q"].double().numpy()
    for h in range(2):
        for qb in range(3):
            rows = slice(qb * 128, min(300, qb * 128 + 128))
            s_blk = sq_blk[rows, h]
            assert len(set(s_blk.tolist())) == 1
            assert s_blk[0] == sq_row[rows, h].max()
            xt = (q64[rows, h].astype(np.float32) - qm[0, h, qb]).astype(np.float32)
            _check_codes(xt, qc_blk[rows, h], s_blk[0])
            # a row holding the block maximum gets the same codes either way
            r_top = int(np.argmax(sq_row[rows, h]))
            np.testing.assert_array_equal(qc_blk[rows, h][r_top], qc_row[rows, h][r_top])


def test_per_block_of_one_row_is_per_row(oracle_mod):
    """With one query row per block and one KV tile per K group, per-block granularity is
    the per-row / per-group granularity: both runs must agree bit for bit."""
    w = W.scaled(W.PREFILL, (40,), (70,), hq=2, hkv=1)
    x = W.make_inputs(w)
    a = _emu(oracle_mod, w, x, bq=1, bkv=32, gk=32, smooth_q=False)
    b = _emu(oracle_mod, w, x, bq=1, bkv=32, smooth_q=False, per_block=True)
    np.testing.assert_array_equal(a, b)
    c = _emu(oracle_mod, w, x, bkv=32, per_block=True)   # 128-row Q blocks: differs
    assert not np.array_equal(a, c)


@pytest.mark.parametrize("nkv", [100, 200])
def test_tiling_one_and_two_kv_tiles_vs_restatement(oracle_mod, nkv):
    """One KV tile reduces to the direct formula; two tiles to the hand expansion of the
    online softmax (the restatement runs the same tile boundaries)."""
    w = W.Workload("t", (6,), (nkv,), 1, 1, 64, "fp16", False, "tiny", 8, varlen=True)
    x = W.make_inputs(w)
    got = oracle_mod.attention_emulated(bits(x["q"]), bits(x["k"]), bits(x["v"]), F16, x["cu_q"],
                                        x["cu_kv"], 1, 1, 64, False)
    ref = NR.mode_q(x["q"].double().numpy(), x["k"].double().numpy(), x["v"].double().numpy(),
                    x["cu_q"], x["cu_kv"], 1, 1, 64, False)
    np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-9)


def test_tile_p448_dump_rebuilds_the_output(oracle_mod):
    """The P448 test hook: with one KV tile (Nkv <= 128) a row's output is the e4m3 codes of
    its dumped P448 times the V codes, times the V scales, over the sum of the unquantized
    P448; the row maximum is 448 (x = log2 448 at the maximal key); invisible keys stay 0."""
    w = W.Workload("dump", (90,), (100,), 2, 1, 64, "fp16", True, "tiny", 5, varlen=True)
    x = W.make_inputs(w)
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), F16, x["cu_q"], x["cu_kv"], 2, 1, 64, True)
    out = oracle_mod.attention_emulated(*args)
    p = oracle_mod.emulated_tile_p448(*args, b=0, h=1, qb=0, kt=0).astype(np.float64)
    _, vamax = oracle_mod.kv_stats(bits(x["k"]), bits(x["v"]), F16, x["cu_kv"], 1, 64)
    vc, sv = oracle_mod.quant_v(bits(x["v"]), F16, x["cu_kv"], 1, 64, vamax)
    vval = oracle_mod.e4m3_decode(vc)[:, 0]                        # [100][64]
    pt = oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(p[:90, :100]))
    for i in range(90):
        vis = i + 10                                               # bottom-right causal
        assert np.all(p[i, vis + 1:] == 0) and np.all(p[i, :vis + 1] > 0)
        assert abs(p[i].max() - 448.0) <= 448.0 * 2.0 ** -20
        want = (pt[i] @ vval) * sv[0, 0] / p[i].sum()
        np.testing.assert_allclose(out[i, 1], want, rtol=1e-6, atol=1e-9)


# ----------------------------------------------------------------- accuracy (ablations)
@pytest.fixture(scope="module")
def outlier_case():
    w = W.scaled(W.PREFILL, (600,), (600,), hq=4, hkv=4)
    x = W.make_inputs(w)
    return w, x


def _emu(oracle_mod, w, x, **kw):
    return oracle_mod.attention_emulated(bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w),
                                         x["cu_q"], x["cu_kv"], w.hq, w.hkv, w.d, w.causal, **kw)


def test_smoothing_ablations_are_directional(oracle_mod, outlier_case):
    """Smoothing K and smoothing Q each reduce the error against exact attention on
    outlier-channel data (the pages' qualitative accuracy claims)."""
    w, x = outlier_case
    ex = oracle_mod.attention_exact(bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w),
                                    x["cu_q"], x["cu_kv"], w.hq, w.hkv, w.d, w.causal)
    e_full = relL1(_emu(oracle_mod, w, x), ex)
    e_noq = relL1(_emu(oracle_mod, w, x, smooth_q=False), ex)
    e_nok = relL1(_emu(oracle_mod, w, x, smooth_k=False), ex)
    e_none = relL1(_emu(oracle_mod, w, x, smooth_q=False, smooth_k=False), ex)
    assert e_full < 0.2
    assert e_noq > 1.5 * e_full and e_nok > 1.5 * e_full and e_none > e_noq


def test_per_thread_granularity_beats_per_block(oracle_mod, outlier_case):
    """Per-thread INT4 scales err less than one scale per block, with or without smoothing;
    the naive scheme (per-block, no smoothing) errs most (the pages' granularity claim)."""
    w, x = outlier_case
    ex = oracle_mod.attention_exact(bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w),
                                    x["cu_q"], x["cu_kv"], w.hq, w.hkv, w.d, w.causal)
    e_thread = relL1(_emu(oracle_mod, w, x), ex)
    e_block = relL1(_emu(oracle_mod, w, x, per_block=True), ex)
    e_naive = relL1(_emu(oracle_mod, w, x, per_block=True, smooth_q=False, smooth_k=False), ex)
    assert e_block > 1.2 * e_thread
    assert e_naive > e_block


def test_int8_path_errs_less_than_int4(oracle_mod, outlier_case):
    """The INT8 grid is 18 times finer than the INT4 one: the SageAttention (v1) path (INT8
    per-block, K smoothed) errs less against exact attention than the method's INT4 path,
    which pays for its 4-bit matrix multiply with the repairs (the pages' trade-off)."""
    w, x = outlier_case
    ex = oracle_mod.attention_exact(bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w),
                                    x["cu_q"], x["cu_kv"], w.hq, w.hkv, w.d, w.causal)
    e_v2 = relL1(_emu(oracle_mod, w, x), ex)
    e_v1 = relL1(_emu(oracle_mod, w, x, **oracle_mod.SAGE1), ex)
    e_v1_int4 = relL1(_emu(oracle_mod, w, x, per_block=True, smooth_q=False), ex)
    assert e_v1 < e_v2 < e_v1_int4


def test_two_level_accumulation_beats_one_level(oracle_mod, outlier_case):
    """Against the same pipeline with an exact accumulator, a reduced-precision
    one-level accumulator errs far more than the two-level FP32 fold."""
    w, x = outlier_case
    exact_acc = _emu(oracle_mod, w, x, acc_bits=60)
    two_level = _emu(oracle_mod, w, x)
    one_level = _emu(oracle_mod, w, x, acc_bits=13)
    e2 = relL1(two_level, exact_acc)
    e1 = relL1(one_level, exact_acc)
    assert e2 < 1e-6
    assert e1 > 10 * e2


def test_mode_q_accuracy_vs_exact_matches_noise_model(oracle_mod):
    """INT4 codes with amax/7 scales leave quantization noise of about 0.1 sigma per
    element; on Gaussian data that is roughly 0.15 of the logit spread, and the output
    error against exact attention follows. The oracle must sit in that band."""
    w = W.TINY
    x = W.make_inputs(w)
    ex = oracle_mod.attention_exact(bits(x["q"]), bits(x["k"]), bits(x["v"]), F16, x["cu_q"],
                                    x["cu_kv"], 2, 2, 64, False)
    emu = _emu(oracle_mod, w, x)
    assert 0.97 < cosine(emu, ex) < 0.999
    assert 0.05 < relL1(emu, ex) < 0.3


# ------------------------------------------------------------------ accuracy against exact attention
# The method's error against exact FP64 attention on the five workloads' distributions (scaled so
# the oracle's two modes finish in seconds), at the K grouping the kernels use (one scale per 32
# keys). These are regression bands of the oracle's own numbers: the INT4 method does not meet
# relative L1 <= 0.06 on these Gaussian inputs at any K grouping (see the next test), while the
# INT8 (v1) path does.
FP64_CASES = {
    "tiny": W.TINY,
    "prefill": W.scaled(W.PREFILL, (1024, 700), (1024, 700), hq=4, hkv=4, name="prefill_s"),
    "gqa": W.scaled(W.GQA_LONG, (2048,), (2048,), hq=8, hkv=2, name="gqa_s"),
    "dit": W.scaled(W.VIDEO_DIT, (1200, 333), (1200, 333), hq=3, hkv=3, name="dit_s"),
    "varlen": W.scaled(W.VARLEN, (300, 77, 129), (500, 129, 1000), hq=8, hkv=2, name="varlen_s"),
}
FP64_BANDS_GK32 = {  # (relative L1, cosine) of Mode Q against Mode E
    "tiny": (0.1844, 0.98223), "prefill": (0.1483, 0.98878), "gqa": (0.1549, 0.98814),
    "dit": (0.1970, 0.97975), "varlen": (0.1957, 0.98101),
}


def _modes(oracle_mod, w, **kw):
    x = W.make_inputs(w)
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)
    return oracle_mod.attention_emulated(*args, **kw), oracle_mod.attention_exact(*args), args


@pytest.mark.parametrize("name", list(FP64_CASES))
def test_method_accuracy_against_exact_attention_bands(oracle_mod, name):
    emu, ex, args = _modes(oracle_mod, FP64_CASES[name])
    r, c = FP64_BANDS_GK32[name]
    assert abs(relL1(emu, ex) - r) <= 0.02 * r, (name, relL1(emu, ex))
    assert abs(cosine(emu, ex) - c) <= 0.002, (name, cosine(emu, ex))
    # the INT8 (v1) path on the same inputs meets cosine >= 0.99 and relative L1 <= 0.06
    v1 = oracle_mod.attention_emulated(*args, **oracle_mod.SAGE1)
    assert relL1(v1, ex) <= 0.06 and cosine(v1, ex) >= 0.99


@pytest.mark.parametrize("name", ["prefill", "varlen"])
def test_finer_k_groups_help_but_do_not_reach_relative_l1_006(oracle_mod, name):
    """A finer K grouping lowers the error monotonically, but even one scale per key leaves the
    INT4 method far above relative L1 0.06 against exact attention."""
    w = FP64_CASES[name]
    x = W.make_inputs(w)
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)
    ex = oracle_mod.attention_exact(*args)
    errs = [relL1(oracle_mod.attention_emulated(*args, gk=gk), ex) for gk in (1, 8, 32, 128)]
    assert all(a < b for a, b in zip(errs, errs[1:])), errs
    assert errs[0] > 0.1, errs
