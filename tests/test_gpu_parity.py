"""GPU parity: the CUDA path against the CPU oracle, through the C ABI.

Gates (per the method's emulation, the oracle's Mode Q):
  * prepass results (means, INT4 codes and scales, e4m3 V codes) bit-exact; DeltaS*c within
    128 units of 2^-24 of c * sum |qmean K~| (plus 2 ulp) of the oracle's FP64 dot product;
  * the raw integer Q K^T accumulators of the tensor-core MMA bit-exact;
  * the output (FP32) within relative L1 1e-3 and max abs 2e-3;
  * fp16/bf16 outputs within one unit in the last place of the oracle's rounded output.
Against exact FP64 attention (Mode E) the GPU must be as accurate as the emulation itself.
"""
from __future__ import annotations


import numpy as np
import pytest
import torch

import oracle
import bit_exact_attention_gb300 as S
from bit_exact_attention_gb300 import workloads as W
from parity_util import (GpuCase, bits, c32_of, check_dsc, check_forward_proven, ds_abs_sum,
                         e4m3_to_f64, kv_tiles, metrics, pad_starts, unit_rows, units_sample)

pytestmark = pytest.mark.gpu

REL_L1, MAX_ABS = 1e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    major, minor = torch.cuda.get_device_capability()
    assert (major, minor) == (10, 3), f"expected an sm_103 GPU, got sm_{major}{minor}"
    oracle.build()
    S.load_library()


# Scaled workloads: the oracle finishes each in seconds; each spans several tiles and a
# ragged tail.
SCALED = {
    "tiny": W.TINY,
    "prefill": W.scaled(W.PREFILL, (700, 300), (700, 300), hq=4, hkv=4, name="prefill_s"),
    "gqa": W.scaled(W.GQA_LONG, (1000,), (1000,), hq=8, hkv=2, name="gqa_s"),
    "dit": W.scaled(W.VIDEO_DIT, (600, 333), (600, 333), hq=3, hkv=3, name="dit_s"),
    "varlen": W.scaled(W.VARLEN, (300, 77, 129), (500, 129, 1000), hq=8, hkv=2, name="varlen_s"),
}


def oracle_ref(w, x, units=None, mode="emu", **kw):
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)
    if mode == "emu":
        return oracle.attention_emulated(*args, units=units, **kw)
    return oracle.attention_exact(*args, units=units)


_cache = {}


def run_case(name):
    if name not in _cache:
        w = SCALED[name]
        x = W.make_inputs(w)
        g = GpuCase(w, x)
        _cache[name] = (w, x, g)
    return _cache[name]


# ------------------------------------------------------------------ prepass
def test_prepass_orders_varlen_sequences_longest_kv_first():
    """The prepass leaves, after the status and format words, the order in which the two-tile
    kernel takes the sequences of a varlen call: a permutation by decreasing K/V length, ties by
    index (the kernel then starts its longest CTAs first)."""
    w = W.scaled(W.VARLEN, (300, 77, 129, 5, 0), (500, 129, 1000, 129, 64), name="order_s")
    x = W.make_inputs(w)
    g = GpuCase(w, x)
    g.prepass()
    torch.cuda.synchronize()
    order = g._buf(g.L.status + 4 * 64, w.batch, torch.int32).cpu().numpy().tolist()
    want = sorted(range(w.batch), key=lambda b: (-w.nkv[b], b))
    assert order == want, (order, want)


@pytest.mark.parametrize("name", list(SCALED))
def test_prepass_codes_bit_exact_delta_s_bounded(name):
    w, x, g = run_case(name)
    g.prepass()
    assert g.status() == (0, 0)
    got = g.gathered()
    dt = W.dtype_code(w)
    kmean, vamax = oracle.kv_stats(bits(x["k"]), bits(x["v"]), dt, x["cu_kv"], w.hkv, w.d)
    qmean, qc, sq = oracle.quant_q(bits(x["q"]), dt, x["cu_q"], w.hq, w.d)
    kc, sk = oracle.quant_k(bits(x["k"]), dt, x["cu_kv"], w.hkv, w.d, kmean=kmean)
    vc, sv = oracle.quant_v(bits(x["v"]), dt, x["cu_kv"], w.hkv, w.d, vamax)
    np.testing.assert_array_equal(got["kmean"], kmean)
    np.testing.assert_array_equal(got["vscale"], sv)
    assert int((got["qcode"] != qc).sum()) == 0, "Q code mismatches"
    np.testing.assert_array_equal(got["qscale"], sq)
    assert int((got["kcode"] != kc).sum()) == 0, "K code mismatches"
    np.testing.assert_array_equal(got["kscale"], sk)
    np.testing.assert_array_equal(got["vcode"], oracle.e4m3_decode(vc))
    # Q block means and DeltaS * c for every (q head, Q block, visited KV tile)
    qp, kp = pad_starts(x["cu_q"]), pad_starts(x["cu_kv"])
    c32 = c32_of(w)
    worst = 0.0
    for b in range(w.batch):
        nqb = (w.nq[b] + 127) // 128
        for h in range(w.hq):
            for qb in range(nqb):
                blk = qp[b] // 128 + qb
                np.testing.assert_array_equal(got["qmean"][h, blk], qmean[b, h, qb])
                hk = h // (w.hq // w.hkv)
                ds = oracle.delta_s(bits(x["k"]), dt, x["cu_kv"], b, w.hkv, hk, w.d, kmean,
                                    qmean[b, h, qb])
                ntiles = kv_tiles(qb, w.nq[b], w.nkv[b], w.causal)
                n = min(w.nkv[b], ntiles * 128)
                absum = ds_abs_sum(x, w, b, hk, kmean, qmean[b, h, qb])
                worst = max(worst, check_dsc(got["dsc"][h, blk, :n], ds[:n], absum[:n], c32))
    print(f"{name}: largest DeltaS*c deviation {worst:.3f} of its bound")


# ------------------------------------------------------------------ integer accumulators
@pytest.mark.parametrize("kernel", ["two_tile", "one_tile"])
@pytest.mark.parametrize("name", ["tiny", "prefill", "dit", "varlen"])
def test_qk_accumulators_bit_exact_and_pv_partial(name, kernel, monkeypatch):
    """S of the tensor-core Q K^T equals the integer product of the oracle's codes exactly, on
    both kernels; the fresh P~V partial matches P~ V in FP64 (the two-tile kernel exposes it
    for the first KV tile only, where the output accumulator starts from it)."""
    if kernel == "one_tile":
        monkeypatch.setenv("SAGE2_ATTN_PP", "0")
    w, x, g = run_case(name)
    g.prepass()
    dt = W.dtype_code(w)
    kmean, vamax = oracle.kv_stats(bits(x["k"]), bits(x["v"]), dt, x["cu_kv"], w.hkv, w.d)
    _, qc, _ = oracle.quant_q(bits(x["q"]), dt, x["cu_q"], w.hq, w.d)
    kc, _ = oracle.quant_k(bits(x["k"]), dt, x["cu_kv"], w.hkv, w.d, kmean=kmean)
    vc, _ = oracle.quant_v(bits(x["v"]), dt, x["cu_kv"], w.hkv, w.d, vamax)
    vval = oracle.e4m3_decode(vc)
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
                s_out, p_out, r_out = g.debug_tile(b, h, qt, kt)
                A = np.zeros((128, Dp), np.int64)
                rows = np.arange(qt * 128, min(w.nq[b], qt * 128 + 128))
                A[: len(rows)] = qc[x["cu_q"][b] + rows, h]
                Kt = np.zeros((128, Dp), np.int64)
                keys = np.arange(kt * 128, min(w.nkv[b], kt * 128 + 128))
                hk = h // (w.hq // w.hkv)
                Kt[: len(keys)] = kc[x["cu_kv"][b] + keys, hk]
                want = A @ Kt.T
                got = s_out.cpu().numpy()
                assert np.array_equal(got, want.astype(np.float64)), (
                    f"{name} b{b} h{h} qt{qt} kt{kt}: {(got != want).sum()} accumulator mismatches")
                checked += 1
                if kernel == "two_tile" and kt > 0:
                    continue
                # the fresh P~V partial: P~ bytes as dumped, V codes from the oracle, FP64
                Vt = np.zeros((128, Dp))
                Vt[: len(keys)] = vval[x["cu_kv"][b] + keys, hk]
                R_ref = e4m3_to_f64(p_out) @ Vt
                R = r_out.cpu().numpy()
                np.testing.assert_allclose(R, R_ref, rtol=1e-5, atol=1e-3 * np.abs(R_ref).max())
    assert checked >= 2


# ------------------------------------------------------------------ outputs
@pytest.mark.parametrize("name", list(SCALED))
def test_forward_matches_emulation_fp32(name):
    w, x, g = run_case(name)
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    emu = oracle_ref(w, x)
    check_forward_proven(g, w, x, out, emu)
    ex = oracle_ref(w, x, mode="exact")
    mg, mq = metrics(out, ex), metrics(emu, ex)
    # the GPU is exactly as accurate as the method it implements
    assert abs(mg["relL1"] - mq["relL1"]) <= 2e-3 * max(1.0, mq["relL1"] * 10), (mg, mq)
    assert abs(mg["cos"] - mq["cos"]) <= 1e-4, (mg, mq)


@pytest.mark.parametrize("name", list(SCALED))
def test_one_tile_kernel_matches_emulation(name, monkeypatch):
    """The method's codes on the one-tile kernel (fresh FP32 partial per key tile, FP32 fold in
    registers), which SAGE2_ATTN_PP=0 selects, hold the same gate as the default two-tile kernel
    (FP32 rescale, then the P~V MMA accumulating into O). Both compute the same P~ codes and row
    sums, so the outputs differ only by where the accumulation rounds: at FP32 level (measured
    2^-20.9 of max|O| at worst on these cases). An accumulator with a 13-bit significand, the
    flaw the two-level scheme repairs, would put the difference near 2^-13."""
    w, x, g = run_case(name)
    default = g.forward(out_dtype=torch.float32).cpu().numpy()
    monkeypatch.setenv("SAGE2_ATTN_PP", "0")
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    check_forward_proven(g, w, x, out, oracle_ref(w, x))
    m2 = metrics(default, out)
    scale = float(np.abs(out).max()) if out.size else 0.0
    assert m2["relL1"] <= 1e-6 and m2["maxabs"] <= 2.0 ** -18 * max(scale, 1e-30), m2


@pytest.mark.parametrize("name", ["tiny", "prefill", "varlen"])
def test_forward_low_precision_output(name):
    w, x, g = run_case(name)
    out = g.forward()
    assert out.dtype == x["q"].dtype
    got = out.float().cpu().numpy().astype(np.float64)
    emu = oracle_ref(w, x)
    want_bits = oracle.round_output(emu, W.dtype_code(w))
    want = torch.from_numpy(want_bits.view(np.int16)).view(x["q"].dtype).double().numpy()
    # The FP32 result may sit up to MAX_ABS from the emulation; rounding both to the
    # output dtype adds at most one unit in the last place of the larger of the two. Rows beyond
    # that must be explained by located P~ midpoint flips (check_forward_proven).
    mant = 7 if w.dtype == "bf16" else 10
    mag = np.maximum(np.abs(want), np.abs(got))
    ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 1e-30))) - mant)
    check_forward_proven(g, w, x, got, want, tol=MAX_ABS + ulp)


def test_dense_entry_point_equals_varlen():
    w, x, g = run_case("prefill")
    # prefill_s has two sequences of different length: use a uniform one for the dense call
    w2 = W.scaled(W.PREFILL, (384, 384), (384, 384), hq=4, hkv=2, name="dense_eq")
    x2 = W.make_inputs(w2)
    g2 = GpuCase(w2, x2)
    a = g2.forward(out_dtype=torch.float32)
    q = x2["q"].view(2, 384, 4, 128).cuda()
    k = x2["k"].view(2, 384, 2, 128).cuda()
    v = x2["v"].view(2, 384, 2, 128).cuda()
    b = S.attn_fwd(q, k, v, causal=True, out_dtype=torch.float32)
    assert torch.equal(a.view(2, 384, 4, 128), b)


def test_repeatable_bit_identical():
    w, x, g = run_case("varlen")
    a = g.forward(out_dtype=torch.float32)
    b = g.forward(out_dtype=torch.float32)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ edge cases
EDGE = [
    # (nq, nkv, hq, hkv, d, causal, dtype)
    ((1,), (1,), 1, 1, 64, False, "fp16"),
    ((1,), (1000,), 2, 1, 128, True, "bf16"),      # one query sees every key (bottom-right)
    ((300,), (100,), 2, 2, 128, True, "bf16"),     # rows with no visible key output 0
    ((100,), (300,), 2, 2, 64, True, "fp16"),
    ((129, 0, 5), (0, 64, 257), 4, 2, 128, False, "bf16"),  # empty sequences
    ((200,), (200,), 8, 1, 32, True, "bf16"),      # D0 = 32, GQA 8
    ((200,), (333,), 2, 2, 80, False, "fp16"),     # D0 = 80
    ((150,), (150,), 2, 2, 96, True, "bf16"),
    ((130,), (260,), 2, 2, 112, False, "bf16"),
]


@pytest.mark.parametrize("kernel", ["two_tile", "one_tile"])
@pytest.mark.parametrize("case", EDGE, ids=[f"e{i}" for i in range(len(EDGE))])
def test_edge_cases(case, kernel, monkeypatch):
    if kernel == "one_tile":
        monkeypatch.setenv("SAGE2_ATTN_PP", "0")
    nq, nkv, hq, hkv, d, causal, dt = case
    w = W.Workload("edge", nq, nkv, hq, hkv, d, dt, causal, "kbias9", 31, varlen=True)
    x = W.make_inputs(w)
    g = GpuCase(w, x)
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    emu = oracle_ref(w, x)
    if np.abs(emu).sum() == 0:
        assert np.all(out == 0)
    else:
        check_forward_proven(g, w, x, out, emu)
    # rows with no visible key are exactly zero
    for b in range(w.batch):
        for i in range(w.nq[b]):
            if w.nkv[b] == 0 or (causal and i + w.nkv[b] - w.nq[b] < 0):
                assert np.all(out[x["cu_q"][b] + i] == 0)


@pytest.mark.parametrize("kernel", ["two_tile", "one_tile"])
@pytest.mark.parametrize("nb", [40, 300])
def test_many_short_sequences(nb, kernel, monkeypatch):
    """Many short varlen sequences of mixed lengths (empty ones included): 40 are taken in the
    prepass's longest-K/V-first order, 300 exceed the sort limit and keep the batch order; both
    must match the oracle element by element."""
    if kernel == "one_tile":
        monkeypatch.setenv("SAGE2_ATTN_PP", "0")
    rng = np.random.default_rng(1000 + nb)
    nq = tuple(int(v) for v in rng.integers(0, 300, nb))
    nkv = tuple(int(v) for v in rng.integers(0, 400, nb))
    w = W.Workload(f"many_{nb}", nq, nkv, 4, 2, 64, "bf16", bool(nb == 40), "kbias9", 37,
                   varlen=True)
    x = W.make_inputs(w)
    g = GpuCase(w, x)
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    check_forward_proven(g, w, x, out, oracle_ref(w, x))


def _random_shapes(n, seed):
    """Seeded ragged problems: 1-3 sequences (empty ones included, the first never empty),
    GQA ratios 1-4, head dims padded to 64 or 128, causal or not."""
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(n):
        nb = int(rng.integers(1, 4))
        nq = tuple(int(rng.integers(0 if b else 1, 900)) for b in range(nb))
        nkv = tuple(int(rng.integers(0 if b else 1, 1500)) for b in range(nb))
        hkv = int(rng.choice([1, 2, 4]))
        hq = hkv * int(rng.choice([1, 2, 4]))
        d = int(rng.choice([40, 64, 96, 128]))
        shapes.append((nq, nkv, hq, hkv, d, bool(rng.integers(0, 2)),
                       "bf16" if rng.integers(0, 2) else "fp16"))
    return shapes


RANDOM_SHAPES = _random_shapes(16, 2024)


@pytest.mark.parametrize("i", range(len(RANDOM_SHAPES)))
def test_two_tile_kernel_agrees_with_one_tile_on_random_shapes(i, monkeypatch):
    """Ragged pairings (a second tile that is empty or sees fewer key tiles, pairs past the end of
    a sequence, sequences with no keys) on the two-tile kernel, against the one-tile kernel: both
    quantize identically, so the outputs agree to FP32 accumulation level and masked rows are 0
    on both."""
    nq, nkv, hq, hkv, d, causal, dt = RANDOM_SHAPES[i]
    w = W.Workload("rand", nq, nkv, hq, hkv, d, dt, causal, "kbias9", 100 + i, varlen=True)
    x = W.make_inputs(w)
    g = GpuCase(w, x)
    a = g.forward(out_dtype=torch.float32).double().cpu().numpy()
    assert g.status() == (0, 0)
    monkeypatch.setenv("SAGE2_ATTN_PP", "0")
    b = g.forward(out_dtype=torch.float32).double().cpu().numpy()
    assert g.status() == (0, 0)
    assert np.all(np.isfinite(a))
    scale = float(np.abs(b).max()) if b.size else 0.0
    assert np.abs(a - b).max(initial=0.0) <= 2.0 ** -18 * max(scale, 1e-30), (
        RANDOM_SHAPES[i], float(np.abs(a - b).max(initial=0.0)), scale)


def test_sm_scale_argument():
    w = W.scaled(W.TINY, (200,), (300,), hq=2, hkv=2)
    x = W.make_inputs(w)
    g = GpuCase(w, x, sm_scale=0.05)
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    emu = oracle.attention_emulated(bits(x["q"]), bits(x["k"]), bits(x["v"]), 0, x["cu_q"],
                                    x["cu_kv"], 2, 2, 64, False, 0.05)
    check_forward_proven(g, w, x, out, emu)


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("wl", [W.PREFILL, W.GQA_LONG, W.VIDEO_DIT, W.VARLEN],
                         ids=["prefill", "gqa_long", "video_dit", "varlen"])
def test_full_size_sampled_units(wl):
    """Full-size workloads, launched as the benchmark launches them; the oracle computes
    >= 32 seeded (sequence, head, Q block) units including every last partial block, the
    first block and a causal-diagonal block."""
    x = W.make_inputs(wl)
    g = GpuCase(wl, x)
    out = g.forward(out_dtype=torch.float32)
    assert g.status() == (0, 0)
    units = units_sample(wl, 32, seed=wl.seed)
    emu = oracle_ref(wl, x, units=units)
    toks, heads = unit_rows(wl, x["cu_q"], units)
    check_forward_proven(g, wl, x, out.cpu().numpy(), emu, rows=(toks, heads))


@pytest.mark.parametrize("wl", [W.PREFILL, W.VARLEN], ids=["prefill", "varlen"])
def test_full_size_full_output(wl):
    """The LLM prefill and varlen workloads at full size, every output element against the
    oracle's emulation (the oracle runs the whole workload on the host cores): relative L1 within
    1e-3 and every element within 2e-3, except rows that are proven to differ only through P~
    codes the hardware exponential rounded to the other side of an e4m3 midpoint. For each such
    row the GPU's own P~ codes of every KV tile are dumped, the row is recomputed from them in
    NumPy with the oracle's logits, V codes and scales, and the recomputation must match the GPU
    row within 2e-3 while every code that differs from the emulation's is one e4m3 step off with
    its exact 448 P within 4 ulp of the midpoint between the two codes."""
    x = W.make_inputs(wl)
    g = GpuCase(wl, x)
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    emu = oracle_ref(wl, x)
    proven = check_forward_proven(g, wl, x, out, emu, max_rows=64)
    m = metrics(out, emu)
    print(f"{wl.name}: relL1 {m['relL1']:.3g}, max abs {m['maxabs']:.3g}; rows above {MAX_ABS}: "
          f"{proven}, each explained by located midpoint flips")


def test_direct_accumulation_matches_the_literal_fold_along_the_sequence(monkeypatch):
    """The default kernel lets the P~V MMA add each block into the FP32 output accumulator after
    an FP32 rescale; the one-tile kernel sums the block into a fresh FP32 partial and folds it,
    O = fl32(alpha O + R). Both see the same P~ codes and row sums, so their outputs differ only
    by FP32 accumulation rounding. A row that visits T key tiles takes at most T rescales and T
    block sums: each rescale or fold rounds once (u = 2^-24 of |O|, |O| <= max|V| in output
    units), and each block sum of the tensor core is gated at 2^-19 of the sum of |products|
    (test_pv_tile_accumulator_is_fp32_class), whose share over the row sums to about 1.1 max|V|;
    with the 32-product steps of the direct form that bounds the difference by
    (6 T + 80) u max|V|. Checked on every row of the long GQA workload at four lengths, with the
    largest difference reported against max|O| to show its growth."""
    growth = []
    for n in (1024, 4096, 16384, 32768):
        w = W.scaled(W.GQA_LONG, (n,), (n,), name=f"gqa_long_n{n}")
        x = W.make_inputs(w)
        g = GpuCase(w, x)
        monkeypatch.delenv("SAGE2_ATTN_PP", raising=False)
        a = g.forward(out_dtype=torch.float32)
        assert g.status() == (0, 0)
        monkeypatch.setenv("SAGE2_ATTN_PP", "0")
        b = g.forward(out_dtype=torch.float32)
        assert g.status() == (0, 0)
        monkeypatch.delenv("SAGE2_ATTN_PP", raising=False)
        diff = (a - b).abs().amax(dim=2).double().cpu().numpy()  # [token, head]
        i = np.arange(n)
        T = i // 128 + 1  # causal with Nq = Nkv: row i visits the key tiles up to its own
        vmax = float(x["v"].abs().max())
        bound = (6.0 * T + 80.0) * 2.0 ** -24 * vmax
        ratio = diff / bound[:, None]
        assert ratio.max() <= 1.0, (n, float(ratio.max()))
        omax = float(b.abs().max())
        growth.append((n, float(diff.max()), float(diff.max()) / omax, float(ratio.max())))
        del g, a, b
        torch.cuda.empty_cache()
    for n, dmax, rel, r in growth:
        print(f"N {n}: max |direct - literal| {dmax:.3g} = 2^{np.log2(max(rel, 1e-30)):.1f} of "
              f"max|O|, {r:.3f} of the bound")
    # FP32-level at every length: far below what a 13-bit accumulator would leave (2^-13)
    assert all(rel < 2.0 ** -14 for _, _, rel, _ in growth), growth


# ------------------------------------------------------------------ failure detection
def test_bounded_wait_reports_timeout_and_context_survives():
    w = W.TINY
    x = W.make_inputs(w)
    g = GpuCase(w, x)
    g.prepass()
    S.debug_timeout(g.ws, 1, 2, 2, 256, 256, 64)
    code, raw = g.status()
    assert code == -5 and (raw & 0xFF00) == 0x100, (code, hex(raw))
    # the context is still usable: a normal forward afterwards is clean and correct
    out = g.forward(out_dtype=torch.float32).cpu().numpy()
    assert g.status() == (0, 0)
    m = metrics(out, oracle_ref(w, x))
    assert m["relL1"] <= REL_L1, m
