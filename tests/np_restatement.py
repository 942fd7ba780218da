"""Independent NumPy/Python restatement of the quantized pipeline for tiny shapes.

Used only to pin the C oracle by brute force. It shares no code with the oracle or
with the CUDA library: number formats come from library casts (numpy float32
arithmetic, ``torch.float8_e4m3fn`` for e4m3 rounding) and the one fused
multiply-add is evaluated exactly with ``fractions.Fraction``. Pure Python loops:
meant for a handful of tokens.

Method (SageAttention2 pages): K smoothed by its channel mean; Q smoothed by the
mean of its block with the Delta-S correction kept for the logits ("SageAttention2:
Efficient Attention with Thorough Outlier Smoothing and Per-thread INT4
Quantization" research note, component 1); INT4-grid codes with per-row Q scales
and per-32-token K scales (component 2); e4m3 P~ and V with a fresh partial per KV
block folded into FP32 (component 3; PMLR v267 zhang25ae, Abstract).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

F32 = np.float32


def fr_to_f32(x: Fraction) -> np.float32:
    """Correctly rounded (nearest-even) Fraction -> float32, normal range."""
    if x == 0:
        return F32(0.0)
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 23)
    r = round(a / quantum)  # Fraction rounding: ties to even
    return F32(float(s * r * quantum))


def fma32(a, b, c) -> np.float32:
    return fr_to_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def e4m3_value(x: np.float32) -> float:
    t = torch.tensor([float(x)], dtype=torch.float32).to(torch.float8_e4m3fn)
    return float(t.to(torch.float64)[0])


def quantize_group(x: np.ndarray, g: int = 7):
    """x: float32 array (any shape), grid [-g, g]. Returns (int codes, float32 scale)."""
    a = F32(np.max(np.abs(x))) if x.size else F32(0)
    if a == 0:
        return np.zeros(x.shape, dtype=np.int64), F32(0)
    inv = F32(g) / a
    t = (x * inv).astype(F32)
    codes = np.clip(np.rint(t), -g, g).astype(np.int64)
    return codes, F32(a / F32(g))


def mode_q(q, k, v, cu_q, cu_kv, hq, hkv, d0, causal, sm_scale=0.0, bq=128, bkv=128, gk=32,
           smooth_q=True, smooth_k=True, per_block=False, qk_bits=4):
    """q, k, v: float64 arrays [tokens, heads, d0] holding the exact fp16/bf16 values.
    Returns the FP64 output before dtype rounding, [total_q, hq, d0].
    Switches: smooth_q / smooth_k off use a zero mean; per_block quantizes each block of bq
    query rows, and each block of bkv keys, with one scale; qk_bits = 8 uses the grid
    [-127, 127] for the Q and K codes instead of [-7, 7]."""
    G = 7 if qk_bits == 4 else 127
    g = hq // hkv
    scale32 = F32(sm_scale) if sm_scale > 0 else F32(1.0 / math.sqrt(d0))
    c32 = F32(1.4426950408889634 * float(scale32))
    L32 = F32(math.log2(448.0))
    B = len(cu_q) - 1
    out = np.zeros((cu_q[-1], hq, d0))
    for b in range(B):
        nq, nkv = cu_q[b + 1] - cu_q[b], cu_kv[b + 1] - cu_kv[b]
        for h in range(hq):
            hk = h // g
            K = k[cu_kv[b]:cu_kv[b + 1], hk, :]
            V = v[cu_kv[b]:cu_kv[b + 1], hk, :]
            kmean = np.array([F32(K[:, c].sum() / nkv) for c in range(d0)], dtype=F32) \
                if (nkv and smooth_k) else np.zeros(d0, F32)
            Kt = (K.astype(F32) - kmean).astype(F32)              # smoothed K, float32
            kcodes = np.zeros((nkv, d0), np.int64)
            ksc = np.zeros(nkv, F32)
            kg = bkv if per_block else gk
            for t0 in range(0, nkv, kg):
                cds, s = quantize_group(Kt[t0:t0 + kg], G)
                kcodes[t0:t0 + kg] = cds
                ksc[t0:t0 + kg] = s
            vamax = np.abs(V).max(axis=0).astype(F32) if nkv else np.zeros(d0, F32)
            vinv = np.array([F32(448.0) / a if a > 0 else F32(0) for a in vamax], dtype=F32)
            vsc = np.array([a / F32(448.0) if a > 0 else F32(0) for a in vamax], dtype=F32)
            vhat = np.array([[e4m3_value(F32(V[j, c]) * vinv[c]) for c in range(d0)]
                             for j in range(nkv)]).reshape(nkv, d0)
            Q = q[cu_q[b]:cu_q[b + 1], h, :]
            for r0 in range(0, nq, bq):
                rows = range(r0, min(r0 + bq, nq))
                qbar = np.array([F32(Q[r0:r0 + bq, c].sum() / len(rows)) for c in range(d0)], F32) \
                    if smooth_q else np.zeros(d0, F32)
                if per_block:
                    blk_codes, blk_scale = quantize_group((Q[r0:r0 + bq].astype(F32) - qbar).astype(F32), G)
                # Delta-S: the exact dot product of the FP32 operands (math.fsum of exact FP64
                # products), rounded to FP32
                dS = [F32(math.fsum(float(qbar[c]) * float(Kt[j, c]) for c in range(d0)))
                      for j in range(nkv)]
                for i in rows:
                    qt = (Q[i].astype(F32) - qbar).astype(F32)
                    qc, qs = (blk_codes[i - r0], blk_scale) if per_block else quantize_group(qt, G)
                    sqc = F32(qs * c32)
                    m = -math.inf
                    lsum = 0.0
                    O = np.zeros(d0, F32)
                    for t0 in range(0, nkv, bkv):
                        js = range(t0, min(t0 + bkv, nkv))
                        sp = {}
                        for j in js:
                            if causal and j > i + (nkv - nq):
                                continue
                            A = int(np.dot(qc, kcodes[j]))
                            mult = F32(sqc * ksc[j])
                            sp[j] = fma32(F32(A), mult, F32(dS[j] * c32))
                        mx = max(sp.values()) if sp else -math.inf
                        m_new = max(m, mx)
                        if m_new == -math.inf:
                            continue
                        alpha = 0.0 if m == -math.inf else 2.0 ** (float(m) - float(m_new))
                        m448 = F32(F32(m_new) - L32)
                        R = np.zeros(d0)
                        ps = 0.0
                        for j, s in sp.items():
                            p448 = F32(2.0 ** float(F32(s - m448)))
                            ps += float(p448)
                            R += e4m3_value(p448) * vhat[j]
                        lsum = alpha * lsum + ps
                        O = (alpha * O.astype(np.float64) + R.astype(F32).astype(np.float64)).astype(F32)
                        m = m_new
                    row = cu_q[b] + i
                    out[row, h] = (O.astype(np.float64) * vsc.astype(np.float64) / lsum) if lsum > 0 else 0.0
    return out
