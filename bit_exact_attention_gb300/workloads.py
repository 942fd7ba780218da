"""Seeded synthetic inputs shaped like the SageAttention2 workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle may take their
inputs from it.

Every tensor is drawn on the CPU with ``torch.Generator().manual_seed(seed)``
in FP32 and cast (round-to-nearest-even) to fp16/bf16, so the GPU and the
oracle see identical bits. Layout: token-major and packed over the batch,
``[total_tokens, heads, D]``; ``cu_q``/``cu_kv`` are prefix sums of the
per-sequence lengths.

Readings of the workload descriptions:
  * ``N(0, s2)`` names a variance: N(0,4) has standard deviation 2.
  * a "channel bias" is one offset per (head, channel), shared by every token
    and every sequence of the batch.
  * "outlier channels": per head, 4 channel indices drawn without replacement
    (independently for Q and for K), each offset by a constant of random sign
    times U(8, 16), shared by every token.
"""
from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    nq: tuple[int, ...]          # per-sequence query lengths
    nkv: tuple[int, ...]         # per-sequence key/value lengths
    hq: int
    hkv: int
    d: int
    dtype: str                   # "fp16" | "bf16"
    causal: bool
    dist: str                    # distribution recipe, see make_inputs
    seed: int
    varlen: bool = False         # packed variable-length call (cu_seqlens)

    @property
    def batch(self) -> int:
        return len(self.nq)

    def metric_ops(self) -> float:
        """4 * Hq * Nq * Nkv * D summed per sequence, halved for causal."""
        ops = sum(4.0 * self.hq * a * b * self.d for a, b in zip(self.nq, self.nkv))
        return ops / 2 if self.causal else ops

    def visible_pairs(self) -> int:
        """Exact count of visible (query, key) pairs per head, all sequences."""
        tot = 0
        for a, b in zip(self.nq, self.nkv):
            if not self.causal:
                tot += a * b
            else:
                off = b - a
                for i in range(a):
                    tot += max(0, min(b, i + off + 1))
        return tot


def _uniform(n, B):
    return tuple([n] * B)


# The five workloads (shapes, dtypes, distributions) the method is measured on.
TINY = Workload("tiny_noncausal_B1_H2_N256_D64_fp16", _uniform(256, 1), _uniform(256, 1),
                2, 2, 64, "fp16", False, "tiny", 0)
PREFILL = Workload("llm_prefill_causal_B2_H32_N4096_D128_bf16", _uniform(4096, 2),
                   _uniform(4096, 2), 32, 32, 128, "bf16", True, "outlier", 1)
GQA_LONG = Workload("gqa_long_causal_B1_Hq32_Hkv8_N32768_D128_bf16", _uniform(32768, 1),
                    _uniform(32768, 1), 32, 8, 128, "bf16", True, "outlier", 2)
VIDEO_DIT = Workload("video_dit_noncausal_B2_H24_N17776_D64_fp16", _uniform(17776, 2),
                     _uniform(17776, 2), 24, 24, 64, "fp16", False, "dit", 3)
VARLEN = Workload("varlen_noncausal_B4_Hq16_Hkv4_D128_bf16", (1024, 3000, 512, 7777),
                  (8192, 4096, 16384, 2048), 16, 4, 128, "bf16", False, "kbias9", 4, varlen=True)

ALL = (TINY, PREFILL, GQA_LONG, VIDEO_DIT, VARLEN)


def scaled(w: Workload, nq, nkv, hq=None, hkv=None, name=None, seed=None, causal=None,
           d=None, varlen=None) -> Workload:
    """Same distribution and dtype at other sizes (parity cases the oracle finishes quickly)."""
    return dataclasses.replace(
        w, name=name or (w.name + "_scaled"), nq=tuple(nq), nkv=tuple(nkv),
        hq=hq if hq is not None else w.hq, hkv=hkv if hkv is not None else w.hkv,
        seed=w.seed if seed is None else seed, causal=w.causal if causal is None else causal,
        d=w.d if d is None else d, varlen=w.varlen if varlen is None else varlen)


def _channel_offsets(gen, heads, d, std):
    return torch.randn(heads, d, generator=gen) * std


def _outliers(gen, heads, d, count=4):
    off = torch.zeros(heads, d)
    for h in range(heads):
        idx = torch.randperm(d, generator=gen)[:count]
        sign = torch.where(torch.rand(count, generator=gen) < 0.5, -1.0, 1.0)
        mag = 8.0 + 8.0 * torch.rand(count, generator=gen)
        off[h, idx] = sign * mag
    return off


def make_inputs(w: Workload):
    """Returns dict(q, k, v: CPU tensors [total, heads, D] of w.dtype; cu_q, cu_kv: lists)."""
    gen = torch.Generator().manual_seed(w.seed)
    tq, tkv = sum(w.nq), sum(w.nkv)
    q = torch.randn(tq, w.hq, w.d, generator=gen)
    k = torch.randn(tkv, w.hkv, w.d, generator=gen)
    v = torch.randn(tkv, w.hkv, w.d, generator=gen)
    if w.dist == "tiny":          # K plus a per-head channel bias ~ N(0, 4)
        k += _channel_offsets(gen, w.hkv, w.d, 2.0)
    elif w.dist == "outlier":     # 4 outlier channels per head in Q and K; K bias ~ N(0, 9)
        q += _outliers(gen, w.hq, w.d)
        k += _outliers(gen, w.hkv, w.d)
        k += _channel_offsets(gen, w.hkv, w.d, 3.0)
    elif w.dist == "dit":         # Q, K ~ N(0, 1.5) each with a channel bias ~ N(0, 4)
        q *= math.sqrt(1.5)
        k *= math.sqrt(1.5)
        q += _channel_offsets(gen, w.hq, w.d, 2.0)
        k += _channel_offsets(gen, w.hkv, w.d, 2.0)
    elif w.dist == "kbias9":      # K channel bias ~ N(0, 9)
        k += _channel_offsets(gen, w.hkv, w.d, 3.0)
    elif w.dist == "plain":
        pass
    else:
        raise ValueError(w.dist)
    dt = DTYPES[w.dtype]
    cu_q = [0]
    for n in w.nq:
        cu_q.append(cu_q[-1] + n)
    cu_kv = [0]
    for n in w.nkv:
        cu_kv.append(cu_kv[-1] + n)
    return {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous(),
            "cu_q": cu_q, "cu_kv": cu_kv}


def as_bits(t: torch.Tensor):
    """Raw 16-bit patterns of an fp16/bf16 CPU tensor as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def dtype_code(w: Workload) -> int:
    """0 for fp16, 1 for bf16 (the code both the library and the oracle use)."""
    return 1 if w.dtype == "bf16" else 0
