"""Helpers for the GPU parity tests: run the library, read its workspace back in the
oracle's layouts, run the oracle on the same seeded inputs, compare.

The oracle only ever sees the seeded inputs; nothing computed by the CUDA path is fed
to it.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import bit_exact_attention_gb300 as S
from bit_exact_attention_gb300 import workloads as W


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def pad_starts(cu):
    return [128 * (cu[b] // 128 + b) for b in range(len(cu) - 1)]


def metrics(a: np.ndarray, r: np.ndarray) -> dict:
    a = np.asarray(a, np.float64).ravel()
    r = np.asarray(r, np.float64).ravel()
    den = np.abs(r).sum()
    cos = float(a @ r / math.sqrt((a @ a) * (r @ r))) if (a @ a) > 0 and (r @ r) > 0 else float(
        np.array_equal(a, r))
    return {"relL1": float(np.abs(a - r).sum() / den) if den > 0 else float(np.abs(a - r).sum()),
            "maxabs": float(np.abs(a - r).max()) if a.size else 0.0, "cos": cos}


def c32_of(w: W.Workload, sm_scale=0.0):
    """c = fl32(log2(e) * fl32(sm_scale)), sm_scale defaulting to 1/sqrt(D0)."""
    s = np.float32(sm_scale) if sm_scale > 0 else np.float32(1.0 / math.sqrt(w.d))
    return np.float32(1.4426950408889634 * float(s))


def kv_tiles(qt, nq, nkv, causal):
    """KV tiles of 128 keys that Q block qt visits (bottom-right causal alignment)."""
    nt = (nkv + 127) // 128
    if not causal:
        return nt
    i_last = min(qt * 128 + 127, nq - 1)
    j_max = i_last + (nkv - nq)
    return 0 if j_max < 0 else min(nt, j_max // 128 + 1)


def e4m3_to_int(u8: torch.Tensor) -> np.ndarray:
    return u8.contiguous().view(torch.float8_e4m3fn).to(torch.float32).cpu().numpy().astype(np.int64)


def e4m3_to_f64(u8: torch.Tensor) -> np.ndarray:
    return u8.contiguous().view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()


class GpuCase:
    """Inputs on the GPU plus a workspace; prepass / attention / debug hooks."""

    def __init__(self, w: W.Workload, x: dict, causal=None, sm_scale=0.0, quant_flags=0):
        self.w, self.x = w, x
        self.quant_flags = quant_flags
        self.causal = w.causal if causal is None else causal
        self.sm_scale = sm_scale
        self.B = w.batch
        self.max_nq, self.max_nkv = max(w.nq), max(w.nkv)
        self.tq, self.tkv = sum(w.nq), sum(w.nkv)
        self.q = x["q"].cuda()
        self.k = x["k"].cuda()
        self.v = x["v"].cuda()
        self.cu_q = torch.tensor(x["cu_q"], dtype=torch.int32, device="cuda")
        self.cu_kv = torch.tensor(x["cu_kv"], dtype=torch.int32, device="cuda")
        self.L = S.workspace_layout(self.B, w.hq, w.hkv, self.max_nq, self.max_nkv, w.d,
                                    self.tq, self.tkv, quant_flags=quant_flags)
        self.ws = S.alloc_workspace(self.L.total_bytes)
        self.off0 = (-self.ws.data_ptr()) % 1024

    def prepass(self):
        S.prepass_varlen(self.q, self.k, self.v, self.cu_q, self.cu_kv, self.max_nq,
                         self.max_nkv, self.ws, causal=self.causal, sm_scale=self.sm_scale,
                         quant_flags=self.quant_flags)

    def attention(self, out_dtype=torch.float32):
        out = torch.empty(self.tq, self.w.hq, self.w.d, dtype=out_dtype, device="cuda")
        S.attention_varlen(out, self.ws, self.cu_q, self.cu_kv, self.w.hkv, self.max_nq,
                           self.max_nkv, self.tkv, causal=self.causal, sm_scale=self.sm_scale)
        return out

    def forward(self, out_dtype=None):
        return S.attn_fwd_varlen(self.q, self.k, self.v, self.cu_q, self.cu_kv, self.max_nq,
                                 self.max_nkv, causal=self.causal, sm_scale=self.sm_scale,
                                 out_dtype=out_dtype, workspace=self.ws,
                                 quant_flags=self.quant_flags)

    def status(self):
        return S.device_status(self.ws)

    def debug_tile(self, b, h, qt, kt):
        return S.debug_tile(self.ws, self.B, self.w.hq, self.w.hkv, self.max_nq, self.max_nkv,
                            self.w.d, self.causal, b, h, qt, kt, sm_scale=self.sm_scale,
                            cu_seqlens_q=self.cu_q, cu_seqlens_kv=self.cu_kv, total_q=self.tq,
                            total_kv=self.tkv, quant_flags=self.quant_flags)

    # ---------------------------------------------------------------- workspace views
    @property
    def code_dtype(self):
        """Q / K codes: e4m3 bytes, or fp16 values for the INT8 path."""
        return torch.float16 if self.L.code_bytes == 2 else torch.uint8

    def code_to_int(self, t: torch.Tensor) -> np.ndarray:
        if self.L.code_bytes == 2:
            f = t.contiguous().to(torch.float64).cpu().numpy()
            assert np.all(f == np.rint(f)), "INT8-path codes must be integers"
            return f.astype(np.int64)
        return e4m3_to_int(t)

    def _buf(self, off, count, dtype):
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return self.ws[self.off0 + off: self.off0 + off + nbytes].view(dtype)

    def views(self):
        L, w = self.L, self.w
        Dp = L.Dp
        return {
            "qcode": self._buf(L.qcode, w.hq * L.Tq * Dp, self.code_dtype).view(w.hq, L.Tq, Dp),
            "kcode": self._buf(L.kcode, w.hkv * L.Tkv * Dp, self.code_dtype).view(w.hkv, L.Tkv, Dp),
            "vcodeT": self._buf(L.vcodeT, w.hkv * Dp * L.Tkv, torch.uint8).view(w.hkv, Dp, L.Tkv),
            "qscale": self._buf(L.qscale, w.hq * L.Tq, torch.float32).view(w.hq, L.Tq),
            "kscale": self._buf(L.kscale, w.hkv * L.Tkv // 32, torch.float32).view(w.hkv, L.Tkv // 32),
            "qmean": self._buf(L.qmean, w.hq * (L.Tq // 128) * Dp, torch.float32).view(w.hq, L.Tq // 128, Dp),
            "kmean": self._buf(L.kmean, self.B * w.hkv * Dp, torch.float32).view(self.B, w.hkv, Dp),
            "vscale": self._buf(L.vscale, self.B * w.hkv * Dp, torch.float32).view(self.B, w.hkv, Dp),
            "dsc": self._buf(L.dsc, w.hq * (L.Tq // 128) * L.nkv_pad, torch.float32).view(
                w.hq, L.Tq // 128, L.nkv_pad),
        }

    def gathered(self):
        """The prepass results in the oracle's (token-major, unpadded) layouts."""
        v = {k: t.cpu() for k, t in self.views().items()}
        w, x = self.w, self.x
        qp, kp = pad_starts(x["cu_q"]), pad_starts(x["cu_kv"])
        Dp = self.L.Dp
        qc = np.zeros((self.tq, w.hq, Dp), np.int64)
        sq = np.zeros((self.tq, w.hq), np.float32)
        kc = np.zeros((self.tkv, w.hkv, Dp), np.int64)
        sk = np.zeros((self.tkv, w.hkv), np.float32)
        vc = np.zeros((self.tkv, w.hkv, Dp), np.float64)
        for b in range(self.B):
            q0, nq = x["cu_q"][b], w.nq[b]
            k0, nkv = x["cu_kv"][b], w.nkv[b]
            qc[q0:q0 + nq] = self.code_to_int(v["qcode"][:, qp[b]:qp[b] + nq]).transpose(1, 0, 2)
            sq[q0:q0 + nq] = v["qscale"][:, qp[b]:qp[b] + nq].numpy().T
            kc[k0:k0 + nkv] = self.code_to_int(v["kcode"][:, kp[b]:kp[b] + nkv]).transpose(1, 0, 2)
            toks = np.arange(nkv)
            sk[k0:k0 + nkv] = v["kscale"][:, (kp[b] + toks) // 32].numpy().T
            vc[k0:k0 + nkv] = e4m3_to_f64(v["vcodeT"][:, :, kp[b]:kp[b] + nkv]).transpose(2, 0, 1)
        return {"qcode": qc, "qscale": sq, "kcode": kc, "kscale": sk, "vcode": vc,
                "kmean": v["kmean"].numpy(), "vscale": v["vscale"].numpy(),
                "qmean": v["qmean"].numpy(), "dsc": v["dsc"].numpy(), "raw": v}


def units_sample(w: W.Workload, n: int, seed: int = 0):
    """>= n (b, h, q-block) units: always the last (possibly partial) block of each sequence,
    the first block, a causal-diagonal block, then seeded random ones."""
    rng = np.random.default_rng(seed)
    units = set()
    for b in range(w.batch):
        nqb = (w.nq[b] + 127) // 128
        if nqb == 0:
            continue
        for h in sorted({0, w.hq - 1}):
            units.add((b, h, nqb - 1))
            units.add((b, h, 0))
            units.add((b, h, nqb // 2))
    while len(units) < n:
        b = int(rng.integers(w.batch))
        nqb = (w.nq[b] + 127) // 128
        if nqb == 0:
            continue
        units.add((b, int(rng.integers(w.hq)), int(rng.integers(nqb))))
    return sorted(units)


def unit_rows(w: W.Workload, cu_q, units):
    """Index arrays (token, head) of the rows the units cover."""
    toks, heads = [], []
    for b, h, qb in units:
        r0, r1 = qb * 128, min(w.nq[b], qb * 128 + 128)
        t = np.arange(cu_q[b] + r0, cu_q[b] + r1)
        toks.append(t)
        heads.append(np.full_like(t, h))
    return np.concatenate(toks), np.concatenate(heads)


# ---------------------------------------------------------------- checks shared by GPU tests
def compare_p_codes(g: GpuCase, w: W.Workload, x: dict, kw: dict):
    """P~ e4m3 codes of a few tiles per sequence (first, middle, last Q tile; first, middle and
    last visited KV tile) from the kernel against the emulation's, for the oracle switches kw.
    Every disagreement must be one e4m3 step, at an exact 448 P within 4 ulp of the rounding
    midpoint between the two codes (the hardware exponential's error). Returns
    (differing codes, compared codes)."""
    import oracle
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)
    n_cmp = n_diff = 0
    for b in range(w.batch):
        nqb = (w.nq[b] + 127) // 128
        for (h, qt) in sorted({(0, 0), (w.hq - 1, nqb - 1), (w.hq // 2, nqb // 2)}):
            if nqb == 0:
                continue
            T = kv_tiles(qt, w.nq[b], w.nkv[b], w.causal)
            for kt in sorted({0, T // 2, T - 1}):
                if kt < 0:
                    continue
                _, p_out, _ = g.debug_tile(b, h, qt, kt)
                nr = min(128, w.nq[b] - qt * 128)
                got = p_out.cpu().numpy()[:nr]
                p448 = oracle.emulated_tile_p448(*args, b, h, qt, kt, **kw)[:nr]
                want = oracle.e4m3_encode(p448.astype(np.float64))
                diff = got != want
                n_cmp += got.size
                n_diff += int(diff.sum())
                if diff.any():
                    # positive e4m3 bytes are ordered like their values: one step = one byte
                    step = np.abs(got[diff].astype(np.int64) - want[diff].astype(np.int64))
                    assert np.all(step == 1), f"b{b} h{h} qt{qt} kt{kt}: codes more than one step off"
                    lo = oracle.e4m3_decode(np.minimum(got[diff], want[diff]))
                    hi = oracle.e4m3_decode(np.maximum(got[diff], want[diff]))
                    mid = (lo + hi) / 2
                    ulp = np.spacing(mid.astype(np.float32)).astype(np.float64)
                    off = np.abs(p448[diff].astype(np.float64) - mid) / ulp
                    assert off.max() <= 4, f"b{b} h{h} qt{qt} kt{kt}: a flip {off.max()} ulp from a midpoint"
    return n_diff, n_cmp


def check_forward_with_flips(out, emu, x, rel_l1=1e-3, max_abs=2e-3):
    """Output against the emulation where P~ code flips may sit on dominant keys: relative L1
    within rel_l1; every element within max_abs or within max|V| / 8 + max_abs (all one-step
    flips of a row together move it by at most max|V| / 8); at most 1% of rows above max_abs."""
    m = metrics(out, emu)
    assert m["relL1"] <= rel_l1, m
    vmax = float(np.abs(x["v"].double().numpy()).max())
    d = np.abs(out - emu)
    assert d.max() <= vmax / 8 + max_abs, (d.max(), vmax)
    rows_off = int((d.reshape(-1, d.shape[-1]).max(axis=1) > max_abs).sum())
    assert rows_off <= max(2, d.shape[0] * d.shape[1] // 100), rows_off
