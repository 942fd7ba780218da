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
# The GPU's DeltaS against the oracle's (the FP64 dot product rounded once): the tensor core
# accumulates the bf16 pieces of both operands in FP32 (about 50 roundings at most for 128
# channels and six piece products, plus 2^-23 for the dropped piece products) and the CUDA-core
# form is a 128-long FP32 chain, so both lie within 128 units of 2^-24 of sum |qmean_d K~_jd|;
# times c, plus the rounding of both sides' products with c.
DS_UNITS = 128


def ds_abs_sum(x: dict, w: W.Workload, b: int, hk: int, kmean, qbar) -> np.ndarray:
    """sum_d |qmean_d| |K~_jd| for the keys of sequence b, kv head hk (K~ = fl32(K - kmean))."""
    k0, k1 = x["cu_kv"][b], x["cu_kv"][b + 1]
    kf = x["k"][k0:k1, hk].float().numpy()
    kt = (kf - (kmean[b, hk, : w.d] if kmean is not None else 0)).astype(np.float32)
    return np.abs(kt).astype(np.float64) @ np.abs(qbar[: w.d]).astype(np.float64)


def check_dsc(got_dsc: np.ndarray, ds_oracle: np.ndarray, abs_sum: np.ndarray, c32) -> float:
    """DeltaS*c of the GPU (FP32) within DS_UNITS * 2^-24 * c * sum|qmean K~| + 2 ulp of the
    oracle's fl32(DeltaS c); returns the largest deviation as a fraction of that bound."""
    want = (ds_oracle * np.float32(c32)).astype(np.float32)
    bound = (DS_UNITS * 2.0 ** -24 * float(c32) * abs_sum +
             2.0 * np.spacing(np.abs(want)).astype(np.float64))
    dev = np.abs(got_dsc.astype(np.float64) - want.astype(np.float64))
    assert np.all(dev <= bound), (float((dev / bound).max()), int(np.argmax(dev / bound)))
    return float((dev / np.maximum(bound, 1e-300)).max()) if dev.size else 0.0


def flip_allowance(dsc_dev_max: float, s_abs_max: float) -> float:
    """FP32 ulps of 448 P by which a P~ decision may sit from an e4m3 midpoint and still differ
    from the emulation: 4 for the hardware exponential, plus the logit shift that a DeltaS
    deviation of at most dsc_dev_max (and one FP32 rounding of logits up to s_abs_max) makes,
    both in the key's own logit and in the row maximum (2 (dev + ulp) in log2 units; 448 P moves
    by that times ln 2 relative, at most 2^24 ulps per unit)."""
    shift = 2.0 * (dsc_dev_max + float(np.spacing(np.float32(s_abs_max))))
    return 4.0 + shift * math.log(2.0) * 2.0 ** 24


def located_flips(got: np.ndarray, p448: np.ndarray, max_ulp: float = 4.0) -> int:
    """The e4m3 codes `got` against the emulation's P448 (fl32 values of 448 P): every code that
    differs from e4m3(P448) must be one e4m3 step off, with P448 within `max_ulp` FP32 ulps of
    the rounding midpoint between the two codes (the hardware exponential's error). Returns the
    number of differing codes."""
    import oracle
    want = oracle.e4m3_encode(p448.astype(np.float64))
    diff = got != want
    if diff.any():
        # positive e4m3 bytes are ordered like their values: one step = one byte
        step = np.abs(got[diff].astype(np.int64) - want[diff].astype(np.int64))
        assert np.all(step == 1), "codes more than one step off"
        lo = oracle.e4m3_decode(np.minimum(got[diff], want[diff]))
        hi = oracle.e4m3_decode(np.maximum(got[diff], want[diff]))
        mid = (lo + hi) / 2
        ulp = np.spacing(mid.astype(np.float32)).astype(np.float64)
        off = np.abs(p448[diff].astype(np.float64) - mid) / ulp
        assert off.max() <= max_ulp, f"a flip {off.max()} ulp from a midpoint"
    return int(diff.sum())


L32 = np.float32(8.8073549220576041)  # fl32(log2(448))


def tile_logits(A, sq_rows, sk_keys, ds_keys, c32, visible):
    """S' = fl32(A * fl32(fl32(sq c) sk) + fl32(DeltaS c)) for rows x keys, -inf where a key is
    not visible. A * mult is exact in FP64 (13 + 24 bits) and the sum with the FP32 addend is
    rounded once more to FP32, which equals the fused multiply-add except when the two terms'
    exponents are more than 16 apart (then both roundings still land within 1 ulp)."""
    sqc = (sq_rows.astype(np.float32) * np.float32(c32)).astype(np.float32)
    mult = (sqc[:, None] * sk_keys.astype(np.float32)[None, :]).astype(np.float32)
    dsc = (ds_keys.astype(np.float32) * np.float32(c32)).astype(np.float32)
    S = (A.astype(np.float64) * mult.astype(np.float64) + dsc.astype(np.float64)[None, :])
    S = S.astype(np.float32)
    S[~visible] = -np.inf
    return S


def fold_rows(S_tiles, P_tiles, V_tiles, sv):
    """The two-level fold of the method for given P~ values, in FP64: with m_j the running row
    maximum after KV tile j, O = sum_j 2^(m_j - m_T) P~_j V_j, l = sum_j 2^(m_j - m_T) sum_k
    P448_jk with P448 = 2^(fl32(S'_jk - fl32(m_j - log2 448))) = 448 * 2^(S' - m_j), output
    O * sv / l (P~ and l both carry the static factor 448); rows with no visible key give 0.
    S_tiles, P_tiles: [rows, keys] per tile; V_tiles: [keys, D]."""
    rows = S_tiles[0].shape[0]
    m = np.full(rows, -np.inf, np.float32)
    ms, rsum = [], []
    for S in S_tiles:
        m = np.maximum(m, S.max(axis=1))
        ms.append(m.copy())
        m448 = np.where(np.isfinite(m), (m - L32).astype(np.float32), np.float32(0))
        arg = (S - m448[:, None]).astype(np.float32)
        rsum.append(np.where(np.isfinite(arg), np.exp2(arg.astype(np.float64)), 0.0).sum(axis=1))
    mT = ms[-1]
    O = np.zeros((rows, V_tiles[0].shape[1]))
    l = np.zeros(rows)
    for mj, rj, P, V in zip(ms, rsum, P_tiles, V_tiles):
        f = np.where(np.isfinite(mj), np.exp2(np.where(np.isfinite(mj), mj.astype(np.float64) -
                                                       mT.astype(np.float64), 0.0)), 0.0)
        O += f[:, None] * (P.astype(np.float64) @ V.astype(np.float64))
        l += f * rj
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(l[:, None] > 0, O * sv[None, :] / l[:, None], 0.0)
    return out


class UnitData:
    """The oracle's quantized operands of one workload: codes, scales, means, DeltaS per
    (sequence, q head, Q block); kw are the oracle's quantization switches (smooth_q, smooth_k,
    per_block, qk_bits) as attention_emulated takes them."""

    def __init__(self, w: W.Workload, x: dict, sm_scale=0.0, **kw):
        import oracle
        self.w, self.x, self.kw, self.sm_scale = w, x, kw, sm_scale
        smooth_q, smooth_k = kw.get("smooth_q", True), kw.get("smooth_k", True)
        per_block, qk_bits = kw.get("per_block", False), kw.get("qk_bits", 4)
        dt = W.dtype_code(w)
        qb, kb, vb = bits(x["q"]), bits(x["k"]), bits(x["v"])
        kmean, vamax = oracle.kv_stats(kb, vb, dt, x["cu_kv"], w.hkv, w.d)
        self.kmean = kmean if smooth_k else None
        self.qmean, self.qc, self.sq = oracle.quant_q(qb, dt, x["cu_q"], w.hq, w.d,
                                                      smooth_q=smooth_q, per_block=per_block,
                                                      qk_bits=qk_bits)
        self.kc, self.sk = oracle.quant_k(kb, dt, x["cu_kv"], w.hkv, w.d, kmean=self.kmean,
                                          gk=128 if per_block else 32, qk_bits=qk_bits)
        vc, self.sv = oracle.quant_v(vb, dt, x["cu_kv"], w.hkv, w.d, vamax)
        self.vval = oracle.e4m3_decode(vc)
        self.c32 = c32_of(w, sm_scale)
        self._ds = {}
        self.kb, self.dt = kb, dt

    def delta_s(self, b, h, qt):
        import oracle
        key = (b, h, qt)
        if key not in self._ds:
            w = self.w
            self._ds[key] = oracle.delta_s(self.kb, self.dt, self.x["cu_kv"], b, w.hkv,
                                           h // (w.hq // w.hkv), w.d, self.kmean,
                                           self.qmean[b, h, qt])
        return self._ds[key]

    def dsc_deviation(self, g: "GpuCase", b, h, qt) -> np.ndarray:
        """|GPU DeltaS*c - oracle fl32(DeltaS c)| for the keys of sequence b seen by Q block qt
        of head h (0 past the visited tiles)."""
        if not hasattr(self, "_gpu_dsc"):
            self._gpu_dsc = g.gathered()["dsc"]
        w = self.w
        n = min(w.nkv[b], kv_tiles(qt, w.nq[b], w.nkv[b], w.causal) * 128)
        blk = pad_starts(self.x["cu_q"])[b] // 128 + qt
        got = self._gpu_dsc[h, blk, :n].astype(np.float64)
        want = (self.delta_s(b, h, qt)[:n] * np.float32(self.c32)).astype(np.float32)
        out = np.zeros(max(w.nkv[b], 1))
        out[:n] = np.abs(got - want.astype(np.float64))
        return out

    def tile(self, b, h, qt, kt, rows):
        """(S' [len(rows), 128], V [128, D0]) of KV tile kt for the given rows of Q tile qt."""
        w, x = self.w, self.x
        nq, nkv = w.nq[b], w.nkv[b]
        hk = h // (w.hq // w.hkv)
        i = qt * 128 + np.asarray(rows)
        keys = kt * 128 + np.arange(128)
        kin = np.minimum(keys, nkv - 1)
        vis = np.broadcast_to(keys[None, :] < nkv, (len(i), 128)).copy()
        if w.causal:
            vis = vis & (keys[None, :] <= (i + nkv - nq)[:, None])
        A = (self.qc[x["cu_q"][b] + i, h].astype(np.int64) @
             self.kc[x["cu_kv"][b] + kin, hk].astype(np.int64).T)
        S = tile_logits(A, self.sq[x["cu_q"][b] + i, h], self.sk[x["cu_kv"][b] + kin, hk],
                        self.delta_s(b, h, qt)[kin], self.c32, vis)
        V = np.where((keys < nkv)[:, None], self.vval[x["cu_kv"][b] + kin, hk], 0.0)
        return S, V[:, : w.d]


def prove_rows_by_codes(g: GpuCase, ud: UnitData, b, h, qt, rows, max_ulp=4.0):
    """Rows of Q tile (b, h, qt) recomputed from the GPU's own P~ codes (dumped tile by tile with
    the debug hook) with the oracle's logits, V codes and scales; every code that differs from
    the emulation's is checked to be a located midpoint flip. Returns (the recomputed rows in
    FP64, differing codes per row)."""
    import oracle
    w, x = ud.w, ud.x
    T = kv_tiles(qt, w.nq[b], w.nkv[b], w.causal)
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)
    S_t, P_t, V_t = [], [], []
    flips = np.zeros(len(rows), np.int64)
    dev = ud.dsc_deviation(g, b, h, qt)
    for kt in range(T):
        S, V = ud.tile(b, h, qt, kt, rows)
        _, p_out, _ = g.debug_tile(b, h, qt, kt)
        got = p_out.cpu().numpy()[rows]
        p448 = oracle.emulated_tile_p448(*args, b, h, qt, kt, sm_scale=ud.sm_scale,
                                         **ud.kw)[rows]
        vis = np.isfinite(S)
        allow = max(max_ulp, flip_allowance(float(dev[: (kt + 1) * 128].max(initial=0.0)),
                                            float(np.abs(S[vis]).max(initial=0.0))))
        for r in range(len(rows)):
            flips[r] += located_flips(got[r][vis[r]], p448[r][vis[r]], allow)
        P_t.append(np.where(vis, e4m3_to_f64(torch.from_numpy(got.copy())), 0.0))
        S_t.append(S)
        V_t.append(V)
    sv = ud.sv[b, h // (w.hq // w.hkv), : w.d]
    return fold_rows(S_t, P_t, V_t, sv), flips


def compare_p_codes(g: GpuCase, w: W.Workload, x: dict, kw: dict):
    """P~ e4m3 codes of a few tiles per sequence (first, middle, last Q tile; first, middle and
    last visited KV tile) from the kernel against the emulation's, for the oracle switches kw.
    Every disagreement must be one e4m3 step, at an exact 448 P within 4 ulp of the rounding
    midpoint between the two codes (the hardware exponential's error). Returns
    (differing codes, compared codes)."""
    import oracle
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)
    ud = UnitData(w, x, **kw)
    n_cmp = n_diff = 0
    for b in range(w.batch):
        nqb = (w.nq[b] + 127) // 128
        for (h, qt) in sorted({(0, 0), (w.hq - 1, nqb - 1), (w.hq // 2, nqb // 2)}):
            if nqb == 0:
                continue
            T = kv_tiles(qt, w.nq[b], w.nkv[b], w.causal)
            dev = ud.dsc_deviation(g, b, h, qt)
            rows = np.arange(min(128, w.nq[b] - qt * 128))
            for kt in sorted({0, T // 2, T - 1}):
                if kt < 0:
                    continue
                _, p_out, _ = g.debug_tile(b, h, qt, kt)
                got = p_out.cpu().numpy()[rows]
                p448 = oracle.emulated_tile_p448(*args, b, h, qt, kt, **kw)[rows]
                S, _ = ud.tile(b, h, qt, kt, rows)
                fin = S[np.isfinite(S)]
                allow = flip_allowance(float(dev[: (kt + 1) * 128].max(initial=0.0)),
                                       float(np.abs(fin).max(initial=0.0)))
                n_cmp += got.size
                n_diff += located_flips(got, p448, allow)
    return n_diff, n_cmp


def check_forward_proven(g: GpuCase, w: W.Workload, x: dict, out, emu, kw=None,
                         rel_l1=1e-3, max_abs=2e-3, max_rows=400, rows=None, tol=None):
    """Output against the emulation: relative L1 within rel_l1 and every element within max_abs,
    except rows proven to differ only through P~ codes on the other side of an e4m3 rounding
    midpoint (prove_rows_by_codes: the row recomputed from the GPU's own codes matches the GPU
    within max_abs, and every code that differs from the emulation's is a located flip).
    tol (default max_abs) may be an array of per-element tolerances shaped like out.
    Returns the number of proven rows."""
    tol = np.full(out.shape, max_abs) if tol is None else np.broadcast_to(tol, out.shape)
    if rows is not None:  # only these (token, head) rows were computed by the oracle
        toks, heads = rows
        m = metrics(out[toks, heads], emu[toks, heads])
        row_over = np.zeros(out.shape[:2], bool)
        row_over[toks, heads] = (np.abs(out[toks, heads] - emu[toks, heads]) >
                                 tol[toks, heads]).any(axis=1)
    else:
        m = metrics(out, emu)
        row_over = (np.abs(out - emu) > tol).any(axis=2) if out.size else np.zeros((0, 0), bool)
    assert m["relL1"] <= rel_l1, m
    off_t, off_h = np.nonzero(row_over)
    assert len(off_t) <= max_rows, f"{len(off_t)} rows above {max_abs}"
    if len(off_t) == 0:
        return 0
    cu = np.asarray(x["cu_q"])
    groups = {}
    for t, h in zip(off_t, off_h):
        b = int(np.searchsorted(cu, t, side="right") - 1)
        i = int(t - cu[b])
        groups.setdefault((b, int(h), i // 128), []).append(i % 128)
    ud = UnitData(w, x, sm_scale=g.sm_scale, **(kw or {}))
    for (b, h, qt), rows in sorted(groups.items()):
        rows = np.asarray(sorted(rows))
        rec, flips = prove_rows_by_codes(g, ud, b, h, qt, rows)
        toks = cu[b] + qt * 128 + rows
        gap = np.abs(rec - out[toks, h]) - tol[toks, h]
        assert np.all(gap <= 0), (b, h, qt, rows, gap.max(axis=1))
        assert np.all(flips >= 1), (b, h, qt, rows, flips)
    return len(off_t)
