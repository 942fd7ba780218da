"""The NumPy restatement of the method's logits and two-level fold that the full-size GPU test
uses to explain rows by their P~ codes (parity_util.tile_logits / fold_rows / UnitData), pinned
on the CPU: fed the emulation's own e4m3 codes, it reproduces the oracle's Mode Q output."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from bit_exact_attention_gb300 import workloads as W
from parity_util import UnitData, bits, fold_rows, kv_tiles

CASES = {
    "prefill": W.scaled(W.PREFILL, (300, 200), (300, 200), hq=2, hkv=2, name="fold_prefill"),
    "varlen": W.scaled(W.VARLEN, (140, 77), (300, 129), hq=4, hkv=2, name="fold_varlen"),
    "gqa_nq_ne_nkv": W.scaled(W.GQA_LONG, (200,), (333,), hq=4, hkv=1, name="fold_gqa"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fold_of_the_emulations_codes_reproduces_mode_q(oracle_mod, name):
    w = CASES[name]
    x = W.make_inputs(w)
    ud = UnitData(w, x)
    args = (bits(x["q"]), bits(x["k"]), bits(x["v"]), W.dtype_code(w), x["cu_q"], x["cu_kv"],
            w.hq, w.hkv, w.d, w.causal)
    emu = oracle_mod.attention_emulated(*args)
    checked = 0
    for b in range(w.batch):
        for h in range(w.hq):
            for qt in range((w.nq[b] + 127) // 128):
                rows = np.arange(min(128, w.nq[b] - qt * 128))
                T = kv_tiles(qt, w.nq[b], w.nkv[b], w.causal)
                if T == 0:
                    continue
                S_t, P_t, V_t = [], [], []
                for kt in range(T):
                    S, V = ud.tile(b, h, qt, kt, rows)
                    p448 = oracle_mod.emulated_tile_p448(*args, b, h, qt, kt)[rows]
                    codes = oracle_mod.e4m3_encode(p448.astype(np.float64))
                    P = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
                    S_t.append(S)
                    P_t.append(np.where(np.isfinite(S), P, 0.0))
                    V_t.append(V)
                sv = ud.sv[b, h // (w.hq // w.hkv), : w.d]
                got = fold_rows(S_t, P_t, V_t, sv)
                want = emu[x["cu_q"][b] + qt * 128 + rows, h]
                np.testing.assert_allclose(got, want, rtol=0, atol=2e-6,
                                           err_msg=f"{name} b{b} h{h} qt{qt}")
                checked += 1
    assert checked >= 4
