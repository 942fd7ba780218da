"""CPU oracle for the SageAttention2 quantized attention forward (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library
and never imports it.

The arithmetic lives in ``sage2_oracle.c`` (plain C + OpenMP, built here with
gcc). This module only builds that file, marshals numpy arrays into it and
returns numpy arrays. See the C file's header for the pages each step follows.

Conventions: inputs are the raw 16-bit patterns of fp16/bf16 tensors as
``np.uint16`` arrays, token-major and packed over the batch
(``[total_tokens, heads, D0]``); ``cu_q``/``cu_kv`` are host int32 prefix sums
of the per-sequence lengths (``B + 1`` entries).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sage2_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsage2_oracle.so")

F16, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA involved). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i, f, sz = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_round_output.argtypes = [P, sz, i, P]
        lib.oracle_num_threads.restype = i
        lib.oracle_attention_exact.argtypes = [P, P, P, i, i, P, P, i, i, i, i, f, i, P, i, P]
        lib.oracle_kv_stats.argtypes = [P, P, i, i, P, i, i, i, P, P]
        lib.oracle_quant_q.argtypes = [P, i, i, P, i, i, i, i, i, i, i, P, P, P]
        lib.oracle_quant_k.argtypes = [P, i, i, P, i, i, i, i, P, i, P, P]
        lib.oracle_quant_v.argtypes = [P, i, i, P, i, i, i, P, P, P]
        lib.oracle_delta_s.argtypes = [P, i, P, i, i, i, i, i, P, P, P]
        lib.oracle_attention_emulated.argtypes = [P, P, P, i, i, P, P, i, i, i, i, i, f, i, i, i,
                                                  i, i, i, i, i, P, i, P, i, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    assert a.dtype == np.uint16, a.dtype
    return a


def _cu(cu) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int32))


def padded_dim(D0: int) -> int:
    """Head dim the method computes in: 64 for D0 <= 64, 128 for D0 <= 128."""
    if D0 <= 64:
        return 64
    if D0 <= 128:
        return 128
    raise ValueError("head dim above 128 is not supported")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- formats
def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_f16_to_f64(int(b)) for b in np.ravel(bits)]).reshape(np.shape(bits))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_bf16_to_f64(int(b)) for b in np.ravel(bits)]).reshape(np.shape(bits))


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ravel(np.asarray(x, dtype=np.float64))
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ravel(np.asarray(c, dtype=np.uint8))
    return np.array([lib.oracle_e4m3_decode(int(v)) for v in flat]).reshape(np.shape(c))


def round_output(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round FP64 values to fp16/bf16 (nearest-even); returns the uint16 bit patterns."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_round_output(_ptr(a), a.size, dtype, _ptr(out))
    return out


# ---------------------------------------------------------------- Mode E
def _units(units) -> tuple[np.ndarray | None, int]:
    if units is None:
        return None, -1
    u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 3))
    return u, len(u)


def attention_exact(q, k, v, dtype, cu_q, cu_kv, Hq, Hkv, D0, causal, sm_scale=0.0,
                    units=None, bq=128, out=None) -> np.ndarray:
    """FP64 softmax(Q K^T * sm_scale) V. Rows outside ``units`` are left as in ``out``."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cq, ck = _cu(cu_q), _cu(cu_kv)
    B = len(cq) - 1
    if out is None:
        out = np.zeros((int(cq[-1]), Hq, D0), dtype=np.float64)
    u, nu = _units(units)
    _load().oracle_attention_exact(_ptr(q), _ptr(k), _ptr(v), dtype, B, _ptr(cq), _ptr(ck), Hq, Hkv,
                                   D0, int(bool(causal)), float(sm_scale), bq, _ptr(u), nu, _ptr(out))
    return out


# ---------------------------------------------------------------- Mode Q steps
def kv_stats(k, v, dtype, cu_kv, Hkv, D0):
    k, v = _u16(k), _u16(v)
    ck = _cu(cu_kv)
    B, Dp = len(ck) - 1, padded_dim(D0)
    kmean = np.zeros((B, Hkv, Dp), np.float32)
    vamax = np.zeros((B, Hkv, Dp), np.float32)
    _load().oracle_kv_stats(_ptr(k), _ptr(v), dtype, B, _ptr(ck), Hkv, D0, Dp, _ptr(kmean), _ptr(vamax))
    return kmean, vamax


def _qmax(qk_bits: int) -> int:
    if qk_bits not in (4, 8):
        raise ValueError("qk_bits is 4 (the INT4 grid) or 8 (the INT8 grid)")
    return (1 << (qk_bits - 1)) - 1


def quant_q(q, dtype, cu_q, Hq, D0, bq=128, smooth_q=True, per_block=False, qk_bits=4):
    q = _u16(q)
    cq = _cu(cu_q)
    B, Dp = len(cq) - 1, padded_dim(D0)
    nqb = max(1, (int(np.max(np.diff(cq))) + bq - 1) // bq) if B else 1
    qmean = np.zeros((B, Hq, nqb, Dp), np.float32)
    codes = np.zeros((int(cq[-1]), Hq, Dp), np.int8)
    sq = np.zeros((int(cq[-1]), Hq), np.float32)
    _load().oracle_quant_q(_ptr(q), dtype, B, _ptr(cq), Hq, D0, Dp, bq, int(bool(smooth_q)),
                           int(bool(per_block)), _qmax(qk_bits), _ptr(qmean), _ptr(codes),
                           _ptr(sq))
    return qmean, codes, sq


def quant_k(k, dtype, cu_kv, Hkv, D0, kmean=None, gk=32, qk_bits=4):
    k = _u16(k)
    ck = _cu(cu_kv)
    B, Dp = len(ck) - 1, padded_dim(D0)
    codes = np.zeros((int(ck[-1]), Hkv, Dp), np.int8)
    sk = np.zeros((int(ck[-1]), Hkv), np.float32)
    km = None if kmean is None else np.ascontiguousarray(kmean, dtype=np.float32)
    _load().oracle_quant_k(_ptr(k), dtype, B, _ptr(ck), Hkv, D0, Dp, gk, _ptr(km), _qmax(qk_bits),
                           _ptr(codes), _ptr(sk))
    return codes, sk


def quant_v(v, dtype, cu_kv, Hkv, D0, vamax):
    v = _u16(v)
    ck = _cu(cu_kv)
    B, Dp = len(ck) - 1, padded_dim(D0)
    codes = np.zeros((int(ck[-1]), Hkv, Dp), np.uint8)
    sv = np.zeros((B, Hkv, Dp), np.float32)
    va = np.ascontiguousarray(vamax, dtype=np.float32)
    _load().oracle_quant_v(_ptr(v), dtype, B, _ptr(ck), Hkv, D0, Dp, _ptr(va), _ptr(codes), _ptr(sv))
    return codes, sv


def delta_s(k, dtype, cu_kv, b, Hkv, hk, D0, kmean, qbar):
    """Delta-S = qbar . fl32(K - kmean) for every key of sequence b, kv head hk: the FP64 dot
    product of the FP32 operands rounded once to FP32."""
    k = _u16(k)
    ck = _cu(cu_kv)
    Dp = padded_dim(D0)
    n = int(ck[b + 1] - ck[b])
    out = np.zeros(max(n, 1), np.float32)
    km = None if kmean is None else np.ascontiguousarray(kmean, dtype=np.float32)
    qb = np.ascontiguousarray(qbar, dtype=np.float32)
    assert qb.size >= Dp
    _load().oracle_delta_s(_ptr(k), dtype, _ptr(ck), b, Hkv, hk, D0, Dp, _ptr(km), _ptr(qb), _ptr(out))
    return out[:n]


# ---------------------------------------------------------------- Mode Q
def attention_emulated(q, k, v, dtype, cu_q, cu_kv, Hq, Hkv, D0, causal, sm_scale=0.0,
                       units=None, bq=128, bkv=128, gk=32, smooth_q=True, smooth_k=True,
                       per_block=False, acc_bits=0, qk_bits=4, out=None) -> np.ndarray:
    """The full quantized pipeline (FP64 result before output rounding).

    Ablations (the defaults are the method): ``smooth_q`` / ``smooth_k`` off skip the Q block
    mean / K channel mean; ``per_block`` gives Q one scale per block of ``bq`` rows and K one
    per block of ``bkv`` keys instead of the per-thread scales; ``acc_bits > 0`` swaps the
    two-level P~V fold for one-level accumulation in an ``acc_bits``-bit significand;
    ``qk_bits=8`` puts the Q and K codes on the INT8 grid [-127, 127] (with ``smooth_q=False,
    per_block=True``: the SageAttention (v1) path, see ``SAGE1``)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cq, ck = _cu(cu_q), _cu(cu_kv)
    B = len(cq) - 1
    if out is None:
        out = np.zeros((int(cq[-1]), Hq, D0), dtype=np.float64)
    u, nu = _units(units)
    _load().oracle_attention_emulated(
        _ptr(q), _ptr(k), _ptr(v), dtype, B, _ptr(cq), _ptr(ck), Hq, Hkv, D0, padded_dim(D0),
        int(bool(causal)), float(sm_scale), bq, bkv, bkv if per_block else gk,
        int(bool(smooth_q)), int(bool(smooth_k)), int(bool(per_block)), _qmax(qk_bits),
        int(acc_bits), _ptr(u), nu, _ptr(out), 0, None)
    return out


# The SageAttention (v1) path as a set of switches of the same emulation: INT8 per-block Q and
# K codes, K smoothed, Q not smoothed (so no Delta-S), P~ and V as in the method.
SAGE1 = dict(qk_bits=8, per_block=True, smooth_q=False)


def emulated_tile_p448(q, k, v, dtype, cu_q, cu_kv, Hq, Hkv, D0, causal, b, h, qb, kt,
                       sm_scale=0.0, bq=128, bkv=128, gk=32, smooth_q=True, smooth_k=True,
                       per_block=False, qk_bits=4) -> np.ndarray:
    """The fl32 P448 = 448 * 2^(S' - m_new) of KV tile kt of unit (b, h, qb), as the Mode-Q
    emulation computes it on the way to its output: [bq][bkv], 0 where a key is not visible
    (rows past the sequence end stay 0). The e4m3 code of P~ is oracle.e4m3_encode of it."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cq, ck = _cu(cu_q), _cu(cu_kv)
    B = len(cq) - 1
    out = np.zeros((int(cq[-1]), Hq, D0), dtype=np.float64)
    dump = np.zeros((bq, bkv), np.float32)
    u, nu = _units([(b, h, qb)])
    _load().oracle_attention_emulated(
        _ptr(q), _ptr(k), _ptr(v), dtype, B, _ptr(cq), _ptr(ck), Hq, Hkv, D0, padded_dim(D0),
        int(bool(causal)), float(sm_scale), bq, bkv, bkv if per_block else gk,
        int(bool(smooth_q)), int(bool(smooth_k)), int(bool(per_block)), _qmax(qk_bits), 0,
        _ptr(u), nu, _ptr(out), int(kt), _ptr(dump))
    return dump
