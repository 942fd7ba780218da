"""GB300-native SageAttention2 quantized exact-attention forward.

Thin Python binding over the C ABI in ``include/sage2_attn.h`` (library
``libsage2_attn.so``, built in-tree for sm_103a). The functions here only check
and marshal arguments -- torch tensors give device pointers and the current
stream -- and every step of the computation runs in the library's kernels. There
is no CPU path: without the built library (or without an sm_103 GPU) every call
raises.

Shapes follow the library: dense ``q [B, Nq, Hq, D]``, ``k, v [B, Nkv, Hkv, D]``;
varlen packed ``[total, H, D]`` with int32 ``cu_seqlens`` on the device.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import BF16, FP16, FP32, Sage2Error, WsLayout  # noqa: F401

__all__ = ["attn_fwd", "attn_fwd_varlen", "prepass", "attention", "prepass_varlen",
           "attention_varlen", "workspace_size", "workspace_layout", "device_status",
           "alloc_workspace", "debug_tile", "debug_timeout", "Sage2Error", "load_library",
           "attn_fwd_noalloc", "noalloc_status", "NOALLOC_SCRATCH_BYTES", "quant_flags",
           "QUANT_NO_SMOOTH_Q", "QUANT_NO_SMOOTH_K", "QUANT_PER_BLOCK", "QUANT_SAGE1",
           "attn_fwd_host", "host_scratch_size", "host_status"]

_DT = {torch.float16: FP16, torch.bfloat16: BF16, torch.float32: FP32}
NOALLOC_SCRATCH_BYTES = 64 << 20  # SAGE2_NOALLOC_SCRATCH_BYTES in include/sage2_attn.h
# sage2_quant_flags in include/sage2_attn.h: accuracy ablations (0 is the method), and the
# SageAttention (v1) path: INT8 per-block Q and K codes, K smoothed, Q not
QUANT_NO_SMOOTH_Q, QUANT_NO_SMOOTH_K, QUANT_PER_BLOCK, QUANT_SAGE1 = 1, 2, 4, 8


def quant_flags(smooth_q: bool = True, smooth_k: bool = True, per_block: bool = False) -> int:
    """The sage2_quant_flags word for one ablation setting (all defaults: the method)."""
    return ((0 if smooth_q else QUANT_NO_SMOOTH_Q) | (0 if smooth_k else QUANT_NO_SMOOTH_K)
            | (QUANT_PER_BLOCK if per_block else 0))


def load_library():
    """Loads (building first if needed) and returns the ctypes library handle."""
    return _lib.lib()


def _code(dtype: torch.dtype) -> int:
    if dtype not in _DT:
        raise TypeError(f"unsupported dtype {dtype}")
    return _DT[dtype]


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(B, Hq, Hkv, max_nq, max_nkv, D, total_q=None, total_kv=None,
                   quant_flags=0) -> int:
    total_q = B * max_nq if total_q is None else total_q
    total_kv = B * max_nkv if total_kv is None else total_kv
    if quant_flags:
        n = _lib.lib().sage2_workspace_size_ex(B, Hq, Hkv, max_nq, max_nkv, D, total_q, total_kv,
                                               int(quant_flags))
    else:
        n = _lib.lib().sage2_workspace_size(B, Hq, Hkv, max_nq, max_nkv, D, total_q, total_kv)
    if n == 0:
        raise Sage2Error(_lib.EINVAL, "sage2_workspace_size")
    return int(n)


def workspace_layout(B, Hq, Hkv, max_nq, max_nkv, D, total_q=None, total_kv=None,
                     quant_flags=0) -> WsLayout:
    total_q = B * max_nq if total_q is None else total_q
    total_kv = B * max_nkv if total_kv is None else total_kv
    L = WsLayout()
    _lib.check(_lib.lib().sage2_workspace_layout_ex(B, Hq, Hkv, max_nq, max_nkv, D, total_q,
                                                    total_kv, int(quant_flags), ctypes.byref(L)),
               "sage2_workspace_layout_ex")
    return L


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def _ws(workspace, nbytes, device):
    if workspace is None:
        workspace = alloc_workspace(nbytes, device)
    _dev(workspace, "workspace")
    if workspace.numel() * workspace.element_size() < nbytes:
        raise Sage2Error(_lib.EWORKSPACE, "workspace")
    return workspace


def _out(out, shape, dtype, device):
    if out is None:
        out = torch.empty(shape, dtype=dtype, device=device)
    _dev(out, "out")
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {tuple(shape)}")
    return out


def attn_fwd(q, k, v, causal=False, sm_scale=0.0, out=None, out_dtype=None, workspace=None,
             stream=None, quant_flags=0):
    """softmax(Q K^T * sm_scale) V the SageAttention2 way; q [B, Nq, Hq, D], k/v [B, Nkv, Hkv, D].

    ``quant_flags`` (see :func:`quant_flags`) selects an accuracy ablation; it runs the packed
    prepass with those switches, then the same attention kernel."""
    if quant_flags:
        B, Nq, Hq, D = q.shape
        _, Nkv, Hkv, _ = k.shape
        dev = q.device
        cu_q = torch.arange(0, (B + 1) * Nq, Nq, dtype=torch.int32, device=dev)
        cu_kv = torch.arange(0, (B + 1) * Nkv, Nkv, dtype=torch.int32, device=dev)
        o = attn_fwd_varlen(q.reshape(B * Nq, Hq, D), k.reshape(B * Nkv, Hkv, D),
                            v.reshape(B * Nkv, Hkv, D), cu_q, cu_kv, Nq, Nkv, causal=causal,
                            sm_scale=sm_scale, out=None if out is None else out.view(B * Nq, Hq, D),
                            out_dtype=out_dtype, workspace=workspace, stream=stream,
                            quant_flags=quant_flags)
        return o.view(B, Nq, Hq, D)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev(t, n)
    B, Nq, Hq, D = q.shape
    _, Nkv, Hkv, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes/dtypes disagree")
    odt = q.dtype if out_dtype is None else out_dtype
    out = _out(out, (B, Nq, Hq, D), odt, q.device)
    ws = _ws(workspace, workspace_size(B, Hq, Hkv, Nq, Nkv, D), q.device)
    _lib.check(_lib.lib().sage2_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _code(q.dtype), _code(out.dtype), B, Hq, Hkv, Nq,
        Nkv, D, int(bool(causal)), float(sm_scale), _ptr(ws), ws.numel(), _stream(stream)),
        "sage2_attn_fwd")
    return out


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_nq, max_nkv, causal=False,
                    sm_scale=0.0, out=None, out_dtype=None, workspace=None, stream=None,
                    quant_flags=0):
    """Packed variable-length form: q [total_q, Hq, D], k/v [total_kv, Hkv, D], cu_seqlens int32 (B+1).

    Nonzero ``quant_flags`` runs :func:`prepass_varlen` with those switches, then
    :func:`attention_varlen`, on one workspace."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cu_seqlens_q, "cu_seqlens_q"),
                 (cu_seqlens_kv, "cu_seqlens_kv")):
        _dev(t, n)
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_kv.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    total_q, Hq, D = q.shape
    total_kv, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    odt = q.dtype if out_dtype is None else out_dtype
    out = _out(out, (total_q, Hq, D), odt, q.device)
    ws = _ws(workspace, workspace_size(B, Hq, Hkv, max_nq, max_nkv, D, total_q, total_kv,
                                       quant_flags), q.device)
    if quant_flags:
        prepass_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_nq, max_nkv, ws, causal=causal,
                       sm_scale=sm_scale, stream=stream, quant_flags=quant_flags)
        attention_varlen(out, ws, cu_seqlens_q, cu_seqlens_kv, Hkv, max_nq, max_nkv, total_kv,
                         causal=causal, sm_scale=sm_scale, stream=stream, quant_flags=quant_flags)
        return out
    _lib.check(_lib.lib().sage2_attn_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _code(q.dtype), _code(out.dtype),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B, Hq, Hkv, max_nq, max_nkv, total_q, total_kv,
        D, int(bool(causal)), float(sm_scale), _ptr(ws), ws.numel(), _stream(stream)),
        "sage2_attn_fwd_varlen")
    return out


def prepass(q, k, v, workspace, causal=False, sm_scale=0.0, stream=None):
    B, Nq, Hq, D = q.shape
    _, Nkv, Hkv, _ = k.shape
    _lib.check(_lib.lib().sage2_prepass(
        _ptr(q), _ptr(k), _ptr(v), _code(q.dtype), B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)),
        float(sm_scale), _ptr(workspace), workspace.numel(), _stream(stream)), "sage2_prepass")


def attention(out, workspace, B, Hq, Hkv, Nq, Nkv, D, causal=False, sm_scale=0.0, stream=None):
    _lib.check(_lib.lib().sage2_attention(
        _ptr(out), _code(out.dtype), B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), float(sm_scale),
        _ptr(workspace), workspace.numel(), _stream(stream)), "sage2_attention")


def prepass_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_nq, max_nkv, workspace,
                   causal=False, sm_scale=0.0, stream=None, quant_flags=0):
    total_q, Hq, D = q.shape
    total_kv, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    if quant_flags:
        _lib.check(_lib.lib().sage2_prepass_varlen_ex(
            _ptr(q), _ptr(k), _ptr(v), _code(q.dtype), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B,
            Hq, Hkv, max_nq, max_nkv, total_q, total_kv, D, int(bool(causal)), float(sm_scale),
            int(quant_flags), _ptr(workspace), workspace.numel(), _stream(stream)),
            "sage2_prepass_varlen_ex")
        return
    _lib.check(_lib.lib().sage2_prepass_varlen(
        _ptr(q), _ptr(k), _ptr(v), _code(q.dtype), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B, Hq,
        Hkv, max_nq, max_nkv, total_q, total_kv, D, int(bool(causal)), float(sm_scale),
        _ptr(workspace), workspace.numel(), _stream(stream)), "sage2_prepass_varlen")


def attention_varlen(out, workspace, cu_seqlens_q, cu_seqlens_kv, Hkv, max_nq, max_nkv,
                     total_kv, causal=False, sm_scale=0.0, stream=None, quant_flags=0):
    total_q, Hq, D = out.shape
    B = cu_seqlens_q.numel() - 1
    if quant_flags:
        _lib.check(_lib.lib().sage2_attention_varlen_ex(
            _ptr(out), _code(out.dtype), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B, Hq, Hkv,
            max_nq, max_nkv, total_q, total_kv, D, int(bool(causal)), float(sm_scale),
            int(quant_flags), _ptr(workspace), workspace.numel(), _stream(stream)),
            "sage2_attention_varlen_ex")
        return
    _lib.check(_lib.lib().sage2_attention_varlen(
        _ptr(out), _code(out.dtype), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B, Hq, Hkv, max_nq,
        max_nkv, total_q, total_kv, D, int(bool(causal)), float(sm_scale), _ptr(workspace),
        workspace.numel(), _stream(stream)), "sage2_attention_varlen")


def device_status(workspace, stream=None) -> tuple[int, int]:
    """(status code, raw status word) after synchronizing the stream."""
    raw = ctypes.c_int(0)
    rc = _lib.lib().sage2_device_status(_ptr(workspace), _stream(stream), ctypes.byref(raw))
    return int(rc), int(raw.value)


def debug_tile(workspace, B, Hq, Hkv, max_nq, max_nkv, D, causal, b, h, qt, kt, sm_scale=0.0,
               cu_seqlens_q=None, cu_seqlens_kv=None, total_q=None, total_kv=None, stream=None,
               quant_flags=0):
    """Raw (S accumulators, P~ bytes, fresh P~V partial) of one KV tile of one work unit. On
    the two-tile kernel (INT4 codes) the partial is returned for kt = 0 only (zeros otherwise);
    see sage2_debug_tile in include/sage2_attn.h."""
    dev = workspace.device
    Dp = 64 if D <= 64 else 128
    s_out = torch.zeros(128, 128, dtype=torch.float32, device=dev)
    p_out = torch.zeros(128, 128, dtype=torch.uint8, device=dev)
    r_out = torch.zeros(128, Dp, dtype=torch.float32, device=dev)
    total_q = B * max_nq if total_q is None else total_q
    total_kv = B * max_nkv if total_kv is None else total_kv
    _lib.check(_lib.lib().sage2_debug_tile_ex(
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B, Hq, Hkv, max_nq, max_nkv, total_q, total_kv,
        D, int(bool(causal)), float(sm_scale), int(quant_flags), _ptr(workspace),
        workspace.numel(), b, h, qt, kt, _ptr(s_out), _ptr(p_out), _ptr(r_out), _stream(stream)),
        "sage2_debug_tile_ex")
    return s_out, p_out, r_out


def debug_timeout(workspace, B, Hq, Hkv, Nq, Nkv, D, stream=None):
    _lib.check(_lib.lib().sage2_debug_timeout(B, Hq, Hkv, Nq, Nkv, D, _ptr(workspace),
                                              workspace.numel(), _stream(stream)),
               "sage2_debug_timeout")


def host_scratch_size(B, Hq, Hkv, Nq, Nkv, D, out_dtype, kv_heads_per_chunk, quant_flags=0):
    n = _lib.lib().sage2_host_scratch_size(B, Hq, Hkv, Nq, Nkv, D, _code(out_dtype),
                                           int(kv_heads_per_chunk), int(quant_flags))
    if n == 0:
        raise Sage2Error(_lib.EINVAL, "sage2_host_scratch_size")
    return int(n)


def attn_fwd_host(q, k, v, out, causal=False, sm_scale=0.0, quant_flags=0, kv_heads_per_chunk=1,
                  scratch=None, stream=None):
    """The forward from host memory: q [B, Nq, Hq, D], k/v [B, Nkv, Hkv, D] and out
    [B, Nq, Hq, D] are CPU tensors (pinned for the transfers to overlap the computation);
    `scratch` a CUDA uint8 tensor of host_scratch_size(...) bytes (allocated if None). Runs in
    chunks of kv_heads_per_chunk kv heads with copies in, computation and copies out overlapped;
    the result equals attn_fwd on the whole problem. Returns the scratch tensor (for
    host_status)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    B, Nq, Hq, D = q.shape
    _, Nkv, Hkv, _ = k.shape
    if k.shape != v.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes/dtypes disagree")
    if tuple(out.shape) != (B, Nq, Hq, D):
        raise ValueError("out shape")
    n = host_scratch_size(B, Hq, Hkv, Nq, Nkv, D, out.dtype, kv_heads_per_chunk, quant_flags)
    if scratch is None:
        scratch = alloc_workspace(n)
    _dev(scratch, "scratch")
    _lib.check(_lib.lib().sage2_attn_fwd_host(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), _code(q.dtype),
        _code(out.dtype), B, Hq, Hkv, Nq, Nkv, D, int(bool(causal)), float(sm_scale),
        int(quant_flags), int(kv_heads_per_chunk), _ptr(scratch), scratch.numel(),
        _stream(stream)), "sage2_attn_fwd_host")
    return scratch


def host_status(scratch, stream=None) -> tuple[int, int]:
    """(status code, raw word) of the chunks of the last attn_fwd_host call on `scratch`."""
    raw = ctypes.c_int(0)
    rc = _lib.lib().sage2_host_status(_ptr(scratch), _stream(stream), ctypes.byref(raw))
    return int(rc), int(raw.value)


def attn_fwd_noalloc(q, k, v, out, causal=False, sm_scale=0.0, stream=None):
    """Forward that allocates no device memory, for callers that cannot allocate (engines
    whose runtime owns every device allocation, allocation-free latency-critical loops).
    Uses the library's built-in scratch (NOALLOC_SCRATCH_BYTES per GPU, held until exit)
    instead of a workspace; ``out`` must be provided. Calls share that scratch, so calls that
    overlap on the GPU race; keep them ordered."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _dev(t, n)
    B, Nq, Hq, D = q.shape
    _, Nkv, Hkv, _ = k.shape
    _lib.check(_lib.lib().sage2_attn_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _code(q.dtype), _code(out.dtype), B, Hq, Hkv, Nq,
        Nkv, D, int(bool(causal)), float(sm_scale), _stream(stream)), "sage2_attn_fwd_noalloc")
    return out


def noalloc_status(stream=None) -> tuple[int, int]:
    """(status code, raw word) of the last attn_fwd_noalloc call on the current device."""
    raw = ctypes.c_int(0)
    rc = _lib.lib().sage2_noalloc_status(_stream(stream), ctypes.byref(raw))
    return int(rc), int(raw.value)
