"""Python binding of the C ABI (include/flattn.h), same names without the
``fl_`` prefix.  Argument marshalling only: tensors are checked for device,
dtype and layout, outputs are allocated with torch when not given, and the
pointers plus the current CUDA stream go to the library.  Every step of the
computation runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import FL_DEBUG_KEY_SPLIT, FL_DEBUG_SKIP_KV_LOAD, MASKS, SCORE_MODS, FlattnError  # noqa: F401


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, ndim: int, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _strides4(t: torch.Tensor):
    s = t.stride()
    return (ctypes.c_int64 * 4)(*[int(x) for x in s])


def _variant_desc(B, Hq, Hkv, Lq, Lk, d, dv, *, mask="none", window=None, prefix=None, doc_offsets=None,
                  doc_causal=False, score_mod="none", alibi_slopes=None, softcap=None, scale=None):
    desc = _lib.new_desc()
    desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = B, Hq, Hkv, Lq, Lk, d, dv
    desc.scale = 0.0 if scale is None else float(scale)
    if mask not in MASKS:
        raise ValueError(f"unknown mask {mask!r}")
    desc.mask_kind = MASKS[mask]
    desc.doc_causal = 1 if doc_causal else 0
    desc.window = 0 if window is None else int(window)
    desc.prefix_len = 0 if prefix is None else int(prefix)
    if score_mod not in SCORE_MODS:
        raise ValueError(f"unknown score_mod {score_mod!r}")
    desc.score_mod = SCORE_MODS[score_mod]
    desc.softcap = 0.0 if softcap is None else float(softcap)
    if alibi_slopes is not None:
        _need(alibi_slopes, "alibi_slopes", 1, torch.float32)
        desc.alibi_slopes = alibi_slopes.data_ptr()
    if doc_offsets is not None:
        _need(doc_offsets, "doc_offsets", 2, torch.int32)
        if not doc_offsets.is_contiguous():
            raise ValueError("doc_offsets must be contiguous")
        desc.doc_offsets = doc_offsets.data_ptr()
        desc.num_docs = doc_offsets.shape[1] - 1
    return desc


def attn_fwd(q, k, v, *, mask: str = "none", window: int | None = None, prefix: int | None = None,
             doc_offsets: torch.Tensor | None = None, doc_causal: bool = False,
             score_mod: str = "none", alibi_slopes: torch.Tensor | None = None,
             softcap: float | None = None, scale: float | None = None,
             out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
             return_lse: bool = True, stream=None, debug_flags: int = 0, debug_arg: int = -1,
             wait_limit_ms: int = 0):
    """fl_attn_fwd: q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] bf16 CUDA tensors (head dim
    contiguous).  Returns (out [B,Hq,Lq,d] bf16, lse [B,Hq,Lq] fp32 or None)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, 4)
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have a contiguous head dimension")
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, Hq, Lq, dv), device=q.device, dtype=torch.bfloat16)
    _need(out, "out", 4)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Lq), device=q.device, dtype=torch.float32)
    if lse is not None:
        _need(lse, "lse", 3, torch.float32)
        if not lse.is_contiguous():
            raise ValueError("lse must be contiguous")
    desc = _variant_desc(B, Hq, Hkv, Lq, Lk, d, dv, mask=mask, window=window, prefix=prefix,
                         doc_offsets=doc_offsets, doc_causal=doc_causal, score_mod=score_mod,
                         alibi_slopes=alibi_slopes, softcap=softcap, scale=scale)
    desc.q_strides, desc.k_strides = _strides4(q), _strides4(k)
    desc.v_strides, desc.o_strides = _strides4(v), _strides4(out)
    desc.stream = _stream_ptr(stream)
    desc.debug_flags, desc.debug_arg, desc.wait_limit_ms = int(debug_flags), int(debug_arg), int(wait_limit_ms)
    st = _lib.lib().fl_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                0 if lse is None else lse.data_ptr(), ctypes.byref(desc))
    _lib.check(st, "fl_attn_fwd")
    return out, lse


def diffattn_fwd(q1, k1, q2, k2, v, lam: float, *, causal: bool = True, scale: float | None = None,
                 out=None, lse=None, return_lse: bool = True, stream=None):
    """fl_diffattn_fwd: q1,k1,q2,k2 [B,H,L,64], v [B,H,L,128] contiguous bf16.
    Returns (out [B,H,L,128] bf16, lse [2,B,H,L] fp32 or None)."""
    for name, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v)):
        _need(t, name, 4)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, H, L, d = q1.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, L, dv), device=q1.device, dtype=torch.bfloat16)
    _need(out, "out", 4)
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    if lse is None and return_lse:
        lse = torch.empty((2, B, H, L), device=q1.device, dtype=torch.float32)
    desc = _lib.new_desc()
    desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = B, H, H, L, L, d, dv
    desc.scale = 0.0 if scale is None else float(scale)
    desc.mask_kind = MASKS["causal" if causal else "none"]
    desc.stream = _stream_ptr(stream)
    st = _lib.lib().fl_diffattn_fwd(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(), v.data_ptr(),
                                    out.data_ptr(), 0 if lse is None else lse.data_ptr(),
                                    ctypes.c_float(float(lam)), ctypes.byref(desc))
    _lib.check(st, "fl_diffattn_fwd")
    return out, lse


def diffattn_bwd(q1, k1, q2, k2, v, dout, lam: float, *, causal: bool = True, scale: float | None = None,
                 dq1=None, dk1=None, dq2=None, dk2=None, dv=None, workspace=None, stream=None):
    """fl_diffattn_bwd: gradients (dq1, dk1, dq2, dk2, dv) of diffattn_fwd's
    out for the output gradient dout [B,H,L,128]; contiguous bf16 tensors."""
    for name, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v), ("dout", dout)):
        _need(t, name, 4)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, H, L, d = q1.shape
    dq1 = torch.empty_like(q1) if dq1 is None else dq1
    dk1 = torch.empty_like(k1) if dk1 is None else dk1
    dq2 = torch.empty_like(q2) if dq2 is None else dq2
    dk2 = torch.empty_like(k2) if dk2 is None else dk2
    dv = torch.empty_like(v) if dv is None else dv
    desc = _lib.new_desc()
    desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = B, H, H, L, L, d, v.shape[-1]
    desc.scale = 0.0 if scale is None else float(scale)
    desc.mask_kind = MASKS["causal" if causal else "none"]
    desc.stream = _stream_ptr(stream)
    need = int(_lib.lib().fl_diffattn_bwd_workspace_size(ctypes.byref(desc)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q1.device, dtype=torch.uint8)
    st = _lib.lib().fl_diffattn_bwd(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(), v.data_ptr(),
                                    dout.data_ptr(), ctypes.c_float(float(lam)), dq1.data_ptr(), dk1.data_ptr(),
                                    dq2.data_ptr(), dk2.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                                    ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                    ctypes.byref(desc))
    _lib.check(st, "fl_diffattn_bwd")
    return dq1, dk1, dq2, dk2, dv


def evoformer_gated_attn_fwd(q, k, v, pair_bias, mask_bias, gate, *, scale: float | None = None,
                             out=None, lse=None, return_lse: bool = True, stream=None):
    """fl_evoformer_gated_attn_fwd: q,k,v,gate [B,N_seq,H,N_res,d] bf16,
    pair_bias [B,H,N_res,N_res] fp32 (or None), mask_bias [B,N_seq,N_res] fp32
    (or None).  Returns (out like q, lse [B,N_seq,H,N_res] fp32 or None)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("gate", gate)):
        _need(t, name, 5)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, Ns, H, Nr, d = q.shape
    if pair_bias is not None:
        _need(pair_bias, "pair_bias", 4, torch.float32)
        if not pair_bias.is_contiguous() or tuple(pair_bias.shape) != (B, H, Nr, Nr):
            raise ValueError("pair_bias must be contiguous [B,H,N_res,N_res]")
    if mask_bias is not None:
        _need(mask_bias, "mask_bias", 3, torch.float32)
        if not mask_bias.is_contiguous() or tuple(mask_bias.shape) != (B, Ns, Nr):
            raise ValueError("mask_bias must be contiguous [B,N_seq,N_res]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", 5)
    if lse is None and return_lse:
        lse = torch.empty((B, Ns, H, Nr), device=q.device, dtype=torch.float32)
    st = _lib.lib().fl_evoformer_gated_attn_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(),
        0 if pair_bias is None else pair_bias.data_ptr(),
        0 if mask_bias is None else mask_bias.data_ptr(),
        gate.data_ptr(), out.data_ptr(), 0 if lse is None else lse.data_ptr(),
        B, Ns, Nr, H, d, ctypes.c_float(0.0 if scale is None else float(scale)), _stream_ptr(stream))
    _lib.check(st, "fl_evoformer_gated_attn_fwd")
    return out, lse


def evoformer_col_gated_attn_fwd(q, k, v, mask_bias, gate, *, scale: float | None = None,
                                 out=None, lse=None, return_lse: bool = True, stream=None):
    """fl_evoformer_col_gated_attn_fwd: q,k,v,gate [B,N_seq,H,N_res,d] bf16,
    mask_bias [B,N_res,N_seq] fp32 (or None).  Attention over the MSA rows of
    every residue column.  Returns (out like q, lse [B,H,N_res,N_seq] fp32 or
    None)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("gate", gate)):
        _need(t, name, 5)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, Ns, H, Nr, d = q.shape
    if mask_bias is not None:
        _need(mask_bias, "mask_bias", 3, torch.float32)
        if not mask_bias.is_contiguous() or tuple(mask_bias.shape) != (B, Nr, Ns):
            raise ValueError("mask_bias must be contiguous [B,N_res,N_seq]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", 5)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nr, Ns), device=q.device, dtype=torch.float32)
    st = _lib.lib().fl_evoformer_col_gated_attn_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(),
        0 if mask_bias is None else mask_bias.data_ptr(),
        gate.data_ptr(), out.data_ptr(), 0 if lse is None else lse.data_ptr(),
        B, Ns, Nr, H, d, ctypes.c_float(0.0 if scale is None else float(scale)), _stream_ptr(stream))
    _lib.check(st, "fl_evoformer_col_gated_attn_fwd")
    return out, lse


def attn_decode_fwd(q, k_cache, v_cache, kv_len=None, *, causal: bool = False, score_mod: str = "none",
                    alibi_slopes=None, softcap: float | None = None, scale: float | None = None,
                    out=None, lse=None, return_lse: bool = True, workspace=None, stream=None):
    """fl_attn_decode_fwd: q [B,Hq,Lq,d], k_cache/v_cache [B,Hkv,Lk,d] bf16
    contiguous, kv_len int32 [B] (or None).  The key-split workspace is
    allocated with torch when not given.  Returns (out [B,Hq,Lq,d] bf16,
    lse [B,Hq,Lq] fp32 or None)."""
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, 4)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", 4)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Lq), device=q.device, dtype=torch.float32)
    if kv_len is not None:
        _need(kv_len, "kv_len", 1, torch.int32)
    desc = _lib.new_desc()
    desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = B, Hq, Hkv, Lq, Lk, d, v_cache.shape[-1]
    desc.scale = 0.0 if scale is None else float(scale)
    desc.mask_kind = MASKS["causal" if causal else "none"]
    if score_mod not in SCORE_MODS:
        raise ValueError(f"unknown score_mod {score_mod!r}")
    desc.score_mod = SCORE_MODS[score_mod]
    desc.softcap = 0.0 if softcap is None else float(softcap)
    if alibi_slopes is not None:
        _need(alibi_slopes, "alibi_slopes", 1, torch.float32)
        desc.alibi_slopes = alibi_slopes.data_ptr()
    desc.stream = _stream_ptr(stream)
    need = int(_lib.lib().fl_attn_decode_workspace_size(ctypes.byref(desc)))
    if need and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_ptr = 0 if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.lib().fl_attn_decode_fwd(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                       0 if lse is None else lse.data_ptr(),
                                       0 if kv_len is None else kv_len.data_ptr(),
                                       ws_ptr, ctypes.c_size_t(ws_bytes), ctypes.byref(desc))
    _lib.check(st, "fl_attn_decode_fwd")
    return out, lse


def attn_bwd(q, k, v, out, dout, lse, *, mask: str = "none", window: int | None = None,
             prefix: int | None = None, doc_offsets: torch.Tensor | None = None, doc_causal: bool = False,
             score_mod: str = "none", alibi_slopes: torch.Tensor | None = None, softcap: float | None = None,
             scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """fl_attn_bwd: gradients (dq, dk, dv) of attn_fwd given its out, lse and
    dout; contiguous bf16 tensors, the forward's variant arguments."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _need(t, name, 4)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _need(lse, "lse", 3, torch.float32)
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    desc = _variant_desc(B, Hq, Hkv, Lq, Lk, d, v.shape[-1], mask=mask, window=window, prefix=prefix,
                         doc_offsets=doc_offsets, doc_causal=doc_causal, score_mod=score_mod,
                         alibi_slopes=alibi_slopes, softcap=softcap, scale=scale)
    desc.stream = _stream_ptr(stream)
    need = int(_lib.lib().fl_attn_bwd_workspace_size(ctypes.byref(desc)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    st = _lib.lib().fl_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                                lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                                ctypes.c_size_t(workspace.numel() * workspace.element_size()), ctypes.byref(desc))
    _lib.check(st, "fl_attn_bwd")
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, kw):
        out, lse = attn_fwd(q, k, v, **kw)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.kw = kw
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = attn_bwd(q, k, v, out, dout.contiguous(), lse, **ctx.kw)
        return dq, dk, dv, None


def attention(q, k, v, **kw):
    """Differentiable fused attention: attn_fwd in the forward, attn_bwd in
    the backward (the variant keyword arguments of attn_fwd)."""
    return _Attention.apply(q, k, v, kw)


class _DiffAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q1, k1, q2, k2, v, lam, causal, scale):
        out, _ = diffattn_fwd(q1, k1, q2, k2, v, lam, causal=causal, scale=scale, return_lse=False)
        ctx.save_for_backward(q1, k1, q2, k2, v)
        ctx.args = (lam, causal, scale)
        return out

    @staticmethod
    def backward(ctx, dout):
        lam, causal, scale = ctx.args
        grads = diffattn_bwd(*ctx.saved_tensors, dout.contiguous(), lam, causal=causal, scale=scale)
        return (*grads, None, None, None)


def diff_attention(q1, k1, q2, k2, v, lam: float, *, causal: bool = True, scale: float | None = None):
    """Differentiable differential attention: diffattn_fwd in the forward,
    diffattn_bwd (gradients of q1, k1, q2, k2 and v) in the backward."""
    return _DiffAttention.apply(q1, k1, q2, k2, v, float(lam), causal, scale)


def sync_status(stream=None) -> int:
    """fl_sync_status: synchronise the stream and return (and clear) the
    device status word; raises FlattnError if a kernel reported a failure."""
    st = _lib.lib().fl_sync_status(_stream_ptr(stream))
    _lib.check(st, "device status")
    return st


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
