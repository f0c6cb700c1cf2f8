"""fl_attn_fwd_noalloc: the allocation-free entry point.

It exists for callers that cannot let a library call cudaMalloc (a process
whose device memory all comes from its own pre-reserved pool, code that must
not allocate while a stream is captured into a CUDA graph, callers with a
hard memory budget).  It runs the same kernel as fl_attn_fwd with the
kernel's status words in a fixed array compiled into the library.

The GPU test calls it through the C ABI twice in a row, on different inputs
and variants, and checks each output against fl_attn_fwd's on the same
inputs within the tolerance every parity test here uses.  This file is named
so that pytest collects it last; it also passes when run alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from flashattention_attn_fwd_gb300 import _lib, synth

ATOL, RTOL, LSE_ATOL = 2e-2, 1e-2, 1e-3


def _desc(B, Hq, Hkv, L, d, stream, **kw):
    desc = _lib.new_desc()
    desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = B, Hq, Hkv, L, L, d, d
    for k, v in kw.items():
        setattr(desc, k, v)
    desc.stream = stream
    return desc


def _run(fn, q, k, v, desc):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), ctypes.byref(desc))
    assert st == _lib.FL_OK, _lib.status_string(st)
    return out, lse


def test_noalloc_rejects_bad_arguments_before_any_cuda_call():
    L = _lib.lib()
    d = _desc(1, 2, 2, 128, 64, None)
    P = 0x10000
    assert L.fl_attn_fwd_noalloc(P, P, P, P, 0, None) == _lib.FL_ERR_INVALID_ARG
    assert L.fl_attn_fwd_noalloc(P, 0, P, P, 0, ctypes.byref(d)) == _lib.FL_ERR_INVALID_ARG
    assert L.fl_attn_fwd_noalloc(P, P + 8, P, P, 0, ctypes.byref(d)) == _lib.FL_ERR_ALIGNMENT
    bad = _desc(1, 2, 2, 128, 96, None)
    assert L.fl_attn_fwd_noalloc(P, P, P, P, 0, ctypes.byref(bad)) == _lib.FL_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_matches_fl_attn_fwd_on_two_calls_in_a_row():
    L = _lib.lib()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    cases = [
        (synth.attn_inputs(2, 4, 4, 300, 64, seed=71), dict(mask_kind=_lib.MASKS["causal"]), None),
        (synth.attn_inputs(1, 8, 2, 520, 64, seed=72),
         dict(score_mod=_lib.SCORE_MODS["alibi"]), synth.alibi_slopes(8)),
    ]
    for (q, k, v), kw, slopes in cases:
        q, k, v = q.to(dev), k.to(dev), v.to(dev)
        B, Hq, Lq, d = q.shape
        Hkv = k.shape[1]
        kw = dict(kw)
        if slopes is not None:
            slopes = slopes.to(dev)
            kw["alibi_slopes"] = slopes.data_ptr()
        ref_o, ref_l = _run(L.fl_attn_fwd, q, k, v, _desc(B, Hq, Hkv, Lq, d, stream, **kw))
        assert L.fl_sync_status(stream) == _lib.FL_OK
        out, lse = _run(L.fl_attn_fwd_noalloc, q, k, v, _desc(B, Hq, Hkv, Lq, d, stream, **kw))
        # query mode: all data pointers NULL -> sync and read the recorded status
        assert L.fl_attn_fwd_noalloc(0, 0, 0, 0, 0, ctypes.byref(_desc(B, Hq, Hkv, Lq, d, stream))) == _lib.FL_OK
        g, r = out.float().cpu().numpy(), ref_o.float().cpu().numpy()
        assert np.isfinite(g).all()
        mae = float(np.abs(g - r).max())
        rel = float(np.linalg.norm(g - r) / np.linalg.norm(r))
        assert mae <= ATOL and rel <= RTOL, (mae, rel)
        assert float((lse - ref_l).abs().max()) <= LSE_ATOL


@pytest.mark.gpu
def test_noalloc_matches_the_oracle():
    """The allocation-free path checked against the fp64 oracle directly."""
    L = _lib.lib()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for (B, Hq, Hkv, S, d), kw, okw in (((1, 4, 4, 300, 64), dict(mask_kind=_lib.MASKS["window"], window=90),
                                         dict(mask="window", window=90)),
                                        ((2, 8, 2, 260, 32), dict(mask_kind=_lib.MASKS["causal"]), dict(mask="causal"))):
        q, k, v = synth.attn_inputs(B, Hq, Hkv, S, d, seed=S + d)
        out, lse = _run(L.fl_attn_fwd_noalloc, q.to(dev), k.to(dev), v.to(dev), _desc(B, Hq, Hkv, S, d, stream, **kw))
        assert L.fl_attn_fwd_noalloc(0, 0, 0, 0, 0, ctypes.byref(_desc(B, Hq, Hkv, S, d, stream))) == _lib.FL_OK
        ro, rl = oracle.attention(q, k, v, **okw)
        g = out.float().cpu().numpy()
        assert np.abs(g - ro).max() <= ATOL and np.linalg.norm(g - ro) / np.linalg.norm(ro) <= RTOL
        assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_ATOL


@pytest.mark.gpu
def test_noalloc_timeout_is_recorded_in_its_own_array_and_cleared():
    """A pipeline wait that runs out (block 0 never loads one key tile, 20 ms
    limit) is recorded in the allocation-free path's own status words: the
    query reports FL_ERR_TIMEOUT once and clears it, fl_sync_status's word is
    untouched, and the next call is correct."""
    L = _lib.lib()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    q, k, v = synth.attn_inputs(1, 2, 2, 512, 64, seed=1)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    bad = _desc(1, 2, 2, 512, 64, stream, debug_flags=_lib.FL_DEBUG_SKIP_KV_LOAD, debug_arg=1, wait_limit_ms=20)
    out = torch.empty_like(qd)
    lse = torch.empty(1, 2, 512, device=dev)
    assert L.fl_attn_fwd_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                 ctypes.byref(bad)) == _lib.FL_OK
    query = _desc(1, 2, 2, 512, 64, stream)
    assert L.fl_attn_fwd_noalloc(0, 0, 0, 0, 0, ctypes.byref(query)) == _lib.FL_ERR_TIMEOUT
    assert L.fl_attn_fwd_noalloc(0, 0, 0, 0, 0, ctypes.byref(query)) == _lib.FL_OK
    assert L.fl_sync_status(stream) == _lib.FL_OK
    out, lse = _run(L.fl_attn_fwd_noalloc, qd, kd, vd, _desc(1, 2, 2, 512, 64, stream))
    assert L.fl_attn_fwd_noalloc(0, 0, 0, 0, 0, ctypes.byref(query)) == _lib.FL_OK
    ro, rl = oracle.attention(q, k, v)
    g = out.float().cpu().numpy()
    assert np.abs(g - ro).max() <= ATOL and np.linalg.norm(g - ro) / np.linalg.norm(ro) <= RTOL
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_ATOL
