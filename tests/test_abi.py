"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/flattn.h declares, agrees with the binding on the descriptor layout,
and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

from flashattention_attn_fwd_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flattn.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_lib.LIB_PATH):
        from flashattention_attn_fwd_gb300.build import build
        build()
    return _lib.lib()


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"FL_API\s+[\w\s\*]+?\b(fl_\w+)\s*\(", txt)))


def test_header_declarations_match_binding():
    assert _declared() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
    assert L.fl_abi_version() == 1
    assert L.fl_attn_desc_size() == ctypes.sizeof(_lib.AttnDesc)


def test_status_strings(L):
    for code in range(7):
        s = _lib.status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert _lib.status_string(99) == "unknown status"


def _desc(**kw):
    d = _lib.new_desc()
    base = dict(B=1, Hq=2, Hkv=2, Lq=128, Lk=128, d=64, dv=64)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


P = 0x10000  # a 16-byte aligned fake device address; never dereferenced


def _attn(L, desc, q=P, k=P, v=P, o=P, lse=0):
    return L.fl_attn_fwd(q, k, v, o, lse, ctypes.byref(desc))


@pytest.mark.parametrize("kw,expect", [
    (dict(B=0), _lib.FL_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), _lib.FL_ERR_INVALID_ARG),
    (dict(Lq=0), _lib.FL_ERR_INVALID_ARG),
    (dict(d=96, dv=96), _lib.FL_ERR_UNSUPPORTED),
    (dict(dv=96), _lib.FL_ERR_UNSUPPORTED),
    (dict(dv=256), _lib.FL_ERR_UNSUPPORTED),
    (dict(mask_kind=9), _lib.FL_ERR_INVALID_ARG),
    (dict(mask_kind=1, Lk=64), _lib.FL_ERR_UNSUPPORTED),
    (dict(mask_kind=2, window=0), _lib.FL_ERR_INVALID_ARG),
    (dict(mask_kind=3, prefix_len=-1), _lib.FL_ERR_INVALID_ARG),
    (dict(mask_kind=4, num_docs=2), _lib.FL_ERR_INVALID_ARG),       # no offsets
    (dict(score_mod=1), _lib.FL_ERR_INVALID_ARG),                   # no slopes
    (dict(score_mod=2, softcap=0.0), _lib.FL_ERR_INVALID_ARG),
    (dict(score_mod=2, softcap=float("inf")), _lib.FL_ERR_INVALID_ARG),
    (dict(score_mod=7), _lib.FL_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.FL_ERR_INVALID_ARG),
])
def test_attn_rejects_bad_descriptor(L, kw, expect):
    assert _attn(L, _desc(**kw)) == expect


def test_attn_rejects_null_and_misaligned(L):
    d = _desc()
    assert _attn(L, d, q=0) == _lib.FL_ERR_INVALID_ARG
    assert _attn(L, d, o=0) == _lib.FL_ERR_INVALID_ARG
    assert L.fl_attn_fwd(P, P, P, P, 0, None) == _lib.FL_ERR_INVALID_ARG
    assert _attn(L, d, k=P + 8) == _lib.FL_ERR_ALIGNMENT
    assert _attn(L, d, lse=P + 2) == _lib.FL_ERR_ALIGNMENT
    d2 = _desc()
    d2.q_strides = (ctypes.c_int64 * 4)(2 * 128 * 68, 128 * 68, 68, 1)  # row stride 136 bytes
    assert _attn(L, d2) == _lib.FL_ERR_ALIGNMENT
    d3 = _desc()
    d3.q_strides = (ctypes.c_int64 * 4)(1, 1, 64, 2)  # channel stride must be 1
    assert _attn(L, d3) == _lib.FL_ERR_INVALID_ARG


def test_diffattn_rejects(L):
    d = _desc(d=64, dv=128)
    f = L.fl_diffattn_fwd
    assert f(P, P, P, P, P, P, 0, ctypes.c_float(float("nan")), ctypes.byref(d)) == _lib.FL_ERR_INVALID_ARG
    assert f(P, 0, P, P, P, P, 0, ctypes.c_float(0.8), ctypes.byref(d)) == _lib.FL_ERR_INVALID_ARG
    bad = _desc(d=64, dv=64)
    assert f(P, P, P, P, P, P, 0, ctypes.c_float(0.8), ctypes.byref(bad)) == _lib.FL_ERR_UNSUPPORTED
    win = _desc(d=64, dv=128, mask_kind=2, window=4)
    assert f(P, P, P, P, P, P, 0, ctypes.c_float(0.8), ctypes.byref(win)) == _lib.FL_ERR_UNSUPPORTED
    gqa = _desc(d=64, dv=128, Hq=4, Hkv=2)
    assert f(P, P, P, P, P, P, 0, ctypes.c_float(0.8), ctypes.byref(gqa)) == _lib.FL_ERR_INVALID_ARG
    assert f(P, P, P, P, P + 4, P, 0, ctypes.c_float(0.8), ctypes.byref(d)) == _lib.FL_ERR_ALIGNMENT


def test_evoformer_rejects(L):
    f = L.fl_evoformer_gated_attn_fwd
    s = ctypes.c_float(0.0)
    assert f(P, P, P, P, P, 0, P, 0, 1, 4, 256, 8, 32, s, None) == _lib.FL_ERR_INVALID_ARG  # no gate
    assert f(P, P, P, P, P, P, P, 0, 1, 4, 256, 8, 48, s, None) == _lib.FL_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, P, P, 0, 0, 4, 256, 8, 32, s, None) == _lib.FL_ERR_INVALID_ARG
    assert f(P, P, P, P + 4, P, P, P, 0, 1, 4, 256, 8, 32, s, None) == _lib.FL_ERR_ALIGNMENT
    assert f(P, P, P, P, P, P, P, 0, 1, 4, 250, 8, 32, s, None) == _lib.FL_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, P, P, 0, 1, 4, 256, 8, 32, ctypes.c_float(float("inf")), None) == _lib.FL_ERR_INVALID_ARG
    assert f(P, P, P, P, P, P, P, 0, 1, 4, 256, 8, 64, s, None) == _lib.FL_ERR_UNSUPPORTED  # row-wise: d = 32


def test_evoformer_col_rejects(L):
    f = L.fl_evoformer_col_gated_attn_fwd
    s = ctypes.c_float(0.0)
    assert f(P, P, P, P, 0, P, 0, 1, 128, 256, 8, 32, s, None) == _lib.FL_ERR_INVALID_ARG  # no gate
    assert f(P, P, P, P, P, P, 0, 1, 128, 256, 8, 48, s, None) == _lib.FL_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, P, 0, 1, 0, 256, 8, 32, s, None) == _lib.FL_ERR_INVALID_ARG
    assert f(P, P, P, P + 4, P, P, 0, 1, 128, 256, 8, 32, s, None) == _lib.FL_ERR_ALIGNMENT
    assert f(P, P, P, P, P, P, 0, 1, 126, 256, 8, 32, s, None) == _lib.FL_ERR_UNSUPPORTED  # N_seq % 4 with a mask
    assert f(P, P, P, P, P, P, P + 2, 1, 128, 256, 8, 32, s, None) == _lib.FL_ERR_ALIGNMENT


def test_decode_rejects(L):
    f = L.fl_attn_decode_fwd
    def dd(**kw):
        base = dict(B=2, Hq=8, Hkv=2, Lq=1, Lk=4096, d=64, dv=64)
        base.update(kw)
        return _desc(**base)
    z = ctypes.c_size_t(0)
    assert f(P, P, P, P, 0, 0, 0, z, None) == _lib.FL_ERR_INVALID_ARG
    assert f(P, 0, P, P, 0, 0, 0, z, ctypes.byref(dd())) == _lib.FL_ERR_INVALID_ARG
    assert f(P, P, P, P, 0, 0, 0, z, ctypes.byref(dd(d=32, dv=32))) == _lib.FL_ERR_UNSUPPORTED
    assert f(P, P, P, P, 0, 0, 0, z, ctypes.byref(dd(dv=128))) == _lib.FL_ERR_UNSUPPORTED
    assert f(P, P, P, P, 0, 0, 0, z, ctypes.byref(dd(Hq=64, Hkv=1, Lq=2))) == _lib.FL_ERR_UNSUPPORTED  # 128 rows
    assert f(P, P, P, P, 0, 0, 0, z, ctypes.byref(dd(mask_kind=2, window=8))) == _lib.FL_ERR_UNSUPPORTED
    assert f(P, P, P, P, 0, 0, 0, z, ctypes.byref(dd(Lq=8, Lk=4))) == _lib.FL_ERR_INVALID_ARG
    assert f(P, P, P + 8, P, 0, 0, 0, z, ctypes.byref(dd())) == _lib.FL_ERR_ALIGNMENT
    assert f(P, P, P, P, 0, P + 2, 0, z, ctypes.byref(dd())) == _lib.FL_ERR_ALIGNMENT
    assert f(P, P, P, P, 0, 0, 0, z, ctypes.byref(dd(score_mod=1))) == _lib.FL_ERR_INVALID_ARG


def test_bwd_rejects(L):
    """fl_attn_bwd's argument checks, all of which return before any CUDA
    call; d = dv in {32, 64, 128} and (d, dv) = (64, 128) pass the dimension
    check and are stopped here only by the workspace size."""
    f = L.fl_attn_bwd
    ws = L.fl_attn_bwd_workspace_size

    def call(desc, ptr=P, nbytes=None, **over):
        args = dict(q=P, k=P, v=P, out=P, dout=P, lse=P, dq=P, dk=P, dv=P, workspace=P)
        args.update(over)
        n = ws(ctypes.byref(desc)) if nbytes is None else nbytes
        return f(*args.values(), ctypes.c_size_t(n), ctypes.byref(desc))

    assert f(P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t(1 << 30), None) == _lib.FL_ERR_INVALID_ARG
    assert call(_desc(), lse=0) == _lib.FL_ERR_INVALID_ARG
    for d, dv in ((96, 96), (32, 64), (128, 64), (64, 32), (256, 256), (16, 16)):
        assert call(_desc(d=d, dv=dv)) == _lib.FL_ERR_UNSUPPORTED, (d, dv)
    assert call(_desc(mask_kind=1, Lk=256)) == _lib.FL_ERR_UNSUPPORTED      # masked Lq != Lk
    assert call(_desc(Lq=130, Lk=130)) == _lib.FL_ERR_UNSUPPORTED           # Lq % 4
    assert call(_desc(score_mod=2, softcap=0.0)) == _lib.FL_ERR_INVALID_ARG
    assert call(_desc(score_mod=1)) == _lib.FL_ERR_INVALID_ARG              # ALiBi without slopes
    assert call(_desc(), dk=P + 8) == _lib.FL_ERR_ALIGNMENT
    assert call(_desc(), lse=P + 2) == _lib.FL_ERR_ALIGNMENT
    for d, dv in ((32, 32), (64, 64), (128, 128), (64, 128)):
        desc = _desc(d=d, dv=dv)
        need = ws(ctypes.byref(desc))
        assert need == 1 * 2 * 128 * (d + 2) * 4
        assert call(desc, nbytes=need - 1) == _lib.FL_ERR_INVALID_ARG, d
        assert call(desc, workspace=0) == _lib.FL_ERR_INVALID_ARG, d


def test_diffattn_bwd_rejects(L):
    """fl_diffattn_bwd's argument checks (none reaches CUDA)."""
    f = L.fl_diffattn_bwd
    ws = L.fl_diffattn_bwd_workspace_size

    def dd(**kw):
        base = dict(B=1, Hq=2, Hkv=2, Lq=256, Lk=256, d=64, dv=128, mask_kind=1)
        base.update(kw)
        return _desc(**base)

    def call(desc, lam=0.8, nbytes=None, **over):
        a = dict(q1=P, k1=P, q2=P, k2=P, v=P, dout=P)
        o = dict(dq1=P, dk1=P, dq2=P, dk2=P, dv=P, workspace=P)
        a.update({k: v for k, v in over.items() if k in a})
        o.update({k: v for k, v in over.items() if k in o})
        n = ws(ctypes.byref(desc)) if nbytes is None else nbytes
        return f(*a.values(), ctypes.c_float(lam), *o.values(), ctypes.c_size_t(n), ctypes.byref(desc))

    rows = 1 * 2 * 256
    assert ws(ctypes.byref(dd())) == rows * (2 * 128 * 2 + 66 * 4 + 8)
    assert f(P, P, P, P, P, P, ctypes.c_float(0.8), P, P, P, P, P, P, ctypes.c_size_t(1 << 30), None) == \
        _lib.FL_ERR_INVALID_ARG
    assert call(dd(), dq2=0) == _lib.FL_ERR_INVALID_ARG
    assert call(dd(), lam=float("nan")) == _lib.FL_ERR_INVALID_ARG
    assert call(dd(Hkv=1)) == _lib.FL_ERR_INVALID_ARG
    assert call(dd(Lk=128)) == _lib.FL_ERR_INVALID_ARG
    assert call(dd(d=32, dv=128)) == _lib.FL_ERR_UNSUPPORTED
    assert call(dd(dv=64)) == _lib.FL_ERR_UNSUPPORTED
    assert call(dd(mask_kind=2, window=8)) == _lib.FL_ERR_UNSUPPORTED
    assert call(dd(score_mod=2, softcap=30.0)) == _lib.FL_ERR_UNSUPPORTED
    assert call(dd(Lq=258, Lk=258)) == _lib.FL_ERR_UNSUPPORTED
    assert call(dd(), dv=P + 8) == _lib.FL_ERR_ALIGNMENT
    assert call(dd(), workspace=P + 4) == _lib.FL_ERR_ALIGNMENT
    assert call(dd(), nbytes=ws(ctypes.byref(dd())) - 1) == _lib.FL_ERR_INVALID_ARG


def test_decode_split_arithmetic():
    """Host split rule (mirrors csrc/decode.h): enough CTAs for four per SM
    (up to 8 query rows per CTA) or sixteen per SM (more rows), every split a
    whole number of 128-key tiles, none past the cache."""
    def split(B, Hkv, Lmax, M, sms):
        tiles = (Lmax + 127) // 128
        per_sm = 4 if M <= 8 else 16
        ns = max(1, min(tiles, -(-per_sm * sms // (B * Hkv))))
        per = -(-tiles // ns)
        return -(-tiles // per), per * 128
    for B, Hkv, Lmax in ((16, 8, 8192), (1, 1, 100), (2, 8, 65536), (64, 8, 1024)):
        for M in (1, 4, 8, 16, 64):
            ns, chunk = split(B, Hkv, Lmax, M, 152)
            assert chunk % 128 == 0 and (ns - 1) * chunk < Lmax <= ns * chunk
    assert split(1, 1, 100, 4, 152) == (1, 128)
    assert split(16, 8, 8192, 4, 152) == (5, 1664)
    assert split(16, 8, 8192, 16, 152) == (16, 512)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_cuda_error(L):
    assert _attn(L, _desc()) == _lib.FL_ERR_CUDA
    assert L.fl_last_error_detail().decode().startswith("cudaGetDevice")
    assert L.fl_sync_status(None) == _lib.FL_ERR_CUDA


def test_python_binding_fails_loudly_without_cuda_tensors():
    from flashattention_attn_fwd_gb300 import attn_fwd
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn_fwd(q, q, q)
