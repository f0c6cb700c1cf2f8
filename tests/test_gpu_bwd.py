"""GPU parity of the backward pass (dq, dk, dv through fl_attn_bwd, with the
forward's out and lse from fl_attn_fwd) against the fp64 backward oracle on
the same bf16 inputs.

Bar per gradient: relative L2 error <= 2e-2 and max-abs error <= 5e-2 of the
gradient's largest magnitude.  The derivation: the kernel rounds P and dS to
bf16 (relative 2^-9 each) before the tensor-core products and uses the
forward's bf16 output in rowsum(dO * O); with fp32 accumulation over at
most a few thousand terms the expected relative L2 error is a few 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from flashattention_attn_fwd_gb300 import attention, attn_bwd, attn_fwd, synth, sync_status

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cmp(g, ref, name):
    g = g.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), name
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(g - ref) / max(nr, 1e-30)
    mae = np.abs(g - ref).max()
    assert rel <= 2e-2, f"{name}: rel-L2 {rel:.3e}"
    assert mae <= 5e-2 * max(np.abs(ref).max(), 1e-6), f"{name}: max-abs {mae:.3e} vs max {np.abs(ref).max():.3e}"


CASES = [
    # (B, Hq, Hkv, L, d, n_docs, kwargs)
    (1, 2, 2, 256, 64, None, dict()),
    (1, 2, 2, 256, 64, None, dict(mask="causal")),
    (2, 2, 2, 300, 64, None, dict(mask="causal")),
    (1, 2, 2, 520, 64, None, dict(mask="window", window=100)),
    (1, 2, 2, 400, 64, None, dict(mask="prefix_lm", prefix=150)),
    (2, 2, 2, 500, 64, 4, dict(mask="document")),
    (2, 2, 2, 500, 64, 4, dict(mask="document", doc_causal=True)),
    (1, 4, 4, 300, 64, None, dict(score_mod="alibi", mask="causal")),
    (1, 2, 2, 300, 64, None, dict(score_mod="softcap", softcap=5.0)),
    (2, 8, 2, 300, 64, None, dict(mask="causal")),
    (1, 6, 2, 260, 64, None, dict()),
    (1, 2, 2, 300, 32, None, dict(mask="causal")),
    (1, 4, 2, 1000, 32, None, dict(score_mod="softcap", softcap=20.0, mask="causal")),
    (2, 4, 4, 1024, 64, None, dict(mask="causal")),
    # d = 128: its own TMEM map (dQ sharing dP^T's columns), one dO buffer
    (1, 2, 2, 256, 128, None, dict()),
    (1, 2, 2, 300, 128, None, dict(mask="causal")),
    (1, 4, 2, 520, 128, None, dict(mask="window", window=100)),
    (1, 2, 2, 400, 128, None, dict(mask="prefix_lm", prefix=150)),
    (2, 2, 2, 500, 128, 4, dict(mask="document", doc_causal=True)),
    (1, 4, 4, 300, 128, None, dict(score_mod="alibi", mask="causal")),
    (1, 2, 2, 300, 128, None, dict(score_mod="softcap", softcap=5.0)),
    (1, 4, 2, 1000, 128, None, dict(score_mod="softcap", softcap=20.0, mask="causal")),
    (2, 8, 2, 1024, 128, None, dict(mask="causal")),
]


def _id(c):
    B, Hq, Hkv, L, d, nd, kw = c
    return f"B{B}H{Hq}x{Hkv}L{L}d{d}" + (f"docs{nd}" if nd else "") + "-" + "-".join(f"{k}{v}" for k, v in kw.items())


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_bwd_parity(case):
    B, Hq, Hkv, L, d, nd, kw = case
    q, k, v = synth.attn_inputs(B, Hq, Hkv, L, d, seed=L + d + 3)
    g = synth.generator(L + 7)
    dout = synth.randn_bf16((B, Hq, L, d), g)
    gkw, okw = dict(kw), dict(kw)
    if nd:
        offs = synth.doc_offsets(B, L, nd, seed=L)
        gkw["doc_offsets"], okw["doc_offsets"] = offs.to(DEV), offs
    if kw.get("score_mod") == "alibi":
        s = synth.alibi_slopes(Hq)
        gkw["alibi_slopes"], okw["slopes"] = s.to(DEV), s
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    out, lse = attn_fwd(qd, kd, vd, **gkw)
    dq, dk, dv = attn_bwd(qd, kd, vd, out, dod, lse, **gkw)
    sync_status()
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, **okw)
    _cmp(dq, rq, "dq")
    _cmp(dk, rk, "dk")
    _cmp(dv, rv, "dv")


def test_autograd_function_matches_oracle():
    B, H, L, d = 1, 2, 256, 64
    q, k, v = synth.attn_inputs(B, H, H, L, d, seed=3)
    dout = synth.randn_bf16((B, H, L, d), synth.generator(4))
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    out = attention(qd, kd, vd, mask="causal")
    out.backward(dout.to(DEV))
    sync_status()
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, mask="causal")
    _cmp(qd.grad, rq, "dq")
    _cmp(kd.grad, rk, "dk")
    _cmp(vd.grad, rv, "dv")


# The benchmark's backward workload at full size (B=4 H=16 L=2048 d=64,
# causal; the same seeds and the same launch configuration the benchmark
# times), plus softcap 30.  Heads are independent (Hq = Hkv), so the oracle's
# exact gradients of a sampled (b, h) slice are those of the whole problem
# restricted to that head; three heads spread over the grid's key-tile-major
# CTA order are compared under the bar above.
@pytest.mark.parametrize("kw", [dict(mask="causal"), dict(mask="causal", score_mod="softcap", softcap=30.0)],
                         ids=["causal", "causal-softcap30"])
def test_bwd_fullsize_sampled_heads(kw):
    B, H, L, d = 4, 16, 2048, 64
    q, k, v = synth.attn_inputs(B, H, H, L, d, seed=90)
    dout = synth.randn_bf16((B, H, L, d), synth.generator(91))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    out, lse = attn_fwd(qd, kd, vd, **kw)
    dq, dk, dv = attn_bwd(qd, kd, vd, out, dod, lse, **kw)
    sync_status()
    okw = {k_: v_ for k_, v_ in kw.items()}
    for b, h in ((0, 0), (1, 7), (3, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        rq, rk, rv = oracle.attention_backward(q[sl], k[sl], v[sl], dout[sl], **okw)
        _cmp(dq[sl], rq, f"dq[{b},{h}]")
        _cmp(dk[sl], rk, f"dk[{b},{h}]")
        _cmp(dv[sl], rv, f"dv[{b},{h}]")


# The d = 128 forward's workload (causal, B 2, H 16, L 4096): dq, dk, dv of
# three sampled heads against the oracle's exact gradients of those heads.
@pytest.mark.parametrize("kw", [dict(mask="causal"), dict(score_mod="softcap", softcap=30.0)],
                         ids=["causal", "softcap30"])
def test_bwd_d128_fullsize_sampled_heads(kw):
    B, H, L, d = 2, 16, 4096, 128
    q, k, v = synth.attn_inputs(B, H, H, L, d, seed=92)
    dout = synth.randn_bf16((B, H, L, d), synth.generator(93))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    out, lse = attn_fwd(qd, kd, vd, **kw)
    dq, dk, dv = attn_bwd(qd, kd, vd, out, dod, lse, **kw)
    sync_status()
    for b, h in ((0, 0), (1, 9), (1, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        rq, rk, rv = oracle.attention_backward(q[sl], k[sl], v[sl], dout[sl], **kw)
        _cmp(dq[sl], rq, f"dq[{b},{h}]")
        _cmp(dk[sl], rk, f"dk[{b},{h}]")
        _cmp(dv[sl], rv, f"dv[{b},{h}]")


# value head dim 128 with query/key head dim 64 (the differential attention
# branches' shape): own TMEM map (dV 128 columns, dK and dQ 64 each)
DV_CASES = [
    (1, 2, 2, 256, dict()),
    (1, 2, 2, 300, dict(mask="causal")),
    (2, 8, 2, 300, dict(mask="causal")),
    (1, 4, 4, 300, dict(score_mod="alibi", mask="causal")),
    (1, 2, 2, 300, dict(score_mod="softcap", softcap=5.0)),
    (1, 2, 2, 520, dict(mask="window", window=100)),
    (2, 4, 4, 1024, dict(mask="causal")),
]


@pytest.mark.parametrize("case", DV_CASES, ids=lambda c: f"B{c[0]}H{c[1]}x{c[2]}L{c[3]}-" +
                         "-".join(f"{k}{v}" for k, v in c[4].items()))
def test_bwd_value_head_dim_128(case):
    B, Hq, Hkv, L, kw = case
    q, k, v = synth.attn_inputs(B, Hq, Hkv, L, 64, dv=128, seed=L + 5)
    dout = synth.randn_bf16((B, Hq, L, 128), synth.generator(L + 9))
    gkw, okw = dict(kw), dict(kw)
    if kw.get("score_mod") == "alibi":
        s = synth.alibi_slopes(Hq)
        gkw["alibi_slopes"], okw["slopes"] = s.to(DEV), s
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    out, lse = attn_fwd(qd, kd, vd, **gkw)
    dq, dk, dv = attn_bwd(qd, kd, vd, out, dod, lse, **gkw)
    sync_status()
    assert dv.shape == v.shape
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, **okw)
    _cmp(dq, rq, "dq")
    _cmp(dk, rk, "dk")
    _cmp(dv, rv, "dv")


DIFF_CASES = [
    # (B, H, L, causal, lambda)
    (1, 2, 256, True, 0.8),
    (1, 2, 300, False, 0.5),
    (2, 4, 520, True, 0.8),
    (1, 2, 260, True, 0.0),
    (1, 2, 384, True, -1.5),
]


@pytest.mark.parametrize("case", DIFF_CASES, ids=lambda c: f"B{c[0]}H{c[1]}L{c[2]}causal{c[3]}lam{c[4]}")
def test_diffattn_bwd_parity(case):
    from flashattention_attn_fwd_gb300 import diffattn_bwd
    B, H, L, causal, lam = case
    q1, k1, q2, k2, v = synth.diff_inputs(B, H, L, seed=L + 21)
    dout = synth.randn_bf16((B, H, L, 128), synth.generator(L + 23))
    dq1, dk1, dq2, dk2, dv = diffattn_bwd(*(t.to(DEV) for t in (q1, k1, q2, k2, v, dout)), lam, causal=causal)
    sync_status()
    ref = oracle.diff_attention_backward(q1, k1, q2, k2, v, dout, lam, causal=causal)
    for name, g, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), (dq1, dk1, dq2, dk2, dv), ref):
        if lam == 0.0 and name in ("dq2", "dk2"):
            assert float(g.abs().max()) == 0.0, name
            continue
        _cmp(g, r, name)


# The differential forward's workload (B 4, H 16, L 4096, causal, lambda
# 0.8): all five gradients of two sampled heads against the oracle (heads
# are independent).
def test_diffattn_bwd_fullsize_sampled_heads():
    from flashattention_attn_fwd_gb300 import diffattn_bwd
    B, H, L, lam = 4, 16, 4096, 0.8
    q1, k1, q2, k2, v = synth.diff_inputs(B, H, L, seed=40)
    dout = synth.randn_bf16((B, H, L, 128), synth.generator(41))
    grads = diffattn_bwd(*(t.to(DEV) for t in (q1, k1, q2, k2, v, dout)), lam, causal=True)
    sync_status()
    for b, h in ((0, 3), (3, 14)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.diff_attention_backward(q1[sl], k1[sl], q2[sl], k2[sl], v[sl], dout[sl], lam, causal=True)
        for name, g, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, ref):
            _cmp(g[sl], r, f"{name}[{b},{h}]")


def test_diff_attention_autograd_matches_oracle():
    from flashattention_attn_fwd_gb300 import diff_attention
    B, H, L, lam = 1, 2, 256, 0.8
    q1, k1, q2, k2, v = synth.diff_inputs(B, H, L, seed=12)
    dout = synth.randn_bf16((B, H, L, 128), synth.generator(13))
    ins = [t.to(DEV).requires_grad_() for t in (q1, k1, q2, k2, v)]
    out = diff_attention(*ins, lam, causal=True)
    out.backward(dout.to(DEV))
    sync_status()
    ref = oracle.diff_attention_backward(q1, k1, q2, k2, v, dout, lam, causal=True)
    for name, t, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), ins, ref):
        _cmp(t.grad, r, name)
