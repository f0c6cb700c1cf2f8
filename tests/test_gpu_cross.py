"""GPU parity when the query and key/value sequences differ in length
(Lq != Lk; the mask must then be NONE), forward and backward, against the
fp64 oracle on the same seeded bf16 inputs.  ALiBi's bias is slope * (j - i)
with i and j the 0-based positions in their own sequences, as in the oracle.

Bars: the forward's (max-abs <= 2e-2, relative L2 <= 1e-2, LSE max-abs
<= 1e-3) and the backward's (per gradient relative L2 <= 2e-2, max-abs
<= 5e-2 of the largest magnitude).
"""
import numpy as np
import pytest

import oracle
from flashattention_attn_fwd_gb300 import attn_bwd, attn_fwd, synth, sync_status

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _inputs(B, Hq, Hkv, Lq, Lk, d, kw, seed):
    q, k, v = synth.attn_inputs(B, Hq, Hkv, Lq, d, seed=seed, Lk=Lk)
    gkw, okw = dict(kw), dict(kw)
    if kw.get("score_mod") == "alibi":
        s = synth.alibi_slopes(Hq)
        gkw["alibi_slopes"], okw["slopes"] = s.to(DEV), s
    return q, k, v, gkw, okw


FWD = [
    # (B, Hq, Hkv, Lq, Lk, d, kwargs)
    (1, 2, 2, 300, 700, 64, dict()),
    (2, 4, 2, 700, 300, 64, dict()),
    (1, 2, 2, 130, 1000, 64, dict(score_mod="alibi")),
    (1, 2, 2, 257, 513, 64, dict(score_mod="softcap", softcap=20.0)),
    (1, 4, 1, 1, 1500, 128, dict()),
    (1, 2, 2, 200, 333, 32, dict()),
]


@pytest.mark.parametrize("case", FWD, ids=lambda c: f"B{c[0]}H{c[1]}x{c[2]}Lq{c[3]}Lk{c[4]}d{c[5]}-" +
                         "-".join(f"{k}{v}" for k, v in c[6].items()))
def test_cross_forward(case):
    B, Hq, Hkv, Lq, Lk, d, kw = case
    q, k, v, gkw, okw = _inputs(B, Hq, Hkv, Lq, Lk, d, kw, seed=Lq + Lk)
    out, lse = attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), **gkw)
    sync_status()
    ro, rl = oracle.attention(q, k, v, **okw)
    g = _np(out)
    assert g.shape == ro.shape and np.isfinite(g).all()
    mae = float(np.abs(g - ro).max())
    rel = float(np.linalg.norm(g - ro) / np.linalg.norm(ro))
    assert mae <= 2e-2 and rel <= 1e-2, f"max-abs {mae:.3e} rel-L2 {rel:.3e}"
    assert float(np.abs(_np(lse) - rl).max()) <= 1e-3


BWD = [
    (1, 2, 2, 256, 520, 64, dict()),
    (2, 4, 2, 516, 300, 64, dict()),
    (1, 2, 2, 300, 700, 64, dict(score_mod="softcap", softcap=5.0)),
    (1, 2, 2, 200, 600, 32, dict(score_mod="alibi")),
]


def _cmp(g, ref, name):
    g = _np(g)
    assert np.isfinite(g).all(), name
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    mae = np.abs(g - ref).max()
    assert rel <= 2e-2, f"{name}: rel-L2 {rel:.3e}"
    assert mae <= 5e-2 * max(np.abs(ref).max(), 1e-6), f"{name}: max-abs {mae:.3e}"


@pytest.mark.parametrize("case", BWD, ids=lambda c: f"B{c[0]}H{c[1]}x{c[2]}Lq{c[3]}Lk{c[4]}d{c[5]}-" +
                         "-".join(f"{k}{v}" for k, v in c[6].items()))
def test_cross_backward(case):
    B, Hq, Hkv, Lq, Lk, d, kw = case
    q, k, v, gkw, okw = _inputs(B, Hq, Hkv, Lq, Lk, d, kw, seed=Lq + 2 * Lk)
    dout = synth.randn_bf16((B, Hq, Lq, d), synth.generator(Lq + 11))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, dout))
    out, lse = attn_fwd(qd, kd, vd, **gkw)
    dq, dk, dv = attn_bwd(qd, kd, vd, out, dod, lse, **gkw)
    sync_status()
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, **okw)
    _cmp(dq, rq, "dq")
    _cmp(dk, rk, "dk")
    _cmp(dv, rv, "dv")
