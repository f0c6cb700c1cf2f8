"""fp64 CPU oracle for the backward pass of the fused attention (test
infrastructure; the same import rules as the rest of ``oracle``).

The Flashlight wiki summary lists the training backward among the open items
(局限与 Future Work: "训练 backward ... 未系统评测"); the pages give no formula,
so this is the plain derivative of the forward definition in
``oracle.attention``, written out with the full probability matrix:

    P      = softmax_j(T),   T = score_mod(scale * Q K^T) with the mask
    dV     = P^T dO
    dP     = dO V^T
    D_i    = sum_j P_ij dP_ij            (= rowsum(dO * O))
    dT     = P * (dP - D)
    dS     = dT * dT/dS                   (1 for none / ALiBi; softcap:
                                          1 - tanh(S / cap)^2)
    dQ     = scale * dS K,   dK = scale * dS^T Q

with S = scale * Q K^T written as S = scale * R, so the scale enters dQ and
dK once.  For GQA the key/value gradients of a group sum over its query
heads.  A row with no visible key contributes nothing.
"""
from __future__ import annotations

import numpy as np

from .attention import _f64, apply_score_mod, softmax_rows, visibility

__all__ = ["attention_backward", "diff_attention_backward"]


def attention_backward(q, k, v, dout, *, scale: float | None = None, mask: str = "none",
                       window: int | None = None, prefix: int | None = None,
                       doc_offsets=None, doc_causal: bool = False,
                       score_mod: str = "none", slopes=None, softcap: float | None = None):
    """(dq, dk, dv) of L = sum(dout * attention(q, k, v, ...)) in float64;
    shapes as ``oracle.attention``'s inputs."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    slopes = None if slopes is None else _f64(slopes)
    offs = None if doc_offsets is None else np.asarray(_f64(doc_offsets), dtype=np.int64)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        vis = visibility(mask, Lq, Lk, window=window, prefix=prefix,
                         offsets=None if offs is None else offs[b], doc_causal=doc_causal)
        for h in range(Hq):
            g = h // grp
            s = scale * (q[b, h] @ k[b, g].T)
            t = apply_score_mod(s, score_mod, slope=None if slopes is None else slopes[h], cap=softcap)
            t = np.where(vis, t, -np.inf)
            P, _ = softmax_rows(t)
            dO = dout[b, h]
            dv[b, g] += P.T @ dO
            dP = dO @ v[b, g].T
            D = np.sum(P * dP, axis=1, keepdims=True)
            dT = P * (dP - D)
            if score_mod == "softcap":
                dT = dT * (1.0 - np.tanh(s / float(softcap)) ** 2)
            dq[b, h] += scale * (dT @ k[b, g])
            dk[b, g] += scale * (dT.T @ q[b, h])
    return dq, dk, dv


def diff_attention_backward(q1, k1, q2, k2, v, dout, lam: float, *, scale: float | None = None,
                            causal: bool = True):
    """(dq1, dk1, dq2, dk2, dv) of L = sum(dout * diff_attention(...)) in
    float64.  The output O1 - lam * O2 is linear in the two branch outputs,
    so branch 1 takes the output gradient dout and branch 2 takes -lam * dout.
    Both branches read the same V, so dv is the sum of the two branch dV's."""
    d = _f64(q1).shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    mask = "causal" if causal else "none"
    dout = _f64(dout)
    dq1, dk1, dv1 = attention_backward(q1, k1, v, dout, scale=scale, mask=mask)
    dq2, dk2, dv2 = attention_backward(q2, k2, v, -float(lam) * dout, scale=scale, mask=mask)
    return dq1, dk1, dq2, dk2, dv1 + dv2
