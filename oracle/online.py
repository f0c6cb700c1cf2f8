"""The single-pass online-softmax formulation, in fp64 (test infrastructure).

The Flashlight technical summary (gist.science), Methodology: "Semantic
Fusion with Algebraic Transformation", says the stable two-pass softmax is
rewritten into one pass that keeps a running maximum and a running sum and
rescales the sum, using e^(x-y) = e^x / e^y, whenever the running maximum
grows; "Tiling-Aware Dimension Elimination and Logical Grids" says the loop
walks contiguous tiles of the key axis.  This module restates that pass over
key tiles of ``block`` columns, carrying (m, l, acc) per query row, so that
tests can pin the two-pass oracle against the pages' claim that both give
the same result.  It is not used to produce expected values.
"""
from __future__ import annotations

import numpy as np

from .attention import _f64, apply_score_mod, visibility


def online_attention(q, k, v, *, block: int = 16, scale=None, mask="none",
                     window=None, prefix=None, doc_offsets=None, doc_causal=False,
                     score_mod="none", slopes=None, softcap=None):
    """Same arguments and results as ``attention.attention`` (no GQA packing
    beyond h // (Hq/Hkv)), computed tile by tile with an online softmax."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, d = q.shape
    Hkv, Lk, dv = k.shape[1], k.shape[2], v.shape[-1]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    slopes = None if slopes is None else _f64(slopes)
    out = np.zeros((B, Hq, Lq, dv))
    lse = np.zeros((B, Hq, Lq))
    for b in range(B):
        offs = None if doc_offsets is None else np.asarray(_f64(doc_offsets)[b], dtype=np.int64)
        vis = visibility(mask, Lq, Lk, window=window, prefix=prefix, offsets=offs,
                         doc_causal=doc_causal)
        for h in range(Hq):
            g = h // grp
            s_full = apply_score_mod(scale * (q[b, h] @ k[b, g].T), score_mod,
                                     slope=None if slopes is None else slopes[h], cap=softcap)
            m = np.full(Lq, -np.inf)
            l = np.zeros(Lq)
            acc = np.zeros((Lq, dv))
            for j0 in range(0, Lk, block):
                j1 = min(Lk, j0 + block)
                t = np.where(vis[:, j0:j1], s_full[:, j0:j1], -np.inf)
                m_new = np.maximum(m, t.max(axis=1))
                base = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp(m - base), 0.0)
                p = np.exp(t - base[:, None])
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ v[b, g, j0:j1]
                m = m_new
            with np.errstate(divide="ignore", invalid="ignore"):
                out[b, h] = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
                lse[b, h] = np.where(l > 0, np.where(np.isfinite(m), m, 0.0)
                                     + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse
