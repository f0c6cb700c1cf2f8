"""Plain fp64 CPU oracle for the fused attention forward and its variants.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or run this module.
It shares no code with the CUDA library and imports nothing from it.

What it computes
----------------
The Flashlight pages state that the fused kernel computes exactly
``softmax(QK^T) V`` (Flashlight technical summary, gist.science, Methodology:
"Tiling-Aware Dimension Elimination and Logical Grids"; Key Contributions:
"Kernel-Level Fusion"), and that the single-pass online softmax is an exact
rewrite of the two-pass stable softmax (same page, Methodology: "Semantic
Fusion with Algebraic Transformation").  The oracle is therefore the plain
definition, written out in the two-pass form, with the full score matrix
materialised for every (batch, head):

    s[i,j]  = scale * sum_c q[i,c] k[j,c]
    t[i,j]  = score_mod(s[i,j], h, i, j) + bias[i,j]
    t[i,j]  = -inf where key j is not visible to query i
    M_i     = max_j t[i,j]
    P[i,j]  = exp(t[i,j] - M_i) / sum_j exp(t[i,j] - M_i)
    O       = P V,      LSE_i = M_i + log sum_j exp(t[i,j] - M_i)

The variants are the ones the Flashlight wiki summary (papers.lqhl.me) lists
under 实验与结果 (Vanilla, ALiBi, Softcap, Causal, Sliding Window, PrefixLM,
Document Mask; MHA/GQA) and under 问题与动机 (differential attention, Evoformer
row-wise gated attention).  The pages print no formula for any variant; the
readings taken here are:

* ALiBi        t = s + m_h (j - i), non-causal, slopes passed by the caller.
* Softcap      t = cap * tanh(s / cap) on the scaled logit.
* Causal       j <= i.
* Window w     i - w < j <= i   (w keys visible, self included).
* Prefix-LM P  j <= i  or  j < P.
* Document     doc(i) == doc(j) (bidirectional in the document); with the
               optional causal bit also j <= i.  Documents are contiguous and
               given by offsets [0, c1, ..., L].
* GQA          query head h reads key/value head h // (Hq / Hkv).
* Differential out = softmax(Q1 K1^T s) V - lambda softmax(Q2 K2^T s) V.
* Evoformer    t = s + pair_bias[h, i, j] + mask_bias[msa_row, j];
               out = sigmoid(gate) * (P V).
* Evoformer, column-wise: for each residue column r, attention over the MSA
               rows s with t = s + mask_bias[r, s'] and no pair bias;
               out = sigmoid(gate) * (P V) (technical summary, Results, names
               the row- and column-wise gated forms).
* Decode      Lq new query rows against a cache of kv_len[b] keys (the rows
               are the last Lq positions of that sequence): keys j < kv_len[b]
               are visible, and with the causal mask only j <= kv_len[b]-Lq+i
               (technical summary, Methodology, and the wiki summary's
               批判性分析 note on the serving path's decode phase; the pages
               evaluate no decode workload, so this is the plain reading).
* A row with no visible key gives O = 0 and LSE = -inf.

All arithmetic is float64 NumPy; a matmul and ``exp``/``log``/``tanh`` are
the only library primitives used.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "MASKS",
    "SCORE_MODS",
    "doc_ids",
    "visibility",
    "apply_score_mod",
    "softmax_rows",
    "attention",
    "attention_rows",
    "diff_attention",
    "diff_attention_rows",
    "evoformer_gated_attention",
    "evoformer_rows",
    "evoformer_col_gated_attention",
    "evoformer_col_rows",
    "decode_attention",
]

MASKS = ("none", "causal", "window", "prefix_lm", "document")
SCORE_MODS = ("none", "alibi", "softcap")


def _f64(x) -> np.ndarray:
    """Anything array-like (numpy, or a CPU torch tensor of any float dtype)
    to a float64 numpy array.  bf16 values convert exactly."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16" or str(x.dtype) == "torch.float16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def doc_ids(offsets, L: int) -> np.ndarray:
    """Document index of every position 0..L-1, for sorted offsets [0, ..., L]."""
    off = np.asarray(offsets, dtype=np.int64)
    return np.searchsorted(off, np.arange(L), side="right") - 1


def visibility(mask: str, Lq: int, Lk: int, *, window: int | None = None,
               prefix: int | None = None, offsets=None,
               doc_causal: bool = False) -> np.ndarray:
    """Boolean [Lq, Lk]: True where key j is visible to query i."""
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    if mask == "none":
        return np.ones((Lq, Lk), dtype=bool)
    if mask == "causal":
        return j <= i
    if mask == "window":
        return (j <= i) & (j > i - int(window))
    if mask == "prefix_lm":
        return (j <= i) | (j < int(prefix))
    if mask == "document":
        dq = doc_ids(offsets, Lq)[:, None]
        dk = doc_ids(offsets, Lk)[None, :]
        vis = dq == dk
        if doc_causal:
            vis &= j <= i
        return vis
    raise ValueError(f"unknown mask {mask!r}")


def apply_score_mod(s: np.ndarray, score_mod: str, *, slope: float | None = None,
                    cap: float | None = None) -> np.ndarray:
    """score_mod applied to the scaled logits s [Lq, Lk] of one head."""
    if score_mod == "none":
        return s
    Lq, Lk = s.shape
    if score_mod == "alibi":
        i = np.arange(Lq, dtype=np.float64)[:, None]
        j = np.arange(Lk, dtype=np.float64)[None, :]
        return s + float(slope) * (j - i)
    if score_mod == "softcap":
        return float(cap) * np.tanh(s / float(cap))
    raise ValueError(f"unknown score_mod {score_mod!r}")


def softmax_rows(t: np.ndarray):
    """Two-pass stable softmax over the last axis.  Returns (P, LSE); rows
    that are entirely -inf give P = 0 and LSE = -inf."""
    M = np.max(t, axis=-1, keepdims=True)
    empty = ~np.isfinite(M)
    Ms = np.where(empty, 0.0, M)
    E = np.exp(t - Ms)
    Z = np.sum(E, axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(Z > 0, E / np.where(Z > 0, Z, 1.0), 0.0)
        lse = np.where(Z[..., 0] > 0, Ms[..., 0] + np.log(np.where(Z[..., 0] > 0, Z[..., 0], 1.0)),
                       -np.inf)
    return P, lse


def _head_scores(qh, kh, scale):
    return scale * (qh @ kh.T)


def attention(q, k, v, *, scale: float | None = None, mask: str = "none",
              window: int | None = None, prefix: int | None = None,
              doc_offsets=None, doc_causal: bool = False,
              score_mod: str = "none", slopes=None, softcap: float | None = None,
              return_probs: bool = False):
    """softmax(score_mod(scale Q K^T) masked) V for q [B,Hq,Lq,d],
    k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv].  Returns (out [B,Hq,Lq,dv],
    lse [B,Hq,Lq]) in float64, and P [B,Hq,Lq,Lk] when return_probs."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    dv = v.shape[-1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    slopes = None if slopes is None else _f64(slopes)
    offs = None if doc_offsets is None else np.asarray(_f64(doc_offsets), dtype=np.int64)
    out = np.zeros((B, Hq, Lq, dv))
    lse = np.zeros((B, Hq, Lq))
    probs = np.zeros((B, Hq, Lq, Lk)) if return_probs else None
    vis_common = None
    if mask != "document":
        vis_common = visibility(mask, Lq, Lk, window=window, prefix=prefix)
    for b in range(B):
        vis = vis_common if vis_common is not None else visibility(
            "document", Lq, Lk, offsets=offs[b], doc_causal=doc_causal)
        for h in range(Hq):
            g = h // grp
            s = _head_scores(q[b, h], k[b, g], scale)
            t = apply_score_mod(s, score_mod,
                                slope=None if slopes is None else slopes[h], cap=softcap)
            t = np.where(vis, t, -np.inf)
            P, l = softmax_rows(t)
            out[b, h] = P @ v[b, g]
            lse[b, h] = l
            if return_probs:
                probs[b, h] = P
    if return_probs:
        return out, lse, probs
    return out, lse


def attention_rows(q, k, v, rows, **kw):
    """The same definition for a list of (b, h, i) query rows only (each row
    computed on its own from the full K/V), for parity checks at sizes where
    the whole score matrix is too large.  Returns (out [n,dv], lse [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    grp = Hq // Hkv
    scale = kw.get("scale")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    mask = kw.get("mask", "none")
    score_mod = kw.get("score_mod", "none")
    slopes = kw.get("slopes")
    slopes = None if slopes is None else _f64(slopes)
    offs = kw.get("doc_offsets")
    offs = None if offs is None else np.asarray(_f64(offs), dtype=np.int64)
    outs, lses = [], []
    for (b, h, i) in rows:
        g = h // grp
        s = scale * (k[b, g] @ q[b, h, i])[None, :]
        j = np.arange(Lk)
        if score_mod == "alibi":
            t = s + slopes[h] * (j - i)[None, :]
        elif score_mod == "softcap":
            t = float(kw["softcap"]) * np.tanh(s / float(kw["softcap"]))
        else:
            t = s
        if mask == "none":
            vis = np.ones(Lk, dtype=bool)
        elif mask == "causal":
            vis = j <= i
        elif mask == "window":
            vis = (j <= i) & (j > i - int(kw["window"]))
        elif mask == "prefix_lm":
            vis = (j <= i) | (j < int(kw["prefix"]))
        elif mask == "document":
            ids = doc_ids(offs[b], max(Lk, i + 1))
            vis = ids[:Lk] == ids[i]
            if kw.get("doc_causal", False):
                vis &= j <= i
        else:
            raise ValueError(mask)
        t = np.where(vis[None, :], t, -np.inf)
        P, l = softmax_rows(t)
        outs.append((P @ v[b, g])[0])
        lses.append(l[0])
    return np.array(outs), np.array(lses)


def diff_attention(q1, k1, q2, k2, v, lam: float, *, scale: float | None = None,
                   causal: bool = True):
    """Differential attention: softmax(s Q1 K1^T) V - lam softmax(s Q2 K2^T) V,
    each branch a plain softmax attention (causal by default) over the shared
    V.  Returns (out, lse1, lse2)."""
    d = _f64(q1).shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    mask = "causal" if causal else "none"
    o1, l1 = attention(q1, k1, v, scale=scale, mask=mask)
    o2, l2 = attention(q2, k2, v, scale=scale, mask=mask)
    return o1 - float(lam) * o2, l1, l2


def diff_attention_rows(q1, k1, q2, k2, v, lam: float, rows, *, scale=None, causal=True):
    d = _f64(q1).shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    mask = "causal" if causal else "none"
    o1, l1 = attention_rows(q1, k1, v, rows, scale=scale, mask=mask)
    o2, l2 = attention_rows(q2, k2, v, rows, scale=scale, mask=mask)
    return o1 - float(lam) * o2, l1, l2


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def evoformer_gated_attention(q, k, v, pair_bias, mask_bias, gate, *,
                              scale: float | None = None):
    """Evoformer MSA row-wise gated self-attention.

    q, k, v, gate : [B, N_seq, H, N_res, d];  pair_bias : [B, H, N_res, N_res]
    (the same for every MSA row);  mask_bias : [B, N_seq, N_res] (added to
    every query row of that MSA row).  Attention runs over the residue axis.
    Returns (out [B,N_seq,H,N_res,d], lse [B,N_seq,H,N_res])."""
    q, k, v, gate = _f64(q), _f64(k), _f64(v), _f64(gate)
    pb, mb = _f64(pair_bias), _f64(mask_bias)
    B, Ns, H, Nr, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.zeros_like(q)
    lse = np.zeros((B, Ns, H, Nr))
    for b in range(B):
        for s in range(Ns):
            for h in range(H):
                t = scale * (q[b, s, h] @ k[b, s, h].T) + pb[b, h] + mb[b, s][None, :]
                P, l = softmax_rows(t)
                out[b, s, h] = _sigmoid(gate[b, s, h]) * (P @ v[b, s, h])
                lse[b, s, h] = l
    return out, lse


def evoformer_rows(q, k, v, pair_bias, mask_bias, gate, rows, *, scale=None):
    """Evoformer output for a list of (b, msa_row, h, i) query rows."""
    q, k, v, gate = _f64(q), _f64(k), _f64(v), _f64(gate)
    pb, mb = _f64(pair_bias), _f64(mask_bias)
    d = q.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    outs, lses = [], []
    for (b, s, h, i) in rows:
        t = (scale * (k[b, s, h] @ q[b, s, h, i]) + pb[b, h, i] + mb[b, s])[None, :]
        P, l = softmax_rows(t)
        outs.append(_sigmoid(gate[b, s, h, i]) * (P @ v[b, s, h])[0])
        lses.append(l[0])
    return np.array(outs), np.array(lses)


def evoformer_col_gated_attention(q, k, v, mask_bias, gate, *, scale: float | None = None):
    """Evoformer MSA column-wise gated self-attention.

    q, k, v, gate : [B, N_seq, H, N_res, d] (the MSA layout of the row-wise
    form);  mask_bias : [B, N_res, N_seq] (added to every query of residue
    column r, per key MSA row).  For every (b, h, r) attention runs over the
    MSA-row axis.  Returns (out [B,N_seq,H,N_res,d], lse [B,H,N_res,N_seq])."""
    q, k, v, gate = _f64(q), _f64(k), _f64(v), _f64(gate)
    mb = _f64(mask_bias)
    B, Ns, H, Nr, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.zeros_like(q)
    lse = np.zeros((B, H, Nr, Ns))
    for b in range(B):
        for h in range(H):
            for r in range(Nr):
                t = scale * (q[b, :, h, r] @ k[b, :, h, r].T) + mb[b, r][None, :]
                P, l = softmax_rows(t)
                out[b, :, h, r] = _sigmoid(gate[b, :, h, r]) * (P @ v[b, :, h, r])
                lse[b, h, r] = l
    return out, lse


def evoformer_col_rows(q, k, v, mask_bias, gate, rows, *, scale=None):
    """Column-wise Evoformer output for a list of (b, msa_row, h, r) query rows."""
    q, k, v, gate = _f64(q), _f64(k), _f64(v), _f64(gate)
    mb = _f64(mask_bias)
    d = q.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    outs, lses = [], []
    for (b, s, h, r) in rows:
        t = (scale * (k[b, :, h, r] @ q[b, s, h, r]) + mb[b, r])[None, :]
        P, l = softmax_rows(t)
        outs.append(_sigmoid(gate[b, s, h, r]) * (P @ v[b, :, h, r])[0])
        lses.append(l[0])
    return np.array(outs), np.array(lses)


def decode_attention(q, k, v, kv_len=None, *, causal: bool = False, scale: float | None = None,
                     score_mod: str = "none", slopes=None, softcap: float | None = None):
    """Decode-phase attention over a key/value cache.

    q [B,Hq,Lq,d]; k [B,Hkv,Lmax,d]; v [B,Hkv,Lmax,dv]; kv_len [B] valid
    cache lengths (None: Lmax for every sequence).  Query row i of sequence
    b sits at position p_i = kv_len[b] - Lq + i; key j is visible when
    j < kv_len[b] and, with ``causal``, j <= p_i.  ALiBi adds m_h (j - p_i).
    Returns (out [B,Hq,Lq,dv], lse [B,Hq,Lq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, d = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    dv = v.shape[-1]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    lens = np.full(B, Lmax, dtype=np.int64) if kv_len is None else np.asarray(_f64(kv_len), dtype=np.int64)
    slopes = None if slopes is None else _f64(slopes)
    out = np.zeros((B, Hq, Lq, dv))
    lse = np.zeros((B, Hq, Lq))
    for b in range(B):
        n = int(lens[b])
        pos = n - Lq + np.arange(Lq)[:, None]
        j = np.arange(Lmax)[None, :]
        vis = j < n
        if causal:
            vis = vis & (j <= pos)
        for h in range(Hq):
            g = h // grp
            s = scale * (q[b, h] @ k[b, g].T)
            if score_mod == "alibi":
                s = s + slopes[h] * (j - pos)
            elif score_mod == "softcap":
                s = float(softcap) * np.tanh(s / float(softcap))
            t = np.where(vis, s, -np.inf)
            P, l = softmax_rows(t)
            out[b, h] = P @ v[b, g]
            lse[b, h] = l
    return out, lse
