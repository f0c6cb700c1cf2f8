"""Scalar pure-Python attention for tiny inputs (test helper).

Written element by element from the definitions stated in the oracle's
header, with no NumPy vectorisation, so that an indexing or broadcasting
mistake in the vectorised oracle shows up as a mismatch.  Inputs are nested
Python lists of floats.
"""
import math


def _visible(mask, i, j, window=None, prefix=None, offsets=None, doc_causal=False):
    if mask == "none":
        return True
    if mask == "causal":
        return j <= i
    if mask == "window":
        return j <= i and j > i - window
    if mask == "prefix_lm":
        return j <= i or j < prefix
    if mask == "document":
        def doc(x):
            dd = 0
            while dd + 1 < len(offsets) and offsets[dd + 1] <= x:
                dd += 1
            return dd
        ok = doc(i) == doc(j)
        if doc_causal:
            ok = ok and j <= i
        return ok
    raise ValueError(mask)


def brute_row(qi, K, V, i, scale, mask="none", score_mod="none", slope=0.0, cap=None,
              bias_row=None, **mk):
    """One query row: returns (out list, lse)."""
    ts = []
    for j in range(len(K)):
        if not _visible(mask, i, j, **mk):
            continue
        s = 0.0
        for c in range(len(qi)):
            s += qi[c] * K[j][c]
        s *= scale
        if score_mod == "alibi":
            s = s + slope * (j - i)
        elif score_mod == "softcap":
            s = cap * math.tanh(s / cap)
        if bias_row is not None:
            s = s + bias_row[j]
        ts.append((j, s))
    if not ts:
        return [0.0] * len(V[0]), -math.inf
    mx = max(t for _, t in ts)
    z = sum(math.exp(t - mx) for _, t in ts)
    out = [0.0] * len(V[0])
    for j, t in ts:
        w = math.exp(t - mx) / z
        for c in range(len(V[0])):
            out[c] += w * V[j][c]
    return out, mx + math.log(z)
