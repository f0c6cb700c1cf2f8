"""FLOP and byte accounting for the roofline (host-side bookkeeping).

FLOPs count the two contractions of every (query, key) pair the method
computes: 2*d for Q K^T and 2*dv for P V.  The headline figure counts whole
128 x 128 tiles of the (query, key) grid that hold at least one visible
pair -- the work a tiled kernel that skips fully-masked tiles must do, the
same for any kernel tiling -- and the exact visible-pair count is reported
beside it.  Algorithmic bytes are every input read once (K/V once per
key/value head; the Evoformer pair bias once, not once per MSA row) plus
every output written once.
"""
from __future__ import annotations

import numpy as np

TILE = 128


def row_intervals(mask: str, L: int, *, window=None, prefix=None, offsets=None, doc_causal=False):
    """Visible-key interval [lo_i, hi_i] of every query row (Lq == Lk == L)."""
    i = np.arange(L, dtype=np.int64)
    if mask == "none":
        lo, hi = np.zeros(L, np.int64), np.full(L, L - 1, np.int64)
    elif mask == "causal":
        lo, hi = np.zeros(L, np.int64), i.copy()
    elif mask == "window":
        lo, hi = np.maximum(i - int(window) + 1, 0), i.copy()
    elif mask == "prefix_lm":
        lo, hi = np.zeros(L, np.int64), np.maximum(i, int(prefix) - 1)
    elif mask == "document":
        off = np.asarray(offsets, dtype=np.int64)
        doc = np.searchsorted(off, i, side="right") - 1
        lo = off[doc]
        hi = i.copy() if doc_causal else off[doc + 1] - 1
    else:
        raise ValueError(mask)
    return lo, np.minimum(hi, L - 1)


def visible_tiles(lo, hi, L: int, tile: int = TILE) -> int:
    """Number of tile x tile blocks holding at least one visible pair."""
    nt = (L + tile - 1) // tile
    marked = np.zeros((nt, nt), dtype=bool)
    for r in range(nt):
        rows = slice(r * tile, min(L, (r + 1) * tile))
        for a, b in zip(lo[rows], hi[rows]):
            if b >= a:
                marked[r, a // tile: b // tile + 1] = True
    return int(marked.sum())


def visible_pairs(lo, hi) -> int:
    return int(np.maximum(hi - lo + 1, 0).sum())


def attn_counts(B, Hq, Hkv, L, d, dv=None, *, mask="none", window=None, prefix=None,
                doc_offsets=None, doc_causal=False):
    """(tile_flops, exact_flops, alg_bytes) of one fused attention forward."""
    dv = d if dv is None else dv
    per_pair = 2 * d + 2 * dv
    tiles = pairs = 0
    batches = range(B) if mask == "document" else [None]
    for b in batches:
        offs = None if b is None else np.asarray(doc_offsets)[b]
        lo, hi = row_intervals(mask, L, window=window, prefix=prefix, offsets=offs, doc_causal=doc_causal)
        mult = 1 if b is not None else B
        tiles += mult * visible_tiles(lo, hi, L)
        pairs += mult * visible_pairs(lo, hi)
    tile_flops = tiles * TILE * TILE * per_pair * Hq
    exact_flops = pairs * per_pair * Hq
    bytes_ = 2 * (B * Hq * L * d + B * Hkv * L * d + B * Hkv * L * dv + B * Hq * L * dv) + 4 * B * Hq * L
    return tile_flops, exact_flops, bytes_


def bwd_counts(B, Hq, Hkv, L, d, *, mask="none", window=None, prefix=None, doc_offsets=None,
               doc_causal=False):
    """Backward pass: five products per visible pair (S = QK^T and dP = dO V^T
    recomputed, dV, dK, dQ), 2*d FLOPs each; bytes read q, k, v, out, dout,
    lse and written dq, dk, dv once."""
    tf, ef, _ = attn_counts(B, Hq, Hkv, L, d, mask=mask, window=window, prefix=prefix,
                            doc_offsets=doc_offsets, doc_causal=doc_causal)
    f = 10 / 4  # 10 d per pair against the forward's 4 d
    bytes_ = 2 * (3 * B * Hq * L * d + 2 * B * Hkv * L * d) + 4 * B * Hq * L + 2 * (B * Hq * L * d + 2 * B * Hkv * L * d)
    return int(tf * f), int(ef * f), bytes_


def diff_bwd_counts(B, H, L, d=64, dv=128, causal=True):
    """Backward of differential attention as fl_diffattn_bwd runs it: per
    branch the forward recomputed (2 d + 2 dv FLOPs per visible pair) and the
    five backward products (S and dP recomputed, dV, dK, dQ: 2 (3 d + 2 dv));
    bytes read q1, k1, q2, k2, v, dout and written their five gradients once."""
    tf, ef, _ = attn_counts(B, H, H, L, d, dv, mask="causal" if causal else "none")
    per_fwd = 2 * d + 2 * dv
    per_all = 2 * (per_fwd + 2 * (3 * d + 2 * dv))
    n = B * H * L
    bytes_ = 2 * (4 * n * d + 2 * n * dv) + 2 * (4 * n * d + n * dv)
    return tf // per_fwd * per_all, ef // per_fwd * per_all, bytes_


def diff_counts(B, H, L, d=64, dv=128, causal=True):
    lo, hi = row_intervals("causal" if causal else "none", L)
    tiles, pairs = visible_tiles(lo, hi, L), visible_pairs(lo, hi)
    per_pair = 2 * (2 * d + 2 * dv)
    tile_flops = B * H * tiles * TILE * TILE * per_pair
    exact_flops = B * H * pairs * per_pair
    bytes_ = 2 * (4 * B * H * L * d + B * H * L * dv + B * H * L * dv) + 4 * 2 * B * H * L
    return tile_flops, exact_flops, bytes_


def evo_counts(B, N_seq, N_res, H, d=32, with_pair_bias=True, with_mask=True):
    lo, hi = row_intervals("none", N_res)
    tiles, pairs = visible_tiles(lo, hi, N_res), visible_pairs(lo, hi)
    per_pair = 4 * d
    n = B * N_seq * H
    tile_flops = n * tiles * TILE * TILE * per_pair
    exact_flops = n * pairs * per_pair
    bytes_ = 2 * 5 * n * N_res * d + 4 * n * N_res
    if with_pair_bias:
        bytes_ += 4 * B * H * N_res * N_res
    if with_mask:
        bytes_ += 4 * B * N_seq * N_res
    return tile_flops, exact_flops, bytes_


def evo_col_counts(B, N_seq, N_res, H, d=32, with_mask=True):
    """Column-wise Evoformer: attention over the N_seq MSA rows of each of the
    B * H * N_res residue columns; no pair bias."""
    lo, hi = row_intervals("none", N_seq)
    tiles, pairs = visible_tiles(lo, hi, N_seq), visible_pairs(lo, hi)
    per_pair = 4 * d
    n = B * H * N_res
    tile_flops = n * tiles * TILE * TILE * per_pair
    exact_flops = n * pairs * per_pair
    bytes_ = 2 * 5 * n * N_seq * d + 4 * n * N_seq
    if with_mask:
        bytes_ += 4 * B * N_res * N_seq
    return tile_flops, exact_flops, bytes_


def decode_counts(B, Hq, Hkv, Lq, d, kv_len, causal=False):
    """Decode over a key/value cache: the FLOPs of the visible (row, key)
    pairs (no tile rounding: the kernel has no 128-row tiles) and the bytes
    of q, the valid part of the K/V cache, out and lse."""
    lens = np.asarray(kv_len, dtype=np.int64)
    if causal:
        pairs = int(sum(sum(n - Lq + i + 1 for i in range(Lq)) for n in lens))
    else:
        pairs = int(lens.sum()) * Lq
    flops = pairs * Hq * 4 * d
    bytes_ = 2 * (2 * B * Hq * Lq * d + 2 * int(lens.sum()) * Hkv * d) + 4 * B * Hq * Lq
    return flops, flops, bytes_


def roofline_time(flops: float, bytes_: float, tflops_peak: float, hbm_gbs: float):
    """(seconds, bound) of the slower of tensor-peak and HBM-peak time."""
    t_tensor = flops / (tflops_peak * 1e12)
    t_hbm = bytes_ / (hbm_gbs * 1e9)
    return (t_tensor, "tensor") if t_tensor >= t_hbm else (t_hbm, "hbm")
