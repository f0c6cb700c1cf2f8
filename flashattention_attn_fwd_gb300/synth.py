"""Seeded synthetic inputs shared by the tests, the benchmark and the CPU oracle.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Everything is drawn on the CPU from a seeded
``torch.Generator`` so that the same call gives the same tensors on every
machine; callers move the tensors to the GPU themselves.

Shapes follow the workloads the Flashlight pages evaluate (sequence lengths
512-16k with head dim 64; the AlphaFold2 Evoformer at 256 residues), see the
Flashlight wiki summary (papers.lqhl.me), sections 设计取舍 and 实验与结果.
"""
from __future__ import annotations

import torch

__all__ = [
    "generator",
    "randn_bf16",
    "attn_inputs",
    "alibi_slopes",
    "doc_offsets",
    "diff_inputs",
    "evo_inputs",
    "evo_col_inputs",
    "decode_inputs",
]


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator) -> torch.Tensor:
    """N(0,1) drawn in fp32, then rounded to bf16 (the values both sides see)."""
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def attn_inputs(B: int, Hq: int, Hkv: int, L: int, d: int, dv: int | None = None,
                seed: int = 0, Lk: int | None = None):
    """q [B,Hq,L,d], k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv]; bf16, N(0,1)."""
    dv = d if dv is None else dv
    Lk = L if Lk is None else Lk
    g = generator(seed)
    q = randn_bf16((B, Hq, L, d), g)
    k = randn_bf16((B, Hkv, Lk, d), g)
    v = randn_bf16((B, Hkv, Lk, dv), g)
    return q, k, v


def alibi_slopes(H: int) -> torch.Tensor:
    """Geometric ALiBi slopes 2^(-8h/H) for h = 1..H (fp32, one per query head)."""
    h = torch.arange(1, H + 1, dtype=torch.float64)
    return torch.pow(2.0, -8.0 * h / H).to(torch.float32)


def doc_offsets(B: int, L: int, n_docs: int, seed: int = 0) -> torch.Tensor:
    """Per batch element, a seeded uniform partition of [0, L) into n_docs
    contiguous, non-empty documents: n_docs-1 distinct cut points drawn
    without replacement from {1..L-1}, sorted.  Returns int32 [B, n_docs+1]
    with offsets[b, 0] = 0 and offsets[b, n_docs] = L."""
    if n_docs < 1 or n_docs > L:
        raise ValueError("need 1 <= n_docs <= L")
    g = generator(seed)
    rows = []
    for _ in range(B):
        perm = torch.randperm(L - 1, generator=g)[: n_docs - 1] + 1
        cuts = torch.sort(perm).values
        rows.append(torch.cat([torch.tensor([0]), cuts, torch.tensor([L])]))
    return torch.stack(rows).to(torch.int32)


def diff_inputs(B: int, H: int, L: int, d: int = 64, dv: int = 128, seed: int = 0):
    """Two query/key branches q1,k1,q2,k2 [B,H,L,d] and a shared v [B,H,L,dv]."""
    g = generator(seed)
    q1 = randn_bf16((B, H, L, d), g)
    k1 = randn_bf16((B, H, L, d), g)
    q2 = randn_bf16((B, H, L, d), g)
    k2 = randn_bf16((B, H, L, d), g)
    v = randn_bf16((B, H, L, dv), g)
    return q1, k1, q2, k2, v


def evo_inputs(B: int, N_seq: int, N_res: int, H: int, d: int = 32, seed: int = 0,
               p_keep: float = 0.9, mask_value: float = -1e9):
    """Evoformer MSA row-attention inputs.

    q, k, v, gate : bf16 [B, N_seq, H, N_res, d], N(0,1) (gate holds logits)
    pair_bias     : fp32 [B, H, N_res, N_res], N(0,1), shared by every MSA row
    mask_bias     : fp32 [B, N_seq, N_res], 0 where the residue is kept
                    (Bernoulli(p_keep)) and ``mask_value`` where it is masked.
    Every MSA row keeps at least one residue, so no softmax row is empty.
    """
    g = generator(seed)
    q = randn_bf16((B, N_seq, H, N_res, d), g)
    k = randn_bf16((B, N_seq, H, N_res, d), g)
    v = randn_bf16((B, N_seq, H, N_res, d), g)
    gate = randn_bf16((B, N_seq, H, N_res, d), g)
    pair_bias = torch.randn(B, H, N_res, N_res, generator=g, dtype=torch.float32)
    keep = torch.rand(B, N_seq, N_res, generator=g) < p_keep
    empty = ~keep.any(dim=-1)
    if bool(empty.any()):
        first = torch.zeros_like(keep)
        first[..., 0] = True
        keep = keep | (first & empty[..., None])
    mask_bias = torch.where(keep, torch.zeros((), dtype=torch.float32),
                            torch.full((), mask_value, dtype=torch.float32))
    return q, k, v, pair_bias, mask_bias, gate


def evo_col_inputs(B: int, N_seq: int, N_res: int, H: int, d: int = 32, seed: int = 0,
                   p_keep: float = 0.9, mask_value: float = -1e9):
    """Evoformer MSA column-attention inputs.

    q, k, v, gate : bf16 [B, N_seq, H, N_res, d], N(0,1) (gate holds logits)
    mask_bias     : fp32 [B, N_res, N_seq], 0 where the MSA row is kept
                    (Bernoulli(p_keep)) and ``mask_value`` where it is masked.
    Every residue column keeps at least one MSA row.
    """
    g = generator(seed)
    q = randn_bf16((B, N_seq, H, N_res, d), g)
    k = randn_bf16((B, N_seq, H, N_res, d), g)
    v = randn_bf16((B, N_seq, H, N_res, d), g)
    gate = randn_bf16((B, N_seq, H, N_res, d), g)
    keep = torch.rand(B, N_res, N_seq, generator=g) < p_keep
    empty = ~keep.any(dim=-1)
    if bool(empty.any()):
        first = torch.zeros_like(keep)
        first[..., 0] = True
        keep = keep | (first & empty[..., None])
    mask_bias = torch.where(keep, torch.zeros((), dtype=torch.float32),
                            torch.full((), mask_value, dtype=torch.float32))
    return q, k, v, mask_bias, gate


def decode_inputs(B: int, Hq: int, Hkv: int, Lq: int, Lmax: int, d: int, seed: int = 0,
                  min_len: int | None = None):
    """Decode-phase inputs: q [B,Hq,Lq,d], a key/value cache k, v
    [B,Hkv,Lmax,d] (bf16 N(0,1)) and int32 kv_len [B], the valid cache length
    of each sequence, uniform in [min_len, Lmax] (a mixed-length serving
    batch; default min_len = Lmax // 4, never below Lq)."""
    g = generator(seed)
    q = randn_bf16((B, Hq, Lq, d), g)
    k = randn_bf16((B, Hkv, Lmax, d), g)
    v = randn_bf16((B, Hkv, Lmax, d), g)
    lo = max(Lq, Lmax // 4 if min_len is None else min_len)
    kv_len = torch.randint(lo, Lmax + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return q, k, v, kv_len
