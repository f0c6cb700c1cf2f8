"""GB300-native fused attention forward for attention variants.

The computation lives in the CUDA library ``libflattn.so`` (C ABI in
``include/flattn.h``); this package holds the build step, a thin ctypes
binding with the same entry-point names, the FLOP/byte accounting used for
the roofline, and the seeded synthetic-input generators.
"""
from .api import (FlattnError, attn_bwd, attn_decode_fwd, attn_fwd, attention, diffattn_bwd,  # noqa: F401
                  diff_attention, diffattn_fwd,
                  evoformer_col_gated_attn_fwd, evoformer_gated_attn_fwd, sync_status)

__all__ = ["attn_fwd", "diffattn_fwd", "diffattn_bwd", "evoformer_gated_attn_fwd", "evoformer_col_gated_attn_fwd",
           "attn_decode_fwd", "attn_bwd", "attention", "diff_attention", "sync_status", "FlattnError"]
