"""The fused forward's block-sparse schedule (fl_attn_schedule walks, on the
host, the same descriptor-derived key-tile ranges the kernel walks) against
an independent count: the (query tile, key tile) blocks of the oracle's
visibility matrix that hold at least one visible pair.  With one MMA issuer
per slot (value head dim <= 64) the schedule must visit exactly those blocks
-- no block mask is built, and no fully masked tile is computed."""
import ctypes

import numpy as np
import pytest

import oracle
from flashattention_attn_fwd_gb300 import _lib, synth


def _visible_blocks(mask, L, **kw):
    offs = kw.pop("offsets", None)
    vis = oracle.visibility(mask, L, L, offsets=offs, **kw)
    nt = (L + 127) // 128
    pad = np.zeros((nt * 128, nt * 128), dtype=bool)
    pad[:L, :L] = vis
    return int(pad.reshape(nt, 128, nt, 128).any(axis=(1, 3)).sum())


def _schedule(B, Hq, Hkv, L, d, dv, doc=None, **kw):
    desc = _lib.new_desc()
    desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = B, Hq, Hkv, L, L, d, dv
    for k, v in kw.items():
        setattr(desc, k, v)
    tiles = (ctypes.c_int64 * 3)()
    buf = None
    if doc is not None:
        buf = np.ascontiguousarray(doc, dtype=np.int32)
        desc.num_docs = buf.shape[1] - 1
        desc.doc_offsets = 0x10000  # validated only; the host copy is read
    st = _lib.lib().fl_attn_schedule(ctypes.byref(desc), None if buf is None else buf.ctypes.data, tiles)
    assert st == _lib.FL_OK, _lib.status_string(st)
    return list(tiles)


CASES = [
    ("none", 1, dict(), {}),
    ("causal", 1, dict(mask_kind=1), {}),
    ("window", 2, dict(mask_kind=2, window=256), dict(window=256)),
    ("window", 2, dict(mask_kind=2, window=37), dict(window=37)),
    ("prefix_lm", 3, dict(mask_kind=3, prefix_len=1024), dict(prefix=1024)),
    ("prefix_lm", 3, dict(mask_kind=3, prefix_len=100), dict(prefix=100)),
]


@pytest.mark.parametrize("L", [128, 300, 2048, 2100])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[3]}")
@pytest.mark.parametrize("heads", [(4, 4), (8, 2)], ids=["mha", "gqa4"])
def test_schedule_visits_exactly_the_visible_blocks(L, case, heads):
    mask, _, dkw, okw = case
    Hq, Hkv = heads
    B = 2
    own, allt, dense = _schedule(B, Hq, Hkv, L, 64, 64, **dkw)
    assert own == B * Hq * _visible_blocks(mask, L, **okw)
    assert dense == B * Hq * ((L + 127) // 128) ** 2
    assert own <= allt <= dense + B * Hq * ((L + 127) // 128)


@pytest.mark.parametrize("L,docs", [(2048, 8), (8192, 8), (1000, 3), (300, 1)])
def test_schedule_document_mask(L, docs):
    B, Hq, Hkv = 2, 8, 2
    offs = synth.doc_offsets(B, L, docs, seed=L).numpy()
    for causal in (0, 1):
        own, _, _ = _schedule(B, Hq, Hkv, L, 64, 64, doc=offs, mask_kind=4, doc_causal=causal)
        want = sum(_visible_blocks("document", L, offsets=offs[b], doc_causal=bool(causal)) for b in range(B))
        assert own == Hq * want


def test_schedule_value_dim_128_walks_the_union():
    """With P written over S (value head dim 128) one MMA thread serves both
    slots, which then walk the union of their ranges: never fewer blocks."""
    own, _, _ = _schedule(1, 4, 4, 2048, 64, 128, mask_kind=1)
    assert own >= 4 * _visible_blocks("causal", 2048)


@pytest.mark.parametrize("L", [256, 300, 2100])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[3]}")
@pytest.mark.parametrize("heads", [(4, 4), (6, 2)], ids=["mha", "gqa3"])
def test_key_split_schedule_visits_the_same_blocks(L, case, heads):
    """Splitting every unit along the key axis (two slots on the same query
    rows, halves of the key range) visits exactly the visible blocks too:
    the halves neither overlap nor leave a gap."""
    mask, _, dkw, okw = case
    Hq, Hkv = heads
    B = 2
    own, allt, _ = _schedule(B, Hq, Hkv, L, 64, 64, debug_flags=_lib.FL_DEBUG_KEY_SPLIT, **dkw)
    assert own == B * Hq * _visible_blocks(mask, L, **okw)
    assert allt >= own
